"""CUDA sampler against the float64 oracle, element by element, through the C ABI.

Kept sets (count and cutoff) and sampled tokens must match exactly; renormalised probabilities
within 1e-5 absolute.  Rows where the oracle reports a knife-edge decision (the mass above a class
within 1e-6 of p, or an e_i within rounding of min_p) are counted, and on them the GPU's answer must
be one of the correct ones: a kept set allowed by the band, and the exact race, probabilities and
log-probabilities over that kept set.  Rows whose two best race keys lie within rounding must still
draw a kept token.
"""
import math

import numpy as np
import pytest
import torch

import nucleus_token_sampler_gb300 as tps
from nucleus_token_sampler_gb300 import workloads

from . import _parity

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


KERNELS = ["cluster", "stream", "auto"]  # auto: a batch of 32+ rows is split between the two kernels


def check(w, rows=None, want_probs=True, logits=None, max_band_frac=0.05, kernels=KERNELS):
    """Both kernels against the oracle; also bit-identical to each other on every row."""
    o = _parity.run_oracle(w, rows=rows, want_probs=want_probs)
    outs = []
    for k in kernels:
        g = _parity.run_gpu(w, want_probs=want_probs, logits=logits, kernel=k)
        rep, fails = _parity.compare(w, g, o, rows=rows, check_probs=want_probs)
        print(w.name, k, rep)
        assert not fails, f"[{k}] " + "\n".join(fails)
        assert rep["band_rows"] <= max(1, max_band_frac * rep["rows"]), rep
        outs.append(g)
    for g in outs[1:]:
        for key in outs[0]:
            assert torch.equal(outs[0][key], g[key]) or (key == "cutoff" and torch.equal(
                torch.nan_to_num(outs[0][key], nan=7.0), torch.nan_to_num(g[key], nan=7.0))), f"kernels differ on {key}"
    return outs[0], o, rep


# Flat rows (logits 1..0 over 128k tokens) have class masses ~1e-5 apart, so a class within 1e-6 of
# p is common there: up to a third of those rows are boundary rows.
BAND_FRAC = {"small": 0.05, "mixed": 0.3, "ties_masked": 0.05}


@pytest.mark.parametrize("name", ["small", "mixed", "ties_masked"])
def test_configs_full(name):
    check(workloads.make(name, device="cpu"), max_band_frac=BAND_FRAC[name])


@pytest.mark.parametrize("B,V,dtype", [(3, 1000, torch.float32), (5, 4099, torch.bfloat16),
                                       (2, 131073, torch.float32), (4, 70001, torch.bfloat16)])
def test_sweep_ragged(B, V, dtype):
    check(workloads.make("sweep", device="cpu", B=B, V=V, dtype=dtype))


def test_decode_full_size_every_row():
    """The benchmark's workload and launch shape (B=1024, V=128,256 fp32), every row checked."""
    w = workloads.make("decode", device="cpu")
    g, o, rep = check(w)
    assert rep["rows"] == 1024
    kept = g["kept"].numpy()
    assert (kept >= 1).all() and (kept <= 50).all()
    assert (g["status"].numpy() == 0).all()


@pytest.mark.parametrize("V", [128256, 256000])
def test_sweep_large_rows_sampled(V):
    w = workloads.make("sweep", device="cpu", B=64, V=V, dtype=torch.bfloat16 if V == 256000 else torch.float32)
    # wide nuclei over 128k-256k tokens: neighbouring classes differ by ~1e-5 of the mass, so many
    # rows have a class within 1e-6 of p (boundary rows, excluded from the exact checks)
    check(w, rows=np.arange(0, 64, 4), max_band_frac=0.6)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_sweep_largest_config_sampled_rows(dtype):
    """The sweep's largest shape, B=4096 x V=256,000 (4.2 GB of fp32 logits), in the launch
    configuration the benchmark times; 24 rows checked against the oracle (probabilities are
    checked at smaller sizes)."""
    w = workloads.make("sweep", device="cpu", B=4096, V=256000, dtype=dtype)
    rows = np.unique(np.concatenate([np.arange(8), np.arange(4096 - 8, 4096),
                                     np.random.default_rng(1).choice(4096, 8, replace=False)]))
    g, _, _ = check(w, rows=rows, want_probs=False, max_band_frac=0.6)
    assert (g["status"].numpy() == 0).all()


def test_largest_vocabulary():
    """V = tps_max_vocab() (2^20 - 1 tokens): too wide for a 16-CTA cluster, so every kernel choice
    that accepts it runs the streaming kernel; rows with and without min-p, greedy and masked."""
    V = tps.max_vocab(torch.float32)
    rng = np.random.default_rng(23)
    z = rng.normal(0, 2.0, size=(4, V))
    z[1, rng.choice(V, 20, replace=False)] += 9.0
    z[3, : V // 2] = -np.inf
    # top-p off over the whole vocabulary; min-p + top-k + top-p on a peaked row; greedy; top-k 1000
    # on a half-masked row (no top-p, so no row sits on a top-p boundary)
    w = _w(z, [0.9, 0.7, 0.0, 1.3], [0, 50, 0, 1000], [1.0, 0.9, 0.9, 1.0], [0.0, 0.05, 0.0, 0.0])
    g, _, rep = check(w, kernels=["stream", "auto"])
    assert rep["band_rows"] == 0 and g["kept"].tolist() == [V, g["kept"][1].item(), 1, 1000]
    with pytest.raises(RuntimeError):
        _parity.run_gpu(w, kernel="cluster")


@pytest.mark.parametrize("kernel", KERNELS)
def test_tiny_vocabularies_grid(kernel):
    fails = []
    nb = 0
    for w in workloads.tiny_grid(777, n_batches=200):
        g = _parity.run_gpu(w, kernel=kernel)
        o = _parity.run_oracle(w)
        rep, f = _parity.compare(w, g, o)
        nb += rep["band_rows"]
        fails += [f"{w.name}: {x}" for x in f]
    assert not fails, "\n".join(fails[:10])
    assert nb <= 40


def test_unaligned_and_strided_rows():
    base = workloads.make("sweep", device="cpu", B=6, V=5003, dtype=torch.bfloat16)
    # bf16 rows starting 2 bytes past a 16-byte boundary, row stride 5011 elements
    big = torch.full((6, 5011 + 1), -3.0, dtype=torch.bfloat16)
    big[:, 1:5004] = base.logits
    dev = big.cuda()
    view = dev[:, 1:5004]
    check(base, logits=view)
    f32 = workloads.make("sweep", device="cpu", B=5, V=777)
    big = torch.zeros((5, 800), dtype=torch.float32)
    big[:, 3:780] = f32.logits
    check(f32, logits=big.cuda()[:, 3:780])


@pytest.mark.parametrize("V", [1, 2, 3, 5, 7, 8, 9, 15, 16, 17, 31, 33, 64, 100])
def test_small_odd_vocab(V):
    for dtype in (torch.float32, torch.bfloat16):
        w = workloads.make("sweep", device="cpu", B=4, V=V, dtype=dtype)
        check(w)


def _w(z, T, k, p, m, seed=1, step=0, dtype=torch.float32):
    z = torch.as_tensor(np.asarray(z, dtype=np.float64)).to(dtype)
    if z.dim() == 1:
        z = z[None]
    B = z.shape[0]
    f = lambda v, dt: torch.as_tensor(np.broadcast_to(np.asarray(v), (B,)).copy()).to(dt)
    return workloads.Workload("edge", z, f(T, torch.float32), f(k, torch.int32), f(p, torch.float32),
                              f(m, torch.float32), f(seed, torch.int64), step)


def test_edge_cases():
    rng = np.random.default_rng(3)
    z = rng.normal(0, 1, 300)
    z[::5] = -np.inf
    rows = [
        (np.array([0.0, np.nan, 1.0]), 1.0, 0, 0.5, 0.0),
        (np.array([0.0, np.inf, 1.0]), 1.0, 0, 0.5, 0.0),
        (np.array([-np.inf, -np.inf, -np.inf]), 1.0, 0, 0.5, 0.0),
        (np.array([0.0, 1.0, 1.0]), np.nan, 0, 0.5, 0.0),
        (np.array([0.0, 1.0, 1.0]), np.inf, 0, 0.5, 0.0),
        (np.array([0.0, 1.0, 1.0]), 1.0, 0, np.nan, 0.0),
        (np.array([0.0, 1.0, 1.0]), 1.0, 0, 0.5, np.inf),
    ]
    for zr, T, k, p, m in rows:
        w = _w(zr, T, k, p, m)
        g, o, _ = check(w)
        assert g["token"][0] == -1
    # greedy with ties (lowest index), p >= 1, p <= 0, tiny p, k = 1 on a tie, min_p = 1 and > 1
    for T, k, p, m in [(0.0, 0, 0.9, 0.0), (-2.0, 5, 0.5, 0.1), (1.0, 0, 1.0, 0.0), (1.0, 0, 7.0, 0.0),
                       (1.0, 0, 0.0, 0.0), (1.0, 0, -1.0, 0.0), (0.8, 0, 1e-8, 0.0), (1.0, 1, 1.0, 0.0),
                       (1.0, 0, 1.0, 1.0), (1.3, 0, 0.9, 5.0), (1e-6, 0, 0.9, 0.0), (1e6, 0, 0.9, 0.0),
                       (0.7, 299, 0.99, 0.0), (0.7, 300, 0.99, 0.0), (0.7, -4, 0.95, 0.2)]:
        zz = z.copy()
        zz[7] = zz[11] = np.nanmax(zz[np.isfinite(zz)]) + 0.5
        check(_w(zz, T, k, p, m))


def test_split_rows_every_outcome():
    """A batch of 48 rows (under four rows per SM) has each row of 200,000 float32 logits streamed
    as six segments, merged by the CTA that finishes a row last: every row status, greedy ties
    across segments, the maximum in any segment, min-p rows, rows for the cluster kernel, and
    ragged, unaligned rows."""
    V, B = 200000, 48
    rng = np.random.default_rng(5)
    z = rng.normal(0, 2.0, size=(B, V))
    z[np.arange(B), rng.integers(0, V, B)] += 9.0       # one leader per row, anywhere
    z[1, 7] = np.nan
    z[2, V - 1] = np.inf
    z[3, :] = -np.inf
    z[4, [10, 60000, 150000, V - 2]] = 50.0              # greedy ties in different segments
    z[5, :] = np.round(z[5, :])                           # big tie classes
    z[6, : V // 2] = -np.inf                              # the first segments fully masked
    T = np.full(B, 0.8)
    T[4] = 0.0
    T[7] = np.nan
    T[8::6] = 0.0
    k = np.where(np.arange(B) % 3 == 0, 40, 0)
    p = np.where(np.arange(B) % 4 == 0, 1.0, 0.9)
    m = np.where(np.arange(B) % 5 == 0, 0.0, 0.05)       # every fifth row goes to the cluster kernel
    w = _w(z, T, k, p, m)
    check(w, max_band_frac=0.1)
    zb = np.zeros((B, V + 3))
    zb[:, 1:V + 1] = z
    base = torch.as_tensor(zb).float().cuda()[:, 1:V + 1]  # rows starting 4 bytes past a 16-byte boundary
    check(w, logits=base, max_band_frac=0.1)


def test_temperature_overflowing_distance():
    """A temperature so small that (zmax - z) / T overflows float to +inf for most of the row: those
    tokens fall in the last fine bin of the general path, where top-k (50 and 300, so the crossing is
    inside that bin, with and without a candidate list), top-p and the top-n outputs must still count
    and list them."""
    V = 128256
    rng = np.random.default_rng(41)
    z = rng.normal(0, 2.0, size=(6, V))
    z[1, rng.choice(V, 4, replace=False)] = z[1].max() + 1e-3  # near-ties at the maximum (finite d)
    z[2, :1000] = np.round(z[2, :1000])                        # integer classes among the leaders
    T = [1e-38, 1e-38, 1e-38, 1e-37, 1e-38, 3e-39]
    k = [50, 50, 300, 300, 0, 1000]
    p = [1.0, 1.0, 1.0, 0.9, 0.5, 1.0]
    w = _w(z, T, k, p, 0.0)
    for kern in KERNELS:
        g = _parity.run_gpu(w, kernel=kern, want_logprob=True, top=8)
        o = _parity.run_oracle(w)
        rep, fails = _parity.compare(w, g, o)
        assert not fails, f"[{kern}] " + "\n".join(fails)
        assert g["kept"].tolist()[0] == 50 and g["kept"].tolist()[2] >= 300


@pytest.mark.parametrize("kernel", KERNELS)
def test_batch_independence_and_determinism(kernel):
    w = workloads.make("mixed", device="cpu", B=16, V=40000)
    g1 = _parity.run_gpu(w, kernel=kernel)
    g2 = _parity.run_gpu(w, kernel=kernel)
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k
    # Same row content at the same row index inside a different batch gives the same outputs.
    w2 = workloads.make("sweep", device="cpu", B=16, V=40000, seed=99)
    keep = [3, 8]
    for t in ("logits",):
        getattr(w2, t)[keep] = getattr(w, t)[keep]
    for t in ("temperature", "top_k", "top_p", "min_p", "seed"):
        getattr(w2, t)[keep] = getattr(w, t)[keep]
    g3 = _parity.run_gpu(w2, kernel=kernel)
    for k in ("token", "status", "cutoff", "kept", "probs"):
        assert torch.equal(g1[k][keep], g3[k][keep]), k


@pytest.mark.parametrize("kernel", KERNELS)
def test_sampled_distribution_million_draws(kernel):
    """10^6 draws on a 5-token case: draw-by-draw equal to the oracle, TV to the exact
    renormalised distribution <= 1e-3."""
    probs = np.array([0.30, 0.25, 0.25, 0.12, 0.08])
    n = 1_000_000
    z = np.tile(np.log(probs), (n, 1))
    w = _w(z, 1.0, 0, 0.9, 0.0, seed=np.arange(n, dtype=np.int64) * 7919 + 5, step=3)
    g = _parity.run_gpu(w, want_probs=False, kernel=kernel)
    o = _parity.run_oracle(w, want_probs=False)
    tok = g["token"].numpy()
    eq = tok == o["token"]
    assert eq.mean() == 1.0 or eq[(o["flags"] & 4) == 0].all()
    exact = probs[:4] / probs[:4].sum()  # p = 0.9 keeps the first four (mass above 0.08 is 0.92)
    freq = np.bincount(tok, minlength=5) / n
    assert freq[4] == 0
    tv = 0.5 * np.abs(freq[:4] - exact).sum()
    print("TV", tv)
    assert tv <= 1e-3


@pytest.mark.parametrize("kernel", KERNELS)
def test_step_changes_draws(kernel):
    w = workloads.make("sweep", device="cpu", B=256, V=1000)
    w.top_p[:] = 1.0
    w.temperature[:] = 2.0
    a = _parity.run_gpu(w, want_probs=False, kernel=kernel)["token"]
    w.step = 1
    b = _parity.run_gpu(w, want_probs=False, kernel=kernel)["token"]
    assert (a != b).float().mean() > 0.5


@pytest.mark.parametrize("kernel", KERNELS)
def test_empty_batch(kernel):
    x = torch.empty((0, 100), device="cuda")
    e = torch.empty(0, device="cuda")
    out = tps.sample(x, e, e.int(), e, e, e.long(), kernel=kernel)
    assert out.shape == (0,)


_ORACLE = {}


def _top_check(w, kernel, top=tps.MAX_TOP):
    key = (w.name, w.B, w.V)
    if w.name == "edge" or key not in _ORACLE:
        _ORACLE[key] = _parity.run_oracle(w)
    o = _ORACLE[key]
    g = _parity.run_gpu(w, kernel=kernel, want_logprob=True, top=top)
    rows = np.arange(w.B)
    okrow = o["status"] == 0
    setband = (o["flags"] & (_parity.TOPP_BAND | _parity.MINP_BAND)) != 0
    fails = _parity.compare_top(w, g, o, rows, okrow, setband)
    assert not fails, f"[{kernel}] " + "\n".join(fails)
    return g, o


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name", ["small", "mixed", "ties_masked"])
def test_top_logprobs(kernel, name):
    """The 32 most probable kept tokens of each row with their ln P (the most the ABI reports):
    list-resolved rows, general-path rows (more than 256 survivors) and rows with ties."""
    _top_check(workloads.make(name, device="cpu"), kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_top_logprobs_big_tie_classes(kernel, dtype):
    """Tie classes larger than a candidate list where the top tokens end: equal logits over the
    whole row, and a few distinct leaders followed by one value shared by most of the row; the
    lowest indices of the tie come first."""
    V = 128256
    rng = np.random.default_rng(11)
    flat = np.zeros(V)
    lead = rng.normal(0, 1, V) - 6.0
    lead[rng.choice(V, 100000, replace=False)] = -1.0
    lead[[5, 900, 77777, 128000]] = [3.0, 2.5, 2.5, 1.0]
    few = flat.copy()
    few[:3] = 1.0
    z = np.stack([flat, flat, lead, lead, lead, few])
    T = [1.0, 0.5, 1.0, 0.8, 1.0, 1.0]
    k = [0, 40, 0, 0, 50, 0]
    p = [0.9, 1.0, 0.95, 1.0, 0.9, 0.999]
    w = _w(z, T, k, p, 0.0, dtype=dtype)
    _top_check(w, kernel)
    _top_check(w, kernel, top=5)


@pytest.mark.gpu
def test_kernels_per_call_follows_the_split_rule():
    f32 = torch.float32
    assert tps.kernels_per_call(f32, 1024, 128256, "auto") == 3   # scratch clear, streaming kernel, cluster kernel
    assert tps.kernels_per_call(f32, 1024, 128256, "stream") == 2  # scratch clear, streaming kernel
    assert tps.kernels_per_call(f32, 1024, 128256, "cluster") == 1
    assert tps.kernels_per_call(f32, 8, 32000, "auto") == 1       # a small batch: the cluster kernel alone


def test_side_stream_with_scalar_parameters():
    """Scalar parameters converted by the binding, and outputs it allocates, are made on the stream
    the caller names, so a call on a side stream while the current stream is busy reads them ready."""
    w = workloads.make("small", device="cpu")
    d = w.to("cuda")
    B = w.B
    scal = dict(temperature=0.9, top_k=40, top_p=0.8, min_p=0.02, seed=1234)
    ws = workloads.Workload("scalar", w.logits, torch.full((B,), 0.9), torch.full((B,), 40, dtype=torch.int32),
                            torch.full((B,), 0.8), torch.full((B,), 0.02), torch.full((B,), 1234, dtype=torch.int64), 7)
    o = _parity.run_oracle(ws, want_probs=False)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    big = torch.randn(4096, 4096, device="cuda")
    for _ in range(3):
        for _ in range(8):
            big = big @ big.T * 1e-3  # keeps the current stream busy while the side stream samples
        r = tps.sample(d.logits, scal["temperature"], scal["top_k"], scal["top_p"], scal["min_p"], scal["seed"], 7,
                       diagnostics=True, stream=side)
        side.synchronize()
        g = {k: v.cpu() for k, v in r.items()}
        rep, fails = _parity.compare(ws, g, o, check_probs=False)
        assert not fails, fails
    torch.cuda.synchronize()
