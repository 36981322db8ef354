"""Penalty kernel (repetition, frequency, presence on raw logits) against the oracle, through the C
ABI: the penalised logits must be identical bit for bit (both sides use the same float32 operations),
and so must the row statuses."""
import numpy as np
import pytest
import torch

import nucleus_token_sampler_gb300 as tps
import oracle
from nucleus_token_sampler_gb300 import workloads

from . import _parity

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def _oracle(z, hist, lens, rep, freq, pres):
    bf16 = z.dtype == torch.bfloat16
    cpu = lambda t: None if t is None else t.cpu().numpy()
    return oracle.penalties(z.float().cpu().numpy(), cpu(hist), cpu(lens), cpu(rep), cpu(freq), cpu(pres), bf16=bf16)


def _gpu(z, hist, lens, rep, freq, pres):
    zz = z.cuda().clone()
    c = lambda t: None if t is None else t.cuda()
    _, st = tps.apply_penalties(zz, c(hist), c(lens), repetition=c(rep), frequency=c(freq), presence=c(pres),
                                status=True)
    torch.cuda.synchronize()
    return zz.cpu(), st.cpu().numpy()


def _same_bits(a_f32, b_f32):
    a, b = np.asarray(a_f32, np.float32), np.asarray(b_f32, np.float32)
    both_nan = np.isnan(a) & np.isnan(b)
    return np.array_equal(np.where(both_nan, 0, a.view(np.uint32)), np.where(both_nan, 0, b.view(np.uint32)))


def _check(z, hist, lens=None, rep=None, freq=None, pres=None):
    want, st_o = _oracle(z, hist, lens, rep, freq, pres)
    got, st_g = _gpu(z, hist, lens, rep, freq, pres)
    assert np.array_equal(st_g, st_o), (st_g, st_o)
    g = got.float().numpy()
    if not _same_bits(g, want):
        bad = np.argwhere(g.view(np.uint32) != want.view(np.uint32))[:5]
        pytest.fail(f"penalised logits differ at {bad.tolist()}: gpu {[g[tuple(i)] for i in bad]} "
                    f"oracle {[want[tuple(i)] for i in bad]}")
    return got


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,V,H", [(64, 128256, 300), (200, 32000, 1000), (8, 151936, 8192)])
def test_penalties_match_oracle(dtype, B, V, H):
    g = torch.Generator().manual_seed(B + V + H)
    z = (2.5 * torch.randn((B, V), generator=g)).to(dtype)
    p = workloads.penalty_inputs(B, V, H, seed=B, bad_rows=4)
    _check(z, p.history, p.hist_len, p.repetition, p.frequency, p.presence)


def test_penalties_edges():
    g = torch.Generator().manual_seed(5)
    # tiny vocabularies, special logits, one token repeated across the whole maximum history
    for V in (1, 2, 5, 33):
        z = torch.randn((3, V), generator=g)
        z[0, 0] = -0.0
        if V > 2:
            z[1, 1], z[1, 2] = float("-inf"), float("inf")
        hist = torch.randint(-1, V + 1, (3, 17), generator=g, dtype=torch.int32)
        _check(z, hist, rep=torch.tensor([1.3, 0.5, 2.0]), freq=torch.tensor([0.2, 0.0, 1.5]),
               pres=torch.tensor([0.1, 0.7, 0.0]))
    z = torch.randn((2, 1000), generator=g)
    hist = torch.zeros((2, tps.MAX_HISTORY), dtype=torch.int32)
    hist[1] = 999
    _check(z, hist, rep=torch.tensor([1.1, 0.9]), freq=torch.tensor([0.001, 0.01]), pres=torch.tensor([0.5, 0.5]))
    # a single penalty given (the others off), no lengths, an empty history, lengths out of range
    z = torch.randn((4, 5000), generator=g)
    hist = torch.randint(0, 5000, (4, 64), generator=g, dtype=torch.int32)
    _check(z, hist, freq=torch.full((4,), 0.3))
    _check(z, hist, rep=torch.full((4,), 1.7))
    _check(z, hist[:, :0], rep=torch.full((4,), 1.7))
    _check(z, hist, lens=torch.tensor([-5, 0, 64, 1000], dtype=torch.int32), pres=torch.full((4,), 2.0))


def test_penalties_strided_rows_and_untouched_padding():
    g = torch.Generator().manual_seed(9)
    base = torch.randn((16, 4160), generator=g)
    z = base[:, :4099]  # row stride 4160 > V
    hist = torch.randint(0, 4099, (16, 50), generator=g, dtype=torch.int32)
    rep = torch.full((16,), 1.4)
    want, _ = _oracle(z.contiguous(), hist, None, rep, None, None)
    dz = base.cuda().clone()
    tps.apply_penalties(dz[:, :4099], hist.cuda(), repetition=rep.cuda())
    torch.cuda.synchronize()
    out = dz.cpu()
    assert _same_bits(out[:, :4099].numpy(), want)
    assert torch.equal(out[:, 4099:], base[:, 4099:]), "the padding past V was written"


def test_penalties_then_sample_moves_the_greedy_choice():
    """The chain penalties -> sampler: a repeated argmax loses the greedy pick (the reason the
    pages put penalties on raw logits, before temperature), and the sampled rows match the oracle's
    chain on the same (bit-identical) penalised logits."""
    w = workloads.make("small", device="cpu", B=8, V=32000)
    z = w.logits.clone()
    top = z.argmax(dim=1)
    hist = top[:, None].repeat(1, 4).to(torch.int32)
    rep = torch.full((8,), 50.0)
    pen = _check(z, hist, rep=rep, freq=torch.full((8,), 5.0))
    w2 = workloads.Workload("penalised", pen, torch.zeros(8), w.top_k, w.top_p, w.min_p, w.seed, w.step)
    g = _parity.run_gpu(w2)
    assert (g["token"] != top.to(torch.int32)).all()
    o = _parity.run_oracle(w2)
    _, fails = _parity.compare(w2, g, o)
    assert not fails, fails


def test_penalties_history_stride_and_grid_stride():
    """A history view whose row stride exceeds H, and more rows than the launch's CTAs (the kernel
    caps the grid at 64 CTAs per SM and strides over the rest)."""
    g = torch.Generator().manual_seed(13)
    B, V = 12000, 1000
    z = torch.randn((B, V), generator=g)
    full = torch.randint(-1, V, (B, 48), generator=g, dtype=torch.int32)
    hist = full[:, :20]  # stride 48 > H = 20
    rep = 1.0 + torch.rand(B, generator=g)
    freq = torch.rand(B, generator=g)
    want, st_o = _oracle(z, hist.contiguous(), None, rep, freq, None)
    zz = z.cuda()
    _, st = tps.apply_penalties(zz, full.cuda()[:, :20], repetition=rep.cuda(), frequency=freq.cuda(), status=True)
    torch.cuda.synchronize()
    assert np.array_equal(st.cpu().numpy(), st_o)
    assert _same_bits(zz.cpu().numpy(), want)
