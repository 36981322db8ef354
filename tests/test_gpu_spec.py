"""Speculative acceptance on the GPU (tps_spec_accept, through the C ABI) against the float64 oracle.

Rows are compared draw by draw with the same uniforms: status and acceptance exactly, the token
exactly.  A row where the oracle flags a decision within rounding (the acceptance test u Q(x) vs
P(x), the two best residual race keys, or a top-p / min-p decision of the target or the draft) must
still give a valid answer: the draft token when it says accepted, otherwise a token the target keeps.
"""
import numpy as np
import pytest
import torch

import nucleus_token_sampler_gb300 as tps
import oracle
from nucleus_token_sampler_gb300 import workloads

from . import _parity

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def _vec(v, B, dt):
    return torch.as_tensor(np.broadcast_to(np.asarray(v), (B,)).copy()).to(dt)


def run_both(zt, zd, tp, dp, x, seeds, step, dtype=torch.float32):
    """GPU and oracle on the same rows; tp / dp = (T, k, p, m) per row or scalars."""
    zt = torch.as_tensor(np.asarray(zt, np.float64)).to(dtype)
    zd = torch.as_tensor(np.asarray(zd, np.float64)).to(dtype)
    B = zt.shape[0]
    tq = [_vec(v, B, d) for v, d in zip(tp, (torch.float32, torch.int32, torch.float32, torch.float32))]
    dq = [_vec(v, B, d) for v, d in zip(dp, (torch.float32, torch.int32, torch.float32, torch.float32))]
    X = _vec(x, B, torch.int32)
    S = _vec(np.asarray(seeds).astype(np.int64), B, torch.int64)
    g = tps.spec_accept(zt.cuda(), zd.cuda(), [t.cuda() for t in tq], [t.cuda() for t in dq], X.cuda(), S.cuda(), step,
                        diagnostics=True)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    o = oracle.spec_accept(zt.double().numpy(), zd.double().numpy(), [t.numpy() for t in tq], [t.numpy() for t in dq],
                           X.numpy(), S.numpy().astype(np.uint64), step)
    return g, o, zt.double().numpy(), tq


def compare(g, o, zt, tq, x):
    """Failure strings and the count of boundary rows."""
    fails = []
    if not np.array_equal(g["status"], o["status"]):
        b = np.nonzero(g["status"] != o["status"])[0][:5]
        fails.append(f"status differs at rows {b.tolist()}: gpu {g['status'][b]} oracle {o['status'][b]}")
    ok = o["status"] == 0
    band = o["flags"] != 0
    exact = ok & ~band
    for name in ("token", "accepted"):
        b = np.nonzero(exact & (g[name] != o[name]))[0]
        if len(b):
            fails.append(f"{name} differs on {len(b)} rows, e.g. row {b[0]}: gpu {g[name][b[0]]} oracle {o[name][b[0]]}")
    if (~ok).any() and not ((g["token"][~ok] == -1).all() and (g["accepted"][~ok] == 0).all()):
        fails.append("failed rows have a token or an acceptance")
    xs = np.asarray(x)
    for b in np.nonzero(ok & band)[0]:
        t = int(g["token"][b])
        if g["accepted"][b] == 1:
            if t != xs[b]:
                fails.append(f"band row {b}: accepted but token {t} != draft token {xs[b]}")
            continue
        T, k, p, m = (float(tq[0][b]), int(tq[1][b]), float(tq[2][b]), float(tq[3][b]))
        if T <= 0:
            if not (0 <= t < zt.shape[1] and zt[b, t] == np.nanmax(zt[b])):
                fails.append(f"band row {b}: greedy target, token {t} is not its maximum")
            continue
        allowed, vals, _ = _parity.valid_kept_classes(zt[b], T, k, p, m)
        lowest = vals[max(allowed) - 1]
        if not (0 <= t < zt.shape[1] and np.isfinite(zt[b, t]) and zt[b, t] >= lowest):
            fails.append(f"band row {b}: rejected, and token {t} is outside every kept set the target allows")
    return fails, int((ok & band).sum())


def draft_tokens(zd, dp, seeds, step):
    """Tokens the draft distribution can produce: the oracle's own draw from it."""
    B = zd.shape[0]
    T, k, p, m = (np.broadcast_to(np.asarray(v), (B,)) for v in dp)
    return oracle.sample(np.asarray(zd, np.float64), T, k, p, m, np.asarray(seeds).astype(np.uint64) + np.uint64(7),
                         step + 1)["token"]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_spec_decode_like_rows(dtype):
    """Decode-shaped rows (V = 128,256): the draft is the target plus noise under other parameters."""
    w = workloads.make("decode", device="cpu", B=64)
    rng = np.random.default_rng(3)
    zt = w.logits.double().numpy()
    zd = zt + rng.normal(0, 0.7, size=zt.shape)
    if dtype == torch.bfloat16:  # compare on the values the GPU sees
        zt = torch.as_tensor(zt).to(torch.bfloat16).double().numpy()
        zd = torch.as_tensor(zd).to(torch.bfloat16).double().numpy()
    B = zt.shape[0]
    tp = (0.7, 50, 0.9, 0.05)
    dp = (rng.choice([0.5, 0.9, 1.2], B), rng.choice([0, 40], B), rng.choice([0.8, 0.95, 1.0], B),
          rng.choice([0.0, 0.02], B))
    seeds = np.arange(B) * 31 + 5
    x = draft_tokens(zd, dp, seeds, 11)
    g, o, ztd, tq = run_both(zt, zd, tp, dp, x, seeds, 11, dtype)
    fails, nb = compare(g, o, ztd, tq, x)
    assert not fails, "\n".join(fails)
    assert nb <= 8, nb
    assert 0 < g["accepted"].sum() < B  # both outcomes occur


def test_spec_tiny_vocabularies():
    """Rows of 2-39 tokens with ties, -inf masks and random parameters on both sides (greedy rows
    included), and draft tokens the draft can produce."""
    fails = []
    nb = 0
    for w in workloads.tiny_grid(4242, n_batches=120):
        zt = w.logits.double().numpy()
        rng = np.random.default_rng(w.V * 101 + w.B)
        zd = zt + np.where(np.isfinite(zt), rng.normal(0, 1.0, size=zt.shape), 0.0)
        zd = np.where(rng.random(zt.shape) < 0.1, -np.inf, zd)
        zd[:, 0] = np.where(np.isfinite(zd[:, 0]), zd[:, 0], 0.0)
        tp = (w.temperature.numpy(), w.top_k.numpy(), w.top_p.numpy(), w.min_p.numpy())
        dp = (rng.choice([0.0, 0.6, 1.0, 1.7], w.B), rng.integers(0, 5, w.B), rng.uniform(0.3, 1.0, w.B),
              rng.choice([0.0, 0.1], w.B))
        seeds = w.seed.numpy()
        x = draft_tokens(zd, dp, seeds, 2)
        x = np.where(x < 0, 0, x)
        g, o, ztd, tq = run_both(zt, zd, tp, dp, x, seeds, 2)
        f, b = compare(g, o, ztd, tq, x)
        fails += [f"{w.name}: {m}" for m in f]
        nb += b
    assert not fails, "\n".join(fails[:10])


def test_spec_special_cases():
    """Identical target and draft accept every draft token; a greedy target returns its maximum;
    disjoint supports never accept; a draft token outside the target's nucleus is never accepted;
    invalid draft tokens and failed rows report their status."""
    rng = np.random.default_rng(9)
    B, V = 48, 3000
    zt = rng.normal(0, 2, size=(B, V))
    seeds = np.arange(B) + 100
    tp = (rng.choice([0.5, 1.0, 2.0], B), rng.choice([0, 3, 100], B), rng.uniform(0.2, 1.0, B), rng.choice([0.0, 0.05], B))
    x = draft_tokens(zt, tp, seeds, 4)
    g, o, ztd, tq = run_both(zt, zt, tp, tp, x, seeds, 4)
    assert (g["accepted"] == 1).all() and (g["token"] == x).all()
    g, o, ztd, tq = run_both(zt, zt, (0.0, 0, 1.0, 0.0), tp, x, seeds, 4)
    assert (g["token"] == ztd.argmax(axis=1)).all()  # the maximum of the float32 logits, lowest index
    za, zb = zt.copy(), zt.copy()
    za[:, V // 2:] = -np.inf
    zb[:, : V // 2] = -np.inf
    xb = draft_tokens(zb, (1.0, 0, 1.0, 0.0), seeds, 4)
    g, o, ztd, tq = run_both(za, zb, (1.0, 0, 1.0, 0.0), (1.0, 0, 1.0, 0.0), xb, seeds, 4)
    fails, _ = compare(g, o, ztd, tq, xb)
    assert not fails, fails
    assert (g["accepted"] == 0).all() and (g["token"] < V // 2).all()
    z3 = np.tile(np.log([0.5, 0.3, 0.2]), (B, 1))
    g, o, ztd, tq = run_both(z3, np.zeros((B, 3)), (1.0, 0, 0.6, 0.0), (1.0, 0, 1.0, 0.0), np.full(B, 2), seeds, 4)
    assert (g["accepted"] == 0).all() and (g["token"] != 2).all()
    zbad = zt[:5].copy()
    zbad[2, 3] = np.nan
    zd = zt[:5].copy()
    zd[3] = -np.inf
    zd[4, 7] = -np.inf
    xbad = np.array([-1, V, 0, 0, 7])
    g, o, ztd, tq = run_both(zbad, zd, (1.0, 0, 1.0, 0.0), (1.0, 0, 1.0, 0.0), xbad, seeds[:5], 4)
    assert g["status"].tolist() == [3, 3, 1, 2, 3] and (g["token"] == -1).all()
    assert np.array_equal(g["status"], o["status"])


def test_spec_million_draws():
    """10^6 rows of a 5-token case: draw by draw equal to the oracle; the acceptance rate is
    sum min(P, Q) and the output frequencies are P (TV <= 1e-3)."""
    n = 1_000_000
    zt = np.log(np.array([0.30, 0.25, 0.25, 0.12, 0.08]))
    zd = np.log(np.array([0.10, 0.40, 0.20, 0.20, 0.10]))
    P = np.array([0.30, 0.25, 0.25, 0.12]) / 0.92  # top-p 0.9 keeps four (the mass above 0.08 is 0.92)
    P = np.append(P, 0.0)
    Q = np.array([0.10, 0.40, 0.20, 0.20, 0.10])
    rng = np.random.default_rng(5)
    x = rng.choice(5, size=n, p=Q)
    seeds = np.arange(n, dtype=np.int64) * 7919 + 3
    g, o, ztd, tq = run_both(np.tile(zt, (n, 1)), np.tile(zd, (n, 1)), (1.0, 0, 0.9, 0.0), (1.0, 0, 1.0, 0.0), x,
                             seeds, 6)
    fails, nb = compare(g, o, ztd, tq, x)
    assert not fails, "\n".join(fails[:5])
    acc = g["accepted"].mean()
    a_exact = np.minimum(P, Q).sum()
    assert abs(acc - a_exact) <= 5 * np.sqrt(a_exact * (1 - a_exact) / n)
    freq = np.bincount(g["token"], minlength=5) / n
    tv = 0.5 * np.abs(freq - P).sum()
    print("acceptance", acc, "exact", a_exact, "TV", tv, "band rows", nb)
    assert tv <= 1e-3
