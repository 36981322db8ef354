"""Checks that pin the float64 oracle to things other than itself.

Each ``check_*`` function takes an ``oracle.Oracle`` (the real build, or a variant with a planted
mistake) and returns a list of failure messages; an empty list means the pin holds.  The pins are:
values the pages print for worked examples (``golden/worked_examples.json``), a brute-force
restatement of the definitions on tiny vocabularies, closed forms and special cases, the sampling
frequencies of the race, and an independent third-party Philox4x32-10.
"""
from __future__ import annotations

import json
import math
import os
import subprocess
import sys

import numpy as np

from . import _bruteforce as bf

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden", "worked_examples.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _logits_of(case):
    if "logits" in case:
        return np.asarray(case["logits"], np.float64)
    if "probs" in case:
        return np.log(np.asarray(case["probs"], np.float64))
    spec = case["logits_spec"]
    V = spec["V"]
    if "linspace" in spec:
        a, b = spec["linspace"]
        return np.linspace(a, b, V)
    z = np.full(V, spec["fill"], np.float64)
    z[: len(spec["head"])] = spec["head"]
    return z


def _run1(o, z, T, p, k=0, m=0.0, seed=1, probs=True, step=0):
    return o.sample(np.asarray(z, np.float64)[None, :], np.float32(T), k, np.float32(p),
                    np.float32(m), seed, step, want_probs=probs)


# -------------------------------------------------------------------------------------------
def check_worked_examples(o):
    fails = []
    for c in _golden()["cases"]:
        z = _logits_of(c)
        # p and T are the printed decimals; the library takes float32, so feed exactly what the GPU
        # would get (np.float32 rounding), which is how the oracle receives them too.
        r = _run1(o, z, c["temperature"], c["top_p"])
        if c.get("boundary_row"):
            if not (r["flags"][0] & 1):
                fails.append(f"{c['id']}: expected a top-p boundary row, flags={r['flags'][0]}")
            continue
        if "kept" in c and int(r["kept"][0]) != c["kept"]:
            fails.append(f"{c['id']}: kept {int(r['kept'][0])} != {c['kept']}")
        if "top_token_prob" in c:
            got = 1.0 / r["z_s"][0]  # e of the top token is 1, so its probability is 1 / Z
            if abs(got - c["top_token_prob"]) > c["tol"]:
                fails.append(f"{c['id']}: top-token probability {got:.6f} != {c['top_token_prob']}")
        if "renormalised" in c:
            # listed in index order (the logits cases are already sorted)
            want = np.asarray(c["renormalised"])
            got = r["probs"][0][: len(want)]
            if np.max(np.abs(got - want)) > c["tol"]:
                fails.append(f"{c['id']}: renormalised {np.round(got, 6)} != {want}")
        if "kept_mass" in c:
            mass = r["z_k"][0] / r["z_s"][0]
            if abs(mass - c["kept_mass"]) > 1e-9:
                fails.append(f"{c['id']}: kept mass {mass} != {c['kept_mass']}")
        if "softmax" in c:
            full = _run1(o, z, c["temperature"], 1.0)["probs"][0]
            if np.max(np.abs(full - np.asarray(c["softmax"]))) > c["softmax_tol"]:
                fails.append(f"{c['id']}: softmax {np.round(full, 4)} != {c['softmax']}")
    return fails


# -------------------------------------------------------------------------------------------
def check_sample_frequencies(o, scale=1):
    """Draw from the race (one row per draw, distinct seeds) and compare with the exact
    renormalised distribution and with the frequencies the pages print."""
    fails = []
    for c in _golden()["sample_frequencies"]:
        z = np.asarray(c["logits"], np.float64)
        n = int(c["draws"]) * scale
        Z = np.tile(z, (n, 1))
        seeds = np.arange(n, dtype=np.uint64) * np.uint64(0x9E3779B97F4A7C15) + np.uint64(12345)
        r = o.sample(Z, np.float32(c["temperature"]), 0, np.float32(c["top_p"]), 0.0, seeds,
                     step=7, want_probs=False)
        exact = _run1(o, z, c["temperature"], c["top_p"])["probs"][0]
        counts = np.bincount(r["token"], minlength=len(z)).astype(np.float64)
        freq = counts / n
        kept = exact > 0
        if counts[~kept].sum() != 0:
            fails.append(f"{c['id']}: sampled a token outside the nucleus")
        # 5-sigma binomial bound against the exact distribution
        sig = np.sqrt(exact * (1 - exact) / n)
        if np.any(np.abs(freq - exact) > 5 * sig + 1e-12):
            fails.append(f"{c['id']}: frequencies {np.round(freq, 4)} vs exact {np.round(exact, 4)}")
        # against the printed run (an independent sample of the same size): sqrt(2) * 5 sigma
        want = np.asarray(c["frequencies"])
        m = len(want)
        sig_p = np.sqrt(exact[:m] * (1 - exact[:m]) / int(c["draws"]))
        if np.any(np.abs(freq[:m] - want) > 5 * np.sqrt(2) * sig_p + 6e-4):
            fails.append(f"{c['id']}: frequencies {np.round(freq[:m], 4)} vs printed {want}")
    return fails


# -------------------------------------------------------------------------------------------
def _tiny_batches(seed=20260, n_batches=300):
    from nucleus_token_sampler_gb300 import workloads
    return workloads.tiny_grid(seed, n_batches=n_batches)


def check_bruteforce(o, n_batches=300):
    """Kept sets, probabilities (1e-12) and sampled tokens against the O(V^2) restatement."""
    fails = []
    rows = excluded = 0
    for w in _tiny_batches(n_batches=n_batches):
        z = w.logits.double().numpy()
        T = w.temperature.numpy()
        P = w.top_p.numpy()
        M = w.min_p.numpy()
        K = w.top_k.numpy()
        S = w.seed.numpy().astype(np.uint64)
        r = o.sample(z, T, K, P, M, S, step=w.step, want_probs=True)
        for b in range(z.shape[0]):
            zl = [float(v) for v in z[b]]
            st, keep, probs = bf.kept_set(zl, float(T[b]), int(K[b]), float(P[b]), float(M[b]))
            rows += 1
            if st in ("nan", "bad_param", "all_masked"):
                continue
            if st == "ok" and bf.boundary_distance(zl, float(T[b]), int(K[b]), float(P[b]),
                                                   float(M[b])) < 1e-9:
                excluded += 1
                continue
            if r["flags"][b] & 2:  # min-p decision within rounding of the cut
                excluded += 1
                continue
            race_band = bool(r["flags"][b] & 4)
            if st == "greedy":  # the greedy kept set is the single argmax, whatever ties it has
                okeep = [i == int(r["token"][b]) for i in range(len(zl))]
            else:
                okeep = [(v > -math.inf) and (v >= r["cutoff"][b]) for v in zl]
            if okeep != keep:
                fails.append(f"{w.name}[{b}]: kept set differs (oracle {sum(okeep)}, brute {sum(keep)})")
                continue
            if np.max(np.abs(np.asarray(probs) - r["probs"][b])) > 1e-12:
                fails.append(f"{w.name}[{b}]: probabilities differ")
            # The race over the brute-force kept set, with the oracle's uniforms as inputs.
            if st == "greedy":
                want = keep.index(True)
            else:
                zmax = max(v for v in zl if v > -math.inf)
                best, want = -math.inf, -1
                for i, kp in enumerate(keep):
                    if not kp:
                        continue
                    u = o.uniform(int(S[b]), b, w.step, i)
                    key = math.log(probs[i]) - math.log(-math.log(u)) if probs[i] > 0 else -math.inf
                    if key > best:
                        best, want = key, i
                del zmax
            if int(r["token"][b]) != want and not race_band:
                fails.append(f"{w.name}[{b}]: token {int(r['token'][b])} != brute {want}")
    if rows == 0 or excluded > 0.2 * rows:
        fails.append(f"brute force: {excluded} of {rows} rows excluded")
    return fails


# -------------------------------------------------------------------------------------------
def check_closed_forms(o):
    fails = []
    rng = np.random.default_rng(5)

    # All logits equal: one class, everything kept, uniform probabilities.
    for V in (1, 2, 7, 1000):
        r = _run1(o, np.full(V, 0.3), 0.8, float(rng.uniform(0.01, 0.99)))
        if int(r["kept"][0]) != V or np.max(np.abs(r["probs"][0] - 1.0 / V)) > 1e-15:
            fails.append(f"equal logits V={V}: kept {int(r['kept'][0])}")

    # Geometric logits z_i = -c i at T = 1: the mass above token i is (1 - r^i) / (1 - r^V).
    for V, c, p in ((50, 0.3, 0.7), (200, 0.05, 0.93), (1000, 0.01, 0.5), (30, 1.7, 0.999)):
        z = -c * np.arange(V, dtype=np.float64)
        rr = math.exp(-c)
        want = sum(1 for i in range(V) if (1 - rr ** i) < p * (1 - rr ** V))
        got = _run1(o, z, 1.0, p)
        if int(got["kept"][0]) != max(want, 1):
            fails.append(f"geometric V={V} c={c} p={p}: kept {int(got['kept'][0])} != {want}")

    # Two classes: n1 tokens at a, n2 at b < a.  Mass above class b = n1 / (n1 + n2 e^{-(a-b)/T}).
    for n1, n2, a, b, T, p in ((3, 5, 1.0, 0.0, 1.0, 0.5), (1, 9, 2.0, 1.5, 0.5, 0.6),
                               (4, 4, 0.0, -1.0, 2.0, 0.45), (2, 100, 5.0, 0.0, 1.0, 0.99)):
        z = np.array([a] * n1 + [b] * n2, np.float64)[rng.permutation(n1 + n2)]
        above = n1 / (n1 + n2 * math.exp(-(a - b) / float(np.float32(T))))
        want = n1 + n2 if above < float(np.float32(p)) else n1
        got = int(_run1(o, z, T, p)["kept"][0])
        if got != want:
            fails.append(f"two classes {n1}/{n2} T={T} p={p}: kept {got} != {want}")

    # Exact dyadic boundary: e = 1, 1/2, 1/2 at p = 1/2; the mass above the tied pair equals p
    # exactly, and 'below p' is strict, so only the top token survives.
    got = _run1(o, np.log(np.array([0.5, 0.25, 0.25])), 1.0, 0.5)
    if int(got["kept"][0]) != 1:
        fails.append(f"dyadic boundary: kept {int(got['kept'][0])} != 1")

    # min-p alone: keep z_i >= zmax + T ln(min_p) (distinct logits, away from the cut).
    for V, T, m in ((500, 0.7, 0.05), (300, 1.3, 0.2), (64, 0.25, 0.5)):
        z = rng.normal(0, 2, V)
        zmax = z.max()
        Tf, mf = float(np.float32(T)), float(np.float32(m))
        thr = zmax + Tf * math.log(mf)
        z = z[np.abs(z - thr) > 1e-6]
        want = int(np.sum(z >= thr))
        got = int(_run1(o, z, T, 1.0, m=m)["kept"][0])
        if got != want:
            fails.append(f"min-p V={V} T={T} m={m}: kept {got} != {want}")

    # top-k alone on distinct logits keeps exactly k; with a tie at the k-th value, the whole tie.
    for V, k in ((100, 1), (100, 50), (1000, 7)):
        z = rng.permutation(V).astype(np.float64) * 0.01
        got = int(_run1(o, z, 1.0, 1.0, k=k)["kept"][0])
        if got != k:
            fails.append(f"top-k V={V} k={k}: kept {got}")
    z = np.array([5.0, 3.0, 4.0, 3.0, 1.0, 3.0])
    if int(_run1(o, z, 1.0, 1.0, k=2)["kept"][0]) != 2 or int(_run1(o, z, 1.0, 1.0, k=3)["kept"][0]) != 5:
        fails.append("top-k with ties at the k-th value")
    # top_k = 1 on two equal maxima keeps both (What do temperature... -- edge cases).
    if int(_run1(o, np.array([1.0, 2.0, 2.0, 0.5]), 1.0, 1.0, k=1)["kept"][0]) != 2:
        fails.append("top_k=1 on a tied maximum")
    # top_k >= V and top_k <= 0 disable the cut.
    for k in (0, -3, 6, 100):
        if int(_run1(o, np.arange(6.0), 1.0, 1.0, k=k)["kept"][0]) != 6:
            fails.append(f"top_k={k} should be off")

    # min_p = 1 keeps exactly the class of the maximum; min_p > 1 is clamped to 1.
    for m in (1.0, 3.0):
        got = _run1(o, np.array([0.0, 2.0, 1.0, 2.0]), 1.0, 1.0, m=m)
        if int(got["kept"][0]) != 2:
            fails.append(f"min_p={m}: kept {int(got['kept'][0])}")

    # p >= 1 keeps every finite token; p <= 0 and tiny p keep the class of the maximum.
    z = rng.normal(0, 1, 300)
    z[::7] = -np.inf
    nf = int(np.isfinite(z).sum())
    for p, want in ((1.0, nf), (1.5, nf), (0.0, 1), (-0.5, 1), (1e-9, 1)):
        got = _run1(o, z, 1.0, p)
        if int(got["kept"][0]) != want:
            fails.append(f"p={p}: kept {int(got['kept'][0])} != {want}")
        if np.any(got["probs"][0][~np.isfinite(z)] != 0):
            fails.append(f"p={p}: a -inf token got probability")

    # Greedy: T <= 0 takes the lowest index of the maximum; probabilities one-hot.
    z = np.array([0.1, 3.0, -1.0, 3.0, 3.0])
    for T in (0.0, -1.0):
        g = _run1(o, z, T, 0.9)
        if int(g["token"][0]) != 1 or g["probs"][0][1] != 1.0 or g["probs"][0].sum() != 1.0:
            fails.append(f"greedy T={T}: token {int(g['token'][0])}")

    # Failure statuses.
    cases = [(np.array([0.0, np.nan, 1.0]), 1.0, 0.5, 0.0, 1),
             (np.array([0.0, np.inf, 1.0]), 1.0, 0.5, 0.0, 1),
             (np.array([-np.inf, -np.inf]), 1.0, 0.5, 0.0, 2),
             (np.array([0.0, 1.0]), np.nan, 0.5, 0.0, 3),
             (np.array([0.0, 1.0]), np.inf, 0.5, 0.0, 3),
             (np.array([0.0, 1.0]), 1.0, np.nan, 0.0, 3),
             (np.array([0.0, 1.0]), 1.0, 0.5, np.nan, 3)]
    for z, T, p, m, st in cases:
        r = _run1(o, z, T, p, m=m)
        if int(r["status"][0]) != st or int(r["token"][0]) != -1 or np.any(r["probs"][0] != 0):
            fails.append(f"status case {z},{T},{p},{m}: status {int(r['status'][0])} != {st}")

    # Precision: on a 128,000-token row with a realistic spread, p = 0.9 keeps far fewer than all
    # tokens (Top-p (Nucleus) Sampling, in depth -- 'What to do next', item 2).
    z = rng.normal(0, 3.0, 128000)
    got = int(_run1(o, z, 1.0, 0.9, probs=False)["kept"][0])
    if not (0 < got < 128000 // 4):
        fails.append(f"128k row at p=0.9 keeps {got}")

    # The empty batch is a no-op.
    r = o.sample(np.zeros((0, 5)), np.zeros(0, np.float32), np.zeros(0, np.int32),
                 np.zeros(0, np.float32), np.zeros(0, np.float32), np.zeros(0, np.uint64))
    if r["token"].shape != (0,):
        fails.append("empty batch")
    return fails


# -------------------------------------------------------------------------------------------
def check_uniform_mapping(o):
    """u = (2 * (x >> 9) + 1) * 2^-24: an odd multiple of 2^-24 strictly inside (0, 1), drawn
    from word (i mod 4) of the Philox block at counter (floor(i / 4), row, step)."""
    fails = []
    us = []
    for t in range(4096):
        seed, row, step = 77 + (t % 5), t % 13, t // 13
        u = o.uniform(seed, row, step, t)
        q = u * 2 ** 24
        if not (0.0 < u < 1.0) or q != math.floor(q) or int(q) % 2 != 1:
            fails.append(f"u={u!r} is not an odd multiple of 2^-24 in (0, 1)")
            break
        blk = o.philox4x32_10([t // 4, row, step & 0xFFFFFFFF, step >> 32], [seed, 0])
        if int(q) >> 1 != int(blk[t % 4]) >> 9:
            fails.append(f"u for token {t} is not taken from word {t % 4} of its block")
            break
        us.append(u)
    us = np.asarray(us)
    if len(us) and abs(us.mean() - 0.5) > 5 * math.sqrt(1 / 12 / len(us)):
        fails.append(f"uniform mean {us.mean()}")
    return fails


_TRITON_SCRIPT = r"""
import json, os, sys
os.environ["TRITON_INTERPRET"] = "1"
import numpy as np, torch, triton, triton.language as tl

@triton.jit
def _k(out_ptr, seed, c0_ptr, c1_ptr, c2_ptr, c3_ptr, N: tl.constexpr):
    offs = tl.arange(0, N)
    a, b, c, d = tl.philox(seed, tl.load(c0_ptr + offs), tl.load(c1_ptr + offs),
                           tl.load(c2_ptr + offs), tl.load(c3_ptr + offs), 10)
    tl.store(out_ptr + offs * 4 + 0, a)
    tl.store(out_ptr + offs * 4 + 1, b)
    tl.store(out_ptr + offs * 4 + 2, c)
    tl.store(out_ptr + offs * 4 + 3, d)

req = json.loads(sys.stdin.read())
res = []
for seed, ctrs in req:
    N = len(ctrs)
    cols = [torch.tensor([c[j] for c in ctrs], dtype=torch.int64).to(torch.uint32) for j in range(4)]
    out = torch.zeros(N * 4, dtype=torch.uint32)
    _k[(1,)](out, seed, *cols, N=N)
    res.append(out.to(torch.int64).view(N, 4).tolist())
print(json.dumps(res))
"""


def triton_philox_available():
    try:
        import triton.language as tl  # noqa: F401
        return hasattr(tl, "philox")
    except Exception:
        return False


def check_philox_vs_triton(o):
    """Compare the oracle's Philox4x32-10 with Triton's own implementation, run on the CPU by
    Triton's interpreter (an independent third-party implementation of the same generator)."""
    rng = np.random.default_rng(11)
    req = []
    for seed in (0, 1, 0xFFFFFFFF, 0x123456789ABCDEF0, int(rng.integers(0, 2**63))):
        ctrs = [[0, 0, 0, 0], [1, 0, 0, 0], [0xFFFFFFFF] * 4]
        ctrs += rng.integers(0, 2**32, size=(5, 4)).tolist()
        req.append([int(seed), [[int(x) for x in c] for c in ctrs]])
    env = dict(os.environ, TRITON_INTERPRET="1")
    out = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT], input=json.dumps(req),
                         capture_output=True, text=True, env=env, timeout=600)
    if out.returncode != 0:
        return [f"triton interpreter failed: {out.stderr[-500:]}"]
    got = json.loads(out.stdout.strip().splitlines()[-1])
    fails = []
    for (seed, ctrs), blocks in zip(req, got):
        key = [seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF]
        for c, want in zip(ctrs, blocks):
            mine = [int(x) for x in o.philox4x32_10(c, key)]
            if mine != [int(x) & 0xFFFFFFFF for x in want]:
                fails.append(f"philox seed={seed:#x} ctr={c}: {mine} != {want}")
    return fails


def check_penalties(o):
    """Repetition / frequency / presence penalties (float32 arithmetic), pinned by hand-worked
    values, identities and invariants of the definition: the pages name the three penalties and
    their place (on raw logits, before temperature) but print no formula or example."""
    fails = []
    f32 = np.float32

    # A hand-worked row (every intermediate is exact in float32):
    #   t0: c=1, 2/2 = 1,    1 - (0.5*1 + 0.25) = 0.25
    #   t1: c=2, -1*2 = -2, -2 - (0.5*2 + 0.25) = -3.25
    #   t2, t3: not in the history, unchanged;  t4: c=3, 3/2 = 1.5, 1.5 - (1.5 + 0.25) = -0.25
    z = np.array([[2.0, -1.0, 0.5, 0.0, 3.0]], f32)
    out, st = o.penalties(z, [[0, 1, 1, 4, 4, 4]], repetition=[2.0], frequency=[0.5], presence=[0.25])
    want = np.array([[0.25, -3.25, 0.5, 0.0, -0.25]], f32)
    if not np.array_equal(out, want) or st[0] != 0:
        fails.append(f"worked row: {out.tolist()} status {st.tolist()}, want {want.tolist()}")

    # Repetition alone: positive logits are divided, negative ones multiplied, zero stays zero.
    out, _ = o.penalties(np.array([[4.0, -4.0, 0.0, 1.5]], f32), [[0, 1, 2]], repetition=[2.0])
    if not np.array_equal(out, np.array([[2.0, -8.0, 0.0, 1.5]], f32)):
        fails.append(f"repetition sign rule: {out.tolist()}")

    # Frequency and presence on integer logits: z - f*c - rho, exactly.
    rng = np.random.default_rng(17)
    zi = rng.integers(-20, 20, size=(3, 50)).astype(f32)
    hist = rng.integers(0, 50, size=(3, 40)).astype(np.int32)
    out, _ = o.penalties(zi, hist, frequency=[0.5, 0.25, 2.0], presence=[1.0, 0.0, 0.5])
    for b, (fq, pr) in enumerate(((0.5, 1.0), (0.25, 0.0), (2.0, 0.5))):
        c = np.bincount(hist[b], minlength=50)
        exp_row = np.where(c > 0, zi[b] - fq * c - pr, zi[b]).astype(f32)
        if not np.array_equal(out[b], exp_row):
            fails.append(f"frequency/presence closed form, row {b}")

    # Penalties off: the row is unchanged, bit for bit (NaN, infinities and -0.0 included).
    zr = rng.normal(0, 3, size=(2, 300)).astype(f32)
    zr[0, :5] = [np.nan, np.inf, -np.inf, -0.0, 0.0]
    hr = rng.integers(0, 300, size=(2, 100)).astype(np.int32)
    out, _ = o.penalties(zr, hr, repetition=[1.0, 1.0], frequency=[0.0, 0.0], presence=[0.0, 0.0])
    if not np.array_equal(out.view(np.uint32), zr.view(np.uint32)):
        fails.append("penalties off changed the logits")

    # The history is a multiset: order does not matter; padding (< 0), ids >= V and entries past the
    # row's length are ignored.
    args = dict(repetition=[1.3, 0.7], frequency=[0.3, 0.1], presence=[0.2, 0.4])
    a, _ = o.penalties(zr, hr, **args)
    b_, _ = o.penalties(zr, hr[:, ::-1].copy(), **args)
    padded = np.concatenate([hr, np.full((2, 7), -1, np.int32), np.full((2, 3), 300, np.int32),
                             rng.integers(0, 300, size=(2, 9)).astype(np.int32)], axis=1)
    c_, _ = o.penalties(zr, padded, hist_len=[100 + 7 + 3, 100 + 10], **args)
    if not (np.array_equal(a, b_, equal_nan=True) and np.array_equal(a, c_, equal_nan=True)):
        fails.append("history order, padding or length changed the result")
    if not np.array_equal(a[:, 5:] != zr[:, 5:], np.stack([np.isin(np.arange(5, 300), hr[i]) for i in range(2)])):
        fails.append("a token outside the history was changed, or one inside was not")

    # One token repeated H times: z/r - (f*H + rho).
    out, _ = o.penalties(np.array([[3.0, 1.0]], f32), np.zeros((1, 64), np.int32), repetition=[1.5],
                         frequency=[0.125], presence=[1.0])
    if out[0, 0] != f32(2.0) - f32(0.125 * 64 + 1.0) or out[0, 1] != f32(1.0):
        fails.append(f"repeated token: {out.tolist()}")

    # Bad parameters leave the row unchanged and report it (status 3); the other rows still run.
    zb = np.tile(np.array([[1.0, -2.0, 3.0]], f32), (6, 1))
    hb = np.zeros((6, 2), np.int32)
    out, st = o.penalties(zb, hb, repetition=[0.0, -1.0, np.nan, 1.0, 1.0, 2.0],
                          frequency=[0.0, 0.0, 0.0, np.inf, 0.0, 0.0], presence=[0.0, 0.0, 0.0, 0.0, np.nan, 0.0])
    if st.tolist() != [3, 3, 3, 3, 3, 0] or not np.array_equal(out[:5], zb[:5]) or out[5, 0] != f32(0.5):
        fails.append(f"bad parameters: status {st.tolist()}")

    # bfloat16 logits: the float32 result rounded to nearest bfloat16, ties to even.  Near 1 the
    # bfloat16 grid is 1 + k/128: 1 + 0.5/128 ties to 1 (k even), 1 + 1.5/128 ties to 1 + 2/128, and
    # 1 + 0.5/128 + 2^-23 rounds up to 1 + 1/128.
    fz = np.array([0.99609375, 0.98828125, f32(0.99609375) - f32(2.0 ** -23)], f32)
    out, _ = o.penalties(np.full((3, 1), 2.0, f32), np.zeros((3, 1), np.int32), frequency=fz, bf16=True)
    want = np.array([1.0, 1.015625, 1.0078125], f32)
    if not np.array_equal(out[:, 0], want):
        fails.append(f"bfloat16 rounding: {out[:, 0].tolist()}, want {want.tolist()}")
    return fails


def _expected_rounds(e_sorted_classes, n_kept_classes):
    """Mean rounds of the rejection draw, by recursion over the classes (descending): with the
    top j classes eligible, one round draws class c with probability m_c / M_j; a kept class ends
    the draw, any other leaves its upper classes (1..c-1) eligible."""
    m = np.asarray(e_sorted_classes, np.float64)
    E = np.ones(len(m) + 1)
    for j in range(n_kept_classes + 1, len(m) + 1):
        M = m[:j].sum()
        E[j] = 1.0 + sum(m[c - 1] / M * E[c - 1] for c in range(n_kept_classes + 1, j + 1))
    return E[len(m)]


def check_rejection(o):
    """The sort-free rejection draw: the page's printed run (frequencies and mean rounds), the exact
    distribution and expected rounds, and membership of every draw in the kept set."""
    fails = []
    for c in _golden()["rejection_frequencies"]:
        z = np.asarray(c["logits"], np.float64)
        n = int(c["draws"])
        seeds = np.arange(n, dtype=np.uint64) * np.uint64(0x9E3779B97F4A7C15) + np.uint64(999)
        r = o.sample(np.tile(z, (n, 1)), np.float32(c["temperature"]), 0, np.float32(c["top_p"]), 0.0, seeds,
                     step=3, draw="rejection")
        exact = _run1(o, z, c["temperature"], c["top_p"])["probs"][0]
        freq = np.bincount(r["token"], minlength=len(z)) / n
        sig = np.sqrt(exact * (1 - exact) / n)
        if np.any(np.abs(freq - exact) > 5 * sig + 1e-12):
            fails.append(f"{c['id']}: frequencies {np.round(freq, 4)} vs exact {np.round(exact, 4)}")
        want = np.asarray(c["frequencies"])
        k = len(want)
        if np.any(np.abs(freq[:k] - want) > 5 * np.sqrt(2) * sig[:k] + 6e-4):
            fails.append(f"{c['id']}: frequencies {np.round(freq[:k], 4)} vs printed {want}")
        # expected rounds: distinct logits here, so every token is its own class
        e = np.exp(-(z.max() - np.sort(z)[::-1]) / np.float64(np.float32(c["temperature"])))
        Er = _expected_rounds(e, int((exact > 0).sum()))
        mr, sr = r["rounds"].mean(), r["rounds"].std() / np.sqrt(n)
        if abs(mr - Er) > 5 * sr + 1e-12:
            fails.append(f"{c['id']}: mean rounds {mr:.4f} vs expected {Er:.4f}")
        if abs(mr - c["mean_rounds"]) > 5 * np.sqrt(2) * sr + 0.005:
            fails.append(f"{c['id']}: mean rounds {mr:.4f} vs printed {c['mean_rounds']}")
    # every draw lies in the kept set; greedy rows match the race; no top-p means one round
    for w in _tiny_batches(n_batches=150):
        args = (w.logits.double().numpy(), w.temperature.numpy(), w.top_k.numpy(), w.top_p.numpy(),
                w.min_p.numpy(), w.seed.numpy().astype(np.uint64), w.step)
        a, b = o.sample(*args), o.sample(*args, draw="rejection")
        zz = w.logits.double().numpy()
        for i in range(w.B):
            if a["status"][i] != 0:
                if b["token"][i] != -1:
                    fails.append(f"{w.name} row {i}: failed row drew a token")
                continue
            t = b["token"][i]
            if not (t >= 0 and np.isfinite(zz[i, t]) and zz[i, t] >= a["cutoff"][i]):
                fails.append(f"{w.name} row {i}: rejection draw {t} outside the kept set")
            if w.temperature[i] <= 0 and t != a["token"][i]:
                fails.append(f"{w.name} row {i}: greedy row differs")
            if w.temperature[i] > 0 and w.top_p[i] >= 1 and b["rounds"][i] != 1:
                fails.append(f"{w.name} row {i}: {b['rounds'][i]} rounds with top-p off")
    return fails


def _philox_word(o, seed, c0, row_word, step, token):
    blk = o.philox4x32_10([c0 & 0xFFFFFFFF, row_word & 0xFFFFFFFF, step & 0xFFFFFFFF, (step >> 32) & 0xFFFFFFFF],
                          [seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF])
    return (2 * (int(blk[token % 4]) >> 9) + 1) * 2.0 ** -24


def check_counter_layouts(o):
    """Where each draw takes its uniforms from (the generator itself is pinned against Triton's
    Philox): the race at counter (i/4, row, step); rejection round r at ((i/4) | (r+1) << 18, row,
    step), so round 0 never reuses the race's counters; speculative acceptance at (i/4, row | 2^31,
    step), with token 2^20 - 1 (word 3 of block 2^18 - 1, above every token index) the acceptance
    test's own uniform."""
    fails = []
    rng = np.random.default_rng(17)
    for _ in range(200):
        seed = int(rng.integers(0, 2**63))
        row, step, tok = int(rng.integers(0, 2**27)), int(rng.integers(0, 2**63)), int(rng.integers(0, 2**20 - 1))
        u_race = o.uniform(seed, row, step, tok)
        if u_race != _philox_word(o, seed, tok // 4, row, step, tok):
            fails.append(f"race uniform of token {tok} not at counter (i/4, row, step)")
        for r in (0, 1, 5):
            u = o.uniform_round(seed, row, step, tok, r)
            if u != _philox_word(o, seed, (tok // 4) | ((r + 1) << 18), row, step, tok):
                fails.append(f"rejection round {r} uniform of token {tok} not at counter ((i/4) | (r+1) << 18, ...)")
        if o.uniform_round(seed, row, step, tok, 0) == u_race:
            fails.append("rejection round 0 reuses the race's uniform")
        u_spec = o.uniform_spec(seed, row, step, tok)
        if u_spec != _philox_word(o, seed, tok // 4, row | 0x80000000, step, tok):
            fails.append(f"speculative uniform of token {tok} not at counter (i/4, row | 2^31, step)")
        if u_spec == u_race:
            fails.append("speculative uniform reuses the race's")
        if o.uniform_spec(seed, row, step, 2**20 - 1) != _philox_word(o, seed, 2**18 - 1, row | 0x80000000, step, 3):
            fails.append("the acceptance uniform is not word 3 of block 2^18 - 1")
        if len(fails) > 5:
            break
    return fails


def _softmax_trunc(z, T, k=0, p=1.0, m=0.0):
    """The renormalised kept distribution written out for small, tie-free rows: min-p, top-k, then
    top-p on the survivors (keep a token iff the mass of more probable survivors is below p)."""
    z = np.asarray(z, np.float64)
    T = float(np.float32(T))
    p = float(np.float32(p))
    e = np.exp((z - z.max()) / T)
    keep = np.ones(len(z), bool)
    if m > 0:
        keep &= e >= min(float(np.float32(m)), 1.0)
    if 0 < k < len(z):
        keep &= z >= np.sort(z)[::-1][k - 1]
    if p < 1:
        order = np.argsort(-z)
        Zs = e[keep].sum()
        above = 0.0
        for i in order:
            if not keep[i]:
                continue
            if above >= p * Zs and z[i] < z.max():
                keep[i] = False
            above += e[i]
    P = np.where(keep, e, 0.0)
    return P / P.sum()


def check_spec_accept(o):
    """Speculative acceptance ("Top-p (Nucleus) Sampling, in depth", 'Logprobs, speculative decoding
    and reproducibility'): the draft token is accepted with probability min(1, P(x)/Q(x)) and a
    rejection draws from the normalised (P - Q)+, which makes the output distributed exactly as P for
    any draft distribution Q; P and Q are the truncated, renormalised distributions."""
    fails = []
    rng = np.random.default_rng(23)
    # --- statistics on small rows, P and Q written out independently of the oracle
    cases = [
        # (target logits, target (T, k, p, m), draft logits, draft (T, k, p, m))
        (np.log([0.5, 0.3, 0.2]), (1.0, 0, 0.6, 0.0), np.zeros(3), (1.0, 0, 1.0, 0.0)),
        ([2.0, 1.0, 0.0, -1.0, 0.5], (0.7, 0, 1.0, 0.0), [0.0, 1.0, 2.0, 0.5, -0.3], (1.3, 3, 1.0, 0.0)),
        ([0.3, 1.7, -0.4, 0.9], (1.1, 0, 0.95, 0.1), [1.2, 0.1, 0.8, -2.0], (0.6, 0, 0.9, 0.0)),
    ]
    n = 200_000
    for ci, (zt, pt, zd, pd) in enumerate(cases):
        zt, zd = np.asarray(zt, np.float64), np.asarray(zd, np.float64)
        P, Q = _softmax_trunc(zt, *pt), _softmax_trunc(zd, *pd)
        x = rng.choice(len(zd), size=n, p=Q)
        seeds = np.arange(n, dtype=np.uint64) * np.uint64(0x9E3779B97F4A7C15) + np.uint64(31 + ci)
        r = o.spec_accept(np.tile(zt, (n, 1)), np.tile(zd, (n, 1)), pt, pd, x, seeds, step=5)
        if (r["status"] != 0).any():
            fails.append(f"case {ci}: failed rows")
            continue
        acc = r["accepted"].mean()
        a_exact = np.minimum(P, Q).sum()
        if abs(acc - a_exact) > 5 * np.sqrt(a_exact * (1 - a_exact) / n) + 1e-9:
            fails.append(f"case {ci}: acceptance rate {acc:.5f} vs sum min(P, Q) = {a_exact:.5f}")
        freq = np.bincount(r["token"], minlength=len(zt)) / n
        sig = np.sqrt(P * (1 - P) / n)
        if np.any(np.abs(freq - P) > 5 * sig + 1e-9):
            fails.append(f"case {ci}: output frequencies {np.round(freq, 4)} vs P {np.round(P, 4)}")
        rej = r["accepted"] == 0
        resid = np.maximum(P - Q, 0)
        if rej.sum() > 1000 and resid.sum() > 0:
            R = resid / resid.sum()
            fr = np.bincount(r["token"][rej], minlength=len(zt)) / rej.sum()
            if np.any(np.abs(fr - R) > 5 * np.sqrt(R * (1 - R) / rej.sum()) + 1e-9):
                fails.append(f"case {ci}: rejected draws {np.round(fr, 4)} vs normalised (P-Q)+ {np.round(R, 4)}")
        if np.any((r["accepted"] == 1) & (r["token"] != x)):
            fails.append(f"case {ci}: an accepted row does not return the draft token")
        if np.any(np.abs(r["p_x"] - P[x]) > 1e-12) or np.any(np.abs(r["q_x"] - Q[x]) > 1e-12):
            fails.append(f"case {ci}: P(x) or Q(x) differs from the written-out distributions")
    # --- special cases
    V = 40
    zt = rng.normal(0, 2, size=(64, V))
    zt[:, 5] = zt[:, 7] = zt.max(axis=1) + 0.5  # tied maxima
    T = rng.choice([0.5, 1.0, 2.0], 64)
    k = rng.choice([0, 3, 10], 64)
    p = rng.uniform(0.2, 1.0, 64)
    m = rng.choice([0.0, 0.05], 64)
    seeds = np.arange(64, dtype=np.uint64) + np.uint64(100)
    own = o.sample(zt, T, k, p, m, seeds, 9)["token"]
    # P == Q: every draft token the draft can produce is accepted
    r = o.spec_accept(zt, zt, (T, k, p, m), (T, k, p, m), own, seeds, step=9)
    if not (r["accepted"] == 1).all() or not (r["token"] == own).all():
        fails.append("identical target and draft: not every draft token accepted")
    # greedy target: always its lowest-index maximum
    r = o.spec_accept(zt, zt, (0.0, 0, 1.0, 0.0), (T, k, p, m), own, seeds, step=9)
    if not (r["token"] == 5).all():
        fails.append("greedy target: not always its lowest-index maximum")
    # disjoint supports: never accepted, the output lies in the target's support
    za, zb = zt.copy(), zt.copy()
    za[:, 20:] = -np.inf
    zb[:, :20] = -np.inf
    xb = o.sample(zb, 1.0, 0, 1.0, 0.0, seeds, 9)["token"]
    r = o.spec_accept(za, zb, (1.0, 0, 1.0, 0.0), (1.0, 0, 1.0, 0.0), xb, seeds, step=9)
    if (r["accepted"] != 0).any() or (r["token"] >= 20).any() or (r["token"] < 0).any():
        fails.append("disjoint supports: a draft token accepted, or the output outside the target's support")
    # truncation is respected: a draft token outside the target's nucleus is never accepted
    z3 = np.tile(np.log([0.5, 0.3, 0.2]), (64, 1))
    r = o.spec_accept(z3, np.zeros((64, 3)), (1.0, 0, 0.6, 0.0), (1.0, 0, 1.0, 0.0), np.full(64, 2), seeds, step=9)
    if (r["accepted"] != 0).any() or (r["token"] == 2).any():
        fails.append("a draft token outside the target's nucleus was accepted")
    # failures: a draft token the draft cannot produce, out of range, a failed target or draft row
    zbad = zt[:4].copy()
    zbad[2, 3] = np.nan
    zd = zt[:4].copy()
    zd[3] = -np.inf
    x = np.array([-1, V, 0, 0])
    r = o.spec_accept(zbad, zd, (1.0, 0, 1.0, 0.0), (1.0, 0, 1.0, 0.0), x, seeds[:4], step=9)
    if r["status"].tolist() != [3, 3, 1, 2] or (r["token"] != -1).any() or (r["accepted"] != 0).any():
        fails.append(f"failed rows: status {r['status'].tolist()} tokens {r['token'].tolist()}")
    zq = np.log(np.array([[0.7, 0.2, 0.1]]))
    r = o.spec_accept(zq, zq, (1.0, 0, 1.0, 0.0), (1.0, 1, 1.0, 0.0), [2], seeds[:1], step=9)
    if r["status"][0] != 3:
        fails.append("a draft token outside the draft's own kept set is not rejected as invalid")
    return fails


ALL_CHECKS = {
    "counter_layouts": check_counter_layouts,
    "spec_accept": check_spec_accept,
    "rejection": check_rejection,
    "penalties": check_penalties,
    "worked_examples": check_worked_examples,
    "sample_frequencies": check_sample_frequencies,
    "bruteforce": check_bruteforce,
    "closed_forms": check_closed_forms,
    "uniform_mapping": check_uniform_mapping,
}
