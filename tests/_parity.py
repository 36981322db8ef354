"""GPU-versus-oracle comparison used by the GPU parity tests."""
from __future__ import annotations

import numpy as np
import torch

import nucleus_token_sampler_gb300 as tps
import oracle

TOPP_BAND, MINP_BAND, RACE_BAND = oracle.FLAG_TOPP_BAND, oracle.FLAG_MINP_BAND, oracle.FLAG_RACE_BAND
PROB_TOL = 1e-5  # absolute, on renormalised probabilities
# absolute, on ln P(token) (plus 1e-6 relative): the kept mass is an exact sum of float expf values
# (relative error ~3e-7 -> ~3e-7 in the log) and the result is stored as a float (ulp 2e-6 at |ln P| = 30)
LOGPROB_TOL = 1e-5


def run_gpu(w, want_probs=True, logits=None, kernel="auto", want_logprob=None, top=None):
    """The library on the GPU.  The log-probability outputs (the sampled token's, and the top 8
    tokens') are requested for the auto kernel (unless want_logprob / top say otherwise), so the
    explicit kernels keep covering the path without them."""
    d = w.to("cuda")
    lg = d.logits if logits is None else logits
    if want_logprob is None:
        want_logprob = kernel == "auto"
    if top is None:
        top = 8 if kernel == "auto" else 0
    r = tps.sample(lg, d.temperature, d.top_k, d.top_p, d.min_p, d.seed, d.step, want_probs=want_probs,
                   diagnostics=True, want_logprob=want_logprob, top_logprobs=top, kernel=kernel)
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in r.items()}


def run_oracle(w, rows=None, want_probs=True):
    z = w.logits if rows is None else w.logits[rows]
    sel = (lambda t: t) if rows is None else (lambda t: t[rows])
    return oracle.sample(z.double().numpy(), sel(w.temperature).numpy(), sel(w.top_k).numpy(),
                         sel(w.top_p).numpy(), sel(w.min_p).numpy(),
                         sel(w.seed).numpy().astype(np.uint64), w.step,
                         row_ids=None if rows is None else np.asarray(rows), want_probs=want_probs)


def expected_top(w, o, rows, j, n):
    """The oracle's n most probable kept tokens of row rows[j] (probability descending, index
    ascending) and their ln P.  The kept set is every finite logit at or above the cutoff (ties
    included); a greedy row keeps its token alone."""
    row = int(rows[j])
    if float(w.temperature[row]) <= 0.0:
        return [int(o["token"][j])], [0.0]
    z = w.logits[row].double().numpy()
    kept = np.nonzero(np.isfinite(z) & (z >= o["cutoff"][j]))[0]
    assert len(kept) == int(o["kept"][j]), "the kept set read off the cutoff disagrees with the oracle's count"
    order = kept[np.lexsort((kept, -z[kept]))][:n]
    return order.tolist(), np.log(o["probs"][j, order]).tolist()


def compare_top(w, g, o, rows, okrow, setband):
    """Top-n tokens and log-probabilities against the oracle, on rows whose kept set is exact."""
    fails = []
    ti = g["top_idx"].numpy()[rows]
    tl = g["top_logprob"].numpy()[rows].astype(np.float64)
    n = ti.shape[1]
    worst = 0.0
    for j in np.nonzero(okrow & ~setband)[0]:
        idx, lp = expected_top(w, o, rows, j, n)
        want = np.full(n, -1, dtype=np.int64)
        want[:len(idx)] = idx
        if not np.array_equal(ti[j], want):
            fails.append(f"top tokens differ at row {rows[j]}: gpu {ti[j].tolist()} oracle {want.tolist()}")
            break
        ref = np.asarray(lp)
        err = np.abs(tl[j, :len(idx)] - ref)
        bad = err > LOGPROB_TOL + 1e-6 * np.abs(ref)
        if bad.any():
            fails.append(f"top log-probability differs by {err.max():.3e} at row {rows[j]}")
            break
        if len(idx) < n and not (tl[j, len(idx):] == -np.inf).all():
            fails.append(f"empty top slots of row {rows[j]} are not -inf")
            break
        worst = max(worst, float(err.max()) if len(err) else 0.0)
    failed = ~okrow
    if failed.any() and not ((ti[failed] == -1).all() and np.isnan(tl[failed]).all()):
        fails.append("failed rows have top tokens")
    return fails


TOPP_TOL = 1e-6     # the top-p band: normalised mass above a class within this of p
MINP_TOL = 1e-12    # the min-p band: e_i within this (relative) of min_p


def valid_kept_classes(z, T, k, p, m):
    """Every kept set a correct sampler may return on one row, as a set of class counts j (the kept
    set is the j largest classes of equal logits).  Exact where the decisions are clear; where the
    oracle's float64 decision sits within the band (top-p: the normalised mass above a class within
    TOPP_TOL of p; min-p: e_i within MINP_TOL of min_p, relative), either outcome is accepted.
    The rules are the sampler's: min-p keeps e_i >= min(m, 1); top-k keeps logits >= the k-th
    largest finite logit; top-p keeps a class of S iff the mass of S above it, over the mass of S,
    is below p; the class of the maximum is always kept; p >= 1 keeps S."""
    fin = np.isfinite(z)
    zf = z[fin]
    vals, counts = np.unique(zf, return_counts=True)
    vals, counts = vals[::-1], counts[::-1]  # classes, largest logit first
    zmax = vals[0]
    e = np.exp(-((zmax - vals) / T))
    mass = counts * e
    n_cls = len(vals)
    lo = hi = n_cls  # classes of S: at least lo, at most hi (S is a prefix of the classes)
    mm = min(m, 1.0)
    if mm > 0:
        sure = e >= mm * (1 + MINP_TOL) if mm > 0 else np.ones(n_cls, bool)
        maybe = e >= mm * (1 - MINP_TOL)
        lo, hi = int(sure.sum()), int(maybe.sum())
    if 0 < k < len(z) and k < len(zf):
        vk = np.sort(zf)[::-1][k - 1]
        nk = int((vals >= vk).sum())
        lo, hi = min(lo, nk), min(hi, nk)
    lo, hi = max(lo, 1), max(hi, 1)
    ok = set()
    for L in range(lo, hi + 1):
        if p >= 1:
            ok.add(L)
            continue
        if p <= 0:
            ok.add(1)
            continue
        Z = mass[:L].sum()
        above = np.concatenate([[0.0], np.cumsum(mass[:L])[:-1]]) / Z
        for j in range(1, L + 1):
            last_ok = j == 1 or above[j - 1] < p + TOPP_TOL
            next_ok = j == L or above[j] >= p - TOPP_TOL
            if last_ok and next_ok:
                ok.add(j)
    return ok, vals, counts


def check_band_row(w, g, rows, j):
    """A boundary row: the GPU's kept set must be one of the correct ones (valid_kept_classes), and
    its token, probabilities and log-probability must be the oracle's over that kept set (the race
    with the same uniforms, renormalised over the same tokens).  Returns failure strings."""
    b = int(rows[j])
    z = w.logits[b].double().numpy()
    T = float(np.float32(w.temperature[b]))
    k = int(w.top_k[b])
    p = float(np.float32(w.top_p[b]))
    m = float(np.float32(w.min_p[b]))
    kept_g = int(g["kept"][b])
    cut_g = float(g["cutoff"][b])
    ok, vals, counts = valid_kept_classes(z, T, k, p, m)
    if cut_g not in set(vals.tolist()):
        return [f"band row {b}: cutoff {cut_g} is not a logit of the row"]
    jg = int((vals >= cut_g).sum())
    if int(counts[:jg].sum()) != kept_g:
        return [f"band row {b}: kept {kept_g} is not the size of the classes at or above the cutoff"]
    if jg not in ok:
        return [f"band row {b}: the GPU keeps {jg} classes; a correct answer keeps one of {sorted(ok)[:8]}"]
    # the oracle over exactly the GPU's kept set: top-k = kept_g selects it (whole classes), nothing else cuts
    want_probs = "probs" in g
    o2 = oracle.sample(z[None], np.float32(T), kept_g, np.float32(1.0), np.float32(0.0),
                       np.asarray([int(w.seed[b])]).astype(np.uint64), w.step, row_ids=np.asarray([b]),
                       want_probs=True)
    fails = []
    if int(o2["kept"][0]) != kept_g:
        return [f"band row {b}: internal: top-k {kept_g} keeps {int(o2['kept'][0])}"]
    tok = int(g["token"][b])
    if (o2["flags"][0] & RACE_BAND) == 0 and tok != int(o2["token"][0]):
        fails.append(f"band row {b}: token {tok}, the race over the GPU's kept set draws {int(o2['token'][0])}")
    if not (np.isfinite(z[tok]) and z[tok] >= cut_g):
        fails.append(f"band row {b}: token {tok} is outside the GPU's kept set")
    if want_probs:
        d = np.abs(g["probs"][b].double().numpy() - o2["probs"][0]).max()
        if d > PROB_TOL:
            fails.append(f"band row {b}: probabilities differ by {d:.3e} from the renormalised kept set")
    if "logprob" in g and (o2["flags"][0] & RACE_BAND) == 0:
        with np.errstate(divide="ignore"):
            ref = float(np.log(o2["probs"][0, tok]))
        err = abs(float(g["logprob"][b]) - ref)
        if err > LOGPROB_TOL + 1e-6 * abs(ref):
            fails.append(f"band row {b}: logprob differs by {err:.3e}")
    if "top_idx" in g:
        n = g["top_idx"].shape[1]
        idx, lp = expected_top(w, o2, [b], 0, n)
        want = np.full(n, -1, dtype=np.int64)
        want[:len(idx)] = idx
        if not np.array_equal(g["top_idx"][b].numpy(), want):
            fails.append(f"band row {b}: top tokens differ")
        else:
            err = np.abs(g["top_logprob"][b].double().numpy()[:len(idx)] - np.asarray(lp))
            if len(idx) and (err > LOGPROB_TOL + 1e-6 * np.abs(np.asarray(lp))).any():
                fails.append(f"band row {b}: top log-probabilities differ by {err.max():.3e}")
    return fails


def compare(w, g, o, rows=None, check_probs=True):
    """Return (report dict, list of failure strings).  Rows the oracle flags as boundary rows are
    not skipped: check_band_row verifies that the GPU's answer is one of the correct ones."""
    B = w.B
    rows = np.arange(B) if rows is None else np.asarray(rows)
    st_g = g["status"].numpy()[rows]
    tok_g = g["token"].numpy()[rows]
    kept_g = g["kept"].numpy()[rows]
    cut_g = g["cutoff"].numpy()[rows].astype(np.float64)
    flags = o["flags"]
    fails = []
    if not np.array_equal(st_g, o["status"]):
        bad = np.nonzero(st_g != o["status"])[0][:5]
        fails.append(f"status differs at rows {rows[bad].tolist()}: gpu {st_g[bad]} oracle {o['status'][bad]}")
    okrow = o["status"] == 0
    setband = (flags & (TOPP_BAND | MINP_BAND)) != 0
    tokband = setband | ((flags & RACE_BAND) != 0)
    chk = okrow & ~setband
    for name, a, b in (("kept", kept_g, o["kept"]),):
        bad = np.nonzero(chk & (a != b))[0]
        if len(bad):
            fails.append(f"{name} differs on {len(bad)} rows, e.g. row {rows[bad[0]]}: gpu {a[bad[0]]} oracle {b[bad[0]]}")
    cut_o = o["cutoff"]
    bad = np.nonzero(chk & (cut_g != cut_o))[0]
    if len(bad):
        fails.append(f"cutoff differs on {len(bad)} rows, e.g. row {rows[bad[0]]}: gpu {cut_g[bad[0]]} oracle {cut_o[bad[0]]}")
    tchk = (o["status"] != 0) | ~tokband
    bad = np.nonzero(tchk & (tok_g != o["token"]))[0]
    if len(bad):
        fails.append(f"token differs on {len(bad)} rows, e.g. row {rows[bad[0]]}: gpu {tok_g[bad[0]]} oracle {o['token'][bad[0]]}")
    # boundary rows: one of the correct answers (kept set within the band, then the exact race over it)
    band_checked = 0
    for j in np.nonzero(okrow & setband)[0]:
        fails += check_band_row(w, g, rows, j)
        band_checked += 1
    # race-margin rows (two race keys within rounding): the token must still be a kept token
    for j in np.nonzero(okrow & ~setband & ((flags & RACE_BAND) != 0))[0]:
        b = int(rows[j])
        zt = float(w.logits[b, int(tok_g[j])]) if 0 <= int(tok_g[j]) < w.V else float("nan")
        if not (np.isfinite(zt) and zt >= cut_o[j]):
            fails.append(f"race-margin row {b}: token {int(tok_g[j])} is outside the kept set")
    if "logprob" in g and "probs" in o:
        # ln P(token) against the float64 oracle's renormalised probability of the same token
        lp = g["logprob"].numpy()[rows].astype(np.float64)
        m = okrow & ~tokband
        if m.any():
            ref = np.log(o["probs"][np.nonzero(m)[0], o["token"][m]])
            err = np.abs(lp[m] - ref)
            tol = LOGPROB_TOL + 1e-6 * np.abs(ref)
            if (err > tol).any():
                i = int(np.argmax(err - tol))
                fails.append(f"logprob differs by {err[i]:.3e} at a row with ln P = {ref[i]:.6f}")
        if (~okrow).any() and not np.isnan(lp[~okrow]).all():
            fails.append("failed rows have a non-NaN logprob")
    if "top_idx" in g and "probs" in o:
        fails += compare_top(w, g, o, rows, okrow, setband)
    maxdp = 0.0
    if check_probs and "probs" in g and "probs" in o:
        pg = g["probs"].numpy()[rows].astype(np.float64)
        po = o["probs"]
        m = chk
        if m.any():
            maxdp = float(np.abs(pg[m] - po[m]).max())
            if maxdp > PROB_TOL:
                fails.append(f"probabilities differ by {maxdp:.3e}")
        sums = pg[okrow].sum(axis=1)
        if okrow.any() and np.abs(sums - 1).max() > 1e-5:
            fails.append(f"probability rows sum to {sums.min()}..{sums.max()}")
        if (~okrow).any() and np.abs(pg[~okrow]).max() != 0:
            fails.append("failed rows have non-zero probabilities")
    rep = {"rows": int(len(rows)), "band_rows": int(setband.sum()), "band_rows_validated": band_checked,
           "topp_band_rows": int(((flags & TOPP_BAND) != 0).sum()), "minp_band_rows": int(((flags & MINP_BAND) != 0).sum()),
           "race_band_rows": int(((flags & RACE_BAND) != 0).sum()), "max_abs_dprob": maxdp}
    return rep, fails
