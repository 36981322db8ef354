"""Brute-force restatement of the sampler chain for tiny vocabularies (O(V^2) per row, pure Python).

Written straight from the pages' definitions, with no sorting and no classes, so that it checks the
oracle's sort-and-walk implementation rather than repeating it:

* temperature divides the logits before the softmax (What do temperature, top-k and top-p each
  do... -- 'A strong answer', the p_i(T) equation);
* min-p keeps p_i >= min_p * max p (Implement batched top-p sampling with temperature -- 'What
  interviewers probe next');
* top-k keeps a token when fewer than k logits are strictly larger (What do temperature... --
  reference sampler: 'ties at the k-th value survive');
* top-p keeps token i iff the mass of strictly more probable survivors is below p (Implement
  batched top-p sampling... -- 'How to approach it'), the maximum always kept (Top-p (Nucleus)
  Sampling, in depth -- 'Boundaries and ties').
"""
from __future__ import annotations

import math


def kept_set(z, T, k, p, m):
    """Return (status, keep list of bools, probs list) for one row, from the definitions."""
    V = len(z)
    if any(math.isnan(v) or v == math.inf for v in z):
        return "nan", None, None
    if not (math.isfinite(T) and math.isfinite(p) and math.isfinite(m)):
        return "bad_param", None, None
    finite = [v > -math.inf for v in z]
    if not any(finite):
        return "all_masked", None, None
    zmax = max(v for v in z if v > -math.inf)
    if T <= 0:
        arg = min(i for i in range(V) if z[i] == zmax)
        keep = [i == arg for i in range(V)]
        return "greedy", keep, [1.0 if i == arg else 0.0 for i in range(V)]
    # Tempered softmax, then each mask on its own.
    w = [math.exp(z[i] / T - zmax / T) if finite[i] else 0.0 for i in range(V)]
    tot = sum(w)
    prob = [x / tot for x in w]
    pmax = max(prob)
    mm = min(m, 1.0)
    s = []
    for i in range(V):
        ok = finite[i]
        if ok and mm > 0:
            ok = prob[i] >= mm * pmax
        if ok and 0 < k < V:
            larger = sum(1 for j in range(V) if finite[j] and z[j] > z[i])
            ok = larger < k
        s.append(ok)
    zs = sum(w[i] for i in range(V) if s[i])
    keep = []
    for i in range(V):
        if not s[i]:
            keep.append(False)
            continue
        if p >= 1.0 or z[i] == zmax:
            keep.append(True)
            continue
        above = sum(w[j] for j in range(V) if s[j] and z[j] > z[i])
        keep.append(above < p * zs)
    zk = sum(w[i] for i in range(V) if keep[i])
    probs = [w[i] / zk if keep[i] else 0.0 for i in range(V)]
    return "ok", keep, probs


def boundary_distance(z, T, k, p, m):
    """Smallest |mass above / Z_S - p| over survivors that are not in the top class (inf if none)."""
    V = len(z)
    finite = [v > -math.inf for v in z]
    zmax = max(v for v in z if v > -math.inf)
    w = [math.exp(z[i] / T - zmax / T) if finite[i] else 0.0 for i in range(V)]
    mm = min(m, 1.0)
    s = []
    for i in range(V):
        ok = finite[i] and (mm <= 0 or w[i] >= mm)
        if ok and 0 < k < V:
            ok = sum(1 for j in range(V) if finite[j] and z[j] > z[i]) < k
        s.append(ok)
    zs = sum(w[i] for i in range(V) if s[i])
    best = math.inf
    if p < 1.0:
        for i in range(V):
            if s[i] and z[i] != zmax:
                above = sum(w[j] for j in range(V) if s[j] and z[j] > z[i])
                best = min(best, abs(above / zs - p))
    return best
