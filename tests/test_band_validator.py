"""The boundary-row validator of the parity harness, checked on the CPU with the oracle standing in
for the GPU: each correct answer on a boundary row passes, and answers outside the band fail.

A boundary row is one where the float64 decision sits within rounding of the cut ("Implement batched
top-p sampling with temperature", 'Why each line is there': the .5/.3/.2 row at p = .8 keeps two
tokens exactly but three with float64 sums).  The parity tests accept either answer there, but only
with the exact race, probabilities and log-probabilities over the kept set the GPU chose.
"""
import numpy as np
import torch

import oracle
from nucleus_token_sampler_gb300 import workloads

from . import _parity


def _w(z, T, k, p, m, seed=5, step=2):
    z = torch.as_tensor(np.asarray(z, dtype=np.float64)).float()
    B = z.shape[0]
    f = lambda v, dt: torch.as_tensor(np.broadcast_to(np.asarray(v), (B,)).copy()).to(dt)
    return workloads.Workload("band", z, f(T, torch.float32), f(k, torch.int32), f(p, torch.float32),
                              f(m, torch.float32), f(seed, torch.int64), step)


def _as_gpu(w, kept_override=None):
    """The oracle's outputs shaped like the GPU's; kept_override[b] = k forces row b's kept set to
    its k largest classes (via top-k, top-p off), i.e. another candidate answer."""
    o = _parity.run_oracle(w)
    g = {k: torch.as_tensor(np.asarray(o[k])) for k in ("token", "status", "kept")}
    g["cutoff"] = torch.as_tensor(o["cutoff"]).float()
    g["probs"] = torch.as_tensor(o["probs"]).float()
    g["logprob"] = torch.as_tensor(np.log(o["probs"][np.arange(w.B), o["token"]])).float()
    for b, kc in (kept_override or {}).items():
        z = w.logits[b].double().numpy()
        vals = np.unique(z[np.isfinite(z)])[::-1]
        cut = vals[kc - 1]
        n = int((z >= cut).sum())
        o2 = oracle.sample(z[None], w.temperature[b:b + 1].numpy(), n, 1.0, 0.0,
                           w.seed[b:b + 1].numpy().astype(np.uint64), w.step, row_ids=[b], want_probs=True)
        g["token"][b] = int(o2["token"][0])
        g["kept"][b] = n
        g["cutoff"][b] = float(cut)
        g["probs"][b] = torch.as_tensor(o2["probs"][0]).float()
        g["logprob"][b] = float(np.log(o2["probs"][0, o2["token"][0]]))
    return g, o


def _rows():
    # row 0: .5/.3/.2 at p = .8 (top-p band: 2 or 3 classes); row 1: min_p = 1 and a second class
    # 1e-30 below the maximum, whose e = exp(-1e-30) is 1 in float64 but below 1 exactly (min-p band:
    # 1 or 2 classes); row 2: a clear row (the band does not apply)
    z = np.full((3, 5), -np.inf)
    z[0, :3] = np.log([0.5, 0.3, 0.2])
    z[1, :2] = [0.0, -1e-30]
    z[2, :4] = [2.0, 1.0, 0.5, -3.0]
    return _w(z, [1.0, 1.0, 1.0], [0, 0, 0], [0.8, 1.0, 0.6], [0.0, 1.0, 0.0])


def test_oracle_answer_passes():
    w = _rows()
    g, o = _as_gpu(w)
    rep, fails = _parity.compare(w, g, o)
    assert not fails, fails
    assert rep["band_rows"] == 2 and rep["band_rows_validated"] == 2, rep


def test_other_answer_inside_the_band_passes():
    w = _rows()
    g, o = _as_gpu(w, {0: 2, 1: 1})  # exact arithmetic's answers
    rep, fails = _parity.compare(w, g, o)
    assert not fails, fails


def test_answer_outside_the_band_fails():
    w = _rows()
    g, o = _as_gpu(w, {0: 1})  # one class at p = .8: the mass above class 2 is .5, far below p
    _, fails = _parity.compare(w, g, o)
    assert any("band row 0" in f for f in fails), fails


def test_wrong_token_on_a_band_row_fails():
    w = _rows()
    g, o = _as_gpu(w, {0: 2})
    g["token"][0] = 2  # outside the two kept classes
    _, fails = _parity.compare(w, g, o)
    assert any("band row 0" in f for f in fails), fails


def test_wrong_probabilities_on_a_band_row_fail():
    w = _rows()
    g, o = _as_gpu(w, {0: 2})
    g["probs"][0] = torch.tensor([0.5, 0.3, 0.2, 0.0, 0.0])  # not renormalised over the two kept classes
    _, fails = _parity.compare(w, g, o)
    assert any("band row 0" in f and "probabilities" in f for f in fails), fails


def test_valid_kept_classes_reference_cases():
    """Cases worked by hand: a clear top-p cut, p >= 1, p <= 0, top-k ties, the min-p band."""
    z = np.log(np.array([0.4, 0.2, 0.2, 0.2]))
    ok, _, _ = _parity.valid_kept_classes(z, 1.0, 0, 0.5, 0.0)
    assert ok == {2}                     # the tied .2 class has mass .4 above it: kept together
    ok, _, _ = _parity.valid_kept_classes(z, 1.0, 0, 1.0, 0.0)
    assert ok == {2}
    ok, _, _ = _parity.valid_kept_classes(z, 1.0, 0, 0.0, 0.0)
    assert ok == {1}
    ok, _, _ = _parity.valid_kept_classes(np.array([3.0, 2.0, 2.0, 1.0]), 1.0, 2, 1.0, 0.0)
    assert ok == {2}                     # top-2 keeps the tie at the 2nd value
    ok, _, _ = _parity.valid_kept_classes(np.array([0.0, -1e-30]), 1.0, 0, 1.0, 1.0)
    assert ok == {1, 2}
    ok, _, _ = _parity.valid_kept_classes(np.array([0.0, -1.0]), 1.0, 0, 1.0, 0.5)
    assert ok == {1}                     # e = .37 is clearly below min_p = .5
