"""tps_sample_noalloc, the sampling entry point for callers that cannot allocate device memory while
they sample (a serving loop that reserves all device memory up front, a host whose allocator belongs
to another framework).  It runs the same kernels as tps_sample_full but keeps the streaming kernel's
per-call scratch in a fixed array compiled into the library instead of drawing it from the device's
memory pool.  Called here through the C ABI and compared with tps_sample_full on the same inputs,
twice in a row (the array keeps the previous call's contents, so each call must clear what it needs).

The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import nucleus_token_sampler_gb300 as tps
from nucleus_token_sampler_gb300 import workloads

from . import _parity

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

TPS_ERR_SCRATCH = 6


def _outputs(B, n_top, dev):
    return {"token": torch.empty(B, dtype=torch.int32, device=dev),
            "status": torch.empty(B, dtype=torch.int32, device=dev),
            "cutoff": torch.empty(B, dtype=torch.float32, device=dev),
            "kept": torch.empty(B, dtype=torch.int32, device=dev),
            "logprob": torch.empty(B, dtype=torch.float32, device=dev),
            "top_idx": torch.empty((B, n_top), dtype=torch.int32, device=dev),
            "top_logprob": torch.empty((B, n_top), dtype=torch.float32, device=dev)}


def _call(fn, d, out, n_top, kernel=0):
    """One call of tps_sample_full or tps_sample_noalloc (same signature) through ctypes."""
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    B, V = d.logits.shape
    rc = fn(P(d.logits), tps.TPS_F32 if d.logits.dtype == torch.float32 else tps.TPS_BF16, B, V, V,
            P(d.temperature), P(d.top_k), P(d.top_p), P(d.min_p), P(d.seed), d.step, P(out["token"]), None,
            P(out["status"]), P(out["cutoff"]), P(out["kept"]), P(out["logprob"]), n_top, P(out["top_idx"]),
            P(out["top_logprob"]), kernel, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return rc, {k: v.cpu() for k, v in out.items()}


@pytest.mark.parametrize("name", ["decode", "mixed"])
def test_no_alloc_matches_the_pool_call(name):
    """The decode batch (B = 1024 x 128,256: whole rows claimed through the scratch's counter) and the
    mixed batch (B = 64, under four rows per SM: every row split into segments whose partial results
    merge through the scratch, and the rows without min-p listed there for the cluster kernel):
    identical tokens, statuses, kept sets and top tokens, log-probabilities within the parity
    tolerance, on two calls in a row."""
    lib = tps.load()
    w = workloads.make(name, device="cpu")
    d = w.to("cuda")
    n_top = 4
    rc, ref = _call(lib.tps_sample_full, d, _outputs(w.B, n_top, "cuda"), n_top)
    assert rc == 0
    for _ in range(2):
        rc, got = _call(lib.tps_sample_noalloc, d, _outputs(w.B, n_top, "cuda"), n_top)
        assert rc == 0, tps.load().tps_status_string(rc)
        for k in ("token", "status", "kept", "top_idx"):
            assert torch.equal(got[k], ref[k]), k
        assert torch.equal(torch.nan_to_num(got["cutoff"], nan=7.0), torch.nan_to_num(ref["cutoff"], nan=7.0))
        for k in ("logprob", "top_logprob"):
            a, b = got[k].double().numpy(), ref[k].double().numpy()
            same = (a == b) | (np.isnan(a) & np.isnan(b))
            close = np.abs(a - b) <= _parity.LOGPROB_TOL + 1e-6 * np.abs(b)
            assert (same | close).all(), k


def test_no_alloc_rejects_a_call_beyond_its_scratch():
    """A call whose scratch would exceed the fixed array is refused before anything is enqueued."""
    lib = tps.load()
    B, V = 2_200_000, 8  # the scratch holds 4 bytes per row (a list of rows): over 8 MiB
    z = torch.zeros((B, V), device="cuda")
    T = torch.ones(B, device="cuda")
    K = torch.zeros(B, dtype=torch.int32, device="cuda")
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    S = torch.zeros(B, dtype=torch.int64, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.tps_sample_noalloc(P(z), tps.TPS_F32, B, V, V, P(T), P(K), P(T), P(T), P(S), 0, P(tok), None, None,
                                None, None, None, 0, None, None, 2, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == TPS_ERR_SCRATCH
    assert b"scratch" in lib.tps_status_string(rc)
