"""The bounded waits of the streaming kernel run out without faulting or hanging the GPU.

tps_sample_stall_test makes CTA 0 withhold the copy of one chunk, so the stage it would fill never
completes -- a flag nothing sets -- and shortens the waits for data and hand-overs to 50 ms (copies
already in flight keep their full limit).  The rows that CTA could not finish must report TIMEOUT
with token -1, every other row must be sampled exactly as the oracle samples it, the call must
return, and the next ordinary call must work."""
import ctypes

import numpy as np
import pytest
import torch

import nucleus_token_sampler_gb300 as tps
from nucleus_token_sampler_gb300 import workloads

from . import _parity

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def test_bounded_waits_run_out_and_report_timeout():
    w = workloads.make("decode", device="cpu", B=512)
    d = w.to("cuda")
    tok = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    st = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = tps.load().tps_sample_stall_test(P(d.logits), tps.TPS_F32, w.B, w.V, P(d.temperature), P(d.top_k),
                                          P(d.top_p), P(d.min_p), P(d.seed), d.step, P(tok), P(st), 2, 50_000_000,
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    tok, st = tok.cpu().numpy(), st.cpu().numpy()
    assert set(np.unique(st).tolist()) <= {0, 4}, np.unique(st)
    timed_out = st == 4
    assert timed_out.any()
    assert (tok[timed_out] == -1).all()
    o = _parity.run_oracle(w, want_probs=False)
    ok = ~timed_out & ((o["flags"] & 7) == 0)
    assert (tok[ok] == o["token"][ok]).all()
    # the context is still usable: an ordinary call samples every row
    g = _parity.run_gpu(w, want_probs=False)
    assert (g["status"].numpy() == 0).all()
    print("rows reported TIMEOUT:", int(timed_out.sum()), "of", w.B)
