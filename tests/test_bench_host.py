"""Host logic of bench.py that runs without a GPU: the CPU baseline leg's sample and its parity
accounting (fed the oracle's own answer, then one with a planted wrong token)."""
import numpy as np
import torch

import bench
import oracle


def test_cpu_baseline_passes_and_parity_accounting():
    args = bench.parse(["--B", "10", "--V", "3000"])
    w = bench.make_workload(args, "cpu")
    o = oracle.sample(w.logits.double().numpy(), w.temperature.numpy(), w.top_k.numpy(), w.top_p.numpy(),
                      w.min_p.numpy(), w.seed.numpy().astype(np.uint64), w.step)
    gpu = {k: torch.as_tensor(np.asarray(o[k])) for k in ("token", "kept", "cutoff", "status")}
    gpu["cutoff"] = gpu["cutoff"].float()
    res = bench.cpu_baseline(w, gpu, seconds=0.0, max_passes=3, chunk=4)
    assert res["parity"]["rows_checked"] == 10
    assert res["parity"]["mismatches_outside_band"] == 0
    assert res["kind"] == "oracle" and res["value"] > 0
    assert "pass" in res["sample"]
    # seconds = 0: the first pass always completes (parity needs every row), and no second starts
    assert res["sample"].startswith("10 rows: 1 pass")
    exact = np.nonzero((o["status"] == 0) & ((o["flags"] & 7) == 0))[0]
    gpu["token"][int(exact[0])] += 1
    res = bench.cpu_baseline(w, gpu, seconds=0.0, max_passes=1, chunk=4)
    assert res["parity"]["mismatches_outside_band"] == 1
