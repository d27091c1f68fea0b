"""The kernels' failure path, exercised without a fault: a bounded wait on
an mbarrier phase that nothing completes runs out, the kernel reports
PKV_DEVERR_TIMEOUT and returns, and the context keeps working (a decode
launched afterwards matches the oracle)."""
import time

import pytest
import torch

import paged_kv_cache_write_gb300 as pkv
from gpu_step import GpuStep, OracleStep, assert_close, f64
from workloads import make_tiny_layer, tiny_plan

pytestmark = pytest.mark.gpu

PKV_DEVERR_TIMEOUT = 16


def test_bounded_wait_runs_out_and_returns():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    pkv.selftest_bounded_wait(err, polls=4096)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 30.0
    assert int(err.item()) == PKV_DEVERR_TIMEOUT
    # the context is intact: a decode afterwards is correct and reports nothing
    plan = tiny_plan([5, 40, 300], [1, 1, 1], n_heads=16, n_kv=4, head_dim=64, block_size=16,
                     num_blocks=64, dtype="bf16", seed=3)
    layer = make_tiny_layer(plan, seed=3)
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.run_write()
    _, dec, _ = g.run()
    assert int(g.err.item()) == 0
    assert_close(f64(dec), o.decode(), "bf16", "after the timeout")
