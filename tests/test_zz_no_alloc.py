"""The decode entry point that allocates nothing (for callers that may not
call cudaMalloc, e.g. code inside a framework that owns all device memory)
gives the same output as the workspace entry point.

Collected last on purpose (file name), so a run that stops at the first
failure has already run every other test.  It must pass both in a fresh
process, where its first call looks up the built-in scratch address, and
after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_step import GpuStep, OracleStep, assert_close, f64, guarded_empty
from workloads import draw_plan, make_layer, tiny_plan, make_tiny_layer

pytestmark = pytest.mark.gpu


def _noalloc(g, max_ctas=0, out=None):
    """Call pkv_paged_attention_decode_noalloc through the C ABI."""
    import paged_kv_cache_write_gb300 as pkv
    fn = pkv.lib.pkv_paged_attention_decode_noalloc
    fn.restype = ctypes.c_int32
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [P, I32, I32, P, P, ctypes.POINTER(pkv.PoolDesc), P, I32, P, I32,
                   ctypes.c_float, I32, P, P, P]
    t = g.t
    nd = g.nd
    q = t["q"][:nd]
    if out is None:
        out = guarded_empty(q.shape, q.dtype)  # canary bands around the output
        out.fill_(float("nan"))
    desc = pkv.pool_desc(t["k_pool"])
    st = fn(q.data_ptr(), nd, q.shape[1], t["k_pool"].data_ptr(), t["v_pool"].data_ptr(),
            ctypes.byref(desc), g.bt.data_ptr(), g.bt.shape[1], g.seq_lens.data_ptr(), g.max_dec,
            g.sh.scale, max_ctas, out.data_ptr(), g.err.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    return st, out


def _bits(t):
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16)


@pytest.mark.parametrize("name", ["toy", "llama-3.2-1b", "llama2-70b-mixed"])
def test_noalloc_decode_matches_workspace_decode(name):
    """Two calls in a row: each output equals the workspace entry point's
    bit for bit (same kernels, same grid, same split) and the float64
    oracle within the dtype's tolerance."""
    from gpu_step import check_canaries
    plan = draw_plan(name)
    layer = make_layer(plan, 0)
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.run_write()
    g.write(g.slots())
    ref = o.decode()
    ws_out = g.decode()
    torch.cuda.synchronize()
    for call in range(2):  # two calls in a row share the built-in scratch
        st, out = _noalloc(g)
        torch.cuda.synchronize()
        check_canaries()
        assert st == 0, f"call {call}: status {st}"
        assert torch.equal(_bits(out), _bits(ws_out)), f"{name} call {call}: not bit-identical"
        assert_close(f64(out), ref, plan.shape.dtype, f"{name} call {call} vs oracle")
    assert int(g.err.item()) == 0


def test_noalloc_rejects_batches_beyond_its_scratch():
    """16 query heads per KV head at head_dim 128 need more split scratch
    than the built-in 8 MiB holds on a full grid (about 10 MB at one CTA
    per SM on 152 SMs; the batch has more units than the grid has CTAs, so
    the grid is full): refused, nothing launched; a 64-CTA grid fits and
    matches the workspace entry point."""
    plan = tiny_plan([300, 9, 1000, 2000, 2000], [1] * 5, n_heads=64, n_kv=4, head_dim=128,
                     block_size=16, num_blocks=400, dtype="bf16", seed=5)
    layer = make_tiny_layer(plan, seed=5)
    g = GpuStep(plan, layer)
    g.write(g.slots())
    marker = torch.full_like(g.t["q"][:g.nd], 7.0)
    st, out = _noalloc(g, out=marker)
    torch.cuda.synchronize()
    assert st == 6  # PKV_ERR_WORKSPACE
    assert torch.all(out == 7.0)  # untouched
    ws_out = g.decode(max_ctas=64)
    o = OracleStep(plan, layer)
    o.run_write()
    ref = o.decode()
    for _ in range(2):
        st, out = _noalloc(g, max_ctas=64)
        torch.cuda.synchronize()
        assert st == 0
        assert torch.equal(_bits(out), _bits(ws_out))
        assert_close(f64(out), ref, "bf16", "max_ctas=64 vs oracle")
