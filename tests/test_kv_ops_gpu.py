"""Slot mapping, KV write and block-table gather on the GPU: bit-exact
against the oracle on every workload shape (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_step import GpuStep, OracleStep, raw
from workloads import SHAPES, draw_plan, make_layer, tiny_plan, make_tiny_layer

pytestmark = pytest.mark.gpu


def _bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32) if a.dtype == np.float32 else a


@pytest.mark.parametrize("name", list(SHAPES))
def test_slot_mapping_and_write_bit_exact(name):
    plan = draw_plan(name)
    layer = make_layer(plan, 0, fill=-3.0)
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    slots_o, kp, vp = o.run_write()
    s = g.slots()
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy(), slots_o)
    g.write(s)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(raw(g.t["k_pool"])), _bits(kp))
    assert np.array_equal(_bits(raw(g.t["v_pool"])), _bits(vp))
    assert int(g.err.item()) == 0
    if plan.shared_prefix_blocks:
        # this step's tokens never land in the shared prefix blocks
        blocks = slots_o // plan.shape.block_size
        assert not np.isin(blocks, plan.shared_prefix_blocks).any()


@pytest.mark.parametrize("name", ["toy", "smollm2-135m", "llama-3.2-1b", "llama-7b"])
def test_gather_matches_oracle(name):
    plan = draw_plan(name)
    layer = make_layer(plan, 1)
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    _, kp, vp = o.run_write()
    g.write(g.slots())
    cu = np.concatenate([[0], np.cumsum(plan.seq_lens)]).astype(np.int32)
    k_out, v_out = g.pkv.kv_gather(g.t["k_pool"], g.t["v_pool"], g.bt, g.seq_lens,
                                   torch.from_numpy(cu).cuda(), int(cu[-1]), err=g.err)
    torch.cuda.synchronize()
    ko, vo = raw(k_out), raw(v_out)
    for b in range(plan.num_seqs):
        ref_k = oracle.gather_kv(kp, plan.block_tables[b], plan.seq_lens[b])
        ref_v = oracle.gather_kv(vp, plan.block_tables[b], plan.seq_lens[b])
        assert np.array_equal(_bits(ko[cu[b]:cu[b + 1]]), _bits(ref_k))
        assert np.array_equal(_bits(vo[cu[b]:cu[b + 1]]), _bits(ref_v))
    assert int(g.err.item()) == 0


@pytest.mark.parametrize("bs", [1, 4, 16, 32])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_write_gather_round_trip_block_sizes(bs, dtype):
    """Whole prompts written through their slots read back exactly, for
    block sizes the attention kernels do not take ("Day 16": byte for
    byte what the naive cache would hand it)."""
    lens = [1, bs, 3 * bs + 1, 40]
    plan = tiny_plan(lens, lens, n_heads=4, n_kv=2, head_dim=16, block_size=bs,
                     num_blocks=4 + sum(-(-l // bs) for l in lens), dtype=dtype, seed=bs)
    layer = make_tiny_layer(plan, seed=bs, fill=7.0)
    g = GpuStep(plan, layer)
    g.write(g.slots())
    cu = plan.cu_new_lens
    k_out, _ = g.pkv.kv_gather(g.t["k_pool"], g.t["v_pool"], g.bt, g.seq_lens,
                               torch.from_numpy(cu).cuda(), int(cu[-1]), err=g.err)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(raw(k_out)), _bits(raw(layer["k"])))
    assert int(g.err.item()) == 0


def test_negative_slots_skip_tokens():
    plan = tiny_plan([20], [20], n_heads=2, n_kv=2, head_dim=16, block_size=16, num_blocks=4)
    layer = make_tiny_layer(plan, fill=5.0)
    g = GpuStep(plan, layer)
    s = g.slots()
    s[::2] = -1
    before = g.t["k_pool"].clone()
    g.write(s)
    torch.cuda.synchronize()
    sc = s.cpu().numpy()
    kp = g.t["k_pool"].reshape(-1, 2, 16).cpu()
    for t, slot in enumerate(sc):
        if slot >= 0:
            assert torch.equal(kp[slot], layer["k"][t])
    untouched = np.setdiff1d(np.arange(kp.shape[0]), sc[sc >= 0])
    assert torch.equal(kp[untouched], before.reshape(-1, 2, 16).cpu()[untouched])


def test_out_of_range_ids_are_reported_not_used():
    """A bad block id / slot is caught by the kernels' own bounds checks:
    the access is skipped and an error bit is set."""
    import paged_kv_cache_write_gb300 as pkv
    plan = tiny_plan([5, 9], [1, 1], n_heads=2, n_kv=2, head_dim=16, block_size=16, num_blocks=4)
    layer = make_tiny_layer(plan)
    g = GpuStep(plan, layer)
    g.bt[1, 0] = 1000  # outside the 4-block pool
    s = g.slots()
    torch.cuda.synchronize()
    assert s[1].item() == -1 and (g.err.item() & pkv.DEVERR["block_id"])
    g.err.zero_()
    bad = s.clone()
    bad[1] = 4 * 16  # one past the last slot
    g.write(bad)
    torch.cuda.synchronize()
    assert g.err.item() & pkv.DEVERR["slot"]
