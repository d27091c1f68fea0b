"""Pools past 4 GiB: blocks whose byte offsets need more than 32 bits (a
LLaMA-2-70B-shaped pool of 163,840 blocks, 5.4 GB for K and as much for V)
are written, copied, read back and attended exactly as the same data at low
block ids ("Day 16: the paged KV cache", the table is the only way to a
block: moving blocks and their table entries changes nothing), bit for bit,
and the outputs match the float64 oracle."""
import numpy as np
import pytest
import torch

from gpu_step import GpuStep, OracleStep, assert_close, f64, guarded_empty
from workloads import make_tiny_layer, tiny_plan

pytestmark = pytest.mark.gpu

BIG_BLOCKS = 163_840  # x 16 tokens x 8 KV heads x 128 dims x 2 bytes = 5.37 GB per pool


def _bits(t):
    return t.view(torch.int16)


def test_pool_beyond_4gib():
    import paged_kv_cache_write_gb300 as pkv
    # six decode rows, then two prefill chunks (one over history, one whole prompt)
    lens = [1, 17, 100, 257, 700, 1500, 600, 300]
    new = [1, 1, 1, 1, 1, 1, 64, 300]
    nb = 400
    plan = tiny_plan(lens, new, n_heads=64, n_kv=8, head_dim=128, block_size=16, num_blocks=nb,
                     dtype="bf16", seed=41)
    layer = make_tiny_layer(plan, seed=41)
    small = GpuStep(plan, layer)
    kp0, vp0 = small.t["k_pool"].clone(), small.t["v_pool"].clone()
    _, dec_ref, pre_ref = small.run()

    # the same blocks at the top of a 163,840-block pool: block i -> off + i
    off = BIG_BLOCKS - nb
    assert off * 16 * 8 * 128 * 2 > 2 ** 32
    shape = (BIG_BLOCKS, 16, 8, 128)
    kb = guarded_empty(shape, torch.bfloat16)  # canary bands past the 5.4 GB pools
    vb = guarded_empty(shape, torch.bfloat16)
    kb[off:] = kp0
    vb[off:] = vp0
    bt = (small.bt.long() + off).int()
    nd, t = small.nd, small.t
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = pkv.slot_mapping(bt, small.seq_lens, small.cu_new, plan.num_new_tokens, 16, BIG_BLOCKS,
                             err=err)
    assert slots.min().item() >= off * 16
    pkv.kv_write(t["k"], t["v"], slots, kb, vb, err=err)
    dec = pkv.paged_attention_decode(t["q"][:nd], kb, vb, bt[:nd], small.seq_lens[:nd],
                                     plan.shape.scale, small.max_dec, err=err)
    pre = pkv.paged_attention_prefill(t["q"][nd:], small.cu_q, kb, vb, bt[nd:],
                                      small.seq_lens[nd:], plan.shape.scale, small.max_q,
                                      small.max_pre, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(_bits(kb[off:]), _bits(t["k_pool"]))
    assert torch.equal(_bits(vb[off:]), _bits(t["v_pool"]))
    assert torch.equal(_bits(dec), _bits(dec_ref))
    assert torch.equal(_bits(pre), _bits(pre_ref))

    o = OracleStep(plan, layer)
    o.run_write()
    assert_close(f64(dec), o.decode(), "bf16", "decode, blocks past 4 GiB")
    rows = [(b, i) for b in range(2) for i in (0, int(new[nd + b]) // 2, int(new[nd + b]) - 1)]
    cu = np.concatenate([[0], np.cumsum(new[nd:])])
    got = np.stack([f64(pre[cu[b] + i]) for b, i in rows])
    ref = np.stack([o.prefill_row(b, i) for b, i in rows])
    assert_close(got, ref, "bf16", "prefill, blocks past 4 GiB")

    # copy-on-write copies of a sequence's blocks into free blocks, all near the top
    free = sorted(set(range(1, nb)) - set(int(x) for x in plan.held_blocks))[:4]
    pairs = torch.tensor([[off + int(plan.block_tables[5, j]), off + f] for j, f in enumerate(free)],
                         dtype=torch.int32, device="cuda")
    pkv.copy_blocks(kb, vb, pairs, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for src, dst in pairs.tolist():
        assert torch.equal(_bits(kb[dst]), _bits(kb[src]))
        assert torch.equal(_bits(vb[dst]), _bits(vb[src]))
