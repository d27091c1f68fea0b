"""Paged decode attention on the GPU against the float64 oracle, through
the C ABI: every workload shape, small ragged cases, split variants, and
the pages' invariants (placement, prefix sharing, garbage in masked slots)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_step import GpuStep, OracleStep, assert_close, f64, raw
from workloads import draw_plan, make_layer, tiny_plan, make_tiny_layer

pytestmark = pytest.mark.gpu

# (shape, layers checked).  All layers of the toy, SmolLM2 and Llama-3.2-1B
# steps; first and last layer of LLaMA-7B; the one 70B layer.  Every decode
# row of each checked layer is compared (all 256 of the 70B step).
CASES = [("toy", [0]), ("smollm2-135m", list(range(30))), ("llama-3.2-1b", list(range(16))),
         ("llama-7b", [0, 31]), ("llama2-70b-mixed", [0]), ("llama2-70b-decode64", [0])]


def _sample_rows(plan, n=24):
    nd = plan.n_decode
    if nd <= n:
        return list(range(nd))
    lens = plan.seq_lens[:nd]
    rng = np.random.default_rng(7)
    pick = set(rng.choice(nd, n - 2, replace=False).tolist())
    pick.add(int(np.argmax(lens)))
    pick.add(int(np.argmin(lens)))
    return sorted(pick)


@pytest.mark.parametrize("name,layers", CASES, ids=[c[0] for c in CASES])
def test_decode_matches_oracle(name, layers):
    plan = draw_plan(name)
    for layer_id in layers:
        layer = make_layer(plan, layer_id, fill=1e30)
        g, o = GpuStep(plan, layer), OracleStep(plan, layer)
        o.run_write()
        _, dec, _ = g.run()
        ref = o.decode()
        assert_close(f64(dec), ref, plan.shape.dtype, f"{name} layer {layer_id}")
        assert int(g.err.item()) == 0


SMALL = [  # (n_heads, n_kv, head_dim, dtype)
    (8, 4, 16, "f32"), (4, 4, 32, "f32"), (16, 2, 64, "f32"), (12, 4, 128, "f32"),
    (9, 3, 64, "bf16"), (32, 8, 64, "bf16"), (64, 8, 128, "bf16"), (8, 8, 128, "bf16"),
    (16, 1, 64, "bf16"), (6, 3, 16, "bf16"), (4, 2, 32, "bf16"),
]


@pytest.mark.parametrize("shape", SMALL, ids=[f"{h}x{k}x{d}-{t}" for h, k, d, t in SMALL])
def test_decode_small_ragged(shape):
    H, K, D, dt = shape
    lens = [1, 2, 15, 16, 17, 31, 33, 64, 100, 257, 700]
    plan = tiny_plan(lens, [1] * len(lens), n_heads=H, n_kv=K, head_dim=D, block_size=16,
                     num_blocks=120, dtype=dt, seed=H * 100 + D)
    layer = make_tiny_layer(plan, seed=D, fill=float("nan"))
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.run_write()
    ref = o.decode()
    for max_ctas in (0, 1, 3, 16):
        _, dec, _ = g.run(max_ctas=max_ctas)
        assert_close(f64(dec), ref, dt, f"max_ctas={max_ctas}")
    assert int(g.err.item()) == 0


def test_decode_empty_and_single_token():
    plan = tiny_plan([0, 1, 1, 5], [0, 1, 1, 1], n_heads=8, n_kv=2, head_dim=64,
                     block_size=16, num_blocks=8, dtype="bf16")
    plan.n_decode = 4
    layer = make_tiny_layer(plan, seed=3)
    g = GpuStep(plan, layer)
    g.write(g.slots())
    dec = g.decode()
    torch.cuda.synchronize()
    out = dec.float().cpu()
    assert torch.count_nonzero(out[0]) == 0  # no keys: zero output
    # one key: the output is that key's value (softmax weight exactly 1)
    kp = g.t["v_pool"].cpu()
    for b in (1, 2):
        blk = int(plan.block_tables[b, 0])
        v0 = kp[blk, 0].float()  # [n_kv, hd]
        for h in range(8):
            assert torch.equal(out[b, h], v0[h // 4])


def _relabel(plan, layer, seed):
    """Move every block to a new physical id (data moved along)."""
    nb = plan.shape.num_blocks
    perm = np.random.default_rng(seed).permutation(nb)
    kp = torch.empty_like(layer["k_pool"])
    vp = torch.empty_like(layer["v_pool"])
    kp[torch.from_numpy(perm)] = layer["k_pool"]
    vp[torch.from_numpy(perm)] = layer["v_pool"]
    return perm, kp, vp


@pytest.mark.parametrize("name", ["toy", "smollm2-135m", "llama-3.2-1b"])
@pytest.mark.parametrize("max_ctas", [0, 5])
def test_decode_bit_identical_under_relabelling(name, max_ctas):
    plan = draw_plan(name)
    layer = make_layer(plan, 2)
    g = GpuStep(plan, layer)
    g.write(g.slots())
    base = g.decode(max_ctas).clone()
    perm, kp, vp = _relabel(plan, {"k_pool": g.t["k_pool"], "v_pool": g.t["v_pool"]}, 11)
    bt2 = torch.from_numpy(perm[plan.block_tables].astype(np.int32)).cuda()
    moved = g.decode(max_ctas, k_pool=kp, v_pool=vp, bt=bt2)
    torch.cuda.synchronize()
    assert torch.equal(base, moved)


def test_decode_shared_prefix_equals_private_copies():
    """SmolLM2 step: the 32-token system prompt in blocks 1 and 2 is shared
    by all 30 tables ("nano-vLLM", How it works); giving every sequence
    private copies of those blocks changes nothing, bit for bit."""
    plan = draw_plan("smollm2-135m")
    layer = make_layer(plan, 0)
    g = GpuStep(plan, layer)
    g.write(g.slots())
    shared = g.decode().clone()
    free = np.setdiff1d(np.arange(plan.shape.num_blocks), plan.held_blocks)
    free = free[free != 0]
    bt = plan.block_tables.copy()
    kp, vp = g.t["k_pool"].clone(), g.t["v_pool"].clone()
    cursor = 0
    for b in range(plan.num_seqs):
        for j in (0, 1):
            new = int(free[cursor])
            cursor += 1
            kp[new] = kp[bt[b, j]]
            vp[new] = vp[bt[b, j]]
            bt[b, j] = new
    private = g.decode(k_pool=kp, v_pool=vp, bt=torch.from_numpy(bt).cuda())
    torch.cuda.synchronize()
    assert torch.equal(shared, private)


@pytest.mark.parametrize("junk", [1e30, float("nan"), float("inf")])
def test_decode_garbage_in_unused_slots(junk):
    """Garbage in every slot no sequence uses (unheld blocks, the dummy block
    0 that pads the tables, tails of last blocks) changes nothing ("nano-vLLM",
    Correctness: the garbage pool proves the mask; NaN included here)."""
    plan = draw_plan("smollm2-135m")
    layer = make_layer(plan, 4)
    g = GpuStep(plan, layer)
    g.write(g.slots())
    clean = g.decode().clone()
    used = np.zeros(plan.shape.num_blocks * plan.shape.block_size, dtype=bool)
    used[oracle.slot_mapping(plan.block_tables, plan.seq_lens, plan.seq_lens,
                             plan.shape.block_size)] = True
    mask = torch.from_numpy(~used).cuda()
    kp = g.t["k_pool"].clone().reshape(used.shape[0], -1)
    vp = g.t["v_pool"].clone().reshape(used.shape[0], -1)
    kp[mask] = junk
    vp[mask] = junk
    dirty = g.decode(k_pool=kp.reshape(g.t["k_pool"].shape), v_pool=vp.reshape(g.t["v_pool"].shape))
    torch.cuda.synchronize()
    assert torch.equal(clean, dirty)


def test_decode_reports_bad_lengths_and_ids():
    import paged_kv_cache_write_gb300 as pkv
    plan = tiny_plan([20, 40], [1, 1], n_heads=4, n_kv=2, head_dim=64, block_size=16,
                     num_blocks=8, dtype="bf16")
    layer = make_tiny_layer(plan)
    g = GpuStep(plan, layer)
    g.bt[0, 1] = -5
    out = g.decode()
    torch.cuda.synchronize()
    assert g.err.item() & pkv.DEVERR["block_id"]
    assert torch.isfinite(out.float()).all()
    g.err.zero_()
    g.seq_lens[1] = 999  # more than the table row holds and than max_seq_len
    out = g.decode()
    torch.cuda.synchronize()
    assert g.err.item() & (pkv.DEVERR["length"] | pkv.DEVERR["table_width"])
    assert torch.isfinite(out.float()).all()


REUSE = [("llama2-70b-decode64", "bf16"), ("llama-3.2-1b", "bf16"), ("smollm2-135m", "bf16"),
         ("toy", "f32")]


@pytest.mark.parametrize("name,dt", REUSE, ids=[r[0] for r in REUSE])
def test_workspace_reused_across_calls_and_grids(name, dt):
    """One workspace serves many calls of different grid sizes without
    clearing: every output row is written each call (outputs start as
    NaN) and each call matches the oracle."""
    plan = draw_plan(name)
    layer = make_layer(plan, 0)
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.run_write()
    g.write(g.slots())
    rows = _sample_rows(plan)
    ref = o.decode(rows=rows)
    sh, nd, t = plan.shape, plan.n_decode, g.t
    ws = torch.full((g.pkv.decode_workspace_bytes(nd, sh.n_heads, sh.head_dim, g.max_dec),),
                    255, dtype=torch.uint8, device="cuda")  # garbage before the first call
    for max_ctas in (0, 3, 16, 0, 7):
        for _ in range(2):
            out = torch.full_like(t["q"][:nd], float("nan"))
            g.pkv.paged_attention_decode(t["q"][:nd], t["k_pool"], t["v_pool"], g.bt[:nd],
                                         g.seq_lens[:nd], sh.scale, g.max_dec, out=out,
                                         workspace=ws, max_ctas=max_ctas, err=g.err)
            torch.cuda.synchronize()
            assert int(g.err.item()) == 0
            assert_close(f64(out)[rows], ref[rows], dt, f"{name} max_ctas={max_ctas}")
            assert not torch.isnan(out.float()).any()


@pytest.mark.parametrize("B", [3000, 9000])
@pytest.mark.parametrize("shape", [(8, 2, 64, "bf16"), (8, 2, 16, "f32")], ids=["bf16", "f32"])
def test_decode_large_batches(B, shape):
    """Batches past the kernel's own plan (2,048 sequences: a plan launch
    splits the work) and past the plan's shared-memory prefix (8,191: the
    prefix lives in the workspace), with empty and one-token sequences:
    plain, planned and append calls agree with the oracle on sampled rows."""
    H, K, D, dt = shape
    rng = np.random.default_rng(B)
    lens = rng.integers(0, 60, size=B)
    lens[::97] = 0
    lens[1::89] = 1
    plan = tiny_plan(lens.tolist(), [1] * B, n_heads=H, n_kv=K, head_dim=D, block_size=16,
                     num_blocks=int(sum((l + 15) // 16 for l in lens)) + 8, dtype=dt, seed=B)
    layer = make_tiny_layer(plan, seed=B, fill=float("nan"))
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.kp, o.vp = o.raw["k_pool"], o.raw["v_pool"]
    rows = sorted(set(rng.choice(B, 40, replace=False).tolist()) | {0, 1, B - 1})
    ref = o.decode(rows=rows)
    t, sh, nd = g.t, g.sh, g.nd
    plain = g.decode()
    ws = torch.zeros(g.pkv.decode_workspace_bytes(nd, H, D, g.max_dec), dtype=torch.uint8,
                     device="cuda")
    g.pkv.decode_plan(t["k_pool"], g.seq_lens, H, g.bt.shape[1], g.max_dec, workspace=ws,
                      err=g.err)
    planned = g.pkv.paged_attention_decode_planned(t["q"], t["k_pool"], t["v_pool"], g.bt,
                                                   g.seq_lens, sh.scale, g.max_dec, workspace=ws,
                                                   err=g.err)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert_close(f64(plain)[rows], ref[rows], dt, f"B={B} plain")
    assert torch.equal(plain.view(torch.int16 if dt == "bf16" else torch.int32),
                       planned.view(torch.int16 if dt == "bf16" else torch.int32))
    for b in np.nonzero(lens == 0)[0][:5]:
        assert torch.count_nonzero(plain[int(b)].float()) == 0
    # append: the step's K/V fused in (sequences of length 0 write nothing),
    # against the oracle after the same write
    sel = [b for b in range(B) if lens[b] > 0]
    slots = np.array([oracle.slot_of(plan.block_tables[b], int(lens[b]) - 1, 16) for b in sel])
    o.kp, o.vp = oracle.kv_write(o.raw["k"][sel], o.raw["v"][sel], slots, o.raw["k_pool"],
                                 o.raw["v_pool"])
    ref_a = o.decode(rows=rows)
    kp, vp = t["k_pool"].clone(), t["v_pool"].clone()
    app = g.pkv.paged_attention_decode_append(t["q"], t["k"], t["v"], kp, vp, g.bt, g.seq_lens,
                                              sh.scale, g.max_dec, err=g.err)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert_close(f64(app)[rows], ref_a[rows], dt, f"B={B} append")
