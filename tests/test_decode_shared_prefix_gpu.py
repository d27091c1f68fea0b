"""Shared-prefix decode on the GPU, through the C ABI: the prefix blocks
every sequence's table starts with are read once per step, and the result
must match the float64 oracle (plain decode over each sequence's own
table) and the plain GPU decode within the dtype's tolerance."""
import numpy as np
import pytest
import torch

import paged_kv_cache_write_gb300 as pkv
from gpu_step import GpuStep, OracleStep, assert_close, f64
from workloads import draw_plan, make_layer, make_tiny_layer, tiny_plan

pytestmark = pytest.mark.gpu

PKV_DEVERR_PREFIX = 32
PKV_DEVERR_BLOCK_ID = 1


def _prefix_decode(g, P, max_ctas=0):
    t = g.t
    nd = g.nd
    return pkv.paged_attention_decode_shared_prefix(
        t["q"][:nd], t["k_pool"], t["v_pool"], g.bt[:nd], g.seq_lens[:nd], g.sh.scale, P,
        g.max_dec, max_ctas=max_ctas, err=g.err)


WORKLOADS = [("smollm2-135m", 0), ("smollm2-135m", 29), ("llama-3.2-1b-sharedprompt", 0),
             ("llama-3.2-1b-sharedprompt", 15)]


@pytest.mark.parametrize("name,layer_id", WORKLOADS, ids=[f"{n}-L{l}" for n, l in WORKLOADS])
def test_shared_prefix_workloads(name, layer_id):
    """SmolLM2 step: 30 sequences share a 2-block (32-token) system prompt;
    Llama-3.2-1B: 64 sequences behind a 64-block (1,024-token) prompt."""
    plan = draw_plan(name)
    P = len(plan.shared_prefix_blocks)
    assert P > 0 and np.all(plan.block_tables[:, :P] == np.array(plan.shared_prefix_blocks))
    layer = make_layer(plan, layer_id, fill=1e30)
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.run_write()
    g.write(g.slots())
    plain = g.decode()
    shared = _prefix_decode(g, P)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    ref = o.decode()
    assert_close(f64(shared), ref, "bf16", f"{name} layer {layer_id}")
    assert_close(f64(shared), f64(plain), "bf16", "vs plain decode")


def _plan_with_prefix(lens, P, H, K, D, dt, seed, num_blocks=160):
    shared = tuple(range(1, 1 + P))
    plan = tiny_plan(lens, [1] * len(lens), n_heads=H, n_kv=K, head_dim=D, block_size=16,
                     num_blocks=num_blocks, dtype=dt, seed=seed, shared=shared)
    bt = plan.block_tables.copy()
    if bt.shape[1] < P:
        bt = np.concatenate([bt, np.zeros((bt.shape[0], P - bt.shape[1]), bt.dtype)], axis=1)
    bt[:, :P] = shared  # every row starts with the shared blocks, short ones too
    plan.block_tables = bt
    return plan


SMALL = [  # (n_heads, n_kv, head_dim, dtype)
    (9, 3, 64, "bf16"), (32, 8, 64, "bf16"), (64, 8, 128, "bf16"), (16, 1, 64, "bf16"),
    (8, 4, 16, "f32"), (12, 4, 128, "f32"), (4, 2, 32, "bf16"),
]


@pytest.mark.parametrize("shape", SMALL, ids=[f"{h}x{k}x{d}-{t}" for h, k, d, t in SMALL])
@pytest.mark.parametrize("P", [1, 2, 5])
def test_shared_prefix_small_ragged(shape, P):
    """Lengths inside, at the end of and past the prefix, empty sequences,
    several grid sizes."""
    H, K, D, dt = shape
    lens = [0, 1, 5, 16, 17, 31, 32, 33, 48, 79, 80, 81, 100, 300, 700]
    plan = _plan_with_prefix(lens, P, H, K, D, dt, seed=H + D + P)
    layer = make_tiny_layer(plan, seed=D + P, fill=float("nan"))
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    # the pools are read as generated (no write step: a length-0 row has no slot)
    o.kp, o.vp = o.raw["k_pool"], o.raw["v_pool"]
    ref = o.decode()
    for max_ctas in (0, 1, 3, 16):
        out = _prefix_decode(g, P, max_ctas)
        torch.cuda.synchronize()
        assert int(g.err.item()) == 0, max_ctas
        assert_close(f64(out), ref, dt, f"P={P} max_ctas={max_ctas}")
        assert torch.count_nonzero(out[0].float()) == 0  # length 0


def test_shared_prefix_zero_blocks_is_plain_decode():
    plan = _plan_with_prefix([3, 40, 200], 2, 32, 8, 64, "bf16", seed=1)
    layer = make_tiny_layer(plan, seed=1)
    g = GpuStep(plan, layer)
    plain = g.decode()
    zero = _prefix_decode(g, 0)
    torch.cuda.synchronize()
    assert torch.equal(plain.view(torch.int16), zero.view(torch.int16))


def test_shared_prefix_mismatch_reported():
    """A row whose visible leading entries are not row 0's is reported."""
    plan = _plan_with_prefix([40, 40, 40], 2, 8, 2, 64, "bf16", seed=2)
    plan.block_tables[1, 1] = plan.block_tables[1, 2]  # row 1's second prefix entry differs
    layer = make_tiny_layer(plan, seed=2)
    g = GpuStep(plan, layer)
    _prefix_decode(g, 2)
    torch.cuda.synchronize()
    assert int(g.err.item()) & PKV_DEVERR_PREFIX


def test_shared_prefix_large_batch():
    """3,000 sequences behind a 3-block prompt (the main kernel's work split
    then comes from a plan launch), lengths inside, at and past the prefix:
    sampled rows against the oracle."""
    rng = np.random.default_rng(3)
    B, P = 3000, 3
    lens = rng.integers(0, 100, size=B).tolist()
    plan = _plan_with_prefix(lens, P, 32, 8, 64, "bf16", seed=4,
                             num_blocks=sum((l + 15) // 16 for l in lens) + 8)
    layer = make_tiny_layer(plan, seed=4)
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.kp, o.vp = o.raw["k_pool"], o.raw["v_pool"]
    rows = sorted(set(rng.choice(B, 40, replace=False).tolist()) | {0, B - 1})
    ref = o.decode(rows=rows)
    out = _prefix_decode(g, P)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert_close(f64(out)[rows], ref[rows], "bf16", "B=3000")


APPEND_SHAPES = [(9, 3, 64, "bf16"), (32, 8, 64, "bf16"), (64, 8, 128, "bf16"), (16, 1, 64, "bf16")]


@pytest.mark.parametrize("shape", APPEND_SHAPES, ids=[f"{h}x{k}x{d}" for h, k, d, _ in APPEND_SHAPES])
@pytest.mark.parametrize("P", [1, 3])
def test_shared_prefix_planned_append_edges(shape, P):
    """Planned shared-prefix decode with the step's K/V fused in, lengths
    inside, at and past the prefix, on whichever kernel the shape selects: a
    token that would land in a shared block is
    reported (PKV_DEVERR_PREFIX) and not written; otherwise outputs and
    pools equal pkv_kv_write of the other sequences' rows followed by the
    planned call without k_new, bit for bit, and match the oracle."""
    import oracle
    from gpu_step import guarded_copy, guarded_empty
    H, K, D, dt = shape
    lens = [0, 5, 16 * P, 16 * P + 1, 40 + 16 * P, 100, 260, 33, 16 * P - 3, 500]
    plan = _plan_with_prefix(lens, P, H, K, D, dt, seed=7 * P + D)
    layer = make_tiny_layer(plan, seed=P + H)
    g = GpuStep(plan, layer)
    nd, t, sh = g.nd, g.t, g.sh
    past = [b for b in range(nd) if lens[b] > 16 * P]
    slots = np.full(nd, -1, dtype=np.int64)
    for b in past:
        slots[b] = oracle.slot_of(plan.block_tables[b], lens[b] - 1, 16)
    k_new, v_new = t["k"][:nd].contiguous(), t["v"][:nd].contiguous()
    kp1, vp1 = guarded_copy(t["k_pool"]), guarded_copy(t["v_pool"])
    kp2, vp2 = guarded_copy(t["k_pool"]), guarded_copy(t["v_pool"])
    ws = guarded_empty((pkv.decode_shared_prefix_workspace_bytes(nd, H, D, g.max_dec, P),),
                       torch.uint8)
    ws.zero_()
    err1 = guarded_empty((1,), torch.int32)
    err1.zero_()
    err2 = guarded_empty((1,), torch.int32)
    err2.zero_()
    pkv.decode_plan(t["k_pool"], g.seq_lens[:nd], H, g.bt.shape[1], g.max_dec, workspace=ws,
                    shared_prefix_blocks=P, err=err1)
    pkv.kv_write(k_new, v_new, torch.from_numpy(slots).cuda(), kp1, vp1, err=err1)
    ref = pkv.paged_attention_decode_planned(t["q"][:nd], kp1, vp1, g.bt[:nd], g.seq_lens[:nd],
                                             sh.scale, g.max_dec, workspace=ws,
                                             shared_prefix_blocks=P, err=err1)
    out = pkv.paged_attention_decode_planned(t["q"][:nd], kp2, vp2, g.bt[:nd], g.seq_lens[:nd],
                                             sh.scale, g.max_dec, workspace=ws, k_new=k_new,
                                             v_new=v_new, shared_prefix_blocks=P, err=err2)
    torch.cuda.synchronize()
    assert int(err1.item()) == 0
    assert int(err2.item()) == PKV_DEVERR_PREFIX  # lengths 5, 16P, 16P - 3 (0 has no token)
    # a reported row's output is unspecified; every other row is compared
    rows = torch.tensor(past, device="cuda")
    assert torch.equal(out[rows].view(torch.int16), ref[rows].view(torch.int16))
    assert torch.equal(kp2.view(torch.int16), kp1.view(torch.int16))
    assert torch.equal(vp2.view(torch.int16), vp1.view(torch.int16))
    o = OracleStep(plan, layer)
    o.kp, o.vp = oracle.kv_write(o.raw["k"][:nd], o.raw["v"][:nd], slots, o.raw["k_pool"],
                                 o.raw["v_pool"])
    assert_close(f64(out)[past], o.decode(rows=past)[past], dt, f"P={P}")


# Long prompts shared by many sequences take the wide prefix pass (one read
# of the prompt per KV head for up to 16 tiles of rows); these shapes are
# past its threshold.  (n_heads, n_kv, head_dim, batch, prefix blocks)
WIDE = [(32, 8, 64, 256, 32), (64, 8, 128, 100, 40), (9, 3, 64, 200, 64), (16, 16, 64, 300, 24)]


def _wide_lens(rng, B, P):
    pre = 16 * P
    lens = rng.integers(pre + 1, pre + 300, size=B)
    # inside, at the end of and just past the prompt; empty
    lens[:8] = [0, 1, pre - 17, pre - 1, pre, pre + 1, pre + 15, pre + 16]
    return rng.permutation(lens).tolist()


@pytest.mark.parametrize("shape", WIDE, ids=[f"{h}x{k}x{d}-B{b}-P{p}" for h, k, d, b, p in WIDE])
def test_shared_prefix_wide_pass(shape):
    """Every row against the oracle and the plain decode."""
    H, K, D, B, P = shape
    rng = np.random.default_rng(H + B)
    lens = _wide_lens(rng, B, P)
    nb = P + sum(max(0, (l + 15) // 16 - P) for l in lens) + 8
    plan = _plan_with_prefix(lens, P, H, K, D, "bf16", seed=B, num_blocks=nb)
    layer = make_tiny_layer(plan, seed=P, fill=float("nan"))
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.kp, o.vp = o.raw["k_pool"], o.raw["v_pool"]
    shared = _prefix_decode(g, P)
    plain = g.decode()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert_close(f64(shared), o.decode(), "bf16", f"wide {shape}")
    assert_close(f64(shared), f64(plain), "bf16", "vs plain decode")


def test_shared_prefix_wide_pass_reports_foreign_tables():
    """A row whose table leaves the prompt where its length reaches is
    reported; rows that stop before the differing entry are not."""
    H, K, D, B, P = 32, 8, 64, 256, 32
    rng = np.random.default_rng(5)
    lens = rng.integers(16 * P + 1, 16 * P + 200, size=B).tolist()
    lens[7] = 16 * 10  # stops before block 10
    nb = P + sum(max(0, (l + 15) // 16 - P) for l in lens) + 8
    plan = _plan_with_prefix(lens, P, H, K, D, "bf16", seed=6, num_blocks=nb)
    layer = make_tiny_layer(plan, seed=6)
    plan.block_tables[7, 10] = plan.block_tables[7, 11]  # beyond its length: not reported
    g = GpuStep(plan, layer)
    _prefix_decode(g, P)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    plan.block_tables[200, 20] = plan.block_tables[200, P]  # inside its length
    g = GpuStep(plan, layer)
    _prefix_decode(g, P)
    torch.cuda.synchronize()
    assert int(g.err.item()) & PKV_DEVERR_PREFIX


@pytest.mark.parametrize("shape", WIDE[:2], ids=[f"{h}x{k}x{d}" for h, k, d, _, _ in WIDE[:2]])
def test_shared_prefix_wide_pass_planned_append(shape):
    """Planned, with the step's K/V fused in: bit-identical to pkv_kv_write
    of the rows past the prompt followed by the planned call without k_new;
    rows ending inside the prompt reported and not written."""
    import oracle
    from gpu_step import guarded_copy, guarded_empty
    H, K, D, B, P = shape
    rng = np.random.default_rng(D + B)
    lens = _wide_lens(rng, B, P)
    nb = P + sum(max(0, (l + 15) // 16 - P) for l in lens) + 8
    plan = _plan_with_prefix(lens, P, H, K, D, "bf16", seed=D, num_blocks=nb)
    layer = make_tiny_layer(plan, seed=D)
    g = GpuStep(plan, layer)
    nd, t, sh = g.nd, g.t, g.sh
    past = [b for b in range(nd) if lens[b] > 16 * P]
    slots = np.full(nd, -1, dtype=np.int64)
    for b in past:
        slots[b] = oracle.slot_of(plan.block_tables[b], lens[b] - 1, 16)
    k_new, v_new = t["k"][:nd].contiguous(), t["v"][:nd].contiguous()
    kp1, vp1 = guarded_copy(t["k_pool"]), guarded_copy(t["v_pool"])
    kp2, vp2 = guarded_copy(t["k_pool"]), guarded_copy(t["v_pool"])
    ws = guarded_empty((pkv.decode_shared_prefix_workspace_bytes(nd, H, D, g.max_dec, P),),
                       torch.uint8)
    ws.zero_()
    errs = [guarded_empty((1,), torch.int32) for _ in range(2)]
    for e in errs:
        e.zero_()
    pkv.decode_plan(t["k_pool"], g.seq_lens[:nd], H, g.bt.shape[1], g.max_dec, workspace=ws,
                    shared_prefix_blocks=P, err=errs[0])
    pkv.kv_write(k_new, v_new, torch.from_numpy(slots).cuda(), kp1, vp1, err=errs[0])
    ref = pkv.paged_attention_decode_planned(t["q"][:nd], kp1, vp1, g.bt[:nd], g.seq_lens[:nd],
                                             sh.scale, g.max_dec, workspace=ws,
                                             shared_prefix_blocks=P, err=errs[0])
    out = pkv.paged_attention_decode_planned(t["q"][:nd], kp2, vp2, g.bt[:nd], g.seq_lens[:nd],
                                             sh.scale, g.max_dec, workspace=ws, k_new=k_new,
                                             v_new=v_new, shared_prefix_blocks=P, err=errs[1])
    torch.cuda.synchronize()
    assert int(errs[0].item()) == 0
    assert int(errs[1].item()) == PKV_DEVERR_PREFIX
    rows = torch.tensor(past, device="cuda")
    assert torch.equal(out[rows].view(torch.int16), ref[rows].view(torch.int16))
    assert torch.equal(kp2.view(torch.int16), kp1.view(torch.int16))
    assert torch.equal(vp2.view(torch.int16), vp1.view(torch.int16))
    o = OracleStep(plan, layer)
    o.kp, o.vp = oracle.kv_write(o.raw["k"][:nd], o.raw["v"][:nd], slots, o.raw["k_pool"],
                                 o.raw["v_pool"])
    assert_close(f64(out)[past], o.decode(rows=past)[past], "bf16", f"wide append {shape}")


def test_shared_prefix_wide_pass_short_rows_nan_slots():
    """No sequence reaches the end of the prompt: its last slots hold NaN,
    which no output may see."""
    H, K, D, B, P = 32, 8, 64, 256, 32
    rng = np.random.default_rng(9)
    lens = rng.integers(0, 16 * P - 5, size=B).tolist()
    plan = _plan_with_prefix(lens, P, H, K, D, "bf16", seed=9, num_blocks=P + 8)
    layer = make_tiny_layer(plan, seed=9, fill=float("nan"))
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.kp, o.vp = o.raw["k_pool"], o.raw["v_pool"]
    out = _prefix_decode(g, P)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert_close(f64(out), o.decode(), "bf16", "short rows")


# Shapes that take the fused launch (prompt runs beside each sequence's own
# blocks, then the prefix merge): (n_heads, n_kv, head_dim, batch, prefix blocks)
FUSED = [(32, 8, 64, 64, 64), (16, 8, 64, 120, 48)]


@pytest.mark.parametrize("shape", FUSED, ids=[f"{h}x{k}x{d}-B{b}-P{p}" for h, k, d, b, p in FUSED])
def test_shared_prefix_fused_launch(shape):
    """Lengths inside, at and past the prompt, NaN in unused slots: every
    row against the oracle; the planned call with the step's K/V fused in
    against pkv_kv_write + the planned call, bit for bit."""
    import oracle
    from gpu_step import guarded_copy, guarded_empty
    H, K, D, B, P = shape
    rng = np.random.default_rng(B + P)
    lens = _wide_lens(rng, B, P)
    nb = P + sum(max(0, (l + 15) // 16 - P) for l in lens) + 8
    plan = _plan_with_prefix(lens, P, H, K, D, "bf16", seed=P, num_blocks=nb)
    layer = make_tiny_layer(plan, seed=B, fill=float("nan"))
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.kp, o.vp = o.raw["k_pool"], o.raw["v_pool"]
    out = _prefix_decode(g, P)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert_close(f64(out), o.decode(), "bf16", f"fused {shape}")

    nd, t, sh = g.nd, g.t, g.sh
    past = [b for b in range(nd) if lens[b] > 16 * P]
    slots = np.full(nd, -1, dtype=np.int64)
    for b in past:
        slots[b] = oracle.slot_of(plan.block_tables[b], lens[b] - 1, 16)
    k_new, v_new = t["k"][:nd].contiguous(), t["v"][:nd].contiguous()
    kp1, vp1 = guarded_copy(t["k_pool"]), guarded_copy(t["v_pool"])
    kp2, vp2 = guarded_copy(t["k_pool"]), guarded_copy(t["v_pool"])
    ws = guarded_empty((pkv.decode_shared_prefix_workspace_bytes(nd, H, D, g.max_dec, P),),
                       torch.uint8)
    ws.zero_()
    errs = [guarded_empty((1,), torch.int32) for _ in range(2)]
    for e in errs:
        e.zero_()
    pkv.decode_plan(t["k_pool"], g.seq_lens[:nd], H, g.bt.shape[1], g.max_dec, workspace=ws,
                    shared_prefix_blocks=P, err=errs[0])
    pkv.kv_write(k_new, v_new, torch.from_numpy(slots).cuda(), kp1, vp1, err=errs[0])
    ref = pkv.paged_attention_decode_planned(t["q"][:nd], kp1, vp1, g.bt[:nd], g.seq_lens[:nd],
                                             sh.scale, g.max_dec, workspace=ws,
                                             shared_prefix_blocks=P, err=errs[0])
    app = pkv.paged_attention_decode_planned(t["q"][:nd], kp2, vp2, g.bt[:nd], g.seq_lens[:nd],
                                             sh.scale, g.max_dec, workspace=ws, k_new=k_new,
                                             v_new=v_new, shared_prefix_blocks=P, err=errs[1])
    torch.cuda.synchronize()
    assert int(errs[0].item()) == 0
    assert int(errs[1].item()) == PKV_DEVERR_PREFIX
    rows = torch.tensor(past, device="cuda")
    assert torch.equal(app[rows].view(torch.int16), ref[rows].view(torch.int16))
    assert torch.equal(kp2.view(torch.int16), kp1.view(torch.int16))
    assert torch.equal(vp2.view(torch.int16), vp1.view(torch.int16))
    # the planned call without k_new on unchanged pools is the unplanned one
    # up to the order of its sums: against the oracle on the written pools
    o.kp, o.vp = oracle.kv_write(o.raw["k"][:nd], o.raw["v"][:nd], slots, o.raw["k_pool"],
                                 o.raw["v_pool"])
    assert_close(f64(app)[past], o.decode(rows=past)[past], "bf16", f"fused append {shape}")


def test_shared_prefix_fused_launch_short_rows():
    """The fused shape with every sequence ending inside the prompt (and
    NaN in the prompt's unreached slots): outputs from the prompt runs
    alone."""
    H, K, D, B, P = FUSED[0]
    rng = np.random.default_rng(11)
    lens = rng.integers(0, 16 * P - 40, size=B).tolist()
    plan = _plan_with_prefix(lens, P, H, K, D, "bf16", seed=11, num_blocks=P + 8)
    layer = make_tiny_layer(plan, seed=11, fill=float("nan"))
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.kp, o.vp = o.raw["k_pool"], o.raw["v_pool"]
    out = _prefix_decode(g, P)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert_close(f64(out), o.decode(), "bf16", "fused short rows")


@pytest.mark.parametrize("shape", [FUSED[0], WIDE[0]], ids=["fused", "wide"])
def test_shared_prefix_bad_prompt_block_reported(shape):
    """A prompt block id past the pool (the same in every table, so the
    prefix stays common) is reported as PKV_DEVERR_BLOCK_ID and read as
    zeros: no fault, no stray write (canary bands), finite outputs."""
    H, K, D, B, P = shape
    rng = np.random.default_rng(17)
    lens = _wide_lens(rng, B, P)
    nb = P + sum(max(0, (l + 15) // 16 - P) for l in lens) + 8
    plan = _plan_with_prefix(lens, P, H, K, D, "bf16", seed=17, num_blocks=nb)
    plan.block_tables[:, P // 2] = nb + 3  # every row: past the pool's end
    layer = make_tiny_layer(plan, seed=17)
    g = GpuStep(plan, layer)
    out = _prefix_decode(g, P)
    torch.cuda.synchronize()
    assert int(g.err.item()) & PKV_DEVERR_BLOCK_ID
    assert torch.isfinite(out.float()).all()
