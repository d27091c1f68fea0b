"""Decode with the step's work split planned once (pkv_decode_plan) and
reused by every layer (pkv_paged_attention_decode_planned), through the C
ABI: bit-identical to the unplanned calls, plain and with append, and
equal to the float64 oracle; empty sequences and bad lengths handled as in
the unplanned call."""
import pytest
import torch

import paged_kv_cache_write_gb300 as pkv
from gpu_step import GpuStep, OracleStep, assert_close, f64
from workloads import draw_plan, make_layer, make_tiny_layer, tiny_plan

pytestmark = pytest.mark.gpu

PKV_DEVERR_LENGTH = 8


def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).reshape(-1)


def _workspace(g, max_ctas=0):
    sh, nd = g.sh, g.nd
    return torch.zeros(pkv.decode_workspace_bytes(nd, sh.n_heads, sh.head_dim, g.max_dec, max_ctas),
                       dtype=torch.uint8, device="cuda")


def _plan(g, ws, max_ctas=0):
    pkv.decode_plan(g.t["k_pool"], g.seq_lens[:g.nd], g.sh.n_heads, g.bt.shape[1], g.max_dec,
                    workspace=ws, max_ctas=max_ctas, err=g.err)


WORKLOADS = ["toy", "smollm2-135m", "llama-3.2-1b", "llama2-70b-decode64"]


@pytest.mark.parametrize("name", WORKLOADS)
@pytest.mark.parametrize("max_ctas", [0, 7])
def test_planned_layers_bit_identical_to_unplanned(name, max_ctas):
    """One plan, three layers' planned calls: each equals the call that
    plans for itself, bit for bit; the first layer also matches the oracle."""
    plan = draw_plan(name)
    nl = 3 if plan.shape.name != "llama2-70b-decode64" else 1
    g0 = None
    ws = None
    for layer_id in range(nl):
        layer = make_layer(plan, layer_id)
        g = GpuStep(plan, layer)
        g.write(g.slots())
        if ws is None:
            g0, ws = g, _workspace(g, max_ctas)
            _plan(g0, ws, max_ctas)
        nd, t = g.nd, g.t
        out = torch.full_like(t["q"][:nd], float("nan"))
        pkv.paged_attention_decode_planned(t["q"][:nd], t["k_pool"], t["v_pool"], g0.bt[:nd],
                                           g0.seq_lens[:nd], g.sh.scale, g.max_dec, workspace=ws,
                                           out=out, max_ctas=max_ctas, err=g.err)
        ref = g.decode(max_ctas=max_ctas)
        torch.cuda.synchronize()
        assert int(g.err.item()) == 0 and int(g0.err.item()) == 0
        assert torch.equal(_bits(out), _bits(ref)), f"{name} layer {layer_id}"
        if layer_id == 0:
            o = OracleStep(plan, layer)
            o.run_write()
            rows = list(range(min(nd, 24)))
            assert_close(f64(out)[rows], o.decode(rows=rows)[rows], plan.shape.dtype, name)


@pytest.mark.parametrize("name", ["smollm2-135m", "llama-3.2-1b"])
def test_planned_append_bit_identical_to_append(name):
    """Planned decode with k_new/v_new equals pkv_paged_attention_decode_append
    bit for bit, outputs and pools (each on its own copy of the pools)."""
    plan = draw_plan(name)
    layer = make_layer(plan, 0)
    g = GpuStep(plan, layer)
    nd, t = g.nd, g.t
    k_new, v_new = t["k"][:nd].contiguous(), t["v"][:nd].contiguous()
    kp1, vp1 = t["k_pool"].clone(), t["v_pool"].clone()
    kp2, vp2 = t["k_pool"].clone(), t["v_pool"].clone()
    ref = pkv.paged_attention_decode_append(t["q"][:nd], k_new, v_new, kp1, vp1, g.bt[:nd],
                                            g.seq_lens[:nd], g.sh.scale, g.max_dec, err=g.err)
    ws = _workspace(g)
    _plan(g, ws)
    out = pkv.paged_attention_decode_planned(t["q"][:nd], kp2, vp2, g.bt[:nd], g.seq_lens[:nd],
                                             g.sh.scale, g.max_dec, workspace=ws, k_new=k_new,
                                             v_new=v_new, err=g.err)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert torch.equal(_bits(out), _bits(ref))
    assert torch.equal(_bits(kp2), _bits(kp1)) and torch.equal(_bits(vp2), _bits(vp1))


@pytest.mark.parametrize("shape", [(32, 8, 64, "bf16"), (64, 8, 128, "bf16"), (8, 4, 16, "f32")],
                         ids=["32x8x64", "64x8x128", "8x4x16-f32"])
def test_planned_empty_sequences_and_bad_length(shape):
    """Length-0 sequences get zero rows (the outputs start as NaN); a
    length above the host's bound is reported by the plan."""
    H, K, D, dt = shape
    lens = [0, 5, 0, 200, 33, 0, 700]
    plan = tiny_plan(lens, [1] * len(lens), n_heads=H, n_kv=K, head_dim=D, block_size=16,
                     num_blocks=120, dtype=dt, seed=D)
    layer = make_tiny_layer(plan, seed=D, fill=float("nan"))
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.kp, o.vp = o.raw["k_pool"], o.raw["v_pool"]
    nd, t = g.nd, g.t
    ws = _workspace(g)
    _plan(g, ws)
    for _ in range(2):
        out = torch.full_like(t["q"][:nd], float("nan"))
        pkv.paged_attention_decode_planned(t["q"][:nd], t["k_pool"], t["v_pool"], g.bt[:nd],
                                           g.seq_lens[:nd], g.sh.scale, g.max_dec, workspace=ws,
                                           out=out, err=g.err)
        torch.cuda.synchronize()
        assert int(g.err.item()) == 0
        assert_close(f64(out), o.decode(), dt, "planned")
        for b in (0, 2, 5):
            assert torch.count_nonzero(out[b].float()) == 0
    bad = g.seq_lens.clone()
    bad[3] = g.max_dec + 5  # above the host's bound: clamped to it and reported
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.decode_plan(t["k_pool"], bad[:nd], H, g.bt.shape[1], g.max_dec, workspace=ws, err=err)
    out = pkv.paged_attention_decode_planned(t["q"][:nd], t["k_pool"], t["v_pool"], g.bt[:nd],
                                             bad[:nd], g.sh.scale, g.max_dec, workspace=ws)
    torch.cuda.synchronize()
    assert int(err.item()) & PKV_DEVERR_LENGTH
    assert not torch.isnan(out[:3].float()).any()  # rows before the bad one are untouched by it


@pytest.mark.parametrize("name", ["smollm2-135m", "llama-3.2-1b-sharedprompt"])
def test_planned_shared_prefix_bit_identical(name):
    """With a shared prefix the planned call equals
    pkv_paged_attention_decode_shared_prefix bit for bit, over two layers
    sharing one plan, and matches the oracle."""
    plan = draw_plan(name)
    P = len(plan.shared_prefix_blocks)
    assert P > 0
    ws = None
    for layer_id in range(2):
        layer = make_layer(plan, layer_id)
        g = GpuStep(plan, layer)
        g.write(g.slots())
        nd, t, sh = g.nd, g.t, g.sh
        if ws is None:
            ws = torch.zeros(pkv.decode_shared_prefix_workspace_bytes(nd, sh.n_heads, sh.head_dim,
                                                                      g.max_dec, P),
                             dtype=torch.uint8, device="cuda")
            pkv.decode_plan(t["k_pool"], g.seq_lens[:nd], sh.n_heads, g.bt.shape[1], g.max_dec,
                            workspace=ws, shared_prefix_blocks=P, err=g.err)
        out = torch.full_like(t["q"][:nd], float("nan"))
        pkv.paged_attention_decode_planned(t["q"][:nd], t["k_pool"], t["v_pool"], g.bt[:nd],
                                           g.seq_lens[:nd], sh.scale, g.max_dec, workspace=ws,
                                           shared_prefix_blocks=P, out=out, err=g.err)
        ref = pkv.paged_attention_decode_shared_prefix(t["q"][:nd], t["k_pool"], t["v_pool"],
                                                       g.bt[:nd], g.seq_lens[:nd], sh.scale, P,
                                                       g.max_dec, err=g.err)
        torch.cuda.synchronize()
        assert int(g.err.item()) == 0
        assert torch.equal(_bits(out), _bits(ref)), f"{name} layer {layer_id}"
        if layer_id == 0:
            o = OracleStep(plan, layer)
            o.run_write()
            rows = list(range(min(nd, 24)))
            assert_close(f64(out)[rows], o.decode(rows=rows)[rows], plan.shape.dtype, name)


def test_planned_shared_prefix_append_bit_identical():
    """Shared prefix with the step's K/V write fused (each new token lands
    after the prefix): outputs and pools bit-identical to pkv_kv_write at
    the new slots followed by the planned shared-prefix call."""
    plan = draw_plan("llama-3.2-1b-sharedprompt")
    P = len(plan.shared_prefix_blocks)
    layer = make_layer(plan, 0)
    g = GpuStep(plan, layer)
    nd, t, sh = g.nd, g.t, g.sh
    k_new, v_new = t["k"][:nd].contiguous(), t["v"][:nd].contiguous()
    kp1, vp1 = t["k_pool"].clone(), t["v_pool"].clone()
    kp2, vp2 = t["k_pool"].clone(), t["v_pool"].clone()
    ws = torch.zeros(pkv.decode_shared_prefix_workspace_bytes(nd, sh.n_heads, sh.head_dim,
                                                              g.max_dec, P),
                     dtype=torch.uint8, device="cuda")
    pkv.decode_plan(t["k_pool"], g.seq_lens[:nd], sh.n_heads, g.bt.shape[1], g.max_dec,
                    workspace=ws, shared_prefix_blocks=P, err=g.err)
    pkv.kv_write(k_new, v_new, g.slots()[:nd], kp1, vp1, err=g.err)
    ref = pkv.paged_attention_decode_planned(t["q"][:nd], kp1, vp1, g.bt[:nd], g.seq_lens[:nd],
                                             sh.scale, g.max_dec, workspace=ws,
                                             shared_prefix_blocks=P, err=g.err)
    out = pkv.paged_attention_decode_planned(t["q"][:nd], kp2, vp2, g.bt[:nd], g.seq_lens[:nd],
                                             sh.scale, g.max_dec, workspace=ws, k_new=k_new,
                                             v_new=v_new, shared_prefix_blocks=P, err=g.err)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert torch.equal(_bits(out), _bits(ref))
    assert torch.equal(_bits(kp2), _bits(kp1)) and torch.equal(_bits(vp2), _bits(vp1))


PKV_DEVERR_PLAN = 64


@pytest.mark.parametrize("case", ["grid", "batch", "unplanned", "replaced"])
def test_planned_call_rejects_a_plan_for_other_sizes(case):
    """A planned call whose plan was made for another grid or batch, or
    whose workspace was never planned or was last used by a call planning
    for itself, computes nothing and reports the plan error; the same
    workspace planned again then gives the right result."""
    plan = draw_plan("smollm2-135m")
    layer = make_layer(plan, 0)
    g = GpuStep(plan, layer)
    g.write(g.slots())
    nd, t = g.nd, g.t
    ws = _workspace(g, 0)  # large enough for either grid
    if case == "grid":
        _plan(g, ws, max_ctas=7)
    elif case == "batch":
        pkv.decode_plan(t["k_pool"], g.seq_lens[:nd - 1], g.sh.n_heads, g.bt.shape[1], g.max_dec,
                        workspace=ws, err=g.err)
    elif case == "replaced":
        _plan(g, ws)
        pkv.paged_attention_decode(t["q"][:nd], t["k_pool"], t["v_pool"], g.bt[:nd], g.seq_lens[:nd],
                                   g.sh.scale, g.max_dec, workspace=ws, err=g.err)
    out = torch.full_like(t["q"][:nd], float("nan"))

    def call():
        pkv.paged_attention_decode_planned(t["q"][:nd], t["k_pool"], t["v_pool"], g.bt[:nd],
                                           g.seq_lens[:nd], g.sh.scale, g.max_dec, workspace=ws,
                                           out=out, err=g.err)

    call()
    torch.cuda.synchronize()
    assert int(g.err.item()) == PKV_DEVERR_PLAN
    assert torch.isnan(out).all()
    g.err.zero_()
    _plan(g, ws)
    call()
    ref = g.decode()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert torch.equal(_bits(out), _bits(ref))


def test_stale_plan_stores_nothing():
    """With k_new / v_new and a plan made for another grid, or with a
    shared prefix the plan was not made for, the planned call reports the
    plan error, leaves both pools untouched and writes no output row (every
    sequence here runs past the 1,024-token prefix)."""
    plan = draw_plan("llama-3.2-1b-sharedprompt")
    P = len(plan.shared_prefix_blocks)
    layer = make_layer(plan, 0)
    g = GpuStep(plan, layer)
    nd, t, sh = g.nd, g.t, g.sh
    assert int(plan.seq_lens[:nd].min()) > P * sh.block_size
    k_new, v_new = t["k"][:nd].contiguous(), t["v"][:nd].contiguous()
    kp0, vp0 = t["k_pool"].clone(), t["v_pool"].clone()
    ws = torch.zeros(pkv.decode_shared_prefix_workspace_bytes(nd, sh.n_heads, sh.head_dim,
                                                              g.max_dec, P),
                     dtype=torch.uint8, device="cuda")
    for plan_ctas, plan_prefix in ((7, P), (0, 0)):
        pkv.decode_plan(t["k_pool"], g.seq_lens[:nd], sh.n_heads, g.bt.shape[1], g.max_dec,
                        workspace=ws, shared_prefix_blocks=plan_prefix, max_ctas=plan_ctas,
                        err=g.err)
        torch.cuda.synchronize()
        assert int(g.err.item()) == 0
        out = torch.full_like(t["q"][:nd], float("nan"))
        pkv.paged_attention_decode_planned(t["q"][:nd], t["k_pool"], t["v_pool"], g.bt[:nd],
                                           g.seq_lens[:nd], sh.scale, g.max_dec, workspace=ws,
                                           k_new=k_new, v_new=v_new, shared_prefix_blocks=P,
                                           out=out, err=g.err)
        torch.cuda.synchronize()
        assert int(g.err.item()) == PKV_DEVERR_PLAN, (plan_ctas, plan_prefix)
        assert torch.isnan(out).all()
        assert torch.equal(_bits(t["k_pool"]), _bits(kp0))
        assert torch.equal(_bits(t["v_pool"]), _bits(vp0))
        g.err.zero_()
