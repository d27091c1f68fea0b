"""Chunked prefill attention on the GPU against the float64 oracle."""
import numpy as np
import pytest
import torch

from gpu_step import GpuStep, OracleStep, assert_close, f64
from workloads import draw_plan, make_layer, tiny_plan, make_tiny_layer

pytestmark = pytest.mark.gpu


@pytest.mark.slow
def test_prefill_70b_mixed_step_every_query():
    """LLaMA-2-70B mixed step: 4 chunks of 512 queries over 0, 1,365, 2,731
    and 4,096 tokens of history; every query of every chunk (all 64 heads)
    against the oracle's chunked prefill (about 20 s of CPU)."""
    import oracle
    plan = draw_plan("llama2-70b-mixed")
    layer = make_layer(plan, 0, fill=1e30)
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.run_write()
    _, _, pre = g.run()
    got = f64(pre)
    nd = plan.n_decode
    cu = (plan.cu_new_lens[nd:] - plan.cu_new_lens[nd]).astype(np.int64)
    ref = oracle.paged_attention_prefill(o.raw["q"][nd:], cu, o.kp, o.vp, plan.block_tables[nd:],
                                         plan.seq_lens[nd:], plan.shape.scale, "bf16")
    for b_rel in range(plan.num_seqs - nd):
        lo, hi = int(cu[b_rel]), int(cu[b_rel + 1])
        assert_close(got[lo:hi], ref[lo:hi], "bf16", f"prefill seq {b_rel}")
    assert int(g.err.item()) == 0


@pytest.mark.parametrize("name", ["smollm2-135m-prompts", "llama-3.2-1b-prompts"])
def test_batched_full_prompt_prefill_sampled(name):
    """Batched full-prompt prefill (history 0): every prompt of a batch of
    users arriving together in one launch; sampled queries of every prompt
    (first, block edges, last, random) against the oracle."""
    plan = draw_plan(name)
    assert plan.n_decode == 0 and np.array_equal(plan.new_lens, plan.seq_lens)
    layer = make_layer(plan, 0, fill=1e30)
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.run_write()
    _, _, pre = g.run()
    got = f64(pre)
    rng = np.random.default_rng(5)
    for b in range(plan.num_seqs):
        c = int(plan.new_lens[b])
        base = int(plan.cu_new_lens[b])
        qs = sorted({0, 1, 15, 16, 17, c - 1} | set(rng.choice(c, 4, replace=False).tolist()))
        ref = np.stack([o.prefill_row(b, i) for i in qs])
        assert_close(got[[base + i for i in qs]], ref, "bf16", f"{name} prompt {b}")
    assert int(g.err.item()) == 0


SMALL = [(8, 4, 16, "f32"), (16, 2, 64, "f32"), (9, 3, 64, "bf16"), (32, 8, 64, "bf16"),
         (64, 8, 128, "bf16"), (8, 8, 128, "bf16"), (16, 1, 64, "bf16"), (4, 2, 32, "bf16"),
         (15, 3, 128, "bf16"), (14, 2, 64, "bf16"), (12, 1, 128, "bf16")]


@pytest.mark.parametrize("shape", SMALL, ids=[f"{h}x{k}x{d}-{t}" for h, k, d, t in SMALL])
def test_prefill_small_ragged(shape):
    H, K, D, dt = shape
    hist = [0, 0, 3, 16, 37, 100]
    chunk = [40, 1, 17, 16, 5, 33]
    lens = [h + c for h, c in zip(hist, chunk)]
    plan = tiny_plan(lens, chunk, n_heads=H, n_kv=K, head_dim=D, block_size=16, num_blocks=64,
                     dtype=dt, seed=D + H)
    plan.n_decode = 0  # every row is a prefill chunk (one of them a single query)
    layer = make_tiny_layer(plan, seed=H, fill=float("nan"))
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.run_write()
    _, _, pre = g.run()
    got = f64(pre)
    for b in range(len(lens)):
        ref = np.stack([o.prefill_row(b, i) for i in range(chunk[b])])
        lo = int(plan.cu_new_lens[b])
        assert_close(got[lo:lo + chunk[b]], ref, dt, f"seq {b}")
    assert int(g.err.item()) == 0


GROUPS = [(9, 3, 64), (15, 3, 128), (12, 2, 64), (21, 3, 128), (13, 1, 64)]


@pytest.mark.parametrize("shape", GROUPS, ids=[f"{h}x{k}x{d}" for h, k, d in GROUPS])
def test_prefill_groups_not_dividing_the_tile(shape):
    """Query heads per KV head that do not divide the 128-row tile (3, 5,
    6, 7, 13): each tile holds floor(128 / rep) queries; chunks spanning
    several tile pairs, with ragged ends, against the oracle on every
    query."""
    H, K, D = shape
    hist = [0, 50, 300]
    chunk = [200, 131, 90]
    lens = [h + c for h, c in zip(hist, chunk)]
    plan = tiny_plan(lens, chunk, n_heads=H, n_kv=K, head_dim=D, block_size=16, num_blocks=96,
                     dtype="bf16", seed=H + D)
    plan.n_decode = 0
    layer = make_tiny_layer(plan, seed=H, fill=float("nan"))
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.run_write()
    _, _, pre = g.run()
    got = f64(pre)
    for b in range(len(lens)):
        ref = np.stack([o.prefill_row(b, i) for i in range(chunk[b])])
        lo = int(plan.cu_new_lens[b])
        assert_close(got[lo:lo + chunk[b]], ref, "bf16", f"seq {b}")
    assert int(g.err.item()) == 0


def test_prefill_chunk_of_one_equals_decode():
    lens = [5, 33, 200]
    for dt, (H, K, D) in (("bf16", (32, 8, 64)), ("f32", (8, 4, 16))):
        plan = tiny_plan(lens, [1, 1, 1], n_heads=H, n_kv=K, head_dim=D, block_size=16,
                         num_blocks=32, dtype=dt)
        layer = make_tiny_layer(plan, seed=9)
        g = GpuStep(plan, layer)
        g.write(g.slots())
        dec = g.decode(max_ctas=1)
        cu = torch.arange(len(lens) + 1, dtype=torch.int32, device="cuda")
        pre = g.pkv.paged_attention_prefill(g.t["q"], cu, g.t["k_pool"], g.t["v_pool"], g.bt,
                                            g.seq_lens, plan.shape.scale, 1, max(lens))
        torch.cuda.synchronize()
        assert_close(f64(pre), f64(dec), dt, "prefill(c=1) vs decode")


@pytest.mark.parametrize("shape", [(32, 8, 64), (9, 3, 128)], ids=["32x8x64", "9x3x128"])
def test_prefill_many_sequences_natural_grid(shape):
    """More sequences than the tcgen05 kernel ranks by work (352): the grid
    falls back to (pair, KV head, sequence) order.  400 chunks of 1..70
    queries over 0..150 tokens of history; sampled queries of every chunk
    against the oracle."""
    H, K, D = shape
    rng = np.random.default_rng(H + D)
    B = 400
    chunk = rng.integers(1, 71, size=B)
    hist = rng.integers(0, 151, size=B)
    lens = (hist + chunk).tolist()
    plan = tiny_plan(lens, chunk.tolist(), n_heads=H, n_kv=K, head_dim=D, block_size=16,
                     num_blocks=int(sum((l + 15) // 16 for l in lens)) + 8, dtype="bf16",
                     seed=H + D)
    plan.n_decode = 0
    layer = make_tiny_layer(plan, seed=D, fill=float("nan"))
    g, o = GpuStep(plan, layer), OracleStep(plan, layer)
    o.run_write()
    _, _, pre = g.run()
    got = f64(pre)
    for b in range(0, B, 7):
        c = int(chunk[b])
        lo = int(plan.cu_new_lens[b])
        qs = sorted({0, c - 1, c // 2})
        ref = np.stack([o.prefill_row(b, i) for i in qs])
        assert_close(got[[lo + i for i in qs]], ref, "bf16", f"seq {b}")
    assert int(g.err.item()) == 0
