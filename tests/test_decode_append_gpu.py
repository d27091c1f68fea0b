"""Decode with append (one launch: store this step's K/V at each sequence's
last position, then attend) on the GPU, through the C ABI.

It must equal the two-call path, kv_write at the decode slots followed by
paged_attention_decode: the pools byte for byte, the outputs bit for bit
for the same max_ctas.  It must also match the float64 oracle (write, then
attend) within the dtype's tolerance."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_write_gb300 as pkv
from gpu_step import assert_close, f64, raw
from workloads import draw_plan, make_layer, make_tiny_layer, tiny_plan

pytestmark = pytest.mark.gpu

PKV_DEVERR_BLOCK_ID = 1
PKV_DEVERR_LENGTH = 8


def _bits(t):
    """The tensor's bytes, flat."""
    return t.contiguous().view(torch.uint8).reshape(-1)


def _decode_slots(plan):
    """Slot of each decode row's new token at position seq_len - 1 (oracle
    arithmetic); -1 (not written) for a sequence of length 0."""
    bs = plan.shape.block_size
    return np.array([oracle.slot_of(plan.block_tables[b], int(L) - 1, bs) if L > 0 else -1
                     for b, L in enumerate(plan.seq_lens[:plan.n_decode])], dtype=np.int64)


def _run_both(plan, layer, max_ctas, max_seq_len=None):
    """(two-call pools, two-call out, fused pools, fused out, err words)."""
    nd = plan.n_decode
    sh = plan.shape
    dev = torch.device("cuda")
    bt = torch.from_numpy(plan.block_tables[:nd]).to(dev)
    sl = torch.from_numpy(plan.seq_lens[:nd]).to(dev)
    q, k, v = (layer[n][:nd].to(dev) for n in ("q", "k", "v"))
    msl = int(plan.seq_lens[:nd].max()) if max_seq_len is None else max_seq_len
    # two calls: kv_write at the decode slots, then decode
    kp1, vp1 = layer["k_pool"].to(dev), layer["v_pool"].to(dev)
    slots = torch.from_numpy(_decode_slots(plan)).to(dev)
    err1 = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.kv_write(k, v, slots, kp1, vp1, err=err1)
    out1 = pkv.paged_attention_decode(q, kp1, vp1, bt, sl, sh.scale, msl, max_ctas=max_ctas,
                                      err=err1)
    # one call
    kp2, vp2 = layer["k_pool"].to(dev), layer["v_pool"].to(dev)
    err2 = torch.zeros(1, dtype=torch.int32, device=dev)
    out2 = pkv.paged_attention_decode_append(q, k, v, kp2, vp2, bt, sl, sh.scale, msl,
                                             max_ctas=max_ctas, err=err2)
    torch.cuda.synchronize()
    return (kp1, vp1), out1, (kp2, vp2), out2, (int(err1.item()), int(err2.item()))


def _sample_rows(plan, n=24):
    nd = plan.n_decode
    if nd <= n:
        return list(range(nd))
    rng = np.random.default_rng(11)
    pick = set(rng.choice(nd, n - 2, replace=False).tolist())
    lens = plan.seq_lens[:nd]
    pick.update((int(np.argmax(lens)), int(np.argmin(lens))))
    return sorted(pick)


def _oracle_decode(plan, layer, rows=None):
    """Oracle: write the decode rows' K/V at their slots, then attend."""
    nd = plan.n_decode
    r = {n: raw(layer[n]) for n in ("q", "k", "v", "k_pool", "v_pool")}
    kp, vp = oracle.kv_write(r["k"][:nd], r["v"][:nd], _decode_slots(plan), r["k_pool"],
                             r["v_pool"])
    return oracle.paged_attention_decode(r["q"][:nd], kp, vp, plan.block_tables[:nd],
                                         plan.seq_lens[:nd], plan.shape.scale, plan.shape.dtype,
                                         rows=rows)


CASES = ["toy", "smollm2-135m", "llama-3.2-1b", "llama-7b", "llama2-70b-mixed"]


@pytest.mark.parametrize("name", CASES)
def test_append_equals_write_then_decode(name):
    plan = draw_plan(name)
    layer = make_layer(plan, 0, fill=1e30)
    pools1, out1, pools2, out2, errs = _run_both(plan, layer, max_ctas=0)
    assert errs == (0, 0)
    assert torch.equal(_bits(pools1[0]), _bits(pools2[0])), "K pools differ"
    assert torch.equal(_bits(pools1[1]), _bits(pools2[1])), "V pools differ"
    assert torch.equal(_bits(out1), _bits(out2)), "outputs differ from the two-call path"
    rows = _sample_rows(plan) if name in ("llama2-70b-mixed", "llama-7b") else None
    ref = _oracle_decode(plan, layer, rows=rows)
    rows = rows if rows is not None else list(range(plan.n_decode))
    assert_close(f64(out2)[rows], ref[rows], plan.shape.dtype, name)
    # the stored rows are this step's k / v, bit for bit
    slots = _decode_slots(plan)
    sh = plan.shape
    kflat = raw(pools2[0].view(sh.num_blocks * sh.block_size, sh.n_kv, sh.head_dim).cpu()[
        torch.from_numpy(slots)])
    assert np.array_equal(kflat, raw(layer["k"][:plan.n_decode]))


SMALL = [  # (n_heads, n_kv, head_dim, dtype)
    (8, 4, 16, "f32"), (12, 4, 128, "f32"), (9, 3, 64, "bf16"), (32, 8, 64, "bf16"),
    (64, 8, 128, "bf16"), (16, 1, 64, "bf16"), (4, 2, 32, "bf16"),
]


@pytest.mark.parametrize("shape", SMALL, ids=[f"{h}x{k}x{d}-{t}" for h, k, d, t in SMALL])
def test_append_small_ragged(shape):
    H, K, D, dt = shape
    lens = [1, 2, 15, 16, 17, 31, 33, 64, 100, 257, 700]
    plan = tiny_plan(lens, [1] * len(lens), n_heads=H, n_kv=K, head_dim=D, block_size=16,
                     num_blocks=120, dtype=dt, seed=H * 10 + D)
    layer = make_tiny_layer(plan, seed=D + 1, fill=float("nan"))
    ref = _oracle_decode(plan, layer)
    for max_ctas in (0, 1, 3, 16):
        pools1, out1, pools2, out2, errs = _run_both(plan, layer, max_ctas)
        assert errs == (0, 0)
        for a, b in zip(pools1, pools2):
            assert torch.equal(_bits(a), _bits(b)), f"pools differ, max_ctas={max_ctas}"
        assert torch.equal(_bits(out1), _bits(out2)), f"outputs differ, max_ctas={max_ctas}"
        assert_close(f64(out2), ref, dt, f"max_ctas={max_ctas}")


def test_append_empty_sequence_writes_nothing():
    # every row carries a k/v row; the two of length 0 have nowhere to put it
    plan = tiny_plan([0, 1, 5, 0, 40], [1] * 5, n_heads=8, n_kv=2, head_dim=64,
                     block_size=16, num_blocks=16, dtype="bf16", seed=4)
    assert plan.n_decode == 5
    layer = make_tiny_layer(plan, seed=9, fill=float("nan"))
    pools1, out1, pools2, out2, errs = _run_both(plan, layer, max_ctas=0)
    assert errs == (0, 0)
    for a, b in zip(pools1, pools2):
        assert torch.equal(_bits(a), _bits(b))
    assert torch.equal(_bits(out1), _bits(out2))
    out = out2.float().cpu()
    assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[3]) == 0


def test_append_bad_block_id_and_bad_length_write_nothing():
    """A last table entry outside the pool, or a length above max_seq_len,
    is reported and nothing is stored for that sequence (the kernel checks
    both before using them as addresses)."""
    plan = tiny_plan([20, 20, 20], [1, 1, 1], n_heads=8, n_kv=2, head_dim=64, block_size=16,
                     num_blocks=16, dtype="bf16", seed=5)
    plan.block_tables = plan.block_tables.copy()
    plan.block_tables[1, 1] = 16 + 5           # last block of sequence 1: out of range
    plan.seq_lens = plan.seq_lens.copy()
    plan.seq_lens[2] = 30                      # above the max_seq_len passed below
    layer = make_tiny_layer(plan, seed=2)
    dev = torch.device("cuda")
    kp, vp = layer["k_pool"].to(dev), layer["v_pool"].to(dev)
    before = [_bits(kp).clone(), _bits(vp).clone()]
    bt = torch.from_numpy(plan.block_tables).to(dev)
    sl = torch.from_numpy(plan.seq_lens).to(dev)
    q, k, v = (layer[n].to(dev) for n in ("q", "k", "v"))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.paged_attention_decode_append(q, k, v, kp, vp, bt, sl, plan.shape.scale, 24, err=err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & PKV_DEVERR_BLOCK_ID and e & PKV_DEVERR_LENGTH
    # only sequence 0's slot changed
    slot0 = int(plan.block_tables[0, 1]) * 16 + 19 - 16
    after = [_bits(kp), _bits(vp)]
    row_bytes = plan.shape.n_kv * plan.shape.head_dim * 2
    for a, b in zip(before, after):
        diff = torch.nonzero(a != b).flatten().cpu().numpy()
        assert diff.size > 0
        assert diff.min() >= slot0 * row_bytes and diff.max() < (slot0 + 1) * row_bytes
