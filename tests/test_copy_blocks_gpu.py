"""Copy-on-write block copy on the GPU against the oracle, through the C
ABI: whole pools bit-exact, bad ids reported and skipped, and the
copy-on-write step of prefix sharing end to end (copy, repoint, append,
attend)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_write_gb300 as pkv
from gpu_step import assert_close, f64, raw

pytestmark = pytest.mark.gpu

PKV_DEVERR_BLOCK_ID = 1


def _pools(nb, bs, n_kv, hd, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    shape = (nb, bs, n_kv, hd)
    return (torch.randn(shape, generator=g).to(dtype), torch.randn(shape, generator=g).to(dtype))


def _pairs(rng, nb, n):
    """n pairs: distinct sources, distinct destinations, no destination a source."""
    ids = rng.permutation(nb)
    return np.stack([ids[:n], ids[n:2 * n]], axis=1).astype(np.int32)


SHAPES = [  # (num_blocks, block_size, n_kv, head_dim, dtype)
    (64, 16, 4, 16, torch.float32), (300, 16, 8, 128, torch.bfloat16),
    (200, 16, 8, 64, torch.bfloat16), (50, 1, 2, 8, torch.float32),
    (80, 4, 3, 64, torch.bfloat16), (40, 32, 1, 128, torch.float32),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"{s[0]}x{s[1]}x{s[2]}x{s[3]}" for s in SHAPES])
def test_copy_blocks_matches_oracle(shape):
    nb, bs, n_kv, hd, dt = shape
    rng = np.random.default_rng(nb + hd)
    kp, vp = _pools(nb, bs, n_kv, hd, dt, seed=nb)
    for n in (1, 7, nb // 2):
        pairs = _pairs(rng, nb, n)
        want_k, want_v = oracle.copy_blocks(raw(kp), raw(vp), pairs)
        gk, gv = kp.cuda(), vp.cuda()
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pkv.copy_blocks(gk, gv, torch.from_numpy(pairs).cuda(), err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert np.array_equal(raw(gk.cpu()), want_k), n
        assert np.array_equal(raw(gv.cpu()), want_v), n


def test_copy_blocks_bad_ids_skipped():
    nb = 32
    kp, vp = _pools(nb, 16, 2, 64, torch.bfloat16, seed=1)
    pairs = np.array([[1, 2], [nb, 3], [4, -1], [5, 6], [-7, 8], [9, nb + 100]], dtype=np.int32)
    want_k, want_v = oracle.copy_blocks(raw(kp), raw(vp), pairs)
    gk, gv = kp.cuda(), vp.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_blocks(gk, gv, torch.from_numpy(pairs).cuda(), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & PKV_DEVERR_BLOCK_ID
    assert np.array_equal(raw(gk.cpu()), want_k)
    assert np.array_equal(raw(gv.cpu()), want_v)


def test_copy_blocks_many_pairs_workload_block():
    """4,096 pairs of LLaMA-2-70B-shaped blocks (32 KB of K and 32 KB of V each)."""
    nb, n = 10000, 4096
    g = torch.Generator(device="cuda").manual_seed(3)
    kp = torch.randn((nb, 16, 8, 128), generator=g, device="cuda").to(torch.bfloat16)
    vp = torch.randn((nb, 16, 8, 128), generator=g, device="cuda").to(torch.bfloat16)
    k0, v0 = kp.clone(), vp.clone()
    pairs = torch.from_numpy(_pairs(np.random.default_rng(0), nb, n)).cuda()
    pkv.copy_blocks(kp, vp, pairs)
    torch.cuda.synchronize()
    src, dst = pairs[:, 0].long(), pairs[:, 1].long()
    assert torch.equal(kp[dst].view(torch.int16), k0[src].view(torch.int16))
    assert torch.equal(vp[dst].view(torch.int16), v0[src].view(torch.int16))
    untouched = torch.ones(nb, dtype=torch.bool, device="cuda")
    untouched[dst] = False
    assert torch.equal(kp[untouched].view(torch.int16), k0[untouched].view(torch.int16))
    assert torch.equal(vp[untouched].view(torch.int16), v0[untouched].view(torch.int16))


def test_copy_on_write_then_append_and_decode():
    """Sequences A and B share a 40-token prefix (blocks P0, P1, P2; P2 is
    half full).  B copies P2 to a free block F, points its table at F and
    appends its token there; A appends nothing.  Decode of both must match
    the oracle doing the same steps, and A's pages must be unchanged."""
    bs, n_kv, hd, H, nb = 16, 2, 64, 8, 12
    kp, vp = _pools(nb, bs, n_kv, hd, torch.bfloat16, seed=21)
    P0, P1, P2, F = 4, 9, 2, 7
    bt = np.array([[P0, P1, P2], [P0, P1, F]], dtype=np.int32)
    lens = np.array([40, 41], dtype=np.int32)     # A: the shared 40; B: 40 + its new token
    g = torch.Generator().manual_seed(8)
    q = torch.randn((2, H, hd), generator=g).to(torch.bfloat16)
    k_new = torch.randn((1, n_kv, hd), generator=g).to(torch.bfloat16)
    v_new = torch.randn((1, n_kv, hd), generator=g).to(torch.bfloat16)
    # oracle: copy, append B's token at position 40 (block F, offset 8), attend
    ok, ov = oracle.copy_blocks(raw(kp), raw(vp), np.array([[P2, F]]))
    slot = oracle.slot_of(bt[1], 40, bs)
    assert slot == F * bs + 8
    ok, ov = oracle.kv_write(raw(k_new), raw(v_new), np.array([slot]), ok, ov)
    ref = oracle.paged_attention_decode(raw(q), ok, ov, bt, lens, hd ** -0.5, "bf16")
    # GPU
    gk, gv = kp.cuda(), vp.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_blocks(gk, gv, torch.tensor([[P2, F]], dtype=torch.int32, device="cuda"), err=err)
    pkv.kv_write(k_new.cuda(), v_new.cuda(), torch.tensor([slot], device="cuda"), gk, gv, err=err)
    out = pkv.paged_attention_decode(q.cuda(), gk, gv, torch.from_numpy(bt).cuda(),
                                     torch.from_numpy(lens).cuda(), hd ** -0.5, 41, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(raw(gk.cpu()), ok) and np.array_equal(raw(gv.cpu()), ov)
    assert_close(f64(out), ref, "bf16", "copy-on-write decode")
    # A's pages are bit-identical to before
    for blk in (P0, P1, P2):
        assert torch.equal(gk[blk].cpu().view(torch.int16), kp[blk].view(torch.int16))
