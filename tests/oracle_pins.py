"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
a worked example from the pages (fixtures under ``tests/golden/``), a closed
form, a library attention routine (torch's scaled_dot_product_attention in
float64 on logically ordered K/V), or an invariant the pages state.  They
are collected by ``test_oracle_pins.py`` and re-run against deliberately
broken copies of the oracle by ``test_oracle_mutations.py``.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle
import oracle.paged as op

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand_pool(rng, nb, bs, n_kv, hd):
    return rng.standard_normal((nb, bs, n_kv, hd)).astype(np.float32)


# ---------------------------------------------------------------- slots / gather


def pin_interleaved_allocation_example():
    """"Build a Mini vLLM" section 2 figure: tables and slots of Seq A / Seq B."""
    g = _golden("mini_vllm_interleaved_tables.json")
    bs = g["block_size"]
    # Allocate the way the figure describes: take turns, one token each;
    # a sequence takes the front of the free list when its count is a
    # multiple of the block size.
    free = list(range(g["num_blocks"]))
    tables = {s: [] for s in g["tokens"]}
    count = {s: 0 for s in g["tokens"]}
    while any(count[s] < n for s, n in g["tokens"].items()):
        for s, n in g["tokens"].items():
            if count[s] < n:
                if count[s] % bs == 0:
                    tables[s].append(free.pop(0))
                count[s] += 1
    assert tables == g["tables"], tables
    for s, n in g["tokens"].items():
        slots = [op.slot_of(g["tables"][s], p, bs) for p in range(n)]
        assert slots == g["slots"][s], (s, slots)
    # the same slots through slot_mapping of a whole-prompt write
    names = list(g["tokens"])
    W = max(len(t) for t in g["tables"].values())
    bt = np.zeros((2, W), dtype=np.int32)
    for i, s in enumerate(names):
        bt[i, :len(g["tables"][s])] = g["tables"][s]
    lens = np.array([g["tokens"][s] for s in names], dtype=np.int32)
    sm = oracle.slot_mapping(bt, lens, lens, bs)
    assert sm.tolist() == g["slots"][names[0]] + g["slots"][names[1]]


def pin_day16_out_of_order_blocks():
    """"Day 16" diagram: block_ids [2, 0], 7 tokens read back in logical order."""
    g = _golden("day16_block_ids_2_0.json")
    bs = g["block_size"]
    nb = 3
    flat = np.arange(nb * bs, dtype=np.int64)  # value = physical flat slot
    pool = flat.reshape(nb, bs, 1, 1)
    got = oracle.gather_kv(pool, np.array(g["table"]), g["tokens"]).reshape(-1)
    assert got.tolist() == g["physical_slots_in_logical_order"], got
    slots = [op.slot_of(g["table"], p, bs) for p in range(g["tokens"])]
    assert slots == g["physical_slots_in_logical_order"]


def pin_write_gather_round_trip():
    """Write every token through its slot, gather back: exact ("Day 16",
    Why it matters: byte for byte what the naive cache would hand it;
    "nano-vLLM" test_kv_pool: values read back exactly through tables)."""
    rng = np.random.default_rng(11)
    for bs in (1, 4, 16):
        nb, n_kv, hd = 40, 2, 3
        lens = np.array([1, bs, 2 * bs + 1, 5 * bs - 1], dtype=np.int32)
        nblk = [-(-int(l) // bs) for l in lens]
        perm = rng.permutation(np.arange(1, nb))
        bt = np.zeros((len(lens), max(nblk)), dtype=np.int32)
        c = 0
        for i, n in enumerate(nblk):
            bt[i, :n] = perm[c:c + n]
            c += n
        toks = [rng.standard_normal((int(l), n_kv, hd)).astype(np.float32) for l in lens]
        k = np.concatenate(toks)
        sm = oracle.slot_mapping(bt, lens, lens, bs)
        sentinel = np.float32(-7.5)
        pool0 = np.full((nb, bs, n_kv, hd), sentinel, dtype=np.float32)
        kp, vp = oracle.kv_write(k, -k, sm, pool0, pool0)
        for i in range(len(lens)):
            assert np.array_equal(oracle.gather_kv(kp, bt[i], lens[i]), toks[i])
            assert np.array_equal(oracle.gather_kv(vp, bt[i], lens[i]), -toks[i])
        # exactly the written slots changed
        touched = np.zeros(nb * bs, dtype=bool)
        touched[sm] = True
        flat = kp.reshape(nb * bs, -1)
        assert np.all(flat[~touched] == sentinel)
        assert len(set(sm.tolist())) == len(sm)


def pin_copy_on_write_shared_prefix():
    """Copy-on-write of a shared prefix block ("Build a Mini vLLM", Key
    Takeaways 6): sequences A and B share physical block P holding the
    first 6 tokens (block size 4: P is full, Q half full and also shared).
    Before B writes its 7th token into the shared, half-full block Q, the
    engine copies Q to a free block F, points B's table at F, then writes.
    A must read back exactly what it had; B its prefix plus the new token."""
    rng = np.random.default_rng(5)
    bs, n_kv, hd, nb = 4, 2, 3, 8
    kp = _rand_pool(rng, nb, bs, n_kv, hd)
    vp = _rand_pool(rng, nb, bs, n_kv, hd)
    P, Q, F = 3, 6, 1
    table_a = np.array([P, Q])
    a_k = oracle.gather_kv(kp, table_a, 6).copy()
    a_v = oracle.gather_kv(vp, table_a, 6).copy()
    kp2, vp2 = oracle.copy_blocks(kp, vp, np.array([[Q, F]]))
    table_b = np.array([P, F])
    new_k = rng.standard_normal((1, n_kv, hd)).astype(np.float32)
    new_v = rng.standard_normal((1, n_kv, hd)).astype(np.float32)
    sm = oracle.slot_mapping(table_b[None], np.array([7]), np.array([1]), bs)
    assert sm.tolist() == [F * bs + 2]
    kp3, vp3 = oracle.kv_write(new_k, new_v, sm, kp2, vp2)
    assert np.array_equal(oracle.gather_kv(kp3, table_a, 6), a_k)
    assert np.array_equal(oracle.gather_kv(vp3, table_a, 6), a_v)
    assert np.array_equal(oracle.gather_kv(kp3, table_b, 7), np.concatenate([a_k, new_k]))
    assert np.array_equal(oracle.gather_kv(vp3, table_b, 7), np.concatenate([a_v, new_v]))
    # only block F changed, and F's first two rows are Q's
    changed = [b for b in range(nb) if not np.array_equal(kp3[b], kp[b])]
    assert changed == [F]
    assert np.array_equal(kp3[F, :2], kp[Q, :2]) and np.array_equal(vp3[F, :2], vp[Q, :2])


def pin_copy_blocks_reads_the_pools_before_the_call():
    """Pairs chained through a block (0 -> 1, 1 -> 2) copy the old
    contents: block 2 receives the old block 1, whatever the pair order;
    a pair with an id outside the pool is skipped."""
    blocks = np.arange(5, dtype=np.float32).reshape(5, 1, 1, 1) * np.ones((5, 2, 1, 2),
                                                                      dtype=np.float32)
    for pairs in ([[0, 1], [1, 2], [7, 3]], [[1, 2], [0, 1], [3, -1]]):
        kp, vp = oracle.copy_blocks(blocks, -blocks, np.array(pairs))
        assert [float(kp[b, 0, 0, 0]) for b in range(5)] == [0.0, 0.0, 1.0, 3.0, 4.0], pairs
        assert np.array_equal(vp, -kp)


def pin_negative_slot_skipped():
    pool = np.zeros((2, 2, 1, 1), dtype=np.float32)
    k = np.array([[[1.0]], [[2.0]]], dtype=np.float32)
    kp, _ = oracle.kv_write(k, k, np.array([-1, 3]), pool, pool)
    assert kp.reshape(-1).tolist() == [0.0, 0.0, 0.0, 2.0]


def pin_bf16_decode_matches_torch():
    """bf16 bit patterns -> values agrees with torch's bfloat16 conversion."""
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.standard_normal(1000).astype(np.float32) * 100,
                           np.array([0.0, -0.0, 1e30, -1e-30, 3.0e38, np.inf, -np.inf], np.float32)])
    t = torch.from_numpy(vals).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    got = oracle.to_float64(bits, "bf16")
    assert np.array_equal(got, t.to(torch.float64).numpy())


# ---------------------------------------------------------------- attention


def pin_worked_example():
    g = _golden("attention_worked_example.json")
    o, p = oracle.attend(np.array(g["q"]), np.array(g["K"]), np.array(g["V"]), g["scale"])
    assert np.allclose(p, g["p"], rtol=0, atol=1e-15), p
    assert np.allclose(o, g["o"], rtol=0, atol=1e-14), o


def pin_closed_forms():
    rng = np.random.default_rng(5)
    hd = 8
    V = rng.standard_normal((9, hd))
    K = rng.standard_normal((9, hd))
    q = rng.standard_normal(hd)
    # one key: the output is that key's value, whatever the score
    o, p = oracle.attend(q, K[:1], V[:1], 0.3)
    assert np.array_equal(o, V[0]) and p.tolist() == [1.0]
    # zero query: uniform weights, output = mean of values
    o, p = oracle.attend(np.zeros(hd), K, V, 0.3)
    assert np.allclose(o, V.mean(0), atol=1e-14) and np.allclose(p, 1 / 9, atol=1e-16)
    # all keys equal: uniform weights
    Ke = np.repeat(K[:1], 9, axis=0)
    o, _ = oracle.attend(q, Ke, V, 0.3)
    assert np.allclose(o, V.mean(0), atol=1e-14)
    # one dominating key: output = its value up to exp(-gap)
    Kd = np.zeros((9, hd))
    Kd[4, 0] = 1.0
    o, p = oracle.attend(np.eye(hd)[0] * 60.0, Kd, V, 1.0)
    assert np.allclose(o, V[4], atol=1e-20 + 9 * math.exp(-60) * np.abs(V).max())
    # probabilities sum to one, are positive, and follow exp of the scores
    o, p = oracle.attend(q, K, V, 0.7)
    assert abs(p.sum() - 1.0) < 1e-15 and np.all(p > 0)
    s = 0.7 * np.array([np.dot(q, K[j]) for j in range(9)])
    assert np.allclose(p[1:] / p[0], np.exp(s[1:] - s[0]), rtol=1e-12)
    # scaling: doubling the scale squares the odds
    _, p2 = oracle.attend(q, K, V, 1.4)
    assert np.allclose(p2[1:] / p2[0], (p[1:] / p[0]) ** 2, rtol=1e-10)
    # no keys: zero output
    o, p = oracle.attend(q, K[:0], V[:0], 0.5)
    assert np.array_equal(o, np.zeros(hd))


def _scatter_logical(rng, lens, nb, bs, n_kv, hd, dummy=True):
    """Place logical per-sequence K/V into a pool block by block (random
    physical blocks) and return pool, tables and the logical arrays."""
    first = 1 if dummy else 0
    nblk = [-(-int(l) // bs) for l in lens]
    perm = rng.permutation(np.arange(first, nb))
    W = max(1, max(nblk))
    bt = np.zeros((len(lens), W), dtype=np.int32)
    kpool = _rand_pool(rng, nb, bs, n_kv, hd)
    vpool = _rand_pool(rng, nb, bs, n_kv, hd)
    logical_k, logical_v, c = [], [], 0
    for i, l in enumerate(lens):
        lk = rng.standard_normal((nblk[i] * bs, n_kv, hd)).astype(np.float32)
        lv = rng.standard_normal((nblk[i] * bs, n_kv, hd)).astype(np.float32)
        for j in range(nblk[i]):
            blk = perm[c]
            c += 1
            bt[i, j] = blk
            kpool[blk] = lk[j * bs:(j + 1) * bs]
            vpool[blk] = lv[j * bs:(j + 1) * bs]
        logical_k.append(lk[:l])
        logical_v.append(lv[:l])
    return kpool, vpool, bt, logical_k, logical_v


def _sdpa(q, K, V, scale, mask=None):
    """torch's attention in float64: q [H, T, hd], K/V [H, L, hd]."""
    return F.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None],
        attn_mask=None if mask is None else torch.from_numpy(mask)[None, None], scale=scale)[0].numpy()


def pin_decode_matches_library_attention():
    """Paged decode == contiguous attention ("Build a Mini vLLM" section 4:
    paged == contiguous; Key Takeaways 3: a gather, not new math), with
    GQA groups expanded by repeat-interleave (section 3)."""
    rng = np.random.default_rng(21)
    for (H, n_kv, hd, bs) in [(8, 4, 16, 16), (9, 3, 8, 4), (4, 4, 8, 8), (8, 1, 4, 2)]:
        lens = [1, 5, bs, 3 * bs + 2]
        kp, vp, bt, lk, lv = _scatter_logical(rng, lens, 64, bs, n_kv, hd)
        q = rng.standard_normal((len(lens), H, hd)).astype(np.float32)
        scale = 1 / math.sqrt(hd)
        got = oracle.paged_attention_decode(q, kp, vp, bt, np.array(lens), scale, "f32")
        rep = H // n_kv
        for b in range(len(lens)):
            K = np.repeat(lk[b].astype(np.float64), rep, axis=1).transpose(1, 0, 2)
            V = np.repeat(lv[b].astype(np.float64), rep, axis=1).transpose(1, 0, 2)
            ref = _sdpa(q[b].astype(np.float64)[:, None, :], K, V, scale)[:, 0, :]
            assert np.allclose(got[b], ref, rtol=0, atol=1e-12), (H, n_kv, b)


def pin_prefill_matches_library_attention():
    """Chunked prefill == causal attention over history + chunk ("Build a
    Mini vLLM" section 4: triu(1) mask; query at position p sees 0..p)."""
    rng = np.random.default_rng(22)
    H, n_kv, hd, bs = 8, 2, 8, 4
    hist = [0, 3, 8, 13]
    chunks = [5, 1, 4, 7]
    lens = [h + c for h, c in zip(hist, chunks)]
    kp, vp, bt, lk, lv = _scatter_logical(rng, lens, 64, bs, n_kv, hd)
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = rng.standard_normal((int(cu[-1]), H, hd)).astype(np.float32)
    scale = 0.4
    got = oracle.paged_attention_prefill(q, cu, kp, vp, bt, np.array(lens), scale, "f32")
    rep = H // n_kv
    for b in range(len(lens)):
        L, c = lens[b], chunks[b]
        K = np.repeat(lk[b].astype(np.float64), rep, axis=1).transpose(1, 0, 2)
        V = np.repeat(lv[b].astype(np.float64), rep, axis=1).transpose(1, 0, 2)
        qb = q[cu[b]:cu[b + 1]].astype(np.float64).transpose(1, 0, 2)
        allowed = np.arange(L)[None, :] <= (L - c + np.arange(c))[:, None]
        ref = _sdpa(qb, K, V, scale, mask=allowed).transpose(1, 0, 2)
        assert np.allclose(got[cu[b]:cu[b + 1]], ref, rtol=0, atol=1e-12), b
    # a chunk with no history: its first query sees only itself
    b0 = 0
    first = got[cu[b0]]
    for h in range(H):
        assert np.array_equal(first[h], lv[b0][0, h // rep].astype(np.float64))


def pin_prefill_equals_sequential_decodes():
    """A chunk of c queries == c decode steps, each over the prefix up to and
    including its own token; a chunk of one == decode."""
    rng = np.random.default_rng(23)
    H, n_kv, hd, bs = 4, 2, 8, 4
    lens = [9, 14]
    chunks = [4, 6]
    kp, vp, bt, _, _ = _scatter_logical(rng, lens, 32, bs, n_kv, hd)
    cu = np.array([0, 4, 10], dtype=np.int32)
    q = rng.standard_normal((10, H, hd)).astype(np.float32)
    got = oracle.paged_attention_prefill(q, cu, kp, vp, bt, np.array(lens), 0.3, "f32")
    for b in range(2):
        for i in range(chunks[b]):
            L_i = lens[b] - chunks[b] + i + 1
            dec = oracle.paged_attention_decode(q[cu[b] + i][None], kp, vp, bt[b:b + 1],
                                                np.array([L_i]), 0.3, "f32")
            assert np.array_equal(got[cu[b] + i], dec[0])
    one = oracle.paged_attention_prefill(q[:2], np.array([0, 1, 2]), kp, vp, bt,
                                         np.array(lens), 0.3, "f32")
    dec = oracle.paged_attention_decode(q[:2], kp, vp, bt, np.array(lens), 0.3, "f32")
    assert np.array_equal(one, dec)


def pin_gqa_equals_mha_on_repeated_kv():
    rng = np.random.default_rng(24)
    H, n_kv, hd, bs = 8, 2, 4, 4
    lens = [6, 11]
    kp, vp, bt, _, _ = _scatter_logical(rng, lens, 16, bs, n_kv, hd)
    q = rng.standard_normal((2, H, hd)).astype(np.float32)
    got = oracle.paged_attention_decode(q, kp, vp, bt, np.array(lens), 0.5, "f32")
    rep = H // n_kv
    mha = oracle.paged_attention_decode(q, np.repeat(kp, rep, axis=2), np.repeat(vp, rep, axis=2),
                                        bt, np.array(lens), 0.5, "f32")
    assert np.array_equal(got, mha)
    # rep == 1 reduces to per-head attention
    got1 = oracle.paged_attention_decode(q[:, :2], kp, vp, bt, np.array(lens), 0.5, "f32")
    for b in range(2):
        for h in range(2):
            K = oracle.gather_kv(kp, bt[b], lens[b])[:, h].astype(np.float64)
            V = oracle.gather_kv(vp, bt[b], lens[b])[:, h].astype(np.float64)
            o, _ = oracle.attend(q[b, h].astype(np.float64), K, V, 0.5)
            assert np.array_equal(got1[b, h], o)


def pin_placement_and_sharing_invariance():
    """Relabelling physical blocks (moving the data along) and sharing a
    prefix block leave the output bit-identical ("Day 16", Why it matters:
    blocks can sit scattered anywhere; "nano-vLLM", How it works: users with
    the same system prompt share blocks 1 and 2)."""
    rng = np.random.default_rng(25)
    H, n_kv, hd, bs, nb = 6, 3, 8, 4, 48
    lens = np.array([9, 13, 4], dtype=np.int32)
    kp, vp, bt, _, _ = _scatter_logical(rng, lens.tolist(), nb, bs, n_kv, hd)
    q = rng.standard_normal((3, H, hd)).astype(np.float32)
    base = oracle.paged_attention_decode(q, kp, vp, bt, lens, 0.35, "f32")
    relabel = rng.permutation(nb)
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[relabel] = kp
    vp2[relabel] = vp
    moved = oracle.paged_attention_decode(q, kp2, vp2, relabel[bt].astype(np.int32), lens, 0.35, "f32")
    assert np.array_equal(base, moved)
    # share: sequence 1's first block becomes a copy shared with sequence 0's
    # first block (same contents); private copies vs a shared id agree
    kp3, vp3 = kp.copy(), vp.copy()
    kp3[bt[1, 0]] = kp[bt[0, 0]]
    vp3[bt[1, 0]] = vp[bt[0, 0]]
    private = oracle.paged_attention_decode(q, kp3, vp3, bt, lens, 0.35, "f32")
    bt_shared = bt.copy()
    bt_shared[1, 0] = bt[0, 0]
    shared = oracle.paged_attention_decode(q, kp3, vp3, bt_shared, lens, 0.35, "f32")
    assert np.array_equal(private, shared)


def pin_garbage_outside_sequence_is_ignored():
    """Huge values and NaN in slots past each length, in padding entries of
    the tables and in unheld blocks change nothing ("nano-vLLM",
    Correctness: the garbage pool proves the mask)."""
    rng = np.random.default_rng(26)
    H, n_kv, hd, bs, nb = 4, 2, 8, 4, 32
    lens = np.array([5, 2, 11], dtype=np.int32)
    kp, vp, bt, _, _ = _scatter_logical(rng, lens.tolist(), nb, bs, n_kv, hd)
    q = rng.standard_normal((3, H, hd)).astype(np.float32)
    base = oracle.paged_attention_decode(q, kp, vp, bt, lens, 0.5, "f32")
    used = np.zeros(nb * bs, dtype=bool)
    used[oracle.slot_mapping(bt, lens, lens, bs)] = True
    for junk in (np.float32(1e30), np.float32(np.nan)):
        kj, vj = kp.copy().reshape(nb * bs, n_kv, hd), vp.copy().reshape(nb * bs, n_kv, hd)
        kj[~used] = junk
        vj[~used] = junk
        btj = bt.copy()
        btj[btj == 0] = 0  # padding entries point at the (garbage) dummy block
        got = oracle.paged_attention_decode(q, kj.reshape(kp.shape), vj.reshape(vp.shape), btj,
                                            lens, 0.5, "f32")
        assert np.array_equal(got, base)


def pin_split_merge_equals_full():
    rng = np.random.default_rng(27)
    H, n_kv, hd, bs = 4, 2, 8, 4
    lens = np.array([1, 7, 16, 33], dtype=np.int32)
    kp, vp, bt, _, _ = _scatter_logical(rng, lens.tolist(), 32, bs, n_kv, hd)
    q = rng.standard_normal((4, H, hd)).astype(np.float32) * 3
    full = oracle.paged_attention_decode(q, kp, vp, bt, lens, 0.5, "f32")
    for P in (4, 8, 12, 64):
        split = oracle.paged_attention_decode_split(q, kp, vp, bt, lens, 0.5, "f32", P)
        assert np.allclose(split, full, rtol=0, atol=1e-13), P
    # merge of two single-key partitions: a two-way softmax
    V = rng.standard_normal((2, hd))
    o = oracle.merge_partials([(V[0], 1.0, 1.0), (V[1], 1.0 + math.log(3), 1.0)])
    assert np.allclose(o, 0.25 * V[0] + 0.75 * V[1], atol=1e-15)


def pin_empty_sequence():
    kp = np.zeros((4, 4, 1, 2), dtype=np.float32)
    q = np.ones((1, 2, 2), dtype=np.float32)
    out = oracle.paged_attention_decode(q, kp, kp, np.zeros((1, 1), np.int32), np.array([0]), 1.0, "f32")
    assert np.array_equal(out, np.zeros((1, 2, 2)))


def pin_bf16_attention_uses_exact_values():
    """bf16 storage is read as its exact value (the oracle and torch agree
    on the dequantised inputs, so results match the f32 path on them)."""
    rng = np.random.default_rng(28)
    H, n_kv, hd, bs = 4, 2, 8, 4
    lens = np.array([6, 9], dtype=np.int32)
    kp, vp, bt, _, _ = _scatter_logical(rng, lens.tolist(), 16, bs, n_kv, hd)
    q = rng.standard_normal((2, H, hd)).astype(np.float32)
    as_bits = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    as_vals = lambda a: torch.from_numpy(a).to(torch.bfloat16).to(torch.float32).numpy()
    got = oracle.paged_attention_decode(as_bits(q), as_bits(kp), as_bits(vp), bt, lens, 0.5, "bf16")
    ref = oracle.paged_attention_decode(as_vals(q), as_vals(kp), as_vals(vp), bt, lens, 0.5, "f32")
    assert np.array_equal(got, ref)


def pin_workload_kv_sizes_match_pages():
    """The workload shapes reproduce the pages' KV sizes per token / block."""
    from workloads import SHAPES
    g = _golden("kv_bytes_per_token.json")
    for name, want in g["per_token_bytes"].items():
        s = SHAPES[name]
        assert 2 * s.layers * s.n_kv * s.head_dim * s.itemsize == want, name
    for name, want in g["per_block_bytes"].items():
        s = SHAPES[name]
        assert 2 * s.layers * s.block_size * s.n_kv * s.head_dim * s.itemsize == want, name


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
