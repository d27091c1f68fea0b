"""Plain float64 definition of paged KV write and paged attention.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing in the CUDA
library imports this module, and the library has no CPU fallback.

Notation follows the pages:
  * a block pool ``pool[num_blocks, block_size, n_kv, head_dim]``
    ("nano-vLLM", How it works: one K and one V tensor per layer,
    [blocks, 16, KV heads, head_dim]);
  * a per-sequence block table mapping logical block ``j`` to a physical
    block id ("Build a Mini vLLM", section 2);
  * the token at logical position ``pos`` lives in block
    ``table[pos // block_size]`` at offset ``pos % block_size``
    ("Build a Mini vLLM", section 2, ``append_slot``; "nano-vLLM", How it
    works: block ``table[n // 16]``, slot ``n % 16``), i.e. at the flat slot
    ``block * block_size + offset`` of the flat pool view
    ``[num_blocks * block_size, n_kv, head_dim]`` ("Day 16", What I added).

Raw arrays are passed with a dtype tag: ``"f32"`` arrays hold float32
values, ``"bf16"`` arrays hold the bfloat16 bit patterns as uint16 (numpy
has no bfloat16).  Copies (write, gather) move raw values, so they are exact
for either dtype; attention converts what it reads to float64 first.
"""
from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------------
# element types
# --------------------------------------------------------------------------


def to_float64(raw: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of raw storage.

    bfloat16 is the upper half of an IEEE-754 binary32: the value of bit
    pattern ``b`` is the float32 whose bits are ``b << 16``.
    """
    if dtype == "f32":
        return np.asarray(raw, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        bits = np.asarray(raw, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


# --------------------------------------------------------------------------
# a1: slot mapping ("Build a Mini vLLM" section 2, append_slot)
# --------------------------------------------------------------------------


def slot_of(table_row, pos: int, block_size: int) -> int:
    """Flat pool slot of the token at logical position ``pos``."""
    block = int(table_row[pos // block_size])
    offset = pos % block_size
    return block * block_size + offset


def slot_mapping(block_tables, seq_lens, new_lens, block_size: int) -> np.ndarray:
    """Slots of this step's new tokens, in token order.

    Sequence ``b`` writes ``new_lens[b]`` tokens, the last ones of its
    ``seq_lens[b]`` tokens: positions ``seq_lens[b] - new_lens[b] ...
    seq_lens[b] - 1``.  A decode step writes one token at position
    ``seq_lens[b] - 1`` ("Build a Mini vLLM" section 4, decode_step: the new
    token's position is the length before the step, and the length is then
    incremented, so ``seq_lens`` here already counts it).
    """
    out = []
    for b in range(len(seq_lens)):
        L, c = int(seq_lens[b]), int(new_lens[b])
        for i in range(c):
            out.append(slot_of(block_tables[b], L - c + i, block_size))
    return np.array(out, dtype=np.int64)


# --------------------------------------------------------------------------
# a2: the scatter write ("Day 16", What I learned 3: pool[slots] = k)
# --------------------------------------------------------------------------


def kv_write(k, v, slots, k_pool, v_pool):
    """Return copies of the pools with token ``t``'s K/V stored at ``slots[t]``.

    The pool is addressed through its flat view ``[num_blocks*block_size,
    n_kv, head_dim]``.  A negative slot marks a padding token that is not
    written (pages silent; the plainest reading of "no slot").
    """
    k_pool = np.array(k_pool, copy=True)
    v_pool = np.array(v_pool, copy=True)
    nb, bs = k_pool.shape[0], k_pool.shape[1]
    for t in range(len(slots)):
        s = int(slots[t])
        if s < 0:
            continue
        if s >= nb * bs:
            raise IndexError(f"slot {s} outside a pool of {nb * bs} slots")
        blk, off = divmod(s, bs)
        k_pool[blk, off] = k[t]
        v_pool[blk, off] = v[t]
    return k_pool, v_pool


def copy_blocks(k_pool, v_pool, pairs):
    """Return copies of the pools where, for each ``(src, dst)`` of
    ``pairs``, physical block ``dst`` holds the contents of block ``src``.

    This is the copy of copy-on-write prefix sharing ("Build a Mini vLLM",
    Key Takeaways 6: real engines share prefix blocks and copy a shared
    block before a sequence writes into it).  All copies read the pools as
    they were before the call, so the result does not depend on the order
    of the pairs.  A pair with an id outside ``[0, num_blocks)`` is skipped
    (pages silent; the kernels report and skip it too).
    """
    src_k = np.array(k_pool, copy=True)
    src_v = np.array(v_pool, copy=True)
    k_out = np.array(k_pool, copy=True)
    v_out = np.array(v_pool, copy=True)
    nb = k_out.shape[0]
    for s, d in np.asarray(pairs, dtype=np.int64).reshape(-1, 2):
        if not (0 <= s < nb and 0 <= d < nb):
            continue
        k_out[d] = src_k[s]
        v_out[d] = src_v[s]
    return k_out, v_out


# --------------------------------------------------------------------------
# the block-table gather ("Build a Mini vLLM" section 3, gather_kv)
# --------------------------------------------------------------------------


def gather_kv(pool, table_row, seq_len: int) -> np.ndarray:
    """The sequence's ``seq_len`` tokens in logical order: [seq_len, n_kv, hd].

    Logical block ``j`` is physical block ``table_row[j]``; concatenating the
    blocks in table order and keeping the first ``seq_len`` rows gives the
    contiguous history.  Table entries past ``ceil(seq_len/block_size)``
    are never read.
    """
    bs = pool.shape[1]
    nblk = -(-int(seq_len) // bs)
    rows = [pool[int(table_row[j])] for j in range(nblk)]
    if not rows:
        return np.zeros((0,) + tuple(pool.shape[2:]), dtype=pool.dtype)
    return np.concatenate(rows, axis=0)[: int(seq_len)]


# --------------------------------------------------------------------------
# attention ("Build a Mini vLLM" section 3, paged_attention)
# --------------------------------------------------------------------------


def kv_head_of(h: int, n_heads: int, n_kv: int) -> int:
    """KV head shared by query head ``h``.

    ``repeat_interleave(REP)`` over the KV-head axis gives query head ``h``
    the copy of KV head ``h // REP``, ``REP = n_heads / n_kv`` ("Build a Mini
    vLLM" section 3; "nano-vLLM", How it works: each group of query heads is
    reshaped onto its shared K/V head).
    """
    return h // (n_heads // n_kv)


def scores(q_vec: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """Scaled dot products ``scale * q . k_j`` for every key row j."""
    return scale * (K @ q_vec)


def attend(q_vec: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Softmax attention of one query over L keys (float64).

    Returns ``(o, p)``: the output ``sum_j p_j V_j`` and the probabilities
    ``p = softmax(scale * K q)``, computed with the row maximum subtracted.
    With no keys the output is zero (pages silent; plainest reading).
    """
    if K.shape[0] == 0:
        return np.zeros(V.shape[1], dtype=np.float64), np.zeros(0, dtype=np.float64)
    s = scores(q_vec, K, scale)
    e = np.exp(s - s.max())
    p = e / e.sum()
    return p @ V, p


def causal_last_key(seq_len: int, chunk: int, i: int) -> int:
    """Last key position (inclusive) that chunk query ``i`` may attend to.

    The chunk holds the last ``chunk`` tokens of a ``seq_len``-token
    sequence, so query ``i`` sits at position ``seq_len - chunk + i`` and
    sees keys ``0 .. seq_len - chunk + i`` (the ``triu(1)`` mask of
    "Build a Mini vLLM" section 4 masks keys strictly after the query).
    """
    return seq_len - chunk + i


def _attend_heads(q_rows, Kc, Vc, n_kv: int, scale: float):
    """All query heads of one token against contiguous K/V [L, n_kv, hd]."""
    H, hd = q_rows.shape
    out = np.zeros((H, hd), dtype=np.float64)
    for h in range(H):
        g = kv_head_of(h, H, n_kv)
        out[h], _ = attend(q_rows[h], Kc[:, g, :], Vc[:, g, :], scale)
    return out


def paged_attention_decode(q, k_pool, v_pool, block_tables, seq_lens, scale, dtype, rows=None):
    """Decode attention: one query token per sequence over its paged history.

    ``q[b]`` ([n_heads, hd]) attends to all ``seq_lens[b]`` tokens of
    sequence ``b``, which include the token written this step ("Build a Mini
    vLLM" section 4: the new token's K/V is written before the gather).
    Returns float64 ``[B, n_heads, hd]`` (only ``rows`` are computed when
    given; the others are left zero).
    """
    B = len(seq_lens)
    H, hd = q.shape[1], q.shape[2]
    n_kv = k_pool.shape[2]
    out = np.zeros((B, H, hd), dtype=np.float64)
    for b in (range(B) if rows is None else rows):
        L = int(seq_lens[b])
        Kc = to_float64(gather_kv(k_pool, block_tables[b], L), dtype)
        Vc = to_float64(gather_kv(v_pool, block_tables[b], L), dtype)
        out[b] = _attend_heads(to_float64(q[b], dtype), Kc, Vc, n_kv, scale)
    return out


def paged_attention_prefill(q, cu_q_lens, k_pool, v_pool, block_tables, seq_lens, scale,
                            dtype, rows=None):
    """Causal attention of each sequence's query chunk over its paged history.

    Sequence ``b`` owns query rows ``cu_q_lens[b] .. cu_q_lens[b+1]-1``
    (``c`` of them); its ``seq_lens[b]`` tokens include the chunk, whose K/V
    was written first.  Query ``i`` attends keys ``0 .. causal_last_key``.
    Returns float64 ``[total_q, n_heads, hd]`` (only sequences in ``rows``
    when given).
    """
    B = len(seq_lens)
    T = int(cu_q_lens[B])
    H, hd = q.shape[1], q.shape[2]
    n_kv = k_pool.shape[2]
    out = np.zeros((T, H, hd), dtype=np.float64)
    for b in (range(B) if rows is None else rows):
        L = int(seq_lens[b])
        lo, hi = int(cu_q_lens[b]), int(cu_q_lens[b + 1])
        c = hi - lo
        Kc = to_float64(gather_kv(k_pool, block_tables[b], L), dtype)
        Vc = to_float64(gather_kv(v_pool, block_tables[b], L), dtype)
        for i in range(c):
            last = causal_last_key(L, c, i)
            out[lo + i] = _attend_heads(to_float64(q[lo + i], dtype), Kc[: last + 1],
                                        Vc[: last + 1], n_kv, scale)
    return out


# --------------------------------------------------------------------------
# a4: split-KV partials and their merge (online-softmax identity)
# --------------------------------------------------------------------------


def partial_attention(q_vec, K, V, scale):
    """Normalised output, maximum score and exp-sum over one key partition.

    ``m = max_j s_j``, ``l = sum_j exp(s_j - m)``,
    ``o = sum_j exp(s_j - m) V_j / l``.
    """
    s = scores(q_vec, K, scale)
    m = s.max()
    e = np.exp(s - m)
    l = e.sum()
    return (e @ V) / l, m, l


def merge_partials(parts):
    """Combine partition results ``(o_s, m_s, l_s)`` into the full softmax.

    With ``M = max_s m_s`` and ``w_s = exp(m_s - M) * l_s`` the full output
    is ``sum_s w_s o_s / sum_s w_s``: each partition's exp-sum is rescaled
    to the common maximum, which is exactly the softmax over the union.
    """
    M = max(m for _, m, _ in parts)
    w = np.array([np.exp(m - M) * l for _, m, l in parts])
    o = sum(wi * oi for wi, (oi, _, _) in zip(w, parts))
    return o / w.sum()


def paged_attention_decode_split(q, k_pool, v_pool, block_tables, seq_lens, scale, dtype,
                                 partition_tokens: int, rows=None):
    """Decode attention computed as key partitions of ``partition_tokens``
    tokens (partition ``s`` covers keys ``[s*P, min((s+1)*P, L))``) merged
    with :func:`merge_partials`.  Equal to :func:`paged_attention_decode` in
    real arithmetic."""
    B = len(seq_lens)
    H, hd = q.shape[1], q.shape[2]
    n_kv = k_pool.shape[2]
    P = int(partition_tokens)
    out = np.zeros((B, H, hd), dtype=np.float64)
    for b in (range(B) if rows is None else rows):
        L = int(seq_lens[b])
        if L == 0:
            continue
        Kc = to_float64(gather_kv(k_pool, block_tables[b], L), dtype)
        Vc = to_float64(gather_kv(v_pool, block_tables[b], L), dtype)
        qb = to_float64(q[b], dtype)
        for h in range(H):
            g = kv_head_of(h, H, n_kv)
            parts = [partial_attention(qb[h], Kc[lo:min(lo + P, L), g], Vc[lo:min(lo + P, L), g], scale)
                     for lo in range(0, L, P)]
            out[b, h] = merge_partials(parts)
    return out
