"""Plant plausible mistakes in the oracle (on the CPU) and check that the
pins catch each one: a pin set that passes a broken oracle pins nothing."""
import numpy as np
import pytest

import oracle.paged as op
from oracle_pins import ALL_PINS

_orig_copy = op.copy_blocks


def _wrong_group(h, n_heads, n_kv):           # h % n_kv instead of h // rep
    return h % n_kv


def _slot_swapped(table_row, pos, bs):        # offset and block index swapped
    return int(table_row[pos % len(table_row)]) * bs + pos // bs


def _slot_off_by_one(table_row, pos, bs):
    return int(table_row[pos // bs]) * bs + (pos + 1) % bs


def _causal_exclusive(seq_len, chunk, i):     # query does not see itself
    return seq_len - chunk + i - 1


def _causal_from_start(seq_len, chunk, i):    # chunk positions counted from 0
    return i


def _scores_unscaled(q_vec, K, scale):
    return K @ q_vec


def _scores_sqrt_scale(q_vec, K, scale):
    return np.sqrt(scale) * (K @ q_vec)


def _gather_off_by_one_len(pool, table_row, seq_len):
    bs = pool.shape[1]
    nblk = -(-int(seq_len) // bs)
    rows = [pool[int(table_row[j])] for j in range(nblk)]
    if not rows:
        return np.zeros((0,) + tuple(pool.shape[2:]), dtype=pool.dtype)
    return np.concatenate(rows, axis=0)[: max(int(seq_len) - 1, 1)]


def _merge_no_rescale(parts):
    w = np.array([l for _, _, l in parts])
    return sum(wi * oi for wi, (oi, _, _) in zip(w, parts)) / w.sum()


def _bf16_truncated_bits(raw, dtype):
    if dtype == "bf16":
        bits = np.asarray(raw, dtype=np.uint16).astype(np.uint32) << np.uint32(15)
        return bits.view(np.float32).astype(np.float64)
    return np.asarray(raw, dtype=np.float32).astype(np.float64)


def _copy_reversed(k_pool, v_pool, pairs):      # dst copied onto src
    return _orig_copy(k_pool, v_pool, np.asarray(pairs).reshape(-1, 2)[:, ::-1])


def _copy_in_place(k_pool, v_pool, pairs):      # later pairs see earlier copies
    k, v = np.array(k_pool, copy=True), np.array(v_pool, copy=True)
    for s, d in np.asarray(pairs).reshape(-1, 2):
        if 0 <= s < k.shape[0] and 0 <= d < k.shape[0]:
            k[d], v[d] = k[s], v[s]
    return k, v


def _copy_k_only(k_pool, v_pool, pairs):        # V left behind
    k, _ = _orig_copy(k_pool, v_pool, pairs)
    return k, np.array(v_pool, copy=True)


MUTANTS = [
    ("kv_head_of", _wrong_group),
    ("slot_of", _slot_swapped),
    ("slot_of", _slot_off_by_one),
    ("causal_last_key", _causal_exclusive),
    ("causal_last_key", _causal_from_start),
    ("scores", _scores_unscaled),
    ("scores", _scores_sqrt_scale),
    ("gather_kv", _gather_off_by_one_len),
    ("merge_partials", _merge_no_rescale),
    ("to_float64", _bf16_truncated_bits),
    ("copy_blocks", _copy_reversed),
    ("copy_blocks", _copy_in_place),
    ("copy_blocks", _copy_k_only),
]


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=[m.__name__ for _, m in MUTANTS])
def test_pins_catch_mutant(monkeypatch, name, mutant):
    import oracle
    monkeypatch.setattr(op, name, mutant)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, mutant)
    failed = []
    for pin in ALL_PINS:
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {mutant.__name__}"
