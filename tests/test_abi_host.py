"""The C-ABI library loads, exports every entry point that include/pkv.h
declares, and rejects bad arguments on the host before any launch (these
calls never touch a GPU, so they run on CPU-only machines)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_write_gb300 import build
    build.build()
    import paged_kv_cache_write_gb300 as m
    return m


def test_header_declares_entry_points():
    names = _declared()
    for need in ("pkv_slot_mapping", "pkv_kv_write", "pkv_kv_gather", "pkv_paged_attention_decode",
                 "pkv_paged_attention_prefill", "pkv_decode_workspace_bytes", "pkv_status_string"):
        assert need in names


def test_library_exports_every_declared_symbol(pkv):
    lib = ctypes.CDLL(pkv.library_path)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_device_error_bits_match_the_header(pkv):
    """The binding's names for the device error bits are the header's
    PKV_DEVERR_* values, one bit each."""
    text = open(HEADER).read()
    bits = {m.group(1).lower(): int(m.group(2))
            for m in re.finditer(r"#define PKV_DEVERR_([A-Z_]+)\s+(\d+)", text)}
    assert bits == pkv.DEVERR
    assert all(v & (v - 1) == 0 for v in bits.values())
    assert len(set(bits.values())) == len(bits)


def test_status_strings(pkv):
    assert pkv.status_string(0) == "ok"
    for s in range(1, 9):
        assert pkv.status_string(s) not in ("ok", "unknown status")
    assert pkv.status_string(1234) == "unknown status"
    assert pkv.abi_version() == 1


def _desc(pkv, **kw):
    d = dict(num_blocks=8, block_size=16, n_kv=2, head_dim=64, dtype=1)
    d.update(kw)
    return pkv.PoolDesc(**d)


FAKE = 0x10000  # a 16-byte-aligned non-null address; never dereferenced


def test_kv_write_host_checks(pkv):
    lib = pkv.lib
    d = _desc(pkv)
    by = ctypes.byref
    assert lib.pkv_kv_write(FAKE, FAKE, FAKE, 4, FAKE, FAKE, None, None, None) == 1
    assert lib.pkv_kv_write(FAKE, FAKE, FAKE, 4, FAKE, FAKE, by(_desc(pkv, dtype=7)), None, None) == 3
    assert lib.pkv_kv_write(FAKE, FAKE, FAKE, -1, FAKE, FAKE, by(d), None, None) == 2
    assert lib.pkv_kv_write(None, FAKE, FAKE, 4, FAKE, FAKE, by(d), None, None) == 1
    assert lib.pkv_kv_write(FAKE + 4, FAKE, FAKE, 4, FAKE, FAKE, by(d), None, None) == 4
    # row of 1 x 6 fp32 = 24 bytes is not a multiple of 16
    assert lib.pkv_kv_write(FAKE, FAKE, FAKE, 4, FAKE, FAKE,
                            by(_desc(pkv, n_kv=1, head_dim=6, dtype=0)), None, None) == 4
    assert lib.pkv_kv_write(None, None, None, 0, None, None, by(d), None, None) == 0
    assert lib.pkv_kv_write(FAKE, FAKE, FAKE, 4, FAKE, FAKE, by(_desc(pkv, num_blocks=0)),
                            None, None) == 2


def test_copy_blocks_host_checks(pkv):
    lib = pkv.lib
    d = _desc(pkv)
    by = ctypes.byref
    assert lib.pkv_copy_blocks(FAKE, FAKE, None, FAKE, 3, None, None) == 1
    assert lib.pkv_copy_blocks(FAKE, FAKE, by(d), FAKE, -1, None, None) == 2
    assert lib.pkv_copy_blocks(FAKE, FAKE, by(d), None, 3, None, None) == 1
    assert lib.pkv_copy_blocks(FAKE + 8, FAKE, by(d), FAKE, 3, None, None) == 4
    assert lib.pkv_copy_blocks(FAKE, FAKE, by(_desc(pkv, dtype=9)), FAKE, 3, None, None) == 3
    assert lib.pkv_copy_blocks(None, None, by(d), None, 0, None, None) == 0


def test_selftest_bounded_wait_host_checks(pkv):
    lib = pkv.lib
    assert lib.pkv_selftest_bounded_wait(0, FAKE, None) == 5
    assert lib.pkv_selftest_bounded_wait(100, None, None) == 1


def test_slot_mapping_host_checks(pkv):
    lib = pkv.lib
    assert lib.pkv_slot_mapping(FAKE, 4, FAKE, FAKE, -1, 3, 16, 8, FAKE, None, None) == 2
    assert lib.pkv_slot_mapping(FAKE, 4, FAKE, FAKE, 2, 3, 0, 8, FAKE, None, None) == 2
    assert lib.pkv_slot_mapping(None, 4, FAKE, FAKE, 2, 3, 16, 8, FAKE, None, None) == 1
    assert lib.pkv_slot_mapping(FAKE, 0, FAKE, FAKE, 2, 3, 16, 8, FAKE, None, None) == 2
    assert lib.pkv_slot_mapping(None, 0, None, None, 0, 0, 16, 8, None, None, None) == 0


def _decode(pkv, **over):
    a = dict(q=FAKE, B=2, H=8, k=FAKE, v=FAKE, desc=_desc(pkv), bt=FAKE, W=4, sl=FAKE, maxlen=64,
             scale=0.125, max_ctas=0, out=FAKE, ws=FAKE, wsb=1 << 40, err=None)
    a.update(over)
    return pkv.lib.pkv_paged_attention_decode(a["q"], a["B"], a["H"], a["k"], a["v"],
                                              ctypes.byref(a["desc"]), a["bt"], a["W"], a["sl"],
                                              a["maxlen"], a["scale"], a["max_ctas"], a["out"],
                                              a["ws"], a["wsb"], a["err"], None)


def test_decode_host_checks(pkv):
    assert _decode(pkv, q=None) == 1
    assert _decode(pkv, H=7) == 2                      # n_heads % n_kv
    assert _decode(pkv, maxlen=65) == 2                # > W * block_size
    assert _decode(pkv, scale=float("nan")) == 5
    assert _decode(pkv, scale=-0.5) == 5                # the score scale must be positive
    assert _decode(pkv, scale=0.0) == 5
    assert _decode(pkv, max_ctas=-1) == 5
    assert _decode(pkv, ws=None) == 6
    assert _decode(pkv, wsb=16) == 6
    assert _decode(pkv, out=FAKE + 8) == 4
    assert _decode(pkv, desc=_desc(pkv, block_size=8), maxlen=32) == 7  # attention needs 16
    assert _decode(pkv, desc=_desc(pkv, head_dim=48)) == 7
    assert _decode(pkv, H=2 * 17) == 7                 # 17 query heads per KV head
    assert _decode(pkv, B=0) == 0


def _prefix(pkv, P, **over):
    a = dict(q=FAKE, B=2, H=8, k=FAKE, v=FAKE, desc=_desc(pkv), bt=FAKE, W=4, sl=FAKE, maxlen=64,
             scale=0.125, max_ctas=0, out=FAKE, ws=FAKE, wsb=1 << 40, err=None)
    a.update(over)
    return pkv.lib.pkv_paged_attention_decode_shared_prefix(
        a["q"], a["B"], a["H"], a["k"], a["v"], ctypes.byref(a["desc"]), a["bt"], a["W"], a["sl"],
        a["maxlen"], P, a["scale"], a["max_ctas"], a["out"], a["ws"], a["wsb"], a["err"], None)


def test_decode_shared_prefix_host_checks(pkv):
    assert _prefix(pkv, -1) == 5
    assert _prefix(pkv, 5) == 5                        # more shared blocks than a table row has
    assert _prefix(pkv, 2, q=None) == 1
    assert _prefix(pkv, 2, H=7) == 2
    assert _prefix(pkv, 2, ws=None) == 6
    assert _prefix(pkv, 2, wsb=16) == 6
    assert _prefix(pkv, 2, desc=_desc(pkv, head_dim=48)) == 7
    assert _prefix(pkv, 2, B=0) == 0


def _append(pkv, **over):
    a = dict(q=FAKE, kn=FAKE, vn=FAKE, B=2, H=8, k=FAKE, v=FAKE, desc=_desc(pkv), bt=FAKE, W=4,
             sl=FAKE, maxlen=64, scale=0.125, max_ctas=0, out=FAKE, ws=FAKE, wsb=1 << 40, err=None)
    a.update(over)
    return pkv.lib.pkv_paged_attention_decode_append(
        a["q"], a["kn"], a["vn"], a["B"], a["H"], a["k"], a["v"], ctypes.byref(a["desc"]), a["bt"],
        a["W"], a["sl"], a["maxlen"], a["scale"], a["max_ctas"], a["out"], a["ws"], a["wsb"],
        a["err"], None)


def test_decode_append_host_checks(pkv):
    assert _append(pkv, kn=None) == 1
    assert _append(pkv, vn=None) == 1
    assert _append(pkv, kn=FAKE + 8) == 4
    assert _append(pkv, vn=FAKE + 4) == 4
    assert _append(pkv, q=None) == 1
    assert _append(pkv, H=7) == 2
    assert _append(pkv, scale=0.0) == 5
    assert _append(pkv, ws=None) == 6
    assert _append(pkv, desc=_desc(pkv, head_dim=48)) == 7
    assert _append(pkv, B=0, kn=None, vn=None) == 0


def test_prefill_host_checks(pkv):
    lib = pkv.lib
    d = _desc(pkv)
    call = lambda **o: lib.pkv_paged_attention_prefill(
        o.get("q", FAKE), o.get("cu", FAKE), o.get("B", 2), o.get("T", 10), o.get("mq", 5), 8, FAKE,
        FAKE, ctypes.byref(o.get("desc", d)), FAKE, 4, FAKE, o.get("ml", 64), 0.125,
        o.get("out", FAKE), None, 0, None, None)
    assert call(cu=None) == 1
    assert call(mq=11) == 2
    assert call(mq=0) == 2
    assert call(T=-1) == 2
    assert call(desc=_desc(pkv, head_dim=40)) == 7
    assert call(B=0) == 0
    assert call(T=0) == 0


def test_workspace_bytes_positive(pkv):
    assert pkv.decode_workspace_bytes(4, 8, 16, 100) > 0
    assert pkv.decode_workspace_bytes(0, 8, 16, 0) > 0


def _plan(pkv, **over):
    a = dict(B=2, H=8, desc=_desc(pkv), W=4, sl=FAKE, maxlen=64, P=0, max_ctas=0, ws=FAKE,
             wsb=1 << 40, err=None)
    a.update(over)
    return pkv.lib.pkv_decode_plan(a["B"], a["H"], ctypes.byref(a["desc"]), a["W"], a["sl"],
                                   a["maxlen"], a["P"], a["max_ctas"], a["ws"], a["wsb"],
                                   a["err"], None)


def test_decode_plan_host_checks(pkv):
    assert _plan(pkv, sl=None) == 1
    assert _plan(pkv, H=7) == 2                        # n_heads % n_kv
    assert _plan(pkv, maxlen=65) == 2                  # > W * block_size
    assert _plan(pkv, B=-1) == 2
    assert _plan(pkv, max_ctas=-1) == 5
    assert _plan(pkv, ws=None) == 6
    assert _plan(pkv, wsb=16) == 6
    assert _plan(pkv, ws=FAKE + 8) == 4
    assert _plan(pkv, desc=_desc(pkv, head_dim=48)) == 7
    assert _plan(pkv, desc=_desc(pkv, dtype=9)) == 3
    assert _plan(pkv, P=-1) == 5
    assert _plan(pkv, P=5) == 5                        # more shared blocks than a table row has
    assert _plan(pkv, B=0, sl=None) == 0


def _planned(pkv, **over):
    a = dict(q=FAKE, kn=None, vn=None, B=2, H=8, k=FAKE, v=FAKE, desc=_desc(pkv), bt=FAKE, W=4,
             sl=FAKE, maxlen=64, P=0, scale=0.125, max_ctas=0, out=FAKE, ws=FAKE, wsb=1 << 40,
             err=None)
    a.update(over)
    return pkv.lib.pkv_paged_attention_decode_planned(
        a["q"], a["kn"], a["vn"], a["B"], a["H"], a["k"], a["v"], ctypes.byref(a["desc"]), a["bt"],
        a["W"], a["sl"], a["maxlen"], a["P"], a["scale"], a["max_ctas"], a["out"], a["ws"],
        a["wsb"], a["err"], None)


def test_decode_planned_host_checks(pkv):
    assert _planned(pkv, kn=FAKE) == 1                 # k_new without v_new
    assert _planned(pkv, vn=FAKE) == 1
    assert _planned(pkv, kn=FAKE, vn=FAKE + 4) == 4
    assert _planned(pkv, q=None) == 1
    assert _planned(pkv, bt=None) == 1
    assert _planned(pkv, H=7) == 2
    assert _planned(pkv, scale=0.0) == 5
    assert _planned(pkv, ws=None) == 6
    assert _planned(pkv, wsb=16) == 6
    assert _planned(pkv, desc=_desc(pkv, head_dim=48)) == 7
    assert _planned(pkv, P=5) == 5
    assert _planned(pkv, B=0) == 0
