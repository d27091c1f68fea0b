"""Paged KV cache write and paged attention for GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/pkv.h`` (``libpkv.so``,
built in-tree by ``paged_kv_cache_write_gb300.build``).  Each function here
has the name of the C entry point without its ``pkv_`` prefix and only
marshals arguments: it checks tensor devices, dtypes and layouts, passes
raw device pointers and the current CUDA stream, and raises on a non-zero
status.  Every step of the computation runs in the library's CUDA kernels;
there is no CPU or PyTorch fallback: the library is loaded on first use
and every call raises ImportError if it has not been built.

PyTorch is used only for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "lib", "library_path", "PoolDesc", "PKV_F32", "PKV_BF16", "DEVERR",
    "slot_mapping", "kv_write", "kv_gather", "copy_blocks", "decode_workspace_bytes",
    "paged_attention_decode", "paged_attention_decode_append",
    "decode_shared_prefix_workspace_bytes", "paged_attention_decode_shared_prefix",
    "decode_plan", "paged_attention_decode_planned", "prefill_workspace_bytes",
    "paged_attention_prefill", "status_string", "abi_version", "paged_attention_decode_noalloc",
    "selftest_bounded_wait",
]

HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(HERE, "libpkv.so")

PKV_F32 = 0
PKV_BF16 = 1
DEVERR = {"block_id": 1, "slot": 2, "table_width": 4, "length": 8, "timeout": 16, "prefix": 32,
          "plan": 64}


class PoolDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("n_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


_lib = None
_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t
_f = ctypes.c_float
_desc = ctypes.POINTER(PoolDesc)


def _load():
    """Load libpkv.so once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(library_path):
        raise ImportError(
            f"{library_path} is missing: build it with "
            "`python -m paged_kv_cache_write_gb300.build` (needs nvcc with sm_103a support)")
    L = ctypes.CDLL(library_path)
    L.pkv_status_string.restype = ctypes.c_char_p
    L.pkv_status_string.argtypes = [_i32]
    L.pkv_abi_version.restype = _i32
    L.pkv_abi_version.argtypes = []
    L.pkv_slot_mapping.restype = _i32
    L.pkv_slot_mapping.argtypes = [_p, _i32, _p, _p, _i32, _i32, _i32, _i32, _p, _p, _p]
    L.pkv_kv_write.restype = _i32
    L.pkv_kv_write.argtypes = [_p, _p, _p, _i32, _p, _p, _desc, _p, _p]
    L.pkv_selftest_bounded_wait.restype = _i32
    L.pkv_selftest_bounded_wait.argtypes = [_i32, _p, _p]
    L.pkv_copy_blocks.restype = _i32
    L.pkv_copy_blocks.argtypes = [_p, _p, _desc, _p, _i32, _p, _p]
    L.pkv_kv_gather.restype = _i32
    L.pkv_kv_gather.argtypes = [_p, _p, _desc, _p, _i32, _p, _p, _i32, _i32, _p, _p, _p, _p]
    L.pkv_decode_workspace_bytes.restype = _sz
    L.pkv_decode_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32]
    L.pkv_paged_attention_decode.restype = _i32
    L.pkv_paged_attention_decode.argtypes = [_p, _i32, _i32, _p, _p, _desc, _p, _i32, _p, _i32,
                                             _f, _i32, _p, _p, _sz, _p, _p]
    L.pkv_decode_shared_prefix_workspace_bytes.restype = _sz
    L.pkv_decode_shared_prefix_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, _i32]
    L.pkv_paged_attention_decode_shared_prefix.restype = _i32
    L.pkv_paged_attention_decode_shared_prefix.argtypes = [_p, _i32, _i32, _p, _p, _desc, _p, _i32,
                                                           _p, _i32, _i32, _f, _i32, _p, _p, _sz,
                                                           _p, _p]
    L.pkv_paged_attention_decode_append.restype = _i32
    L.pkv_paged_attention_decode_append.argtypes = [_p, _p, _p, _i32, _i32, _p, _p, _desc, _p,
                                                    _i32, _p, _i32, _f, _i32, _p, _p, _sz, _p, _p]
    L.pkv_decode_plan.restype = _i32
    L.pkv_decode_plan.argtypes = [_i32, _i32, _desc, _i32, _p, _i32, _i32, _i32, _p, _sz, _p, _p]
    L.pkv_paged_attention_decode_planned.restype = _i32
    L.pkv_paged_attention_decode_planned.argtypes = [_p, _p, _p, _i32, _i32, _p, _p, _desc, _p,
                                                     _i32, _p, _i32, _i32, _f, _i32, _p, _p, _sz,
                                                     _p, _p]
    L.pkv_prefill_workspace_bytes.restype = _sz
    L.pkv_prefill_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32, _i32]
    L.pkv_paged_attention_prefill.restype = _i32
    L.pkv_paged_attention_prefill.argtypes = [_p, _p, _i32, _i32, _i32, _i32, _p, _p, _desc, _p,
                                              _i32, _p, _i32, _f, _p, _p, _sz, _p, _p]
    _lib = L
    return L


def __getattr__(name):
    # `pkv.lib` loads the library on first access
    if name == "lib":
        return _load()
    raise AttributeError(name)


def status_string(status: int) -> str:
    return _load().pkv_status_string(int(status)).decode()


def abi_version() -> int:
    return int(_load().pkv_abi_version())


class PkvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {status_string(status)} (status {status})")
        self.status = status


def _check(fn: str, status: int):
    if status != 0:
        raise PkvError(fn, status)


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return PKV_F32
    if t == torch.bfloat16:
        return PKV_BF16
    raise TypeError(f"unsupported dtype {t}: float32 or bfloat16")


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _opt(t, name, dtype=None):
    return None if t is None else _dev(t, name, dtype)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def pool_desc(k_pool: torch.Tensor) -> PoolDesc:
    if k_pool.dim() != 4:
        raise ValueError("pool must be [num_blocks, block_size, n_kv, head_dim]")
    nb, bs, nkv, hd = k_pool.shape
    return PoolDesc(nb, bs, nkv, hd, _dtype_code(k_pool.dtype))


def slot_mapping(block_tables, seq_lens, cu_new_lens, num_tokens: int, block_size: int,
                 num_blocks: int, *, out=None, err=None, stream=None):
    """int64 [num_tokens] flat pool slot of each token written this step."""
    B, W = block_tables.shape
    if out is None:
        out = torch.empty(num_tokens, dtype=torch.int64, device=block_tables.device)
    _check("pkv_slot_mapping", _load().pkv_slot_mapping(
        _dev(block_tables, "block_tables", torch.int32), W, _dev(seq_lens, "seq_lens", torch.int32),
        _dev(cu_new_lens, "cu_new_lens", torch.int32), B, int(num_tokens), int(block_size),
        int(num_blocks), _dev(out, "out", torch.int64), _opt(err, "err", torch.int32),
        _stream(stream)))
    return out


def kv_write(k, v, slot_mapping, k_pool, v_pool, *, err=None, stream=None):
    """Scatter k/v [T, n_kv, head_dim] into the pools at slot_mapping [T]."""
    desc = pool_desc(k_pool)
    if tuple(v_pool.shape) != tuple(k_pool.shape) or v_pool.dtype != k_pool.dtype:
        raise ValueError("k_pool and v_pool must have the same shape and dtype")
    T = k.shape[0]
    if tuple(k.shape) != (T, desc.n_kv, desc.head_dim) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k, v must be [T, n_kv, head_dim] matching the pool")
    if slot_mapping.shape[0] != T:
        raise ValueError("slot_mapping must have one entry per token")
    _check("pkv_kv_write", _load().pkv_kv_write(
        _dev(k, "k", k_pool.dtype), _dev(v, "v", k_pool.dtype),
        _dev(slot_mapping, "slot_mapping", torch.int64), T, _dev(k_pool, "k_pool"),
        _dev(v_pool, "v_pool"), ctypes.byref(desc), _opt(err, "err", torch.int32),
        _stream(stream)))


def selftest_bounded_wait(err, polls: int = 4096, *, stream=None):
    """Run one wait that nothing completes, bounded by ``polls``; the
    kernel ORs the timeout bit into the device int32 ``err`` and returns."""
    _check("pkv_selftest_bounded_wait", _load().pkv_selftest_bounded_wait(
        int(polls), _dev(err, "err", torch.int32), _stream(stream)))


def copy_blocks(k_pool, v_pool, block_pairs, *, err=None, stream=None):
    """Copy whole blocks of both pools: for each row (src, dst) of the
    int32 [n, 2] ``block_pairs``, block dst becomes a copy of block src
    (copy-on-write).  Destinations must be distinct and not sources."""
    desc = pool_desc(k_pool)
    if block_pairs.dim() != 2 or block_pairs.shape[1] != 2:
        raise ValueError("block_pairs must be [n, 2]")
    _check("pkv_copy_blocks", _load().pkv_copy_blocks(
        _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"), ctypes.byref(desc),
        _dev(block_pairs, "block_pairs", torch.int32), int(block_pairs.shape[0]),
        _opt(err, "err", torch.int32), _stream(stream)))


def kv_gather(k_pool, v_pool, block_tables, seq_lens, cu_seq_lens, total_tokens: int, *,
              k_out=None, v_out=None, err=None, stream=None):
    """Contiguous [total_tokens, n_kv, head_dim] K and V in logical order."""
    desc = pool_desc(k_pool)
    B, W = block_tables.shape
    shape = (int(total_tokens), desc.n_kv, desc.head_dim)
    if k_out is None:
        k_out = torch.empty(shape, dtype=k_pool.dtype, device=k_pool.device)
    if v_out is None:
        v_out = torch.empty(shape, dtype=k_pool.dtype, device=k_pool.device)
    _check("pkv_kv_gather", _load().pkv_kv_gather(
        _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"), ctypes.byref(desc),
        _dev(block_tables, "block_tables", torch.int32), W, _dev(seq_lens, "seq_lens", torch.int32),
        _dev(cu_seq_lens, "cu_seq_lens", torch.int32), B, int(total_tokens),
        _dev(k_out, "k_out", k_pool.dtype), _dev(v_out, "v_out", k_pool.dtype),
        _opt(err, "err", torch.int32), _stream(stream)))
    return k_out, v_out


def decode_workspace_bytes(num_seqs, n_heads, head_dim, max_seq_len, max_ctas=0, block_size=16):
    return int(_load().pkv_decode_workspace_bytes(num_seqs, n_heads, head_dim, max_seq_len, max_ctas,
                                              block_size))


def paged_attention_decode(q, k_pool, v_pool, block_tables, seq_lens, scale: float,
                           max_seq_len: int | None = None, *, out=None, workspace=None,
                           max_ctas: int = 0, err=None, stream=None):
    """Decode attention [B, n_heads, head_dim] over the paged history.

    ``max_seq_len`` is a host-side bound on ``seq_lens`` (reading it from
    the device synchronises; pass it when known).  ``workspace`` is a
    device uint8 tensor of at least ``decode_workspace_bytes(...)`` bytes
    (allocated here when omitted).
    """
    desc = pool_desc(k_pool)
    B, H, hd = q.shape
    W = block_tables.shape[1]
    if max_seq_len is None:
        max_seq_len = int(seq_lens.max().item()) if B else 0
    if out is None:
        out = torch.empty_like(q)
    need = decode_workspace_bytes(B, H, hd, max_seq_len, max_ctas, desc.block_size)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check("pkv_paged_attention_decode", _load().pkv_paged_attention_decode(
        _dev(q, "q", k_pool.dtype), B, H, _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"),
        ctypes.byref(desc), _dev(block_tables, "block_tables", torch.int32), W,
        _dev(seq_lens, "seq_lens", torch.int32), int(max_seq_len), float(scale), int(max_ctas),
        _dev(out, "out", k_pool.dtype), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _opt(err, "err", torch.int32),
        _stream(stream)))
    return out


def decode_shared_prefix_workspace_bytes(num_seqs, n_heads, head_dim, max_seq_len,
                                         shared_prefix_blocks, max_ctas=0, block_size=16):
    return int(_load().pkv_decode_shared_prefix_workspace_bytes(
        num_seqs, n_heads, head_dim, max_seq_len, shared_prefix_blocks, max_ctas, block_size))


def paged_attention_decode_shared_prefix(q, k_pool, v_pool, block_tables, seq_lens, scale: float,
                                         shared_prefix_blocks: int,
                                         max_seq_len: int | None = None, *, out=None,
                                         workspace=None, max_ctas: int = 0, err=None,
                                         stream=None):
    """Decode attention where the first ``shared_prefix_blocks`` table
    entries of every sequence are the same blocks, read once per step."""
    desc = pool_desc(k_pool)
    B, H, hd = q.shape
    W = block_tables.shape[1]
    if max_seq_len is None:
        max_seq_len = int(seq_lens.max().item()) if B else 0
    if out is None:
        out = torch.empty_like(q)
    need = decode_shared_prefix_workspace_bytes(B, H, hd, max_seq_len, shared_prefix_blocks,
                                                max_ctas, desc.block_size)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check("pkv_paged_attention_decode_shared_prefix",
           _load().pkv_paged_attention_decode_shared_prefix(
               _dev(q, "q", k_pool.dtype), B, H, _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"),
               ctypes.byref(desc), _dev(block_tables, "block_tables", torch.int32), W,
               _dev(seq_lens, "seq_lens", torch.int32), int(max_seq_len),
               int(shared_prefix_blocks), float(scale), int(max_ctas),
               _dev(out, "out", k_pool.dtype), _dev(workspace, "workspace"),
               workspace.numel() * workspace.element_size(), _opt(err, "err", torch.int32),
               _stream(stream)))
    return out


def paged_attention_decode_append(q, k_new, v_new, k_pool, v_pool, block_tables, seq_lens,
                                  scale: float, max_seq_len: int | None = None, *, out=None,
                                  workspace=None, max_ctas: int = 0, err=None, stream=None):
    """Store this step's ``k_new``/``v_new`` [B, n_kv, head_dim] at each
    sequence's last position (``seq_lens[b] - 1``) and return decode
    attention [B, n_heads, head_dim] over the updated pages, in one launch.
    Same as ``kv_write`` at those slots followed by ``paged_attention_decode``.
    """
    desc = pool_desc(k_pool)
    B, H, hd = q.shape
    W = block_tables.shape[1]
    if k_new.shape != (B, desc.n_kv, hd) or v_new.shape != k_new.shape:
        raise ValueError(f"k_new/v_new must be {(B, desc.n_kv, hd)}")
    if max_seq_len is None:
        max_seq_len = int(seq_lens.max().item()) if B else 0
    if out is None:
        out = torch.empty_like(q)
    need = decode_workspace_bytes(B, H, hd, max_seq_len, max_ctas, desc.block_size)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check("pkv_paged_attention_decode_append", _load().pkv_paged_attention_decode_append(
        _dev(q, "q", k_pool.dtype), _dev(k_new, "k_new", k_pool.dtype),
        _dev(v_new, "v_new", k_pool.dtype), B, H, _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"),
        ctypes.byref(desc), _dev(block_tables, "block_tables", torch.int32), W,
        _dev(seq_lens, "seq_lens", torch.int32), int(max_seq_len), float(scale), int(max_ctas),
        _dev(out, "out", k_pool.dtype), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _opt(err, "err", torch.int32),
        _stream(stream)))
    return out


def decode_plan(k_pool, seq_lens, n_heads: int, max_blocks_per_seq: int, max_seq_len: int, *,
                workspace, shared_prefix_blocks: int = 0, max_ctas: int = 0, err=None,
                stream=None):
    """Split a decode step's blocks over the decode grid once, into
    ``workspace``, for every layer's ``paged_attention_decode_planned``
    (same lengths, tables, shapes, shared prefix and ``max_ctas`` until the
    step ends)."""
    desc = pool_desc(k_pool)
    B = seq_lens.shape[0]
    _check("pkv_decode_plan", _load().pkv_decode_plan(
        B, int(n_heads), ctypes.byref(desc), int(max_blocks_per_seq),
        _dev(seq_lens, "seq_lens", torch.int32), int(max_seq_len), int(shared_prefix_blocks),
        int(max_ctas),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _opt(err, "err", torch.int32), _stream(stream)))
    return workspace


def paged_attention_decode_planned(q, k_pool, v_pool, block_tables, seq_lens, scale: float,
                                   max_seq_len: int, *, workspace, k_new=None, v_new=None,
                                   shared_prefix_blocks: int = 0, out=None, max_ctas: int = 0,
                                   err=None, stream=None):
    """``paged_attention_decode`` (with ``k_new``/``v_new``,
    ``paged_attention_decode_append``; with ``shared_prefix_blocks``,
    ``paged_attention_decode_shared_prefix``) using the plan
    ``decode_plan`` left in ``workspace``."""
    desc = pool_desc(k_pool)
    B, H, hd = q.shape
    W = block_tables.shape[1]
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if k_new is not None and (k_new.shape != (B, desc.n_kv, hd) or v_new.shape != k_new.shape):
        raise ValueError(f"k_new/v_new must be {(B, desc.n_kv, hd)}")
    if out is None:
        out = torch.empty_like(q)
    _check("pkv_paged_attention_decode_planned", _load().pkv_paged_attention_decode_planned(
        _dev(q, "q", k_pool.dtype),
        None if k_new is None else _dev(k_new, "k_new", k_pool.dtype),
        None if v_new is None else _dev(v_new, "v_new", k_pool.dtype), B, H,
        _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"), ctypes.byref(desc),
        _dev(block_tables, "block_tables", torch.int32), W,
        _dev(seq_lens, "seq_lens", torch.int32), int(max_seq_len), int(shared_prefix_blocks),
        float(scale), int(max_ctas), _dev(out, "out", k_pool.dtype), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _opt(err, "err", torch.int32),
        _stream(stream)))
    return out


def prefill_workspace_bytes(num_seqs, total_q, n_heads, head_dim, max_seq_len):
    return int(_load().pkv_prefill_workspace_bytes(num_seqs, total_q, n_heads, head_dim, max_seq_len))


def paged_attention_prefill(q, cu_q_lens, k_pool, v_pool, block_tables, seq_lens, scale: float,
                            max_q_len: int | None = None, max_seq_len: int | None = None, *,
                            out=None, workspace=None, err=None, stream=None):
    """Causal chunked-prefill attention [total_q, n_heads, head_dim]."""
    desc = pool_desc(k_pool)
    T, H, hd = q.shape
    B, W = block_tables.shape
    if max_q_len is None:
        max_q_len = int((cu_q_lens[1:] - cu_q_lens[:-1]).max().item()) if B else 0
    if max_seq_len is None:
        max_seq_len = int(seq_lens.max().item()) if B else 0
    if out is None:
        out = torch.empty_like(q)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size())
    _check("pkv_paged_attention_prefill", _load().pkv_paged_attention_prefill(
        _dev(q, "q", k_pool.dtype), _dev(cu_q_lens, "cu_q_lens", torch.int32), B, T,
        int(max_q_len), H, _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"), ctypes.byref(desc),
        _dev(block_tables, "block_tables", torch.int32), W,
        _dev(seq_lens, "seq_lens", torch.int32), int(max_seq_len), float(scale),
        _dev(out, "out", k_pool.dtype), ws_ptr, ws_bytes, _opt(err, "err", torch.int32),
        _stream(stream)))
    return out


def paged_attention_decode_noalloc(q, k_pool, v_pool, block_tables, seq_lens, scale: float,
                                   max_seq_len: int, *, out=None, max_ctas: int = 0, err=None,
                                   stream=None):
    """Decode attention using the library's built-in scratch instead of a
    caller workspace (for callers that cannot allocate device memory).

    Same result as :func:`paged_attention_decode`.  Calls overlapping on
    the GPU share the built-in scratch and race; the first call on a
    device should come before any stream capture.
    """
    L = _load()
    fn = L.pkv_paged_attention_decode_noalloc
    fn.restype = _i32
    fn.argtypes = [_p, _i32, _i32, _p, _p, _desc, _p, _i32, _p, _i32, _f, _i32, _p, _p, _p]
    desc = pool_desc(k_pool)
    B, H, hd = q.shape
    if out is None:
        out = torch.empty_like(q)
    _check("pkv_paged_attention_decode_noalloc", fn(
        _dev(q, "q", k_pool.dtype), B, H, _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"),
        ctypes.byref(desc), _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(seq_lens, "seq_lens", torch.int32), int(max_seq_len),
        float(scale), int(max_ctas), _dev(out, "out", k_pool.dtype),
        _opt(err, "err", torch.int32), _stream(stream)))
    return out
