"""Helpers shared by the GPU parity tests: run one step of the hot path
through the C ABI (via the ctypes binding) and the same step through the
CPU oracle, on the same seeded inputs."""
from __future__ import annotations

import functools
import inspect
import math

import numpy as np
import torch

import oracle

TOL = {"f32": dict(max_abs=1e-5, mean_abs=1e-5), "bf16": dict(max_abs=2e-2, mean_abs=2e-3)}

# ---------------------------------------------------------------- canaries
# Guard bands stand in for a memory checker's out-of-bounds detection:
# device tensors the tests hand to the kernels (inputs, pools, outputs,
# workspaces) sit inside larger buffers with CANARY bytes of a fixed random
# pattern on each side, and every call through the binding is followed by
# a check that no pattern byte changed.

CANARY = 4096  # bytes on each side (keeps the tensor 16- and 256-byte aligned)
_LIVE = []     # (buffer, payload bytes) of the running test
_PATTERNS = {}


def _pattern(device):
    key = str(device)
    if key not in _PATTERNS:
        g = torch.Generator(device="cpu").manual_seed(0xC0FFEE)
        _PATTERNS[key] = torch.randint(0, 256, (CANARY,), dtype=torch.uint8,
                                       generator=g).to(device)
    return _PATTERNS[key]


def guarded_empty(shape, dtype, device="cuda"):
    """Uninitialised device tensor with canary bands on both sides."""
    shape = tuple(int(x) for x in shape)
    n = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
    buf = torch.empty(n + 2 * CANARY, dtype=torch.uint8, device=device)
    pat = _pattern(buf.device)
    buf[:CANARY] = pat
    buf[CANARY + n:] = pat
    _LIVE.append((buf, n))
    return buf[CANARY:CANARY + n].view(dtype).view(shape)


def guarded_copy(t, device="cuda"):
    """Device copy of ``t`` with canary bands on both sides."""
    out = guarded_empty(t.shape, t.dtype, device)
    out.copy_(t)
    return out


def check_canaries():
    """Raise if any guard band of the running test changed."""
    if not _LIVE:
        return
    torch.cuda.synchronize()
    for buf, n in _LIVE:
        pat = _pattern(buf.device)
        if not (torch.equal(buf[:CANARY], pat) and torch.equal(buf[CANARY + n:], pat)):
            raise AssertionError(f"a kernel wrote outside a {n}-byte tensor (canary changed)")


def _ws_bytes(pkv, name, a):
    """Workspace the binding would allocate for call `name` (bound args a)."""
    q = a["q"]
    B, H, hd = q.shape
    msl = a.get("max_seq_len")
    if msl is None:
        msl = int(a["seq_lens"].max().item()) if B else 0
    if name == "paged_attention_decode_shared_prefix":
        return pkv.decode_shared_prefix_workspace_bytes(B, H, hd, msl, a["shared_prefix_blocks"],
                                                        a.get("max_ctas", 0))
    return pkv.decode_workspace_bytes(B, H, hd, msl, a.get("max_ctas", 0))


_OUT_LIKE_Q = ("paged_attention_decode", "paged_attention_decode_append",
               "paged_attention_decode_shared_prefix", "paged_attention_decode_planned",
               "paged_attention_prefill", "paged_attention_decode_noalloc")
_WS = ("paged_attention_decode", "paged_attention_decode_append",
       "paged_attention_decode_shared_prefix")
_WRAPPED = _OUT_LIKE_Q + ("slot_mapping", "kv_write", "kv_gather", "copy_blocks", "decode_plan")


def start_guarding(monkeypatch, pkv):
    """Wrap the binding's entry points for one test: outputs and workspaces
    the binding would allocate come from guarded buffers, and the canaries
    of every guarded tensor are checked after each call."""
    _LIVE.clear()
    for name in _WRAPPED:
        fn = getattr(pkv, name)
        sig = inspect.signature(fn)

        @functools.wraps(fn)
        def wrapper(*args, __fn=fn, __sig=sig, __name=name, **kwargs):
            bound = __sig.bind(*args, **kwargs)
            bound.apply_defaults()
            a = bound.arguments
            if __name in _OUT_LIKE_Q and a.get("out") is None:
                a["out"] = guarded_empty(a["q"].shape, a["q"].dtype, a["q"].device)
            if __name in _WS and a.get("workspace") is None:
                a["workspace"] = guarded_empty((_ws_bytes(pkv, __name, a),), torch.uint8,
                                               a["q"].device)
            if __name == "slot_mapping" and a.get("out") is None:
                a["out"] = guarded_empty((a["num_tokens"],), torch.int64,
                                         a["block_tables"].device)
            if __name == "kv_gather":
                shape = (int(a["total_tokens"]), a["k_pool"].shape[2], a["k_pool"].shape[3])
                for k in ("k_out", "v_out"):
                    if a.get(k) is None:
                        a[k] = guarded_empty(shape, a["k_pool"].dtype, a["k_pool"].device)
            result = __fn(*bound.args, **bound.kwargs)
            check_canaries()
            return result

        monkeypatch.setattr(pkv, name, wrapper)


def stop_guarding():
    check_canaries()
    _LIVE.clear()


def raw(t: torch.Tensor) -> np.ndarray:
    """Oracle storage view of a CPU tensor: float32 values or bf16 bits."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    tol = TOL[dtype]
    mx, mean = float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0
    assert mx <= tol["max_abs"], f"{what}: max abs err {mx:.3g} > {tol['max_abs']}"
    assert mean <= tol["mean_abs"], f"{what}: mean abs err {mean:.3g} > {tol['mean_abs']}"
    return mx, mean


class GpuStep:
    """One step (slot mapping, KV write, decode rows, prefill rows) of one
    layer on the GPU, through the library's C ABI."""

    def __init__(self, plan, layer: dict, device="cuda"):
        import paged_kv_cache_write_gb300 as pkv
        self.pkv = pkv
        self.plan = plan
        sh = plan.shape
        self.sh = sh
        self.bt = guarded_copy(torch.from_numpy(plan.block_tables), device)
        self.seq_lens = guarded_copy(torch.from_numpy(plan.seq_lens), device)
        self.cu_new = guarded_copy(torch.from_numpy(plan.cu_new_lens), device)
        self.t = {n: guarded_copy(v, device) for n, v in layer.items()}
        nd = plan.n_decode
        self.nd = nd
        self.max_dec = int(plan.seq_lens[:nd].max()) if nd else 0
        if plan.num_seqs > nd:
            cu = plan.cu_new_lens[nd:] - plan.cu_new_lens[nd]
            self.cu_q = guarded_copy(torch.from_numpy(cu.astype(np.int32)), device)
            self.max_q = int(plan.new_lens[nd:].max())
            self.max_pre = int(plan.seq_lens[nd:].max())
        self.err = guarded_empty((1,), torch.int32, device)
        self.err.zero_()

    def slots(self):
        p = self.plan
        return self.pkv.slot_mapping(self.bt, self.seq_lens, self.cu_new, p.num_new_tokens,
                                     self.sh.block_size, self.sh.num_blocks, err=self.err)

    def write(self, slots):
        t = self.t
        self.pkv.kv_write(t["k"], t["v"], slots, t["k_pool"], t["v_pool"], err=self.err)

    def decode(self, max_ctas=0, k_pool=None, v_pool=None, bt=None):
        t = self.t
        nd = self.nd
        return self.pkv.paged_attention_decode(
            t["q"][:nd], t["k_pool"] if k_pool is None else k_pool,
            t["v_pool"] if v_pool is None else v_pool, (self.bt if bt is None else bt)[:nd],
            self.seq_lens[:nd], self.sh.scale, self.max_dec, max_ctas=max_ctas, err=self.err)

    def prefill(self):
        t = self.t
        nd = self.nd
        return self.pkv.paged_attention_prefill(
            t["q"][nd:], self.cu_q, t["k_pool"], t["v_pool"], self.bt[nd:], self.seq_lens[nd:],
            self.sh.scale, self.max_q, self.max_pre, err=self.err)

    def run(self, max_ctas=0):
        s = self.slots()
        self.write(s)
        dec = self.decode(max_ctas) if self.nd else None
        pre = self.prefill() if self.plan.num_seqs > self.nd else None
        torch.cuda.synchronize()
        return s, dec, pre


class OracleStep:
    """The same step on the CPU oracle (float64)."""

    def __init__(self, plan, layer: dict):
        self.plan = plan
        self.dtype = plan.shape.dtype
        self.raw = {n: raw(v) for n, v in layer.items()}

    def run_write(self):
        p = self.plan
        slots = oracle.slot_mapping(p.block_tables, p.seq_lens, p.new_lens, p.shape.block_size)
        kp, vp = oracle.kv_write(self.raw["k"], self.raw["v"], slots, self.raw["k_pool"],
                                 self.raw["v_pool"])
        self.slots, self.kp, self.vp = slots, kp, vp
        return slots, kp, vp

    def decode(self, rows=None):
        p = self.plan
        nd = p.n_decode
        return oracle.paged_attention_decode(self.raw["q"][:nd], self.kp, self.vp,
                                             p.block_tables[:nd], p.seq_lens[:nd], p.shape.scale,
                                             self.dtype, rows=rows)

    def prefill_row(self, b_rel: int, i: int):
        """Output of query i of prefill sequence b_rel (relative to the
        prefill rows), computed one query at a time as a decode over the
        prefix up to and including its own token."""
        p = self.plan
        nd = p.n_decode
        b = nd + b_rel
        c = int(p.new_lens[b])
        L_i = int(p.seq_lens[b]) - c + i + 1
        t = int(p.cu_new_lens[b]) + i
        out = oracle.paged_attention_decode(self.raw["q"][t:t + 1], self.kp, self.vp,
                                            p.block_tables[b:b + 1], np.array([L_i]),
                                            p.shape.scale, self.dtype)
        return out[0]
