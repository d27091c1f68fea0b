#!/usr/bin/env python
"""Throughput of the paged-KV hot path on one GB300 (or N, one process each).

A step is one pass of the whole hot path over one batch: the slot mapping
of the step's new tokens, and per layer the KV write, paged decode
attention (persistent split kernel + merge) and chunked-prefill attention.
By default the decode rows' KV write is fused into the decode launch
(pkv_paged_attention_decode_append), so the separate KV write and the slot
mapping cover only the prefill chunks; --separate-write runs the plain
write-then-decode sequence instead.  The default workload is one layer of a LLaMA-2-70B-shaped
(GQA-8) mixed step: 256 decode sequences with log-normal lengths
(median 1024, clipped to 16..8192) plus 4 prefill sequences each with a
512-token causal chunk over 0..4096 tokens of paged history, in a pool of
65,536 16-token blocks.  Inputs are seeded synthetic data (workloads/).

Reported (one JSON line from rank 0):
  value      algorithmic HBM bytes of the step / device time (GB/s), inputs
             resident in HBM; every step reads ~1.7 GB of KV, more than the
             129 MB L2, so no flush is needed between steps
  e2e        the same metric with the step's inputs copied from pinned host
             memory and its outputs copied back inside the timed region
  roofline   the decode kernels (the dominant launches) against the measured
             HBM copy bandwidth; prefill_roofline against the measured bf16
             tensor peak
  cpu_baseline  the float64 CPU oracle on a bounded sample of the workload

--impl reference times the CPU oracle (the reference implementation of
this build) on the same workload and metric.
"""
from __future__ import annotations

import os

# The CPU oracle's BLAS calls run single-threaded so the baseline's core
# count is exact (set before numpy is imported).
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import argparse  # noqa: E402
import json  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("paged decode attn: KV GB/s read (% of GB300 HBM peak), decode tokens/s per step")
WORKLOAD = "llama2-70b-mixed"
WORKLOAD_LABEL = "llama2-70b-gqa8-mixed-decode256-prefill4x512"
# DRAM bytes (read + written) per KV byte touched by the decode kernel,
# measured with ncu (dram__bytes_read.sum + dram__bytes_write.sum) on the
# llama2-70b-decode64 workload (70B shape) and one layer of the
# llama-3.2-1b workload; keyed by (dtype, n_heads, n_kv, head_dim).  Valid
# only for the decode kernel as it was captured: drop the entries when the
# kernel changes and capture again.
DECODE_DRAM_PER_KV_BYTE = {("bf16", 64, 8, 128): 1.01791, ("bf16", 32, 8, 64): 1.02860}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
THROTTLE_BITS = {  # nvidia-smi clocks_event_reasons bit -> name
    0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
    0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
    0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting",
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every kernel from the host each step instead of replaying "
                         "the step as a CUDA graph")
    ap.add_argument("--separate-write", action="store_true",
                    help="write every new token with kv_write, then run plain decode "
                         "(instead of the fused decode-with-append launch)")
    ap.add_argument("--shared-prefix", action="store_true",
                    help="decode with the shared-prefix path (the workload's common prompt "
                         "blocks read once per step); the K/V write is fused only when the "
                         "step's work split is planned once (several layers, no --no-plan)")
    ap.add_argument("--no-plan", action="store_true",
                    help="let every decode call split its work itself instead of planning the "
                         "split once per step for all layers")
    ap.add_argument("--layers", type=int, default=0,
                    help="layers materialised per step (0 = the workload's own count)")
    return ap.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------ accounting


def step_accounting(plan):
    """Algorithmic bytes and FLOPs of one layer of the step.

    decode:  each decode sequence's KV (K and V, every token once, shared
             blocks once), its query and output rows, the table entries it
             uses and its length;
    prefill: the same for the prefill sequences' full history + chunk;
    write:   the new K/V rows read and written into the pool, their slots.
    prefill FLOPs: 4 * head_dim * n_heads * sum over queries of visible keys.
    """
    sh = plan.shape
    e = sh.itemsize
    row = sh.n_kv * sh.head_dim * e              # one token's K (or V)
    qrow = sh.n_heads * sh.head_dim * e
    nd = plan.n_decode
    bs = sh.block_size

    def kv_bytes(rows):
        held = set()
        tokens = 0
        for b in rows:
            L = int(plan.seq_lens[b])
            nb = -(-L // bs)
            for j in range(nb):
                blk = int(plan.block_tables[b, j])
                if blk in held:
                    continue  # a shared block is read once
                held.add(blk)
                tokens += min(bs, L - j * bs)
        return tokens * row * 2

    dec_rows = range(nd)
    pre_rows = range(nd, plan.num_seqs)
    dec = kv_bytes(dec_rows) + 2 * nd * qrow + sum(4 * (-(-int(plan.seq_lens[b]) // bs)) + 4
                                                    for b in dec_rows)
    tq = int(plan.new_lens[nd:].sum())
    pre = kv_bytes(pre_rows) + 2 * tq * qrow + sum(4 * (-(-int(plan.seq_lens[b]) // bs)) + 8
                                                    for b in pre_rows)
    T = plan.num_new_tokens
    write = T * row * 2 * 2 + T * 8
    flops = 0
    for b in pre_rows:
        L, c = int(plan.seq_lens[b]), int(plan.new_lens[b])
        vis = sum(L - c + i + 1 for i in range(c))
        flops += 4 * sh.head_dim * sh.n_heads * vis
    return dict(decode_bytes=dec, prefill_bytes=pre, write_bytes=write, prefill_flops=flops,
                decode_kv_bytes=kv_bytes(dec_rows))


# ---------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    def __init__(self, index: int, period_ms: int = 50):
        self.cmd = ["nvidia-smi", f"--id={index}",
                    "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active",
                    "--format=csv,noheader,nounits", f"-lms={period_ms}"]
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 4:
                continue
            try:
                sm, smax = float(parts[0]), float(parts[1])
                reasons = int(parts[3], 16) if parts[3].startswith("0x") else int(parts[3])
            except ValueError:
                continue
            self.samples.append((sm, smax, reasons))
        return False

    def summary(self):
        if not getattr(self, "samples", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        busy = [s for s in self.samples if not (s[2] & 0x1)] or self.samples
        names = set()
        for _, _, r in busy:
            for bit, name in THROTTLE_BITS.items():
                if r & bit and name != "gpu_idle":
                    names.add(name)
        return {"sm_mhz": float(np.median([s[0] for s in busy])),
                "sm_max_mhz": float(max(s[1] for s in busy)), "reasons": sorted(names),
                "samples": len(busy)}


# ----------------------------------------------------------- distributed


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------ CPU oracle


def oracle_sample(plan, layer, n_decode: int, n_prefill_queries: int, offset: int = 0):
    """Time the float64 oracle on a bounded sample of the step: n_decode
    decode sequences and n_prefill_queries prefill queries (spread over the
    prefill chunks).  Returns (seconds, algorithmic bytes of the sample)."""
    import torch
    import oracle

    def raw(t):
        t = t.contiguous()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()

    sh = plan.shape
    dt = sh.dtype
    row = sh.n_kv * sh.head_dim * sh.itemsize
    qrow = sh.n_heads * sh.head_dim * sh.itemsize
    kp, vp = raw(layer["k_pool"]), raw(layer["v_pool"])
    q = raw(layer["q"])
    nd = plan.n_decode
    rows = [(offset + i) % nd for i in range(min(n_decode, nd))] if nd else []
    pre = []
    npre = plan.num_seqs - nd
    for j in range(n_prefill_queries if npre else 0):
        b = nd + j % npre
        c = int(plan.new_lens[b])
        pre.append((b, ((offset + j) * 97) % c))
    t0 = time.perf_counter()
    if rows:
        oracle.paged_attention_decode(q[:nd], kp, vp, plan.block_tables[:nd], plan.seq_lens[:nd],
                                      sh.scale, dt, rows=rows)
    for b, i in pre:
        c = int(plan.new_lens[b])
        Li = int(plan.seq_lens[b]) - c + i + 1
        t = int(plan.cu_new_lens[b]) + i
        oracle.paged_attention_decode(q[t:t + 1], kp, vp, plan.block_tables[b:b + 1],
                                      np.array([Li]), sh.scale, dt)
    secs = time.perf_counter() - t0
    nbytes = sum(int(plan.seq_lens[b]) * row * 2 + 2 * qrow for b in rows)
    nbytes += sum((int(plan.seq_lens[b]) - int(plan.new_lens[b]) + i + 1) * row * 2 + 2 * qrow
                  for b, i in pre)
    return secs, nbytes, len(rows), len(pre)


def pages_method_sample(plan, layer, rows, outputs=None):
    """Time the pages' own method on the CPU for decode rows ``rows``: per
    sequence, gather its blocks through the table into contiguous K and V,
    repeat each KV head onto its query heads, and attend with einsum and
    softmax in fp32 PyTorch ("Build a Mini vLLM" section 3, gather_kv and
    paged_attention; written fresh here, sharing nothing with the kernels
    or the oracle).  Returns (seconds, algorithmic bytes); each row's output
    is appended to ``outputs`` when a list is given."""
    import torch
    sh = plan.shape
    rep = sh.n_heads // sh.n_kv
    kp = layer["k_pool"].float()
    vp = layer["v_pool"].float()
    q = layer["q"].float()
    row = sh.n_kv * sh.head_dim * sh.itemsize
    t0 = time.perf_counter()
    for b in rows:
        L = int(plan.seq_lens[b])
        nb = -(-L // sh.block_size)
        ids = torch.from_numpy(plan.block_tables[b, :nb].astype(np.int64))
        K = kp.index_select(0, ids).reshape(-1, sh.n_kv, sh.head_dim)[:L]
        V = vp.index_select(0, ids).reshape(-1, sh.n_kv, sh.head_dim)[:L]
        K = K.repeat_interleave(rep, dim=1)
        V = V.repeat_interleave(rep, dim=1)
        s = torch.einsum("hd,lhd->hl", q[b], K) * sh.scale
        o = torch.einsum("hl,lhd->hd", torch.softmax(s, dim=-1), V)
        if outputs is not None:
            outputs.append(o)
    secs = time.perf_counter() - t0
    return secs, sum(int(plan.seq_lens[b]) * row * 2 for b in rows)


# --------------------------------------------------------------- arms


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from workloads import draw_plan, make_layer
    plan = draw_plan(args.workload)
    layer = make_layer(plan, 0)
    n_dec, n_pre = 8, 4
    for w in range(args.warmup):
        oracle_sample(plan, layer, n_dec, n_pre, offset=w)
    total_s, total_b = 0.0, 0
    for k in range(args.steps):
        s, b, nr, npq = oracle_sample(plan, layer, n_dec, n_pre, offset=(args.warmup + k) * n_dec)
        total_s += s
        total_b += b
    gbs = total_b / total_s / 1e9
    sample = (f"per step: {nr} decode sequences (rotating) and {npq} prefill queries of one "
              f"layer of the {workload_config(plan)['workload']} step, float64 numpy oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(plan, None, "cpu oracle"),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(plan, n_layers=None, launch="cuda_graph"):
    sh = plan.shape
    from workloads import TIMED_LAYERS
    return {"workload": WORKLOAD_LABEL if plan.shape.name == WORKLOAD else plan.shape.name,
            "layers_timed": n_layers or TIMED_LAYERS[sh.name], "layers_model": sh.layers,
            "decode_seqs": int(plan.n_decode), "prefill_seqs": int(plan.num_seqs - plan.n_decode),
            "prefill_chunk_tokens": int(plan.new_lens[plan.n_decode:].max()) if plan.num_seqs > plan.n_decode else 0,
            "n_heads": sh.n_heads, "n_kv": sh.n_kv, "head_dim": sh.head_dim,
            "block_size": sh.block_size, "num_blocks": sh.num_blocks, "dtype": sh.dtype,
            "sum_seq_len": int(plan.seq_lens.sum()),
            "l2": "inputs larger than L2 (each step reads >100 MB of KV), no flush",
            "launch": launch}


def run_gb300(args, rank, world, local):
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from paged_kv_cache_write_gb300 import build as _b
    _b.build()
    import paged_kv_cache_write_gb300 as pkv
    from workloads import TIMED_LAYERS, draw_plan, make_layer

    plan = draw_plan(args.workload)
    sh = plan.shape
    n_layers = args.layers if args.layers > 0 else TIMED_LAYERS[sh.name]
    acc = step_accounting(plan)
    layers_cpu = [make_layer(plan, l) for l in range(n_layers)]
    L = [{n: t.to(dev) for n, t in lay.items()} for lay in layers_cpu]
    if rank != 0 or args.no_cpu_baseline:
        layers_cpu = layers_cpu[:1] if rank == 0 else []
    nd = plan.n_decode
    has_pre = plan.num_seqs > nd
    bt = torch.from_numpy(plan.block_tables).to(dev)
    seq_lens = torch.from_numpy(plan.seq_lens).to(dev)
    cu_new = torch.from_numpy(plan.cu_new_lens).to(dev)
    T = plan.num_new_tokens
    max_dec = int(plan.seq_lens[:nd].max()) if nd else 0
    if has_pre:
        cu_q = torch.from_numpy((plan.cu_new_lens[nd:] - plan.cu_new_lens[nd]).astype(np.int32)).to(dev)
        max_q = int(plan.new_lens[nd:].max())
        max_pre = int(plan.seq_lens[nd:].max())
    slots = torch.empty(T, dtype=torch.int64, device=dev)
    P = len(plan.shared_prefix_blocks) if args.shared_prefix else 0
    ws_bytes = (pkv.decode_shared_prefix_workspace_bytes(nd, sh.n_heads, sh.head_dim, max_dec, P)
                if P else pkv.decode_workspace_bytes(nd, sh.n_heads, sh.head_dim, max_dec))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    dec_out = [torch.empty((nd, sh.n_heads, sh.head_dim), dtype=sh.torch_dtype, device=dev) for _ in L]
    pre_out = [torch.empty((T - nd, sh.n_heads, sh.head_dim), dtype=sh.torch_dtype, device=dev)
               for _ in L] if has_pre else None
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    ev_dec, ev_pre = [], []

    # the step's decode K/V write rides in the decode launch (with a shared
    # prefix, only in the once-per-step planned call)
    fused = not args.separate_write and (P == 0 or (not args.no_plan and len(L) > 1))
    # the decode rows' work split, planned once per step for all its layers
    # (a one-layer step plans inside its call: a separate plan would not be
    # shared by anything)
    planned = not args.no_plan and len(L) > 1

    def decode_plan(sl_):
        pkv.decode_plan(L[0]["k_pool"], sl_[:nd], sh.n_heads, bt.shape[1], max_dec, workspace=ws,
                        shared_prefix_blocks=P, err=err)

    def decode_call(q, k_pool, v_pool, bt_, sl_, out, k_new=None, v_new=None):
        if planned:
            pkv.paged_attention_decode_planned(q, k_pool, v_pool, bt_, sl_, sh.scale, max_dec,
                                               workspace=ws, k_new=k_new, v_new=v_new,
                                               shared_prefix_blocks=P, out=out, err=err)
        elif P:
            pkv.paged_attention_decode_shared_prefix(q, k_pool, v_pool, bt_, sl_, sh.scale, P,
                                                     max_dec, out=out, workspace=ws, err=err)
        elif k_new is not None:
            pkv.paged_attention_decode_append(q, k_new, v_new, k_pool, v_pool, bt_, sl_, sh.scale,
                                              max_dec, out=out, workspace=ws, err=err)
        else:
            pkv.paged_attention_decode(q, k_pool, v_pool, bt_, sl_, sh.scale, max_dec, out=out,
                                       workspace=ws, err=err)

    def step_head(inputs=None):
        src_bt, src_sl, src_cu = (bt, seq_lens, cu_new) if inputs is None else inputs[:3]
        if has_pre or not fused:
            pkv.slot_mapping(src_bt, src_sl, src_cu, T, sh.block_size, sh.num_blocks, out=slots,
                             err=err)
        if planned and nd:
            decode_plan(src_sl)

    def layer_decode(li, inputs=None, timed=False, outs=None):
        lay = L[li]
        src_bt, src_sl = (bt, seq_lens) if inputs is None else inputs[:2]
        q, k, v = (lay["q"], lay["k"], lay["v"]) if inputs is None else inputs[3][li]
        if not fused:  # the decode rows' tokens come first in the step's token order
            pkv.kv_write(k[:nd], v[:nd], slots[:nd], lay["k_pool"], lay["v_pool"], err=err)
        if timed:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
        if fused:
            decode_call(q[:nd], lay["k_pool"], lay["v_pool"], src_bt[:nd], src_sl[:nd],
                        (outs or dec_out)[li], k_new=k[:nd], v_new=v[:nd])
        else:
            decode_call(q[:nd], lay["k_pool"], lay["v_pool"], src_bt[:nd], src_sl[:nd],
                        (outs or dec_out)[li])
        if timed:
            e1.record(stream)
            ev_dec.append((e0, e1))

    def layer_prefill(li, inputs=None, timed=False, outs=None):
        lay = L[li]
        src_bt, src_sl = (bt, seq_lens) if inputs is None else inputs[:2]
        q, k, v = (lay["q"], lay["k"], lay["v"]) if inputs is None else inputs[3][li]
        pkv.kv_write(k[nd:], v[nd:], slots[nd:], lay["k_pool"], lay["v_pool"], err=err)
        if timed:
            e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e2.record(stream)
        pkv.paged_attention_prefill(q[nd:], cu_q, lay["k_pool"], lay["v_pool"], src_bt[nd:],
                                    src_sl[nd:], sh.scale, max_q, max_pre, out=(outs or pre_out)[li],
                                    err=err)
        if timed:
            e3.record(stream)
            ev_pre.append((e2, e3))

    def step(timed=False, inputs=None):
        step_head(inputs)
        for li in range(len(L)):
            if nd:
                layer_decode(li, inputs, timed)
            if has_pre:
                layer_prefill(li, inputs, timed)

    # (prefix runs + their combine) + (plan above 2,048 sequences) + main + merge;
    # planned: one plan kernel per step, then (prefix runs + combine +) main + merge per layer
    dec_launches = (((2 if planned or nd <= 2048 else 3) + (2 if P else 0)) if nd else 0)
    plan_launches = 1 if planned and nd else 0
    if fused:
        launches_per_step = (plan_launches + (1 if has_pre else 0) +
                             n_layers * (dec_launches + (2 if has_pre else 0)))
    else:
        launches_per_step = plan_launches + 1 + n_layers * ((1 if nd else 0) + dec_launches +
                                                            (2 if has_pre else 0))

    def decode_all():
        if planned:
            decode_plan(seq_lens)
        for li, lay in enumerate(L):
            decode_call(lay["q"][:nd], lay["k_pool"], lay["v_pool"], bt[:nd], seq_lens[:nd],
                        dec_out[li])

    def prefill_all():
        for li, lay in enumerate(L):
            pkv.paged_attention_prefill(lay["q"][nd:], cu_q, lay["k_pool"], lay["v_pool"], bt[nd:],
                                        seq_lens[nd:], sh.scale, max_q, max_pre, out=pre_out[li],
                                        err=err)

    def capture(fn):
        """Warm fn up on a side stream, then record it as a CUDA graph."""
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    def time_graph(g, reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} during warm-up")
    use_graph = not args.no_graph
    if use_graph:
        g_step = capture(step)
        for _ in range(max(args.warmup, 3)):
            g_step.replay()
        torch.cuda.synchronize()

    # ---- device-resident timing
    barrier(world)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        start.record(stream)
        for _ in range(args.steps):
            if use_graph:
                g_step.replay()
            else:
                step(timed=True)
        stop.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = start.elapsed_time(stop)
    ms_max = max_over_ranks(ms, world, dev)
    ms_step = ms_max / args.steps
    if use_graph:
        # per-call durations of the dominant kernels: graphs of one layer-loop
        # of decode calls and of prefill calls, replayed right after the step
        reps = max(10, args.steps // 2)
        dec_ms = time_graph(capture(decode_all), reps) / n_layers if nd else None
        pre_ms = time_graph(capture(prefill_all), reps) / n_layers if has_pre else None
    else:
        dec_ms = float(np.mean([a.elapsed_time(b) for a, b in ev_dec])) if ev_dec else None
        pre_ms = float(np.mean([a.elapsed_time(b) for a, b in ev_pre])) if ev_pre else None

    per_layer = acc["decode_bytes"] + acc["prefill_bytes"] + acc["write_bytes"]
    step_bytes = per_layer * n_layers
    value = world * step_bytes / (ms_step * 1e-3) / 1e9

    # ---- copy-on-write block copy: held blocks onto free ones of layer 0's
    # pools (free blocks are outside every sequence, so the step is untouched)
    cow = None
    free = np.setdiff1d(np.arange(1 if sh.dummy_block0 else 0, sh.num_blocks), plan.held_blocks)
    n_cow = int(min(4096, len(free), len(plan.held_blocks)))
    if n_cow > 0:
        crng = np.random.default_rng(99)
        pairs = np.stack([crng.choice(plan.held_blocks, n_cow, replace=False),
                          crng.choice(free, n_cow, replace=False)], axis=1).astype(np.int32)
        pairs_d = torch.from_numpy(pairs).to(dev)

        def cow_call():
            pkv.copy_blocks(L[0]["k_pool"], L[0]["v_pool"], pairs_d, err=err)

        for _ in range(3):
            cow_call()
        reps = 20
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(reps):
            cow_call()
        c1.record(stream)
        torch.cuda.synchronize()
        cow_ms = c0.elapsed_time(c1) / reps
        block_bytes = sh.block_size * sh.n_kv * sh.head_dim * sh.itemsize
        cow_bytes = 2 * 2 * n_cow * block_bytes  # K and V, read and written
        cow = {"pairs": n_cow, "bytes_per_launch": cow_bytes, "ms_per_launch": cow_ms,
               "achieved": cow_bytes / (cow_ms * 1e-3) / 1e9, "unit": "GB/s",
               "timing": "CUDA events around 20 back-to-back launches after 3 warm-up launches"}

    # ---- end to end: step inputs from pinned host memory, outputs back
    e2e = None
    if not args.no_e2e:
        host_in = [t.cpu().pin_memory() for t in (bt, seq_lens, cu_new)]
        host_layers = [[lay[n].cpu().pin_memory() for n in ("q", "k", "v")] for lay in L]
        host_out = [o.cpu().pin_memory() for o in dec_out] + ([o.cpu().pin_memory() for o in pre_out]
                                                              if has_pre else [])
        # two sets of device inputs and outputs, alternating between steps, so
        # a step's copies overlap its neighbours' compute
        dev_in = [[torch.empty_like(t) for t in (bt, seq_lens, cu_new)] for _ in range(2)]
        dev_layers = [[[torch.empty_like(lay[n]) for n in ("q", "k", "v")] for lay in L]
                      for _ in range(2)]
        dev_dec = [dec_out, [torch.empty_like(o) for o in dec_out]]
        dev_pre = [pre_out, [torch.empty_like(o) for o in pre_out] if has_pre else None]
        h2d = sum(t.numel() * t.element_size() for t in host_in) + sum(
            t.numel() * t.element_size() for lay in host_layers for t in lay)
        d2h = sum(t.numel() * t.element_size() for t in host_out)
        h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        steps_per_graph = 8  # the graph's first step cannot overlap the one before it

        def e2e_steps():
            # Step i uses buffer set i % 2.  Its copies in start once step i-2
            # has finished computing from that set, so they land while step
            # i-1 computes and its compute waits for them once (one wait per
            # step keeps the kernels of a step chained back to back); the
            # first step of the graph instead starts each layer's decode rows,
            # then prefill rows, as soon as they have landed.  Each part's
            # output goes back on a second stream once it is computed, and
            # step i+2 overwrites those outputs only after that copy.  Every
            # step copies all its inputs in and all its outputs out.
            main = torch.cuda.current_stream(dev)
            h2d_s.wait_stream(main)
            d2h_s.wait_stream(main)
            computed = [None] * steps_per_graph
            copied_out = [None] * steps_per_graph
            for i in range(steps_per_graph):
                b = i % 2
                if i >= 2:
                    h2d_s.wait_event(computed[i - 2])
                ev_d, ev_p = [], []
                with torch.cuda.stream(h2d_s):
                    for d, h in zip(dev_in[b], host_in):
                        d.copy_(h, non_blocking=True)
                    for dl, hl in zip(dev_layers[b], host_layers):
                        for part, evs in ((slice(0, nd), ev_d), (slice(nd, None), ev_p)):
                            for d, h in zip(dl, hl):
                                d[part].copy_(h[part], non_blocking=True)
                            e = torch.cuda.Event()
                            e.record(h2d_s)
                            evs.append(e)
                if i >= 2:
                    main.wait_event(copied_out[i - 2])
                inputs = (dev_in[b][0], dev_in[b][1], dev_in[b][2], dev_layers[b])
                main.wait_event(ev_d[0] if i == 0 else ev_p[-1])  # tables first / everything
                step_head(inputs)
                for li in range(len(L)):
                    for run, outs, evs, off, on in ((layer_decode, dev_dec[b], ev_d, 0, nd > 0),
                                                    (layer_prefill, dev_pre[b], ev_p, len(dec_out),
                                                     has_pre)):
                        if not on:
                            continue
                        if i == 0:
                            main.wait_event(evs[li])
                        run(li, inputs, outs=outs)
                        e = torch.cuda.Event()
                        e.record(main)
                        d2h_s.wait_event(e)
                        with torch.cuda.stream(d2h_s):
                            host_out[off + li].copy_(outs[li], non_blocking=True)
                computed[i] = torch.cuda.Event()
                computed[i].record(main)
                copied_out[i] = torch.cuda.Event()
                copied_out[i].record(d2h_s)
            main.wait_stream(h2d_s)
            main.wait_stream(d2h_s)

        for _ in range(2):
            e2e_steps()
        torch.cuda.synchronize()
        run_e2e = capture(e2e_steps).replay if use_graph else e2e_steps
        barrier(world)
        e_reps = max(1, args.steps // (3 * steps_per_graph))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(e_reps):
            run_e2e()
        s1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(s0.elapsed_time(s1), world, dev) / (e_reps * steps_per_graph)
        e2e = {"value": world * step_bytes / (e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "ms_per_step": e_ms, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "copies": f"every step copies all its inputs in and all its outputs out; inputs "
                         f"and outputs double-buffered so a step's copies (one stream in, one "
                         f"out, each layer's outputs as soon as computed) overlap its "
                         f"neighbours' compute; timed over {e_reps} x {steps_per_graph} steps"}

    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} in the timed region")

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    peaks, src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    tc = float(peaks["bf16_tflops"])
    roof = None
    if dec_ms:
        ach = acc["decode_bytes"] / (dec_ms * 1e-3) / 1e9
        ratio = DECODE_DRAM_PER_KV_BYTE.get((sh.dtype, sh.n_heads, sh.n_kv, sh.head_dim))
        traffic = ratio * acc["decode_kv_bytes"] if ratio else None
        roof = {"bound": "hbm", "kernel": ("paged_attention_decode_shared_prefix (prefix + split "
                                           "kernel + merge)" if P else
                                           "paged_attention_decode (split kernel + merge)"),
                "timing": ("CUDA events around graph replays of one layer loop of decode calls, "
                           "after the step's timed region" if use_graph else
                           "CUDA events around every decode call inside the timed region"),
                "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "peak_source": f"hbm_gbs of {src}", "traffic": traffic,
                "traffic_note": ("dram__bytes_read.sum + dram__bytes_write.sum of the decode "
                                 "kernel per KV byte, from one ncu capture of this shape, "
                                 "times this call's KV bytes"
                                 if traffic else "no capture of this shape's current kernel"),
                "algorithmic_bytes_per_launch": acc["decode_bytes"], "ms_per_launch": dec_ms}
    pre_roof = None
    if pre_ms:
        tf = acc["prefill_flops"] / (pre_ms * 1e-3) / 1e12
        pre_roof = {"bound": "tensor", "kernel": "paged_attention_prefill", "achieved": tf,
                    "peak": tc, "unit": "TFLOP/s", "frac": tf / tc,
                    "peak_source": f"bf16_tflops of {src}", "flops_per_launch": acc["prefill_flops"],
                    "ms_per_launch": pre_ms,
                    "traffic": None, "traffic_note": "tensor-bound: DRAM bytes are not its limit"}
    cpu = None
    if not args.no_cpu_baseline and layers_cpu:
        # passes over layer 0 (every decode sequence, 64 prefill queries
        # per pass, rotating) until about 10 s of CPU work are done
        secs = nbytes = nr = npq = passes = 0
        while secs < 10.0 and passes < 50:
            s_, b_, r_, p_ = oracle_sample(plan, layers_cpu[0], nd, 64, offset=passes * 64)
            secs, nbytes, nr, npq, passes = secs + s_, nbytes + b_, nr + r_, npq + p_, passes + 1
        cpu = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{passes} passes over layer 0: {nr} decode sequences + {npq} prefill "
                         f"queries in all ({nbytes / 1e6:.0f} MB of KV), float64 numpy oracle, "
                         f"{secs:.1f} s on one core"}
    pages_cpu = None
    if not args.no_cpu_baseline and layers_cpu and nd:
        import torch as _t
        psecs = pbytes = ppasses = 0
        while psecs < 5.0 and ppasses < 20:
            s_, b_ = pages_method_sample(plan, layers_cpu[0], range(nd))
            psecs, pbytes, ppasses = psecs + s_, pbytes + b_, ppasses + 1
        pages_cpu = {"value": pbytes / psecs / 1e9, "unit": "GB/s", "cores": _t.get_num_threads(),
                     "kind": "the pages' method: per-sequence gather + einsum attention, "
                             "fp32 PyTorch on the CPU",
                     "sample": f"{ppasses} passes over layer 0's {nd} decode sequences, "
                               f"{psecs:.1f} s"}
    dec_tok_s = world * nd / (ms_step * 1e-3 * (sh.layers / n_layers)) if nd else None
    n_pre_tok = int(plan.new_lens[nd:].sum())
    pre_tok_s = (world * n_pre_tok / (ms_step * 1e-3 * (sh.layers / n_layers))
                 if has_pre else None)
    # the roofline object describes the step's dominant kernel
    dominant = roof
    if pre_roof and (roof is None or pre_ms > dec_ms):
        dominant = pre_roof
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if sh.dtype == "bf16" else "f32",
        "data": "synthetic (seeded; workloads/)",
        "config": workload_config(plan, n_layers, "cuda_graph" if use_graph else "eager"),
        "decode_write": ("fused into the decode launch" if fused
                         else "separate kv_write launch"),
        "decode_shared_prefix_blocks": P,
        "decode_plan": ("once per step for all timed layers (decode_plan + decode_planned)"
                        if planned else "inside each decode call"),
        "decode_tokens_per_s": dec_tok_s,
        "decode_tokens_per_s_note": f"{nd} decode tokens per step of {sh.layers} layers, "
                                    f"{n_layers} timed layer(s) scaled by {sh.layers / n_layers:g}",
        "percent_of_hbm_peak_step": 100.0 * value / world / hbm,
        "prefill_tokens_per_s": pre_tok_s,
        "roofline": dominant, "decode_roofline": roof, "prefill_roofline": pre_roof,
        "cpu_baseline": cpu, "cpu_pages_method": pages_cpu, "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "bytes_per_step": step_bytes,
        "copy_blocks": (dict(cow, peak=hbm, frac=cow["achieved"] / hbm,
                             peak_source=f"hbm_gbs of {src}") if cow else None),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_gb300(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
