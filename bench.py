#!/usr/bin/env python
"""Throughput of the paged-KV hot path on one GB300 (or N, one process each).

A step is one pass of the whole hot path over one batch: the slot mapping
of the step's new tokens, and per layer the KV write, paged decode
attention (persistent split kernel + merge) and chunked-prefill attention.
By default the decode rows' KV write is fused into the decode launch
(pkv_paged_attention_decode_append), so the separate KV write and the slot
mapping cover only the prefill chunks; --separate-write runs the plain
write-then-decode sequence instead.  The default workload is one layer of a
LLaMA-2-70B-shaped (GQA-8) mixed step: 256 decode sequences with log-normal
lengths (median 1024, clipped to 16..8192) plus 4 prefill sequences each
with a 512-token causal chunk over 0..4096 tokens of paged history, in a
pool of 65,536 16-token blocks.  Inputs are seeded synthetic data
(workloads/).

Each timed step replays two CUDA graphs back to back, the decode half
(work-split plan, then per layer the decode call with the step's K/V write
fused in) and the prefill half (slot mapping, per layer the prefill chunks'
KV write and the prefill call), with CUDA events on the launching stream
around each half.

Reported (one JSON line from rank 0):
  value      the metric: algorithmic bytes of the decode attention calls
             (KV read + queries + outputs + tables + lengths + the fused
             K/V rows) / their device time, summed over the timed steps;
             inputs resident in HBM; every step reads ~1.7 GB of KV, more
             than the 129 MB L2, so no flush is needed between steps
  ms_per_step  the whole step (decode half + prefill half)
  e2e        the same metric with each step's decode inputs copied from
             pinned host memory and its outputs copied back inside the
             timed region
  roofline   the decode call (the dominant launches) against the measured
             HBM copy bandwidth; prefill_roofline against the measured bf16
             tensor peak
  per_config the decode call of each of the five workload shapes (toy,
             SmolLM2-135M, Llama-3.2-1B, LLaMA-7B, LLaMA-2-70B), median of
             at least 50 graph replays, with its error against the oracle
  cpu_baseline  the float64 CPU oracle on a bounded sample of the workload

--impl reference times the float64 CPU oracle, the reference arm, on the
same workload and metric.
"""
from __future__ import annotations

import os

# The CPU oracle's BLAS calls run single-threaded so the baseline's core
# count is exact (set before numpy is imported).
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")

import argparse  # noqa: E402
import hashlib  # noqa: E402
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
# the five workload shapes whose decode call is timed and checked per config
PER_CONFIG = ("toy", "smollm2-135m", "llama-3.2-1b", "llama-7b", "llama2-70b-mixed")
L2_BYTES = 126 * 2 ** 20
# Sources of the decode kernels; the traffic ratios below are valid only for
# the sources whose hash they carry.
DECODE_SOURCES = ("attention.cuh", "device.cuh", "tcgen05.cuh", "decode.cu", "decode_mma64.cu")
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per algorithmic
# byte of the fused write + decode call, from one ncu capture of the shape
# named in "capture", keyed by (dtype, n_heads, n_kv, head_dim), valid for
# the decode sources with the given hash only (a different hash reports
# traffic null; tests/test_bench_host.py fails while a recorded hash is stale).
DECODE_TRAFFIC: dict = {
    ("bf16", 64, 8, 128): {"ratio": 1.0141, "source_sha256": "63ed210e029b166d",
                           "capture": "llama2-70b-decode64, decode + merge, 2 calls"},
    ("bf16", 32, 8, 64): {"ratio": 1.0164, "source_sha256": "63ed210e029b166d",
                          "capture": "llama-3.2-1b (2 layers), decode + merge, 4 calls"},
    ("bf16", 32, 32, 128): {"ratio": 1.0013, "source_sha256": "63ed210e029b166d",
                            "capture": "llama-7b (2 layers), decode + merge, 4-5 calls"},
}
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
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-config decode timings and oracle checks")
    ap.add_argument("--per-config", default=",".join(PER_CONFIG),
                    help="comma-separated workloads timed per config")
    ap.add_argument("--reps", type=int, default=50,
                    help="minimum graph replays per timed call (median reported)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every kernel from the host each step instead of replaying "
                         "the step's halves as CUDA graphs")
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


def decode_source_hash() -> str:
    """sha256 (first 16 hex digits) of the decode kernels' sources."""
    csrc = os.path.join(ROOT, "paged_kv_cache_write_gb300", "csrc")
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def host_info():
    """Host cores this process may run on, and the BLAS threads numpy uses."""
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        cores = os.cpu_count() or 1
    blas = int(os.environ.get("OPENBLAS_NUM_THREADS", "0") or 0) or None
    return {"host_cores": cores, "blas_threads": blas}


# ------------------------------------------------------------ accounting


def step_accounting(plan):
    """Algorithmic bytes and FLOPs of one layer of the step.

    decode:  each decode sequence's KV (K and V, every token once, shared
             blocks once), its query and output rows, the table entries it
             uses and its length;
    append:  with the write fused into the decode call, each decode row's
             new K and V read once and stored once;
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
                decode_kv_bytes=kv_bytes(dec_rows), append_bytes=nd * row * 2 * 2,
                decode_write_bytes=nd * row * 2 * 2 + nd * 8)


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


def _raw(t):
    """Oracle storage view of a CPU tensor: float32 values or bf16 bits."""
    import torch
    t = t.contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def oracle_sample(plan, layer, n_decode: int, n_prefill_queries: int, offset: int = 0):
    """Time the float64 oracle on a bounded sample of the step: n_decode
    decode sequences and n_prefill_queries prefill queries (spread over the
    prefill chunks).  Returns (seconds, algorithmic bytes of the sample,
    sequences, queries); bytes count what the GPU calls count per row: the
    row's K and V, its query and output, its table entries and length."""
    import oracle

    sh = plan.shape
    dt = sh.dtype
    row = sh.n_kv * sh.head_dim * sh.itemsize
    qrow = sh.n_heads * sh.head_dim * sh.itemsize
    bs = sh.block_size
    kp, vp = _raw(layer["k_pool"]), _raw(layer["v_pool"])
    q = _raw(layer["q"])
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
    nbytes = sum(int(plan.seq_lens[b]) * row * 2 + 2 * qrow + 4 * (-(-int(plan.seq_lens[b]) // bs))
                 + 4 for b in rows)
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


def oracle_decode_error(plan, layer_cpu, out_gpu):
    """Max and mean |GPU - oracle| of a layer's decode rows: the oracle
    writes the step's new K/V rows into the pools, then attends."""
    import oracle
    nd = plan.n_decode
    r = {n: _raw(t) for n, t in layer_cpu.items()}
    slots = oracle.slot_mapping(plan.block_tables[:nd], plan.seq_lens[:nd], plan.new_lens[:nd],
                                plan.shape.block_size)
    kp, vp = oracle.kv_write(r["k"][:nd], r["v"][:nd], slots, r["k_pool"], r["v_pool"])
    t0 = time.perf_counter()
    ref = oracle.paged_attention_decode(r["q"][:nd], kp, vp, plan.block_tables[:nd],
                                        plan.seq_lens[:nd], plan.shape.scale, plan.shape.dtype)
    secs = time.perf_counter() - t0
    got = out_gpu.double().cpu().numpy()
    d = np.abs(got - ref)
    return {"max_abs": float(d.max()), "mean_abs": float(d.mean()), "rows": int(nd),
            "oracle_s": secs}


# --------------------------------------------------------------- arms


def workload_config(plan, n_layers=None):
    sh = plan.shape
    from workloads import TIMED_LAYERS
    return {"workload": WORKLOAD_LABEL if plan.shape.name == WORKLOAD else plan.shape.name,
            "layers_timed": n_layers or TIMED_LAYERS[sh.name], "layers_model": sh.layers,
            "decode_seqs": int(plan.n_decode), "prefill_seqs": int(plan.num_seqs - plan.n_decode),
            "prefill_chunk_tokens": int(plan.new_lens[plan.n_decode:].max()) if plan.num_seqs > plan.n_decode else 0,
            "n_heads": sh.n_heads, "n_kv": sh.n_kv, "head_dim": sh.head_dim,
            "block_size": sh.block_size, "num_blocks": sh.num_blocks, "dtype": sh.dtype,
            "sum_seq_len": int(plan.seq_lens.sum()),
            "l2": "inputs larger than L2 (each step reads >100 MB of KV), no flush"}


def run_reference(args, rank, world):
    """The float64 oracle on the host cores: decode attention of a rotating
    sample of the workload's decode sequences per step (the metric's
    decode KV GB/s)."""
    if rank != 0:
        return 0
    from workloads import draw_plan, make_layer
    plan = draw_plan(args.workload)
    layer = make_layer(plan, 0)
    n_dec = 8
    for w in range(args.warmup):
        oracle_sample(plan, layer, n_dec, 0, offset=w)
    total_s, total_b = 0.0, 0
    for k in range(args.steps):
        s, b, nr, npq = oracle_sample(plan, layer, n_dec, 0, offset=(args.warmup + k) * n_dec)
        total_s += s
        total_b += b
    gbs = total_b / total_s / 1e9
    sample = (f"per step: {nr} decode sequences (rotating) and {npq} prefill queries of one "
              f"layer of the {workload_config(plan)['workload']} step, float64 numpy oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(plan),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample, **host_info()},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _events(torch):
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def capture(torch, dev, fn):
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


def time_replays(torch, stream, run, reps, flush=None, min_seconds=0.0, est_ms=None):
    """Per-replay device times (ms) of ``run``: CUDA events on ``stream``
    around each replay, ``flush`` (an L2 flush) between replays outside the
    events.  At least ``reps`` replays, more to fill ``min_seconds``."""
    n = reps
    if est_ms and min_seconds > 0:
        n = max(reps, min(4000, int(min_seconds * 1e3 / max(est_ms, 1e-3))))
    evs = []
    for _ in range(n):
        if flush is not None:
            flush()
        a, b = _events(torch)
        a.record(stream)
        run()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def summarize(ms):
    a = np.asarray(ms, dtype=np.float64)
    return {"median": float(np.median(a)), "min": float(a.min()), "max": float(a.max()),
            "mean": float(a.mean()), "reps": int(a.size)}


class DecodeCalls:
    """The decode half of one step on the GPU, every layer: the work split
    planned once for all layers (several layers), then per layer the
    decode call with the step's K/V rows written in the same launch
    (pkv_paged_attention_decode_append / _planned with k_new, v_new)."""

    def __init__(self, pkv, torch, plan, layers, dev, *, fused=True, planned=None,
                 shared_prefix=False, err=None):
        nd = plan.n_decode
        sh = plan.shape
        self.pkv, self.sh, self.nd, self.layers = pkv, sh, nd, layers
        self.bt = torch.from_numpy(plan.block_tables[:nd]).to(dev)
        self.sl = torch.from_numpy(plan.seq_lens[:nd]).to(dev)
        self.max_dec = int(plan.seq_lens[:nd].max()) if nd else 0
        self.P = len(plan.shared_prefix_blocks) if shared_prefix else 0
        self.planned = (len(layers) > 1) if planned is None else planned
        self.fused = fused and (self.P == 0 or self.planned)
        ws_bytes = (pkv.decode_shared_prefix_workspace_bytes(nd, sh.n_heads, sh.head_dim,
                                                             self.max_dec, self.P)
                    if self.P else pkv.decode_workspace_bytes(nd, sh.n_heads, sh.head_dim,
                                                              self.max_dec))
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        self.out = [torch.empty((nd, sh.n_heads, sh.head_dim), dtype=sh.torch_dtype, device=dev)
                    for _ in layers]
        self.err = err if err is not None else torch.zeros(1, dtype=torch.int32, device=dev)

    def launches(self):
        """Kernel launches of one call of run() (the plan's, the prefix
        runs' and combine's, the main kernel and the merge per layer)."""
        if not self.nd:
            return 0
        per_layer = (2 if self.planned or self.nd <= 2048 else 3) + (2 if self.P else 0)
        return (1 if self.planned else 0) + len(self.layers) * per_layer

    def call(self, li, q, k, v, bt, sl, out):
        pkv, sh, nd, P = self.pkv, self.sh, self.nd, self.P
        lay = self.layers[li]
        kn, vn = (k[:nd], v[:nd]) if self.fused else (None, None)
        if self.planned:
            pkv.paged_attention_decode_planned(q[:nd], lay["k_pool"], lay["v_pool"], bt, sl,
                                               sh.scale, self.max_dec, workspace=self.ws,
                                               k_new=kn, v_new=vn, shared_prefix_blocks=P,
                                               out=out, err=self.err)
        elif P:
            pkv.paged_attention_decode_shared_prefix(q[:nd], lay["k_pool"], lay["v_pool"], bt, sl,
                                                     sh.scale, P, self.max_dec, out=out,
                                                     workspace=self.ws, err=self.err)
        elif kn is not None:
            pkv.paged_attention_decode_append(q[:nd], kn, vn, lay["k_pool"], lay["v_pool"], bt,
                                              sl, sh.scale, self.max_dec, out=out,
                                              workspace=self.ws, err=self.err)
        else:
            pkv.paged_attention_decode(q[:nd], lay["k_pool"], lay["v_pool"], bt, sl, sh.scale,
                                       self.max_dec, out=out, workspace=self.ws, err=self.err)

    def plan_call(self, sl):
        self.pkv.decode_plan(self.layers[0]["k_pool"], sl, self.sh.n_heads, self.bt.shape[1],
                             self.max_dec, workspace=self.ws, shared_prefix_blocks=self.P,
                             err=self.err)

    def run(self, inputs=None, outs=None, before_layer=None):
        """One decode half.  inputs: (bt, seq_lens, [(q, k, v) per layer])
        device tensors (default: the resident ones); before_layer(li) runs
        ahead of layer li's call (e.g. a separate KV write)."""
        if not self.nd:
            return
        bt, sl = (self.bt, self.sl) if inputs is None else inputs[:2]
        if self.planned:
            self.plan_call(sl)
        for li, lay in enumerate(self.layers):
            q, k, v = (lay["q"], lay["k"], lay["v"]) if inputs is None else inputs[2][li]
            if before_layer is not None:
                before_layer(li)
            self.call(li, q, k, v, bt, sl, (outs or self.out)[li])


def per_config_entry(torch, pkv, dev, stream, local, name, args, hbm, peak_src, layers=None,
                     layers_cpu0=None, plan=None, shared_prefix=False):
    """The decode call of one workload shape, as its step makes it: every
    layer's call (work split planned once when there are several layers,
    the step's K/V write fused in) replayed as one CUDA graph at least
    args.reps times after 5 warm-up replays; per-layer time = median replay
    / layers.  L2 is flushed between replays when a replay's bytes would
    not push the previous replay's data out of L2.  Layer 0's output is
    compared with the float64 oracle on every decode row."""
    from workloads import TIMED_LAYERS, draw_plan, make_layer, make_layer_on_device
    if plan is None:
        plan = draw_plan(name)
    sh = plan.shape
    n_layers = TIMED_LAYERS[sh.name]
    if layers is None:
        layers_cpu0 = make_layer(plan, 0)
        layers = [{n: t.to(dev) for n, t in layers_cpu0.items()}]
        layers += [make_layer_on_device(plan, li, dev) for li in range(1, n_layers)]
    dc = DecodeCalls(pkv, torch, plan, layers, dev, shared_prefix=shared_prefix)
    acc = step_accounting(plan)
    per_layer_bytes = acc["decode_bytes"] + (acc["append_bytes"] if dc.fused else 0)
    replay_bytes = per_layer_bytes * len(layers)
    g = capture(torch, dev, dc.run)
    flush_buf = None
    if replay_bytes < 4 * L2_BYTES:
        flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    flush = (lambda: flush_buf.fill_(1)) if flush_buf is not None else None
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    est = float(np.median(time_replays(torch, stream, g.replay, 5, flush)))
    with ClockSampler(local) as clk:
        ms = time_replays(torch, stream, g.replay, args.reps, flush, min_seconds=0.4, est_ms=est)
    if int(dc.err.item()) != 0:
        raise RuntimeError(f"{name}: device error bits {int(dc.err.item())}")
    s = summarize(ms)
    layer_ms = s["median"] / len(layers)
    gbs = per_layer_bytes / (layer_ms * 1e-3) / 1e9
    err = oracle_decode_error(plan, layers_cpu0, dc.out[0]) if layers_cpu0 is not None else None
    return {
        "workload": sh.name, "dtype": sh.dtype, "layers_timed": len(layers),
        "layers_model": sh.layers, "decode_seqs": int(plan.n_decode),
        "call": ("decode_plan once per step + paged_attention_decode_planned with k_new/v_new "
                 "per layer" if dc.planned else
                 "paged_attention_decode_append (work split planned inside the call)")
                + (f", shared prefix of {dc.P} blocks read once per chunk of sequences"
                   if dc.P else ""),
        "algorithmic_bytes_per_layer": int(per_layer_bytes),
        "kv_bytes_per_layer": int(acc["decode_kv_bytes"]),
        "ms_per_layer": layer_ms, "replay_ms": s, "gbs": gbs, "peak": hbm,
        "frac": gbs / hbm, "peak_source": f"hbm_gbs of {peak_src}",
        "decode_tokens_per_s": plan.n_decode / (layer_ms * 1e-3 * sh.layers),
        "tokens_per_s_note": f"{plan.n_decode} decode tokens per step of {sh.layers} layers",
        "l2": ("L2 flushed (256 MiB written) between replays" if flush_buf is not None else
               f"a replay reads {replay_bytes / 1e6:.0f} MB, more than 4x L2: no flush"),
        "clocks": clk.summary(), "error_vs_oracle": err,
        "launches_per_replay": dc.launches(),
    }


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
    nd = plan.n_decode
    has_pre = plan.num_seqs > nd
    bt = torch.from_numpy(plan.block_tables).to(dev)
    seq_lens = torch.from_numpy(plan.seq_lens).to(dev)
    cu_new = torch.from_numpy(plan.cu_new_lens).to(dev)
    T = plan.num_new_tokens
    if has_pre:
        cu_q = torch.from_numpy((plan.cu_new_lens[nd:] - plan.cu_new_lens[nd]).astype(np.int32)).to(dev)
        max_q = int(plan.new_lens[nd:].max())
        max_pre = int(plan.seq_lens[nd:].max())
    slots = torch.empty(T, dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    pre_out = [torch.empty((T - nd, sh.n_heads, sh.head_dim), dtype=sh.torch_dtype, device=dev)
               for _ in L] if has_pre else None
    dec = DecodeCalls(pkv, torch, plan, L, dev, fused=not args.separate_write,
                      planned=not args.no_plan and len(L) > 1, shared_prefix=args.shared_prefix,
                      err=err)
    fused = dec.fused

    def slot_call(src_bt, src_sl, src_cu):
        pkv.slot_mapping(src_bt, src_sl, src_cu, T, sh.block_size, sh.num_blocks, out=slots,
                         err=err)

    def decode_half(inputs=None, outs=None):
        """Per layer: (separate write of the decode rows) + the decode call."""
        if not nd:
            return
        src = None if inputs is None else (inputs[0][:nd], inputs[1][:nd], inputs[3])
        before = None
        if not fused:
            slot_call(*((bt, seq_lens, cu_new) if inputs is None else inputs[:3]))

            def before(li):  # the decode rows' tokens come first in the step's token order
                lay = L[li]
                k, v = (lay["k"], lay["v"]) if inputs is None else inputs[3][li][1:]
                pkv.kv_write(k[:nd], v[:nd], slots[:nd], lay["k_pool"], lay["v_pool"], err=err)
        dec.run(src, outs, before)

    def prefill_half(inputs=None, outs=None):
        """Slot mapping (when the decode half did not make it), then per
        layer the prefill chunks' KV write and the prefill call."""
        if not has_pre:
            return
        src_bt, src_sl, src_cu = (bt, seq_lens, cu_new) if inputs is None else inputs[:3]
        if fused:
            slot_call(src_bt, src_sl, src_cu)
        for li, lay in enumerate(L):
            q, k, v = (lay["q"], lay["k"], lay["v"]) if inputs is None else inputs[3][li]
            pkv.kv_write(k[nd:], v[nd:], slots[nd:], lay["k_pool"], lay["v_pool"], err=err)
            pkv.paged_attention_prefill(q[nd:], cu_q, lay["k_pool"], lay["v_pool"], src_bt[nd:],
                                        src_sl[nd:], sh.scale, max_q, max_pre,
                                        out=(outs or pre_out)[li], err=err)

    def prefill_calls():
        for li, lay in enumerate(L):
            pkv.paged_attention_prefill(lay["q"][nd:], cu_q, lay["k_pool"], lay["v_pool"], bt[nd:],
                                        seq_lens[nd:], sh.scale, max_q, max_pre, out=pre_out[li],
                                        err=err)

    dec_launches = dec.launches() + (0 if fused else 1 + n_layers)
    pre_launches = (1 + 2 * n_layers) if has_pre else 0
    launches_per_step = dec_launches + pre_launches

    for _ in range(max(args.warmup, 3)):
        decode_half()
        prefill_half()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} during warm-up")
    use_graph = not args.no_graph
    if use_graph:
        g_dec = capture(torch, dev, decode_half) if nd else None
        g_pre = capture(torch, dev, prefill_half) if has_pre else None
        run_dec = g_dec.replay if g_dec else (lambda: None)
        run_pre = g_pre.replay if g_pre else (lambda: None)
        for _ in range(max(args.warmup, 3)):
            run_dec()
            run_pre()
        torch.cuda.synchronize()
    else:
        run_dec, run_pre = decode_half, prefill_half

    # ---- device-resident timing: K steps, events around each half
    barrier(world)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        for e0, e1, e2 in ev:
            e0.record(stream)
            run_dec()
            e1.record(stream)
            run_pre()
            e2.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = ev[0][0].elapsed_time(ev[-1][2])
    dec_step_ms = [e0.elapsed_time(e1) for e0, e1, _ in ev]
    pre_step_ms = [e1.elapsed_time(e2) for _, e1, e2 in ev]
    ms_max = max_over_ranks(ms, world, dev)
    ms_step = ms_max / args.steps
    dec_total_ms = max_over_ranks(float(np.sum(dec_step_ms)), world, dev)
    dec_bytes_step = (acc["decode_bytes"] + (acc["append_bytes"] if fused else 0)) * n_layers
    value = world * dec_bytes_step * args.steps / (dec_total_ms * 1e-3) / 1e9 if nd else 0.0
    step_bytes = (acc["decode_bytes"] + acc["prefill_bytes"] + acc["write_bytes"]) * n_layers

    # ---- per-call durations of the dominant kernels: graphs of one layer
    # loop of decode calls and of prefill calls, median of >= args.reps replays
    dec_call = pre_call = None
    if nd:
        g_d = capture(torch, dev, dec.run)
        for _ in range(5):
            g_d.replay()
        dec_call = summarize(time_replays(torch, stream, g_d.replay, args.reps))
    if has_pre:
        g_p = capture(torch, dev, prefill_calls)
        for _ in range(5):
            g_p.replay()
        pre_call = summarize(time_replays(torch, stream, g_p.replay, args.reps))

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

        for _ in range(5):
            cow_call()
        c = summarize(time_replays(torch, stream, cow_call, args.reps))
        block_bytes = sh.block_size * sh.n_kv * sh.head_dim * sh.itemsize
        cow_bytes = 2 * 2 * n_cow * block_bytes  # K and V, read and written
        cow = {"pairs": n_cow, "bytes_per_launch": cow_bytes, "ms_per_launch": c["median"],
               "ms": c, "achieved": cow_bytes / (c["median"] * 1e-3) / 1e9, "unit": "GB/s",
               "timing": f"median of {c['reps']} event-timed launches after 5 warm-up launches"}

    # ---- end to end: the decode half with its inputs from pinned host
    # memory and its outputs back, every step
    e2e = None
    if not args.no_e2e and nd:
        host_in = [t.cpu().pin_memory() for t in (bt, seq_lens, cu_new)]
        host_layers = [[lay[n].cpu().pin_memory() for n in ("q", "k", "v")] for lay in L]
        host_out = [o.cpu().pin_memory() for o in dec.out]
        # two sets of device inputs and outputs, alternating between steps, so
        # a step's copies overlap its neighbours' compute
        dev_in = [[torch.empty_like(t) for t in (bt, seq_lens, cu_new)] for _ in range(2)]
        dev_layers = [[[torch.empty_like(lay[n]) for n in ("q", "k", "v")] for lay in L]
                      for _ in range(2)]
        dev_out = [dec.out, [torch.empty_like(o) for o in dec.out]]
        # the fused step needs the decode rows' tables and lengths; a separate
        # write first maps the slots of every token (whole tables, cu_new_lens)
        in_parts = ([slice(0, nd), slice(0, nd)] if fused else
                    [slice(None), slice(None), slice(None)])
        h2d = (sum(t[p].numel() * t.element_size() for t, p in zip(host_in, in_parts)) +
               sum(t[:nd].numel() * t.element_size() for lay in host_layers for t in lay))
        d2h = sum(t.numel() * t.element_size() for t in host_out)
        h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        steps_per_graph = 8  # the graph's first step cannot overlap the one before it

        def e2e_steps():
            # Step i uses buffer set i % 2.  Its copies in start once step i-2
            # has finished computing from that set, so they land while step
            # i-1 computes, and its compute waits for them once.  Each
            # layer's output goes back on a second stream once it is
            # computed, and step i+2 overwrites those outputs only after
            # that copy.  Every step copies all its decode inputs in (the
            # tables, lengths and each layer's q, k, v rows) and all its
            # outputs out.
            main = torch.cuda.current_stream(dev)
            h2d_s.wait_stream(main)
            d2h_s.wait_stream(main)
            computed = [None] * steps_per_graph
            copied_out = [None] * steps_per_graph
            for i in range(steps_per_graph):
                b = i % 2
                if i >= 2:
                    h2d_s.wait_event(computed[i - 2])
                with torch.cuda.stream(h2d_s):
                    for d, h, p in zip(dev_in[b], host_in, in_parts):
                        d[p].copy_(h[p], non_blocking=True)
                    for dl, hl in zip(dev_layers[b], host_layers):
                        for d, h in zip(dl, hl):
                            d[:nd].copy_(h[:nd], non_blocking=True)
                    landed = torch.cuda.Event()
                    landed.record(h2d_s)
                if i >= 2:
                    main.wait_event(copied_out[i - 2])
                main.wait_event(landed)
                inputs = (dev_in[b][0], dev_in[b][1], dev_in[b][2], dev_layers[b])
                decode_half(inputs, outs=dev_out[b])
                e = torch.cuda.Event()
                e.record(main)
                d2h_s.wait_event(e)
                with torch.cuda.stream(d2h_s):
                    for li in range(len(L)):
                        host_out[li].copy_(dev_out[b][li], non_blocking=True)
                computed[i] = torch.cuda.Event()
                computed[i].record(main)
                copied_out[i] = torch.cuda.Event()
                copied_out[i].record(d2h_s)
            main.wait_stream(h2d_s)
            main.wait_stream(d2h_s)

        for _ in range(2):
            e2e_steps()
        torch.cuda.synchronize()
        run_e2e = capture(torch, dev, e2e_steps).replay if use_graph else e2e_steps
        run_e2e()
        torch.cuda.synchronize()
        barrier(world)
        e_reps = max(10, args.steps // steps_per_graph)
        e_ms = time_replays(torch, stream, run_e2e, e_reps)
        e_step = max_over_ranks(float(np.sum(e_ms)), world, dev) / (e_reps * steps_per_graph)
        e2e = {"value": world * dec_bytes_step / (e_step * 1e-3) / 1e9, "unit": "GB/s",
               "ms_per_step": e_step, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h),
               "copies": f"every step copies its decode inputs in (tables, lengths, each layer's "
                         f"q, k, v rows) and its outputs out; double-buffered so a step's copies "
                         f"(one stream in, one out) overlap its neighbours' compute; timed over "
                         f"{e_reps} graphs x {steps_per_graph} steps"}

    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} in the timed region")

    peaks, src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    tc = float(peaks["bf16_tflops"])

    # ---- per config: the decode call of each workload shape
    per_config = None
    if rank == 0 and not args.no_per_config:
        per_config = {}
        for name in [n for n in args.per_config.split(",") if n]:
            if name == sh.name and n_layers == TIMED_LAYERS[sh.name]:
                ent = per_config_entry(torch, pkv, dev, stream, local, name, args, hbm, src,
                                       layers=L, layers_cpu0=layers_cpu[0], plan=plan)
            else:
                ent = per_config_entry(torch, pkv, dev, stream, local, name, args, hbm, src)
            per_config[name] = ent
            torch.cuda.empty_cache()
    # ---- shared-prefix decode: 64 Llama-3.2-1B users behind one 1,024-token
    # prompt, the prompt's blocks counted once in the algorithmic bytes
    shared_prefix = None
    if rank == 0 and not args.no_per_config and "llama-3.2-1b" in args.per_config.split(","):
        shared_prefix = per_config_entry(torch, pkv, dev, stream, local,
                                         "llama-3.2-1b-sharedprompt", args, hbm, src,
                                         shared_prefix=True)
        torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    src_hash = decode_source_hash()
    roof = None
    if nd:
        dms = float(np.median(dec_step_ms)) / n_layers
        per_launch = acc["decode_bytes"] + (acc["append_bytes"] if fused else 0)
        ach = per_launch / (dms * 1e-3) / 1e9
        rec = DECODE_TRAFFIC.get((sh.dtype, sh.n_heads, sh.n_kv, sh.head_dim))
        traffic = None
        note = "no ncu capture of the current decode kernel for this shape"
        if rec and rec["source_sha256"] == src_hash and fused and not args.shared_prefix:
            traffic = rec["ratio"] * per_launch
            note = (f"dram__bytes_read.sum + dram__bytes_write.sum per algorithmic byte "
                    f"({rec['ratio']:.4f}) from {rec['capture']}, times this call's bytes")
        elif rec:
            note = "the recorded capture was of other decode sources or another call"
        roof = {"bound": "hbm",
                "kernel": ("paged_attention_decode_shared_prefix (prefix runs + combine + split "
                           "kernel + merge)" if dec.P else
                           "paged_attention_decode with the K/V write fused (split kernel + merge)"),
                "timing": ("median over the timed steps of CUDA events on the launching stream "
                           "around the step's decode half"
                           + (f" ({n_layers} layers, per layer)" if n_layers > 1 else "")),
                "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "peak_source": f"hbm_gbs of {src}", "traffic": traffic, "traffic_note": note,
                "decode_source_sha256": src_hash,
                "algorithmic_bytes_per_launch": per_launch, "ms_per_launch": dms,
                "replays": ({"ms_per_layer": dec_call["median"] / n_layers, "ms": dec_call,
                             "achieved": per_launch / (dec_call["median"] / n_layers * 1e-3) / 1e9,
                             "timing": f"median of {dec_call['reps']} replays of a graph of the "
                                       f"layer loop of decode calls"} if dec_call else None)}
    pre_roof = None
    if has_pre:
        pms = float(np.median(pre_step_ms)) / n_layers
        tf = acc["prefill_flops"] / (pre_call["median"] / n_layers * 1e-3) / 1e12
        pre_roof = {"bound": "tensor", "kernel": "paged_attention_prefill", "achieved": tf,
                    "peak": tc, "unit": "TFLOP/s", "frac": tf / tc,
                    "peak_source": f"bf16_tflops of {src}", "flops_per_launch": acc["prefill_flops"],
                    "ms_per_launch": pre_call["median"] / n_layers, "ms": pre_call,
                    "timing": f"median of {pre_call['reps']} replays of a graph of the layer loop "
                              f"of prefill calls",
                    "prefill_half_ms_per_step": pms,
                    "traffic": None, "traffic_note": "tensor-bound: DRAM bytes are not its limit"}
    cpu = None
    if not args.no_cpu_baseline:
        # passes over layer 0's decode sequences until about 10 s of CPU work
        secs = nbytes = nr = passes = 0
        while secs < 10.0 and passes < 50 and nd:
            s_, b_, r_, _ = oracle_sample(plan, layers_cpu[0], nd, 0, offset=passes * 64)
            secs, nbytes, nr, passes = secs + s_, nbytes + b_, nr + r_, passes + 1
        if secs > 0:
            cpu = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                   "sample": f"{passes} passes over layer 0's decode sequences: {nr} sequences in "
                             f"all ({nbytes / 1e6:.0f} MB of KV), float64 numpy oracle, "
                             f"{secs:.1f} s on one thread", **host_info()}
    pages_cpu = None
    if not args.no_cpu_baseline and nd:
        psecs = pbytes = ppasses = 0
        while psecs < 5.0 and ppasses < 20:
            s_, b_ = pages_method_sample(plan, layers_cpu[0], range(nd))
            psecs, pbytes, ppasses = psecs + s_, pbytes + b_, ppasses + 1
        pages_cpu = {"value": pbytes / psecs / 1e9, "unit": "GB/s", "cores": torch.get_num_threads(),
                     "kind": "the pages' method: per-sequence gather + einsum attention, "
                             "fp32 PyTorch on the CPU",
                     "sample": f"{ppasses} passes over layer 0's {nd} decode sequences, "
                               f"{psecs:.1f} s", **host_info()}
    dec_tok_s = (world * nd / (float(np.median(dec_step_ms)) * 1e-3 * (sh.layers / n_layers))
                 if nd else None)
    n_pre_tok = int(plan.new_lens[nd:].sum())
    pre_tok_s = (world * n_pre_tok / (ms_step * 1e-3 * (sh.layers / n_layers))
                 if has_pre else None)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if sh.dtype == "bf16" else "f32",
        "data": "synthetic (seeded; workloads/)",
        "config": workload_config(plan, n_layers),
        "value_note": ("decode attention calls' algorithmic bytes / their device time (events "
                       "around each step's decode half, summed over the timed steps); "
                       "ms_per_step is the whole step"),
        "launch": "cuda_graph per step half" if use_graph else "eager",
        "decode_write": ("fused into the decode launch" if fused
                         else "separate kv_write launch"),
        "decode_shared_prefix_blocks": dec.P,
        "decode_plan": ("once per step for all timed layers (decode_plan + decode_planned)"
                        if dec.planned else "inside each decode call"),
        "decode_ms_per_step": float(np.median(dec_step_ms)),
        "prefill_ms_per_step": float(np.median(pre_step_ms)) if has_pre else None,
        "decode_tokens_per_s": dec_tok_s,
        "decode_tokens_per_s_note": f"{nd} decode tokens per step of {sh.layers} layers, "
                                    f"{n_layers} timed layer(s) scaled by {sh.layers / n_layers:g}",
        "percent_of_hbm_peak": 100.0 * value / world / hbm,
        "step_gbs": world * step_bytes / (ms_step * 1e-3) / 1e9,
        "step_gbs_note": "all algorithmic bytes of the step (decode, prefill, writes) / step time",
        "prefill_tokens_per_s": pre_tok_s,
        "roofline": roof or pre_roof, "prefill_roofline": pre_roof,
        "per_config": per_config,
        "decode_shared_prefix": shared_prefix,
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
