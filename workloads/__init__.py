"""Seeded synthetic inputs for the paged KV cache write and paged attention.

This module is shared by the tests, the benchmark and the smoke check, and
feeds both the CUDA library and the CPU oracle.  It only *draws* inputs:
sequence lengths, block tables (which physical blocks each sequence was
handed), query/key/value values and pool contents.  It holds none of the
method's arithmetic: no slot computation, no scatter, no gather, no softmax.

Shapes follow the model families the pages measure or size:

* ``toy``            mini-vLLM toy model ("Build a Mini vLLM", section 1:
                     8 query heads, 4 KV heads, head_dim 16, 16-token blocks).
* ``smollm2-135m``   SmolLM2-135M as served by "nano-vLLM" (How it works:
                     pool [blocks, 16, 3 KV heads, 64], 30 layers, block 0 is a
                     dummy, a shared 32-token system prompt in blocks 1 and 2).
* ``llama-3.2-1b``   Llama-3.2-1B ("Day 16" / "Day 38": 16 layers, 8 KV heads,
                     32 query heads, head_dim 64, 16-token blocks, bf16).
* ``llama-7b``       LLaMA-7B MHA ("Build a Mini vLLM", section 1 table).
* ``llama2-70b-mixed`` LLaMA-2-70B GQA-8 ("Build a Mini vLLM", section 1
                     table), one layer of a mixed decode + chunked-prefill step.

Recipe:
  * lengths and tables: ``numpy.random.default_rng(1000 + config_id)``;
  * values: ``torch.Generator('cpu').manual_seed(2000 + 1000*config_id + layer)``,
    N(0, 1) in fp32, cast (round-to-nearest-even) to bf16 where the shape is bf16;
  * block tables: sequences take consecutive runs of a seeded permutation of
    the non-dummy block ids; padding entries hold block 0;
  * pool: every block handed to some sequence is filled with N(0, 1) values
    (all of its slots, including a last block's unused tail); blocks nobody
    holds are filled with ``fill`` (0 for timing, a large sentinel or NaN in
    masking tests);
  * timing-only layers (``make_layer_on_device``: the layers after the first
    of a many-layer step, whose outputs nothing checks): the same shapes and
    distribution, drawn by a ``torch.Generator`` on the GPU seeded with
    ``7000 + 1000*config_id + layer`` (drawing gigabytes of pool on the host
    would dominate the benchmark's run time).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

__all__ = ["Shape", "SHAPES", "CONFIG_IDS", "draw_plan", "make_layer", "make_layer_on_device", "Plan"]


@dataclass(frozen=True)
class Shape:
    name: str
    dtype: str          # "f32" or "bf16"
    layers: int         # layers of one step of this model family
    n_heads: int
    n_kv: int
    head_dim: int
    block_size: int
    num_blocks: int
    dummy_block0: bool  # block 0 reserved (never handed out, pads short tables)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def itemsize(self) -> int:
        return 4 if self.dtype == "f32" else 2


SHAPES = {
    "toy": Shape("toy", "f32", 4, 8, 4, 16, 16, 64, True),
    "smollm2-135m": Shape("smollm2-135m", "bf16", 30, 9, 3, 64, 16, 1024, True),
    "llama-3.2-1b": Shape("llama-3.2-1b", "bf16", 16, 32, 8, 64, 16, 32768, True),
    "llama-7b": Shape("llama-7b", "bf16", 32, 32, 32, 128, 16, 2048, False),
    "llama2-70b-mixed": Shape("llama2-70b-mixed", "bf16", 80, 64, 8, 128, 16, 65536, True),
    # the prefill half of the 70B mixed step alone, in a small pool (profiling)
    "llama2-70b-prefill": Shape("llama2-70b-prefill", "bf16", 80, 64, 8, 128, 16, 2048, True),
    # 64 of the 70B step's decode sequences in an 8,192-block pool (profiling)
    "llama2-70b-decode64": Shape("llama2-70b-decode64", "bf16", 80, 64, 8, 128, 16, 8192, True),
    # batched full-prompt prefill: every user arriving together is prefilled
    # in one pass (history 0), the SmolLM2 server's 30 users and a
    # Llama-3.2-1B batch of 32 prompts
    "smollm2-135m-prompts": Shape("smollm2-135m-prompts", "bf16", 30, 9, 3, 64, 16, 1024, True),
    "llama-3.2-1b-prompts": Shape("llama-3.2-1b-prompts", "bf16", 16, 32, 8, 64, 16, 8192, True),
    # 64 users behind one long common prompt (1,024 tokens, 64 shared blocks)
    "llama-3.2-1b-sharedprompt": Shape("llama-3.2-1b-sharedprompt", "bf16", 16, 32, 8, 64, 16,
                                       4096, True),
}
CONFIG_IDS = {"toy": 1, "smollm2-135m": 2, "llama-3.2-1b": 3, "llama-7b": 4, "llama2-70b-mixed": 5,
              "llama2-70b-prefill": 6, "llama2-70b-decode64": 7, "smollm2-135m-prompts": 8,
              "llama-3.2-1b-prompts": 9, "llama-3.2-1b-sharedprompt": 10}

# Layers materialised (each with its own pool) in one timed step.  The toy
# step is one layer.  One 70B pool of 65,536 blocks is 4.3 GB, so that step
# is timed on one layer and per-step token rates are scaled by its 80 layers.
TIMED_LAYERS = {"toy": 1, "smollm2-135m": 30, "llama-3.2-1b": 16, "llama-7b": 32, "llama2-70b-mixed": 1,
                "llama2-70b-prefill": 1, "llama2-70b-decode64": 1, "smollm2-135m-prompts": 30,
                "llama-3.2-1b-prompts": 16, "llama-3.2-1b-sharedprompt": 16}


@dataclass
class Plan:
    """Lengths and block tables of one step (shared by every layer)."""
    shape: Shape
    seq_lens: np.ndarray        # int32 [B], tokens after this step's write
    new_lens: np.ndarray        # int32 [B], tokens written this step (1 = decode)
    block_tables: np.ndarray    # int32 [B, W], padded with block 0
    held_blocks: np.ndarray     # int64 [n], every block id some sequence holds
    n_decode: int               # rows [0, n_decode) decode, the rest prefill
    shared_prefix_blocks: tuple = field(default_factory=tuple)

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def cu_new_lens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.new_lens)]).astype(np.int32)

    @property
    def num_new_tokens(self) -> int:
        return int(self.new_lens.sum())


def _blocks_held(length: int, block_size: int) -> int:
    # A sequence of `length` tokens holds ceil(length / block_size) blocks
    # ("Build a Mini vLLM", section 2: on-demand allocation).
    return -(-int(length) // block_size)


def draw_plan(name: str, *, num_seqs: int | None = None) -> Plan:
    """Seeded lengths and block tables for one of the named shapes.

    ``num_seqs`` overrides the batch for the uniform-length shapes (used by
    small test cases); the default is each shape's own batch.
    """
    sh = SHAPES[name]
    cid = CONFIG_IDS[name]
    rng = np.random.default_rng(1000 + cid)
    bs = sh.block_size
    shared: tuple = ()
    n_decode = None
    if name == "toy":
        lens = np.array([7, 16, 33, 100], dtype=np.int64)
    elif name == "smollm2-135m":
        b = 30 if num_seqs is None else num_seqs
        # prompt (>= the shared 32-token system prompt) + generated tokens;
        # the lower bound 33 keeps this step's new token out of the shared blocks.
        lens = rng.integers(33, 613, size=b)
        shared = (1, 2)
    elif name == "llama-3.2-1b":
        b = 64 if num_seqs is None else num_seqs
        lens = rng.integers(512, 2049, size=b)
    elif name == "llama-7b":
        b = 16 if num_seqs is None else num_seqs
        lens = np.full(b, 2048, dtype=np.int64)
    elif name == "llama2-70b-mixed":
        b = 256 if num_seqs is None else num_seqs
        raw = rng.lognormal(mean=math.log(1024.0), sigma=1.0, size=b)
        dec = np.clip(np.rint(raw), 16, 8192).astype(np.int64)
        hist = np.array([0, 1365, 2731, 4096], dtype=np.int64)
        lens = np.concatenate([dec, hist + 512])
        n_decode = b
    elif name == "llama2-70b-prefill":
        lens = np.array([0, 1365, 2731, 4096], dtype=np.int64) + 512
        n_decode = 0
    elif name == "llama2-70b-decode64":
        b = 64 if num_seqs is None else num_seqs
        raw = rng.lognormal(mean=math.log(1024.0), sigma=1.0, size=b)
        lens = np.clip(np.rint(raw), 16, 8192).astype(np.int64)
    elif name == "smollm2-135m-prompts":
        # the SmolLM2 server's prompts (system prompt + question) of 30 users
        # arriving together, each prefilled whole
        b = 30 if num_seqs is None else num_seqs
        lens = rng.integers(33, 613, size=b)
        n_decode = 0
    elif name == "llama-3.2-1b-prompts":
        b = 32 if num_seqs is None else num_seqs
        lens = rng.integers(128, 2049, size=b)
        n_decode = 0
    elif name == "llama-3.2-1b-sharedprompt":
        # a 1,024-token common prompt (blocks 1..64) plus each user's own
        # 16..512 tokens, so every step's token lands in a private block
        b = 64 if num_seqs is None else num_seqs
        lens = 1024 + rng.integers(16, 513, size=b)
        shared = tuple(range(1, 65))
    else:
        raise KeyError(name)

    B = lens.shape[0]
    if n_decode is None:
        n_decode = B
    new_lens = np.ones(B, dtype=np.int64)
    new_lens[n_decode:] = 512
    if name.endswith("-prompts"):
        new_lens[:] = lens  # the whole prompt is this step's chunk (history 0)

    first_free = 1 if sh.dummy_block0 else 0
    first_private = first_free + len(shared)
    perm = rng.permutation(np.arange(first_private, sh.num_blocks, dtype=np.int64))
    nblocks = np.array([_blocks_held(l, bs) for l in lens], dtype=np.int64)
    W = int(nblocks.max())
    tables = np.zeros((B, W), dtype=np.int64)
    held = set(shared)
    cursor = 0
    for i in range(B):
        row = list(shared)
        need = int(nblocks[i]) - len(row)
        if cursor + need > perm.shape[0]:
            raise ValueError(f"{name}: pool of {sh.num_blocks} blocks is too small")
        row += perm[cursor:cursor + need].tolist()
        cursor += need
        tables[i, :len(row)] = row
        held.update(row)
    return Plan(sh, lens.astype(np.int32), new_lens.astype(np.int32),
                tables.astype(np.int32), np.array(sorted(held), dtype=np.int64),
                n_decode, shared)


def make_layer(plan: Plan, layer: int = 0, *, fill: float = 0.0, device="cpu"):
    """Seeded values of one layer: new q/k/v for this step and the pools.

    Returns a dict of torch tensors (created on the CPU, then moved to
    ``device``):
      q      [T, n_heads, head_dim]   T = number of tokens written this step
      k, v   [T, n_kv, head_dim]      this step's new keys / values
      k_pool, v_pool [num_blocks, block_size, n_kv, head_dim]
    """
    sh = plan.shape
    g = torch.Generator(device="cpu").manual_seed(2000 + 1000 * CONFIG_IDS[sh.name] + layer)
    T = plan.num_new_tokens
    dt = sh.torch_dtype
    q = torch.randn(T, sh.n_heads, sh.head_dim, generator=g).to(dt)
    k = torch.randn(T, sh.n_kv, sh.head_dim, generator=g).to(dt)
    v = torch.randn(T, sh.n_kv, sh.head_dim, generator=g).to(dt)
    pool_shape = (sh.num_blocks, sh.block_size, sh.n_kv, sh.head_dim)
    held = torch.from_numpy(plan.held_blocks)
    k_pool = torch.full(pool_shape, fill, dtype=dt)
    v_pool = torch.full(pool_shape, fill, dtype=dt)
    k_pool[held] = torch.randn(len(held), *pool_shape[1:], generator=g).to(dt)
    v_pool[held] = torch.randn(len(held), *pool_shape[1:], generator=g).to(dt)
    out = dict(q=q, k=k, v=v, k_pool=k_pool, v_pool=v_pool)
    if device != "cpu":
        out = {n: t.to(device) for n, t in out.items()}
    return out


def tiny_plan(lengths, new_lens, *, n_heads, n_kv, head_dim, block_size, num_blocks,
              dtype="f32", seed=0, dummy_block0=True, shared=()) -> Plan:
    """A hand-sized plan for small parity and edge cases (same table recipe)."""
    sh = Shape("tiny", dtype, 1, n_heads, n_kv, head_dim, block_size, num_blocks, dummy_block0)
    rng = np.random.default_rng(seed)
    lens = np.asarray(lengths, dtype=np.int64)
    B = lens.shape[0]
    first_private = (1 if dummy_block0 else 0) + len(shared)
    perm = rng.permutation(np.arange(first_private, num_blocks, dtype=np.int64))
    nblocks = np.array([_blocks_held(l, block_size) for l in lens], dtype=np.int64)
    W = max(1, int(nblocks.max()) if B else 1)
    tables = np.zeros((B, W), dtype=np.int64)
    held, cursor = set(shared), 0
    for i in range(B):
        row = list(shared)[: int(nblocks[i])]
        need = int(nblocks[i]) - len(row)
        if cursor + need > perm.shape[0]:
            raise ValueError("pool too small")
        row += perm[cursor:cursor + need].tolist()
        cursor += need
        tables[i, :len(row)] = row
        held.update(row)
    new = np.asarray(new_lens, dtype=np.int64)
    n_decode = 0  # leading rows that write one token (decode); the rest are prefill chunks
    while n_decode < B and new[n_decode] == 1:
        n_decode += 1
    return Plan(sh, lens.astype(np.int32), new.astype(np.int32), tables.astype(np.int32),
                np.array(sorted(held), dtype=np.int64), n_decode, tuple(shared))


def make_tiny_layer(plan: Plan, seed: int = 0, *, fill: float = 0.0, device="cpu"):
    """Values for a ``tiny_plan`` (same recipe as ``make_layer``)."""
    sh = plan.shape
    g = torch.Generator(device="cpu").manual_seed(5000 + seed)
    T = plan.num_new_tokens
    dt = sh.torch_dtype
    q = torch.randn(T, sh.n_heads, sh.head_dim, generator=g).to(dt)
    k = torch.randn(T, sh.n_kv, sh.head_dim, generator=g).to(dt)
    v = torch.randn(T, sh.n_kv, sh.head_dim, generator=g).to(dt)
    pool_shape = (sh.num_blocks, sh.block_size, sh.n_kv, sh.head_dim)
    held = torch.from_numpy(plan.held_blocks)
    k_pool = torch.full(pool_shape, fill, dtype=dt)
    v_pool = torch.full(pool_shape, fill, dtype=dt)
    if len(held):
        k_pool[held] = torch.randn(len(held), *pool_shape[1:], generator=g).to(dt)
        v_pool[held] = torch.randn(len(held), *pool_shape[1:], generator=g).to(dt)
    out = dict(q=q, k=k, v=v, k_pool=k_pool, v_pool=v_pool)
    if device != "cpu":
        out = {n: t.to(device) for n, t in out.items()}
    return out


def make_layer_on_device(plan: Plan, layer: int, device):
    """A timing-only layer drawn directly on ``device``: the shapes and
    N(0, 1) values of ``make_layer`` (held blocks filled, the rest zero),
    from a device generator seeded per (shape, layer)."""
    sh = plan.shape
    g = torch.Generator(device=device)
    g.manual_seed(7000 + 1000 * CONFIG_IDS[sh.name] + layer)
    T = plan.num_new_tokens
    dt = sh.torch_dtype

    def draw(*shape):
        return torch.randn(*shape, generator=g, device=device).to(dt)

    q = draw(T, sh.n_heads, sh.head_dim)
    k = draw(T, sh.n_kv, sh.head_dim)
    v = draw(T, sh.n_kv, sh.head_dim)
    pool_shape = (sh.num_blocks, sh.block_size, sh.n_kv, sh.head_dim)
    held = torch.from_numpy(plan.held_blocks).to(device)
    k_pool = torch.zeros(pool_shape, dtype=dt, device=device)
    v_pool = torch.zeros(pool_shape, dtype=dt, device=device)
    k_pool[held] = draw(len(held), *pool_shape[1:])
    v_pool[held] = draw(len(held), *pool_shape[1:])
    return dict(q=q, k=k, v=v, k_pool=k_pool, v_pool=v_pool)
