/*
 * pkv.h - C ABI of the GB300 (sm_103a) paged KV cache library.
 *
 * The library implements the data-parallel hot path of a paged-KV-cache
 * serving engine:
 *
 *   pkv_slot_mapping              where this step's new tokens go
 *   pkv_kv_write                  scatter the new K/V into the block pool
 *   pkv_paged_attention_decode    one query token per sequence over its pages
 *   pkv_paged_attention_prefill   a causal query chunk over paged history
 *   pkv_kv_gather                 block table -> contiguous K/V (test/debug)
 *
 * and, around those: pkv_paged_attention_decode_append (the step's K/V
 * stored and attended in one launch), pkv_paged_attention_decode_shared_prefix
 * (a common prompt prefix read once per step), pkv_decode_plan +
 * pkv_paged_attention_decode_planned (the decode work split made once per
 * step for every layer), pkv_copy_blocks (copy-on-write),
 * pkv_paged_attention_decode_noalloc (decode without a caller workspace),
 * the workspace size queries, pkv_status_string, pkv_abi_version and
 * pkv_selftest_bounded_wait (the kernels' bounded-wait failure path).
 *
 * Sources of the operations (page title, section):
 *   - "Build a Mini vLLM: Paged KV Cache and Continuous Batching From
 *     Scratch", section 2 (KVPool, BlockManager.append_slot), section 3
 *     (gather_kv, paged_attention), section 4 (prefill / decode_step);
 *   - "Day 16: the paged KV cache, real K/V through scattered blocks",
 *     What I added today (flat per-layer pool indexed by slot) and What I
 *     learned 1-3 (one block table shared by every layer; the table grows
 *     once per step; write is a scatter, read is a gather);
 *   - "nano-vLLM", How it works (pool [blocks, 16, KV heads, head_dim] per
 *     layer, K/V written at block table[n // 16], slot n % 16, masked
 *     attention with query heads grouped onto their shared K/V head) and
 *     Correctness (masked slots must not reach the output).
 *
 * Conventions shared by every call
 * --------------------------------
 *  Memory.  Every pointer argument except `pool` (a host struct) is DEVICE
 *  memory owned by the caller, contiguous and row-major.  Tensors read or
 *  written as 16-byte vectors (q, k, v, pools, out) must be 16-byte
 *  aligned.  The library never allocates device memory and never
 *  synchronises the device.  The only state it keeps between calls is
 *  host-side, per device: cached launch set-up (each kernel's shared-memory
 *  opt-in and occupancy, the SM count), held in atomics; and, for
 *  pkv_paged_attention_decode_noalloc alone, one fixed device array
 *  compiled into the library and its looked-up address (see that entry).
 *
 *  Streams.  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *  default stream).  Every call only enqueues work on that stream and
 *  returns; results are visible to later work on the same stream.  Calls
 *  are thread-safe, except that pkv_paged_attention_decode_noalloc calls
 *  whose kernels overlap on the GPU race on its shared array (see there).
 *
 *  Pool layout.  One pool per layer for K and one for V, each
 *  [num_blocks, block_size, n_kv, head_dim] of `dtype`.  Slot
 *  s = block * block_size + offset addresses row s of the flat view
 *  [num_blocks * block_size, n_kv, head_dim].  Block tables, sequence
 *  lengths and slot mappings are shared by all layers of a step; pass the
 *  same device arrays to each layer's call.
 *
 *  Block tables.  int32 [num_seqs, max_blocks_per_seq]; row b lists the
 *  physical blocks of sequence b in logical order.  Entries at index
 *  >= ceil(seq_lens[b] / block_size) are never used as block ids (short
 *  rows may be padded with any value, e.g. a dummy block 0; the decode
 *  may load them along with the entries it uses, from within the
 *  [num_seqs, max_blocks_per_seq] array).  Several rows may name
 *  the same block (shared prefix): it is read, never written, by attention.
 *
 *  Errors.  Argument checks run on the host before anything is enqueued;
 *  a failing check returns its status and enqueues nothing.  Data held in
 *  device memory (block ids, slots, lengths) cannot be checked before
 *  launch: kernels check every value before using it as an address, skip
 *  the access (reading zeros / writing nothing) and, if `err_word` is not
 *  NULL, atomically OR one of the PKV_DEVERR_* bits into *err_word (a
 *  device int32 the caller zeroes).  Kernels never trap.  PKV_ERR_CUDA is
 *  returned if a launch fails.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_NULL = 1,        /* a required pointer is NULL                      */
  PKV_ERR_SHAPE = 2,       /* a size is negative or sizes disagree            */
  PKV_ERR_DTYPE = 3,       /* unknown dtype code                              */
  PKV_ERR_ALIGN = 4,       /* a vector-accessed pointer is not 16-byte aligned */
  PKV_ERR_RANGE = 5,       /* a host-side value is out of range               */
  PKV_ERR_WORKSPACE = 6,   /* workspace missing or smaller than required      */
  PKV_ERR_UNSUPPORTED = 7, /* head_dim / block_size / group not compiled in   */
  PKV_ERR_CUDA = 8         /* a CUDA launch or attribute call failed          */
} pkv_status;

typedef enum pkv_dtype {
  PKV_F32 = 0,   /* IEEE binary32 */
  PKV_BF16 = 1   /* bfloat16; attention accumulates in fp32, rounds RNE   */
} pkv_dtype;

/* Bits OR-ed into *err_word by kernels that meet bad device-resident data. */
#define PKV_DEVERR_BLOCK_ID    1  /* block table entry outside [0, num_blocks)       */
#define PKV_DEVERR_SLOT        2  /* slot >= num_blocks * block_size                 */
#define PKV_DEVERR_TABLE_WIDTH 4  /* a length needs more blocks than a table row has */
#define PKV_DEVERR_LENGTH      8  /* a length < 0, > max_seq_len, or < its chunk      */
#define PKV_DEVERR_TIMEOUT    16  /* a pipeline wait gave up (kernel returned early) */
#define PKV_DEVERR_PREFIX     32  /* a table does not start with the declared shared prefix */
#define PKV_DEVERR_PLAN       64  /* a planned call whose plan was made for other sizes     */

/* Shape of one layer's K pool (the V pool has the same shape). */
typedef struct pkv_pool_desc {
  int32_t num_blocks;
  int32_t block_size;  /* tokens per block                                   */
  int32_t n_kv;        /* KV heads                                           */
  int32_t head_dim;
  int32_t dtype;       /* pkv_dtype                                          */
} pkv_pool_desc;

/* Human-readable name of a status code (static string, never NULL). */
const char* pkv_status_string(int32_t status);

/* ABI version of this library: 1. */
int32_t pkv_abi_version(void);

/*
 * pkv_slot_mapping - flat pool slot of every token written this step.
 *
 * "Build a Mini vLLM" section 2 (append_slot): the token at logical
 * position p of a sequence lives in block table[p // block_size] at offset
 * p % block_size.  Sequence b writes its last n_b = cu_new_lens[b+1] -
 * cu_new_lens[b] tokens, at positions seq_lens[b] - n_b .. seq_lens[b]-1
 * (seq_lens counts the tokens after this step's write: a decode step has
 * n_b = 1 and its token at position seq_lens[b] - 1).
 *
 *   block_tables   int32 [num_seqs, max_blocks_per_seq]
 *   seq_lens       int32 [num_seqs]
 *   cu_new_lens    int32 [num_seqs + 1], cu_new_lens[0] = 0, nondecreasing,
 *                  cu_new_lens[num_seqs] = num_tokens
 *   slot_mapping   int64 [num_tokens] (output):
 *                  block * block_size + offset, or -1 where the data were
 *                  bad (err_word records why)
 *   num_blocks     pool size, used to range-check block ids
 */
pkv_status pkv_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* seq_lens, const int32_t* cu_new_lens,
                            int32_t num_seqs, int32_t num_tokens,
                            int32_t block_size, int32_t num_blocks,
                            int64_t* slot_mapping, int32_t* err_word, void* stream);

/*
 * pkv_kv_write - scatter this step's new K and V into the pools.
 *
 * "Day 16", What I learned 3 (write: pool[slots] = k) and "Build a Mini
 * vLLM" section 4 (prefill / decode_step store each token's K/V at its
 * slot before attention reads it).  For every token t with
 * slot_mapping[t] >= 0:
 *     k_pool_flat[slot_mapping[t]] = k[t],  v_pool_flat[slot_mapping[t]] = v[t]
 * copied bit for bit.  A negative slot skips the token (padding).  Slots
 * must be distinct within one call (otherwise which token lands is
 * unspecified).
 *
 *   k, v      [num_tokens, n_kv, head_dim] of pool->dtype, 16-byte aligned
 *   k_pool, v_pool  pools described by *pool, 16-byte aligned
 *   n_kv * head_dim * sizeof(dtype) must be a multiple of 16 bytes.
 */
pkv_status pkv_kv_write(const void* k, const void* v, const int64_t* slot_mapping,
                        int32_t num_tokens, void* k_pool, void* v_pool,
                        const pkv_pool_desc* pool, int32_t* err_word, void* stream);

/*
 * pkv_kv_gather - the block-table gather of "Build a Mini vLLM" section 3
 * (gather_kv): each sequence's first seq_lens[b] tokens, in logical order,
 * copied into contiguous rows cu_seq_lens[b] .. cu_seq_lens[b+1]-1 of
 * k_out / v_out [total_tokens, n_kv, head_dim].  Bit-exact copies.  The
 * attention calls never materialise this; it exists for tests and debugging.
 *
 *   cu_seq_lens  int32 [num_seqs + 1], cu_seq_lens[b+1]-cu_seq_lens[b] = seq_lens[b]
 */
pkv_status pkv_kv_gather(const void* k_pool, const void* v_pool, const pkv_pool_desc* pool,
                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* seq_lens, const int32_t* cu_seq_lens,
                         int32_t num_seqs, int32_t total_tokens,
                         void* k_out, void* v_out, int32_t* err_word, void* stream);

/*
 * pkv_copy_blocks - copy whole physical blocks of both pools (the copy of
 * copy-on-write prefix sharing).
 *
 * "Build a Mini vLLM", Key Takeaways 6: real engines share the blocks of a
 * common prefix between sequences and copy a shared block before one of
 * them writes into it.  For every pair i:
 *     k_pool[block_pairs[i][1]] = k_pool[block_pairs[i][0]]  (all
 *     block_size x n_kv x head_dim elements, bit for bit), and the same for v_pool
 * The caller then points the writing sequence's table entry at the
 * destination.  Destinations must be distinct and must not be the source
 * of any pair in the same call (then the result is that of copying from
 * the pools as they were before the call); otherwise which bytes land is
 * unspecified.  A pair with an id outside [0, num_blocks) is skipped and
 * reported as PKV_DEVERR_BLOCK_ID.
 *
 *   block_pairs  int32 [num_pairs][2] (source, destination), device memory
 *   k_pool, v_pool  16-byte aligned; n_kv * head_dim * sizeof(dtype) a
 *                   multiple of 16 bytes
 */
pkv_status pkv_copy_blocks(void* k_pool, void* v_pool, const pkv_pool_desc* pool,
                           const int32_t* block_pairs, int32_t num_pairs, int32_t* err_word,
                           void* stream);

/*
 * Workspace for pkv_paged_attention_decode and
 * pkv_paged_attention_decode_append, in bytes (never 0): room for a
 * per-sequence work prefix and two partial results per CTA of the largest
 * grid the current device can run.  max_seq_len and max_ctas are
 * accepted for forward compatibility; block_size must be 16.
 */
size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t n_heads, int32_t head_dim,
                                  int32_t max_seq_len, int32_t max_ctas,
                                  int32_t block_size);

/*
 * pkv_paged_attention_decode - one query token per sequence attends to the
 * sequence's whole history, read in place through its block table.
 *
 * "Build a Mini vLLM" section 3 (paged_attention) and section 4
 * (decode_step): for sequence b and query head h, with kv head
 * g = h / (n_heads / n_kv) (repeat-interleave grouping) and
 * K_b[j] = k_pool[block_tables[b][j / bs]][j % bs][g]:
 *     out[b][h] = sum_{j < seq_lens[b]} softmax_j(scale * q[b][h] . K_b[j]) V_b[j]
 * seq_lens[b] counts this step's token (write it with pkv_kv_write
 * first).  A sequence of length 0 gets a zero output.  Slots past the
 * length and table entries past ceil(len / bs) are never read, so
 * garbage or NaN there cannot reach the output.
 *
 * Work split.  All (sequence, KV-head group, 16-token block) units of the
 * batch are divided into equal contiguous ranges, one per CTA of a
 * persistent grid (max_ctas CTAs if 0 < max_ctas < the device's resident
 * capacity, else one full wave).  A sequence whose units fall inside one
 * range is finished by that CTA; one that spans several ranges is merged
 * from the per-range partial results with log-sum-exp weights.  Split
 * points depend only on logical block positions, the lengths and max_ctas,
 * never on physical block ids, so the output is bit-identical under any
 * physical placement or sharing of blocks.  max_ctas = 1 computes every
 * sequence unsplit.  Small batches (max_ctas = 0, the longest sequence at
 * most 64 blocks, and at most two waves of CTAs) are latency-bound rather
 * than bandwidth-bound; for them each (sequence, KV-head group) is instead
 * split over one thread-block cluster of up to 8 CTAs (about 4 blocks
 * each, contiguous, split points fixed by the length alone), whose partial
 * results are combined in distributed shared memory within the same
 * launch.  Either way the split depends only on logical positions, and
 * identical calls give identical bits.
 *
 *   q, out     [num_seqs, n_heads, head_dim] of pool->dtype
 *   scale      positive and finite (else PKV_ERR_RANGE)
 *   workspace  device scratch of at least pkv_decode_workspace_bytes(...)
 *   Supported: head_dim 16, 32, 64, 128 (f32 and bf16; bf16 64 and 128
 *              run on tensor cores);
 *              block_size 16; n_heads % n_kv == 0, n_heads / n_kv <= 16.
 */
pkv_status pkv_paged_attention_decode(const void* q, int32_t num_seqs, int32_t n_heads,
                                      const void* k_pool, const void* v_pool,
                                      const pkv_pool_desc* pool,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* seq_lens, int32_t max_seq_len,
                                      float scale, int32_t max_ctas, void* out,
                                      void* workspace, size_t workspace_bytes,
                                      int32_t* err_word, void* stream);

/*
 * pkv_paged_attention_decode_shared_prefix - decode attention that reads a
 * prefix shared by every sequence once per step.
 *
 * "nano-vLLM", Where the time went and Next steps 3: with a common prompt,
 * gathering per user reads the shared prefix blocks once per user; a kernel
 * that reads blocks in place should read them once.  The caller declares
 * that the first shared_prefix_blocks entries of every row of
 * block_tables are the same blocks (row 0's entries are used).  The
 * prefix keys are read once per chunk of sequences (as many as the
 * library's shape for the call holds: up to 16 tiles of query rows) and
 * every sequence's query rows attend over the prefix tokens they can see
 * (min(seq_lens[b], shared_prefix_blocks * bs)) in runs of the prefix
 * blocks, several sequences' rows sharing each tensor-core tile; the
 * blocks after the prefix are walked as in pkv_paged_attention_decode and
 * each sequence's runs and own parts are combined with log-sum-exp
 * weights.  The output is the same attention as
 * pkv_paged_attention_decode (within the dtype's tolerance; not bit-equal:
 * the sums are taken in another order).  A row whose first entries differ
 * from row 0's, where the sequence reaches them, is reported as
 * PKV_DEVERR_PREFIX.  shared_prefix_blocks = 0 is plain decode.
 *
 *   shared_prefix_blocks  0 .. max_blocks_per_seq (else PKV_ERR_RANGE)
 *   workspace   at least pkv_decode_shared_prefix_workspace_bytes(...)
 *               (the decode workspace plus up to 16 prefix partials per
 *               query row, at most 1,024 per query head, and 16 bytes
 *               per sequence and query head)
 *   everything else as for pkv_paged_attention_decode
 */
size_t pkv_decode_shared_prefix_workspace_bytes(int32_t num_seqs, int32_t n_heads,
                                                int32_t head_dim, int32_t max_seq_len,
                                                int32_t shared_prefix_blocks, int32_t max_ctas,
                                                int32_t block_size);

pkv_status pkv_paged_attention_decode_shared_prefix(const void* q, int32_t num_seqs,
                                                    int32_t n_heads, const void* k_pool,
                                                    const void* v_pool,
                                                    const pkv_pool_desc* pool,
                                                    const int32_t* block_tables,
                                                    int32_t max_blocks_per_seq,
                                                    const int32_t* seq_lens, int32_t max_seq_len,
                                                    int32_t shared_prefix_blocks, float scale,
                                                    int32_t max_ctas, void* out, void* workspace,
                                                    size_t workspace_bytes, int32_t* err_word,
                                                    void* stream);

/*
 * pkv_paged_attention_decode_append - write this step's K/V and run decode
 * attention, in one launch.
 *
 * "Day 16", What I added (append(layer, k, v) stores the step's K/V and
 * returns the full history for attention) and "nano-vLLM", Where the time
 * went (at small batches the step is dominated by per-operation launch
 * cost; fusing operations removes it).  The result is exactly that of
 *     pkv_kv_write(k_new, v_new, slots) ; pkv_paged_attention_decode(...)
 * with slots[b] = block_tables[b][(seq_lens[b]-1) / bs] * bs
 * + (seq_lens[b]-1) % bs: the pools receive the same bytes and the output
 * is bit-identical to the two calls with the same max_ctas.  Sequences of
 * length 0 write nothing; a sequence whose length is out of range (see the
 * PKV_DEVERR_* bits) or whose last table entry is not a valid block id
 * writes nothing either.  The new row reaches the attention straight from
 * k_new / v_new; the pool copy is stored alongside.
 *
 *   k_new, v_new  [num_seqs, n_kv, head_dim] of pool->dtype, 16-byte aligned
 *   k_pool, v_pool  written at each sequence's last position only
 *   everything else as for pkv_paged_attention_decode (same workspace size)
 */
pkv_status pkv_paged_attention_decode_append(const void* q, const void* k_new, const void* v_new,
                                             int32_t num_seqs, int32_t n_heads, void* k_pool,
                                             void* v_pool, const pkv_pool_desc* pool,
                                             const int32_t* block_tables,
                                             int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                             int32_t max_seq_len, float scale, int32_t max_ctas,
                                             void* out, void* workspace, size_t workspace_bytes,
                                             int32_t* err_word, void* stream);

/*
 * pkv_decode_plan / pkv_paged_attention_decode_planned - the work split of
 * a decode step computed once and reused by every layer.
 *
 * "Day 16: the paged KV cache", What I learned 1-2: one block table serves
 * every layer and grows once per step, at layer 0, so the lengths and
 * tables a decode step reads are the same for all layers.  pkv_decode_plan turns seq_lens into
 * the split of the step's blocks over the decode grid (which CTA walks
 * which blocks) and leaves it in `workspace`; each layer's
 * pkv_paged_attention_decode_planned then reads that plan instead of
 * computing it, and reads its plan, its first table entries and (bf16
 * pools with head_dim 64 or 128) the K/V of its first blocks before
 * waiting for the kernel launched just before it (programmatic dependent
 * launch), so that work overlaps the previous kernel's end.  Those early
 * reads never touch a sequence's last block, the only block a decode step
 * writes: a kernel that can still be running when a planned call starts
 * (one that lets its dependents launch early, as this library's decode
 * kernels do) must not write any other block of the planned call's
 * sequences.  Queries, outputs and every write wait for that kernel.  The outputs are those
 * of pkv_paged_attention_decode (k_new and v_new both NULL) or
 * pkv_paged_attention_decode_append (both given), bit for bit; with
 * shared_prefix_blocks > 0 they are those of
 * pkv_paged_attention_decode_shared_prefix (preceded, when k_new and v_new
 * are given, by pkv_kv_write of each sequence's new token at its last
 * slot; the prefix runs and their combine are launched by each planned
 * call; the plan covers the blocks after the prefix and, for the fused
 * launch, where each sequence's parts are), bit for bit.
 *
 * Contract: the planned calls pass the same num_seqs, n_heads, pool shape,
 * max_blocks_per_seq, seq_lens (pointer and contents), max_seq_len and
 * max_ctas as the plan call, and block_tables, seq_lens and the plan part
 * of the workspace stay unchanged from the plan call to the last planned
 * call (the decode writes only the partial-result part of the workspace,
 * so one workspace serves a whole step's layers in stream order).  The
 * plan reports bad lengths (PKV_DEVERR_LENGTH / _TABLE_WIDTH) once.  A
 * planned call whose batch, shared prefix or grid (max_ctas, device)
 * differs from its plan's reports PKV_DEVERR_PLAN, stores no k_new / v_new
 * row and writes no output that depends on the plan (with a shared prefix,
 * the rows of sequences that end inside the prefix, which the plan does
 * not cover, may still be written); so does one whose workspace was never
 * planned or was last used by a call that plans for itself
 * (pkv_paged_attention_decode and the like).
 *
 *   shared_prefix_blocks  as for pkv_paged_attention_decode_shared_prefix
 *              (0 = none; the same value for the plan and its calls).  With
 *              a shared prefix and k_new / v_new, every sequence's new
 *              token must fall after the prefix (a private block); a
 *              sequence wholly inside the prefix gets no write and is
 *              reported as PKV_DEVERR_PREFIX
 *   workspace  at least pkv_decode_workspace_bytes(...) bytes (with a
 *              shared prefix, pkv_decode_shared_prefix_workspace_bytes),
 *              16-byte aligned (the same workspace for the plan and its
 *              calls)
 *   everything else as for pkv_paged_attention_decode(_append)
 */
pkv_status pkv_decode_plan(int32_t num_seqs, int32_t n_heads, const pkv_pool_desc* pool,
                           int32_t max_blocks_per_seq, const int32_t* seq_lens,
                           int32_t max_seq_len, int32_t shared_prefix_blocks, int32_t max_ctas,
                           void* workspace, size_t workspace_bytes, int32_t* err_word,
                           void* stream);

pkv_status pkv_paged_attention_decode_planned(const void* q, const void* k_new,
                                              const void* v_new, int32_t num_seqs,
                                              int32_t n_heads, void* k_pool, void* v_pool,
                                              const pkv_pool_desc* pool,
                                              const int32_t* block_tables,
                                              int32_t max_blocks_per_seq,
                                              const int32_t* seq_lens, int32_t max_seq_len,
                                              int32_t shared_prefix_blocks, float scale,
                                              int32_t max_ctas, void* out, void* workspace,
                                              size_t workspace_bytes, int32_t* err_word,
                                              void* stream);

/*
 * pkv_paged_attention_prefill - causal attention of a query chunk over the
 * sequence's paged history (chunked prefill).
 *
 * "Build a Mini vLLM" section 4 (prefill: the chunk's K/V is written to
 * the pool first, then causal attention with the triu(1) mask): sequence b
 * owns query rows cu_q_lens[b] .. cu_q_lens[b+1]-1 (c_b of them), the
 * last c_b of its seq_lens[b] tokens.  Query i sits at position
 * p_i = seq_lens[b] - c_b + i and attends keys 0 .. p_i:
 *     out[t][h] = sum_{j <= p_i} softmax_j(scale * q[t][h] . K_b[j]) V_b[j]
 * with the same GQA grouping as decode.  A chunk of one query is a decode.
 *
 *   q, out      [total_q, n_heads, head_dim] of pool->dtype
 *   cu_q_lens   int32 [num_seqs + 1], cu_q_lens[num_seqs] = total_q
 *   max_q_len   host upper bound on every c_b; max_seq_len on seq_lens[b]
 *   workspace   may be NULL (this version needs none); pass
 *               pkv_prefill_workspace_bytes(...) bytes for forward compatibility
 *   Supported: as for decode.
 */
size_t pkv_prefill_workspace_bytes(int32_t num_seqs, int32_t total_q, int32_t n_heads,
                                   int32_t head_dim, int32_t max_seq_len);

pkv_status pkv_paged_attention_prefill(const void* q, const int32_t* cu_q_lens,
                                       int32_t num_seqs, int32_t total_q, int32_t max_q_len,
                                       int32_t n_heads, const void* k_pool, const void* v_pool,
                                       const pkv_pool_desc* pool,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, int32_t max_seq_len,
                                       float scale, void* out,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t* err_word, void* stream);

/*
 * pkv_paged_attention_decode_noalloc - decode attention for callers that
 * cannot allocate device memory.
 *
 * The pages have no counterpart of this entry point.  It computes exactly
 * what pkv_paged_attention_decode computes, with the same arguments minus
 * the workspace, for callers that may not call cudaMalloc or have no
 * scratch to lend: a plug-in inside a framework that owns all device
 * memory through its own arena (a raw cudaMalloc bypasses its accounting
 * and synchronises the whole device), a per-token loop that cannot afford
 * that synchronisation, or a plain C caller without an allocator.
 *
 * Its scratch is one array of PKV_NOALLOC_SCRATCH_BYTES compiled into the
 * library; every GPU that loads the library holds it until the process
 * exits.  The first call on each device looks up the array's device
 * address (make that first call before any stream capture); the address is
 * then cached for the life of the process.  cudaDeviceReset tears the
 * module down and may reload the array elsewhere, so do not call this
 * entry point on a device after resetting it.  The call itself allocates
 * nothing.  Nothing in the array must start at zero.
 * Calls whose kernels overlap on the GPU (e.g. issued on two streams)
 * race on the shared array: issue them on one stream.  A batch needing
 * more scratch than the array holds returns PKV_ERR_WORKSPACE without
 * launching (a smaller max_ctas shrinks the need).
 */
#define PKV_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

pkv_status pkv_paged_attention_decode_noalloc(const void* q, int32_t num_seqs, int32_t n_heads,
                                              const void* k_pool, const void* v_pool,
                                              const pkv_pool_desc* pool,
                                              const int32_t* block_tables,
                                              int32_t max_blocks_per_seq,
                                              const int32_t* seq_lens, int32_t max_seq_len,
                                              float scale, int32_t max_ctas, void* out,
                                              int32_t* err_word, void* stream);

/*
 * pkv_selftest_bounded_wait - check the kernels' failure path on this GPU.
 *
 * The pages have no counterpart of this entry point.  Every wait in the
 * kernels (on an mbarrier phase: a shared-memory stage filled, a stage
 * released) is bounded; when the bound runs out the kernel ORs
 * PKV_DEVERR_TIMEOUT into the error word, lets its own copies land and
 * returns, so the context stays usable.  This launches one thread that
 * waits, with that same wait, on a phase nothing completes, for at most
 * `polls` polls (each try_wait may park the thread briefly), then reports
 * the timeout.  Nothing faults or hangs.
 *
 *   polls     >= 1 (else PKV_ERR_RANGE); a few thousand end in well under a
 *             second
 *   err_word  device int32, required (PKV_ERR_NULL)
 */
pkv_status pkv_selftest_bounded_wait(int32_t polls, int32_t* err_word, void* stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif /* PKV_H */
