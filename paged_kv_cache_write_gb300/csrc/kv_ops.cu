// Slot mapping, scatter write and block-table gather.
//
// "Build a Mini vLLM" section 2 (append_slot: block table[pos // bs],
// offset pos % bs) and section 3 (gather_kv); "Day 16", What I learned 3
// (write is a scatter into the flat per-layer pool, read is a gather).
//
// All three are pure data movement: 16-byte vector copies of token rows
// (n_kv * head_dim elements, contiguous in both the source and the pool's
// flat slot view), one grid-stride loop over (token, vector) pairs so that
// consecutive threads touch consecutive 16-byte words of one row.
#include <cuda_runtime.h>

#include "device.cuh"
#include "host_cache.h"
#include "launch.h"

namespace pkv {

namespace {

constexpr int kThreads = 256;

// Index of the sequence owning row `t` of a ragged batch: the b with
// cu[b] <= t < cu[b+1] (cu nondecreasing, cu[0] = 0).
__device__ __forceinline__ int find_seq(const int32_t* __restrict__ cu, int num_seqs, int t) {
  int lo = 0, hi = num_seqs;  // answer in [lo, hi)
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid;
  }
  return lo;
}

__global__ void slot_mapping_kernel(const int32_t* __restrict__ block_tables, int W,
                                    const int32_t* __restrict__ seq_lens,
                                    const int32_t* __restrict__ cu_new, int num_seqs,
                                    int num_tokens, int bs, int num_blocks,
                                    int64_t* __restrict__ slots, int32_t* err) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < num_tokens;
       t += gridDim.x * blockDim.x) {
    const int b = find_seq(cu_new, num_seqs, t);
    const int L = __ldg(seq_lens + b);
    const int c = __ldg(cu_new + b + 1) - __ldg(cu_new + b);
    const int pos = L - c + (t - __ldg(cu_new + b));
    int64_t slot = -1;
    if (L < 0 || c > L || pos < 0) {
      report(err, PKV_DEVERR_LENGTH);
    } else if (pos / bs >= W) {
      report(err, PKV_DEVERR_TABLE_WIDTH);
    } else {
      const int blk = __ldg(block_tables + (int64_t)b * W + pos / bs);
      if (blk < 0 || blk >= num_blocks) {
        report(err, PKV_DEVERR_BLOCK_ID);
      } else {
        slot = (int64_t)blk * bs + pos % bs;
      }
    }
    slots[t] = slot;
  }
}

// One thread per 16-byte word of K and of V: word w of token t.
__global__ void kv_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                const int64_t* __restrict__ slots, int64_t num_tokens,
                                int words_per_row, uint4* __restrict__ k_pool,
                                uint4* __restrict__ v_pool, int64_t num_slots, int32_t* err) {
  const int64_t total = num_tokens * words_per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / words_per_row;
    const int w = static_cast<int>(i - t * words_per_row);
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;  // padding token
    if (s >= num_slots) {
      if (w == 0) report(err, PKV_DEVERR_SLOT);
      continue;
    }
    const uint4 kw = __ldg(k + i);
    const uint4 vw = __ldg(v + i);
    k_pool[s * words_per_row + w] = kw;
    v_pool[s * words_per_row + w] = vw;
  }
}

// Copy-on-write block copy: CTA i copies block pairs[i][0] onto block
// pairs[i][1] in both pools.  The K and V blocks are one run of 16-byte
// words (K first, then V); each thread moves kCopyUnroll words per pass
// with all loads issued before any store, streaming past the caches (the
// copied data is not read again by this kernel).
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 8;

__global__ void __launch_bounds__(kCopyThreads)
    copy_blocks_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                       const int32_t* __restrict__ pairs, int64_t words_per_block,
                       int num_blocks, int32_t* err) {
  const int src = __ldg(pairs + 2 * int64_t(blockIdx.x));
  const int dst = __ldg(pairs + 2 * int64_t(blockIdx.x) + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0) report(err, PKV_DEVERR_BLOCK_ID);
    return;
  }
  const int64_t n = 2 * words_per_block;
  const uint4* ks = k_pool + src * words_per_block;
  const uint4* vs = v_pool + src * words_per_block;
  uint4* kd = k_pool + dst * words_per_block;
  uint4* vd = v_pool + dst * words_per_block;
  for (int64_t base = threadIdx.x; base < n; base += int64_t(kCopyThreads) * kCopyUnroll) {
    uint4 x[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t i = base + int64_t(u) * kCopyThreads;
      if (i < n) x[u] = i < words_per_block ? __ldcs(ks + i) : __ldcs(vs + (i - words_per_block));
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t i = base + int64_t(u) * kCopyThreads;
      if (i < n) {
        if (i < words_per_block) __stcs(kd + i, x[u]);
        else __stcs(vd + (i - words_per_block), x[u]);
      }
    }
  }
}

__global__ void kv_gather_kernel(const uint4* __restrict__ k_pool, const uint4* __restrict__ v_pool,
                                 int words_per_row, int bs, int num_blocks,
                                 const int32_t* __restrict__ block_tables, int W,
                                 const int32_t* __restrict__ seq_lens,
                                 const int32_t* __restrict__ cu, int num_seqs,
                                 int64_t total_tokens, uint4* __restrict__ k_out,
                                 uint4* __restrict__ v_out, int32_t* err) {
  const int64_t total = total_tokens * words_per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / words_per_row;
    const int w = static_cast<int>(i - r * words_per_row);
    const int b = find_seq(cu, num_seqs, static_cast<int>(r));
    const int pos = static_cast<int>(r - __ldg(cu + b));
    uint4 kw = make_uint4(0, 0, 0, 0), vw = kw;
    if (pos >= __ldg(seq_lens + b)) {
      if (w == 0) report(err, PKV_DEVERR_LENGTH);
    } else if (pos / bs >= W) {
      if (w == 0) report(err, PKV_DEVERR_TABLE_WIDTH);
    } else {
      const int blk = __ldg(block_tables + (int64_t)b * W + pos / bs);
      if (blk < 0 || blk >= num_blocks) {
        if (w == 0) report(err, PKV_DEVERR_BLOCK_ID);
      } else {
        const int64_t src = ((int64_t)blk * bs + pos % bs) * words_per_row + w;
        kw = __ldg(k_pool + src);
        vw = __ldg(v_pool + src);
      }
    }
    k_out[i] = kw;
    v_out[i] = vw;
  }
}

// Grid-stride grid for `work` 16-byte words: at most 8 CTAs per SM of the
// current device.
int grid_for(int64_t work) {
  int64_t blocks = (work + kThreads - 1) / kThreads;
  const int64_t cap = int64_t(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<int>(blocks);
}

}  // namespace

cudaError_t launch_slot_mapping(const int32_t* block_tables, int32_t W, const int32_t* seq_lens,
                                const int32_t* cu_new_lens, int32_t num_seqs, int32_t num_tokens,
                                int32_t block_size, int32_t num_blocks, int64_t* slot_mapping,
                                int32_t* err, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  slot_mapping_kernel<<<grid_for(num_tokens), kThreads, 0, stream>>>(
      block_tables, W, seq_lens, cu_new_lens, num_seqs, num_tokens, block_size, num_blocks,
      slot_mapping, err);
  return cudaGetLastError();
}

cudaError_t launch_kv_write(const void* k, const void* v, const int64_t* slot_mapping,
                            int32_t num_tokens, void* k_pool, void* v_pool, const PoolShape& pool,
                            int32_t* err, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int words = static_cast<int>(pool.row_bytes() / 16);
  const int64_t work = int64_t(num_tokens) * words;
  kv_write_kernel<<<grid_for(work), kThreads, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping, num_tokens, words,
      static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool),
      int64_t(pool.num_blocks) * pool.block_size, err);
  return cudaGetLastError();
}

// Self-test of the bounded waits: one thread waits on an mbarrier phase
// that nothing completes, with the same wait the kernels use but at most
// `polls` polls, then reports PKV_DEVERR_TIMEOUT and returns.
__global__ void bounded_wait_selftest_kernel(uint32_t polls, int32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  if (!mbar_wait(&bar, 0, polls)) report(err, PKV_DEVERR_TIMEOUT);
}

cudaError_t launch_bounded_wait_selftest(uint32_t polls, int32_t* err, cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(polls, err);
  return cudaGetLastError();
}

cudaError_t launch_copy_blocks(void* k_pool, void* v_pool, const PoolShape& pool,
                               const int32_t* pairs, int32_t num_pairs, int32_t* err,
                               cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int64_t words = int64_t(pool.block_size) * pool.row_bytes() / 16;
  copy_blocks_kernel<<<num_pairs, kCopyThreads, 0, stream>>>(
      static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), pairs, words, pool.num_blocks,
      err);
  return cudaGetLastError();
}

cudaError_t launch_kv_gather(const void* k_pool, const void* v_pool, const PoolShape& pool,
                             const int32_t* block_tables, int32_t W, const int32_t* seq_lens,
                             const int32_t* cu_seq_lens, int32_t num_seqs, int32_t total_tokens,
                             void* k_out, void* v_out, int32_t* err, cudaStream_t stream) {
  if (total_tokens == 0) return cudaSuccess;
  const int words = static_cast<int>(pool.row_bytes() / 16);
  const int64_t work = int64_t(total_tokens) * words;
  kv_gather_kernel<<<grid_for(work), kThreads, 0, stream>>>(
      static_cast<const uint4*>(k_pool), static_cast<const uint4*>(v_pool), words,
      pool.block_size, pool.num_blocks, block_tables, W, seq_lens, cu_seq_lens, num_seqs,
      total_tokens, static_cast<uint4*>(k_out), static_cast<uint4*>(v_out), err);
  return cudaGetLastError();
}

}  // namespace pkv
