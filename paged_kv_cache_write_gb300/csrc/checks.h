// Host-side argument checks shared by the extern "C" entry points (abi.cu
// and decode_noalloc.cu), so every entry point that takes the same
// arguments refuses the same arguments with the same status.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pkv.h"
#include "launch.h"

namespace pkv {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline pkv_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return PKV_OK;
  cudaGetLastError();  // clear a sticky launch-configuration error
  return PKV_ERR_CUDA;
}

// A pool descriptor: known dtype, positive sizes, 16-byte token rows and a
// flat slot index that fits in int32.
inline pkv_status check_pool(const pkv_pool_desc* pool, PoolShape* out) {
  if (pool == nullptr) return PKV_ERR_NULL;
  if (pool->dtype != PKV_F32 && pool->dtype != PKV_BF16) return PKV_ERR_DTYPE;
  if (pool->num_blocks <= 0 || pool->block_size <= 0 || pool->n_kv <= 0 || pool->head_dim <= 0)
    return PKV_ERR_SHAPE;
  *out = PoolShape{pool->num_blocks, pool->block_size, pool->n_kv, pool->head_dim, pool->dtype};
  if (out->row_bytes() % 16 != 0) return PKV_ERR_ALIGN;
  if ((int64_t)pool->num_blocks * pool->block_size > INT32_MAX) return PKV_ERR_RANGE;
  return PKV_OK;
}

// Arguments common to decode and prefill attention.  num_seqs == 0 passes
// before the pointer checks (nothing will be read).
inline pkv_status check_attention(const void* q, int32_t num_seqs, int32_t n_heads,
                                  const void* k_pool, const void* v_pool,
                                  const pkv_pool_desc* pool, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                  int32_t max_seq_len, float scale, const void* out,
                                  PoolShape* shape) {
  pkv_status st = check_pool(pool, shape);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || n_heads <= 0 || max_blocks_per_seq < 0 || max_seq_len < 0)
    return PKV_ERR_SHAPE;
  if (n_heads % shape->n_kv != 0) return PKV_ERR_SHAPE;
  if (!(scale > 0.f) || scale == __builtin_inff()) return PKV_ERR_RANGE;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !k_pool || !v_pool || !block_tables || !seq_lens || !out) return PKV_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
    return PKV_ERR_ALIGN;
  if (max_blocks_per_seq == 0 && max_seq_len > 0) return PKV_ERR_SHAPE;
  if ((int64_t)max_seq_len > (int64_t)max_blocks_per_seq * shape->block_size) return PKV_ERR_SHAPE;
  return PKV_OK;
}

// check_attention plus what every decode entry point adds: a non-negative
// grid cap and a compiled-in shape.
inline pkv_status check_decode(const void* q, int32_t num_seqs, int32_t n_heads,
                               const void* k_pool, const void* v_pool, const pkv_pool_desc* pool,
                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* seq_lens, int32_t max_seq_len, float scale,
                               int32_t max_ctas, const void* out, PoolShape* shape) {
  pkv_status st = check_attention(q, num_seqs, n_heads, k_pool, v_pool, pool, block_tables,
                                  max_blocks_per_seq, seq_lens, max_seq_len, scale, out, shape);
  if (st != PKV_OK) return st;
  if (max_ctas < 0) return PKV_ERR_RANGE;
  if (!decode_supported(*shape, n_heads)) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

}  // namespace pkv
