// Internal launcher interface between the C ABI (abi.cu) and the kernels.
// Arguments here are already validated by the ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

struct PoolShape {
  int32_t num_blocks, block_size, n_kv, head_dim, dtype;
  int32_t elem_bytes() const { return dtype == 0 ? 4 : 2; }
  int64_t row_bytes() const { return int64_t(n_kv) * head_dim * elem_bytes(); }
};

cudaError_t launch_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* seq_lens, const int32_t* cu_new_lens,
                                int32_t num_seqs, int32_t num_tokens, int32_t block_size,
                                int32_t num_blocks, int64_t* slot_mapping, int32_t* err,
                                cudaStream_t stream);

cudaError_t launch_kv_write(const void* k, const void* v, const int64_t* slot_mapping,
                            int32_t num_tokens, void* k_pool, void* v_pool, const PoolShape& pool,
                            int32_t* err, cudaStream_t stream);

cudaError_t launch_bounded_wait_selftest(uint32_t polls, int32_t* err, cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_pool, void* v_pool, const PoolShape& pool,
                               const int32_t* pairs, int32_t num_pairs, int32_t* err,
                               cudaStream_t stream);

cudaError_t launch_kv_gather(const void* k_pool, const void* v_pool, const PoolShape& pool,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, const int32_t* cu_seq_lens, int32_t num_seqs,
                             int32_t total_tokens, void* k_out, void* v_out, int32_t* err,
                             cudaStream_t stream);

// Attention problem shared by decode and prefill.
struct AttnArgs {
  const void* q;
  void* out;
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* cu_q_lens;  // prefill only
  int32_t num_seqs, n_heads, max_blocks_per_seq, max_seq_len, max_q_len, total_q;
  PoolShape pool;
  float scale;
  int32_t max_ctas;  // decode: persistent grid cap (0 = one full wave)
  // decode with append: this step's K/V per sequence [num_seqs, n_kv,
  // head_dim], stored at position seq_lens[b] - 1 (null: plain decode;
  // then k_pool / v_pool are only read)
  const void* k_new;
  const void* v_new;
  // decode: leading table entries shared by every sequence (0: none)
  int32_t prefix_blocks;
  // decode: kPlanInCall (plan inside the call), kPlanOnly (compute the
  // plan into the workspace, nothing else) or kPlanned (use the plan a
  // kPlanOnly call with the same arguments left in the workspace)
  int32_t decode_plan;
  void* workspace;
  size_t workspace_bytes;
  int32_t* err;
};

enum : int32_t { kPlanInCall = 0, kPlanOnly = 1, kPlanned = 2 };

// Decode support / sizing.
bool decode_supported(const PoolShape& pool, int32_t n_heads);
size_t decode_workspace_bytes(int32_t num_seqs, int32_t n_heads, int32_t head_dim,
                              int32_t max_seq_len, int32_t max_ctas,
                              int32_t shared_prefix_blocks);
cudaError_t launch_decode(const AttnArgs& a, cudaStream_t stream);
// Workspace the decode launch for `a` needs on the current device (0 on error).
size_t decode_workspace_bytes_exact(const AttnArgs& a);

bool prefill_supported(const PoolShape& pool, int32_t n_heads);
cudaError_t launch_prefill(const AttnArgs& a, cudaStream_t stream);

// tcgen05 prefill (bf16, head_dim 64/128, 1/2/4/8/16 query heads per KV head).
bool prefill_tc_supported(const PoolShape& pool, int32_t n_heads);
cudaError_t launch_prefill_tc(const AttnArgs& a, cudaStream_t stream);

}  // namespace pkv
