// Decode: the tensor-core path for bf16 head_dim 128 and the dispatch of
// every decode entry point to the per-type paths (kernels in attention.cuh).
#include "attention.cuh"

namespace pkv {

using namespace attn;

bool decode_supported(const PoolShape& pool, int32_t n_heads) {
  if (pool.block_size != kBS || pool.n_kv <= 0 || n_heads % pool.n_kv != 0) return false;
  if (n_heads / pool.n_kv > kMaxRep) return false;
  if (pool.dtype == PKV_BF16) return use_mma(pool) || simt_head_dim(pool.head_dim);
  return pool.dtype == PKV_F32 && simt_head_dim(pool.head_dim);
}

// Upper bound of the decode workspace over every grid this device can run.
size_t decode_workspace_bytes(int32_t num_seqs, int32_t n_heads, int32_t head_dim, int32_t, int32_t,
                              int32_t shared_prefix_blocks) {
  // rows per head group <= n_heads, head groups <= n_heads; at most 16
  // resident CTAs per SM
  return DecodeWs(num_seqs, size_t(sm_count()) * 16, size_t(n_heads), head_dim,
                  shared_prefix_blocks > 0
                      ? prefix_slots(max_prefix_runs(num_seqs, shared_prefix_blocks)) * n_heads
                      : 0,
                  shared_prefix_blocks > 0 ? n_heads : 0)
      .total;
}

cudaError_t launch_decode(const AttnArgs& a, cudaStream_t s) {
  const PoolShape& pool = a.pool;
  const int hg = decode_group(pool);
  if (use_mma(pool)) {
    if (pool.head_dim == 64) return launch_decode_mma64(a, hg, s);
    return DecodeLaunch<__nv_bfloat16, 128, 16, true>::run(a, hg, s);
  }
  if (pool.head_dim <= 32) return launch_decode_simt_narrow(a, hg, s);
  return launch_decode_simt_wide(a, hg, s);
}

size_t decode_workspace_bytes_exact(const AttnArgs& a) {
  const PoolShape& pool = a.pool;
  const int hg = decode_group(pool);
  if (use_mma(pool)) {
    if (pool.head_dim == 64) return exact_workspace_mma64(a, hg);
    return decode_exact_workspace<__nv_bfloat16, 128, 16, true>(a, hg);
  }
  if (pool.head_dim <= 32) return exact_workspace_simt_narrow(a, hg);
  return exact_workspace_simt_wide(a, hg);
}

}  // namespace pkv
