// Decode on the CUDA cores for fp32 pools with head_dim 64 / 128, with 4 or
// 16 query rows per warp by GQA ratio (kernels in attention.cuh).
#include "attention.cuh"

namespace pkv {
namespace attn {

cudaError_t launch_decode_simt_wide(const AttnArgs& a, int hg, cudaStream_t s) {
  const int rep = a.n_heads / a.pool.n_kv;
  if (a.pool.head_dim == 64) return by_rep_simt<DecodeLaunch, float, 64>(rep, a, s, hg);
  return by_rep_simt<DecodeLaunch, float, 128>(rep, a, s, hg);
}

size_t exact_workspace_simt_wide(const AttnArgs& a, int hg) {
  const bool small = a.n_heads / a.pool.n_kv <= 4;
  if (a.pool.head_dim == 64)
    return small ? decode_exact_workspace<float, 64, 4, false>(a, hg)
                 : decode_exact_workspace<float, 64, 16, false>(a, hg);
  return small ? decode_exact_workspace<float, 128, 4, false>(a, hg)
               : decode_exact_workspace<float, 128, 16, false>(a, hg);
}

}  // namespace attn
}  // namespace pkv
