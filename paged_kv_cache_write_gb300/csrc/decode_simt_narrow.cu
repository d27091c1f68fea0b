// Decode on the CUDA cores for head_dim 16 / 32 (fp32 pools, and bf16 ones
// too narrow for the tensor-core tile), with 4 or 16 query rows per warp by
// GQA ratio (kernels in attention.cuh).
#include "attention.cuh"

namespace pkv {
namespace attn {

namespace {

template <typename T>
cudaError_t launch_narrow(const AttnArgs& a, int hg, cudaStream_t s) {
  const int rep = a.n_heads / a.pool.n_kv;
  if (a.pool.head_dim == 16) return by_rep_simt<DecodeLaunch, T, 16>(rep, a, s, hg);
  return by_rep_simt<DecodeLaunch, T, 32>(rep, a, s, hg);
}

template <typename T>
size_t workspace_narrow(const AttnArgs& a, int hg) {
  const bool small = a.n_heads / a.pool.n_kv <= 4;
  if (a.pool.head_dim == 16)
    return small ? decode_exact_workspace<T, 16, 4, false>(a, hg)
                 : decode_exact_workspace<T, 16, 16, false>(a, hg);
  return small ? decode_exact_workspace<T, 32, 4, false>(a, hg)
               : decode_exact_workspace<T, 32, 16, false>(a, hg);
}

}  // namespace

cudaError_t launch_decode_simt_narrow(const AttnArgs& a, int hg, cudaStream_t s) {
  if (a.pool.dtype == PKV_F32) return launch_narrow<float>(a, hg, s);
  return launch_narrow<__nv_bfloat16>(a, hg, s);
}

size_t exact_workspace_simt_narrow(const AttnArgs& a, int hg) {
  if (a.pool.dtype == PKV_F32) return workspace_narrow<float>(a, hg);
  return workspace_narrow<__nv_bfloat16>(a, hg);
}

}  // namespace attn
}  // namespace pkv
