// Decode on the tensor cores for bf16 head_dim 64 (kernels in attention.cuh).
#include "attention.cuh"

namespace pkv {
namespace attn {

cudaError_t launch_decode_mma64(const AttnArgs& a, int hg, cudaStream_t s) {
  return DecodeLaunch<__nv_bfloat16, 64, 16, true>::run(a, hg, s);
}

size_t exact_workspace_mma64(const AttnArgs& a, int hg) {
  return decode_exact_workspace<__nv_bfloat16, 64, 16, true>(a, hg);
}

}  // namespace attn
}  // namespace pkv
