// Chunked prefill with warp-level MMA (bf16) or CUDA-core FMAs (fp32 and
// the other head sizes): the shapes the tcgen05 kernel (prefill_tc.cu) does
// not take, and the dispatch between the two.
#include "attention.cuh"

namespace pkv {

using namespace attn;

bool prefill_supported(const PoolShape& pool, int32_t n_heads) { return decode_supported(pool, n_heads); }

cudaError_t launch_prefill(const AttnArgs& a, cudaStream_t s) {
  const PoolShape& pool = a.pool;
  const int rep = a.n_heads / pool.n_kv;
  if (prefill_tc_supported(pool, a.n_heads)) return launch_prefill_tc(a, s);
  if (use_mma(pool)) {
    if (pool.head_dim == 64) return PrefillLaunch<__nv_bfloat16, 64, 16, true>::run(a, s);
    return PrefillLaunch<__nv_bfloat16, 128, 16, true>::run(a, s);
  }
  if (pool.dtype == PKV_F32) {
    switch (pool.head_dim) {
      case 16: return by_rep_simt<PrefillLaunch, float, 16>(rep, a, s, 0);
      case 32: return by_rep_simt<PrefillLaunch, float, 32>(rep, a, s, 0);
      case 64: return by_rep_simt<PrefillLaunch, float, 64>(rep, a, s, 0);
      default: return by_rep_simt<PrefillLaunch, float, 128>(rep, a, s, 0);
    }
  }
  switch (pool.head_dim) {
    case 16: return by_rep_simt<PrefillLaunch, __nv_bfloat16, 16>(rep, a, s, 0);
    default: return by_rep_simt<PrefillLaunch, __nv_bfloat16, 32>(rep, a, s, 0);
  }
}

}  // namespace pkv
