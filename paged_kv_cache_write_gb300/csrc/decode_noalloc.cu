// pkv_paged_attention_decode_noalloc: the decode attention of
// pkv_paged_attention_decode for callers that cannot allocate device memory.
//
// Who needs it.  Some callers may not call cudaMalloc, or hold no workspace
// to lend: a plug-in running inside a serving framework that owns every
// byte of device memory through its own arena (a raw cudaMalloc escapes the
// framework's accounting and implicitly synchronises the whole device,
// stalling every other stream), a per-token inner loop where that
// synchronisation is unaffordable, or a plain C caller with no allocator
// at all.  This entry point takes the same inputs and outputs as
// pkv_paged_attention_decode but no workspace argument: its scratch (the
// per-sequence work prefix and the split partial results) lives in one
// fixed array compiled into the library.
//
// The array is a file-scope __device__ variable of
// PKV_NOALLOC_SCRATCH_BYTES (8 MiB).  Every GPU that loads the library
// holds one copy of it from module load until the process exits.  In host
// code its name only stands in for the symbol; it is not a device address
// (passing it to a kernel would fault, or silently use the wrong memory
// where the GPU can reach host memory).  The device address is looked up
// with cudaGetSymbolAddress, once per device, with that device current,
// during the first call on that device; make that first call before any
// stream capture.  The cached address is kept for the life of the process:
// cudaDeviceReset destroys the context that holds the array and a later
// context may load it at another address, so a device that was reset must
// not be given to this entry point again.
//
// All calls share the one array.  Nothing in it needs to start at zero:
// each call writes the work prefix and every partial slot before reading
// them, so a call never sees a previous call's contents.  Two calls whose
// kernels overlap on the GPU (for example on two streams) race on the
// array: issue them on one stream, or use pkv_paged_attention_decode with
// separate workspaces.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pkv.h"
#include "checks.h"
#include "launch.h"
#include "nvtx.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};  // device address of g_decode_scratch, per device

// Device address of the scratch array on the current device (looked up on
// the first call for that device).
pkv_status scratch_on_current_device(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return PKV_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_paged_attention_decode_noalloc(
    const void* q, int32_t num_seqs, int32_t n_heads, const void* k_pool, const void* v_pool,
    const pkv_pool_desc* pool, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* seq_lens, int32_t max_seq_len, float scale, int32_t max_ctas, void* out,
    int32_t* err_word, void* stream) {
  PKV_NVTX_RANGE("pkv_paged_attention_decode_noalloc");
  // The argument checks of pkv_paged_attention_decode (one shared function,
  // so the two entry points refuse the same arguments with the same status).
  pkv::PoolShape shape;
  const pkv_status chk = pkv::check_decode(q, num_seqs, n_heads, k_pool, v_pool, pool,
                                           block_tables, max_blocks_per_seq, seq_lens,
                                           max_seq_len, scale, max_ctas, out, &shape);
  if (chk != PKV_OK) return chk;
  if (num_seqs == 0) return PKV_OK;

  void* scratch = nullptr;
  const pkv_status st = scratch_on_current_device(&scratch);
  if (st != PKV_OK) return st;

  pkv::AttnArgs a{};
  a.q = q;
  a.out = out;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.cu_q_lens = nullptr;
  a.num_seqs = num_seqs;
  a.n_heads = n_heads;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_seq_len = max_seq_len;
  a.max_q_len = 1;
  a.total_q = num_seqs;
  a.pool = shape;
  a.scale = scale;
  a.max_ctas = max_ctas;
  a.workspace = scratch;
  a.workspace_bytes = PKV_NOALLOC_SCRATCH_BYTES;
  a.err = err_word;
  // Too much work for the fixed array: refuse rather than overrun it.
  const size_t need = pkv::decode_workspace_bytes_exact(a);
  if (need == 0) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  if (need > PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
  const cudaError_t e = pkv::launch_decode(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}
