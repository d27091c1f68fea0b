// extern "C" entry points declared in include/pkv.h: host-side argument
// checks, then the kernel launches on the caller's stream.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pkv.h"
#include "checks.h"
#include "launch.h"
#include "nvtx.h"

namespace {

using pkv::PoolShape;
using pkv::aligned16;
using pkv::check_attention;
using pkv::check_pool;
using pkv::from_cuda;

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

const char* pkv_status_string(int32_t status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_NULL: return "a required pointer is NULL";
    case PKV_ERR_SHAPE: return "invalid or inconsistent sizes";
    case PKV_ERR_DTYPE: return "unknown dtype";
    case PKV_ERR_ALIGN: return "pointer or row size not 16-byte aligned";
    case PKV_ERR_RANGE: return "value out of range";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_UNSUPPORTED: return "unsupported head_dim / block_size / head grouping";
    case PKV_ERR_CUDA: return "CUDA launch failed";
    default: return "unknown status";
  }
}

int32_t pkv_abi_version(void) { return 1; }

pkv_status pkv_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* seq_lens, const int32_t* cu_new_lens, int32_t num_seqs,
                            int32_t num_tokens, int32_t block_size, int32_t num_blocks,
                            int64_t* slot_mapping, int32_t* err_word, void* stream) {
  PKV_NVTX_RANGE("pkv_slot_mapping");
  if (num_seqs < 0 || num_tokens < 0 || max_blocks_per_seq < 0) return PKV_ERR_SHAPE;
  if (block_size <= 0 || num_blocks <= 0) return PKV_ERR_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (num_seqs == 0) return PKV_ERR_SHAPE;
  if (!block_tables || !seq_lens || !cu_new_lens || !slot_mapping) return PKV_ERR_NULL;
  if (max_blocks_per_seq == 0) return PKV_ERR_SHAPE;
  return from_cuda(pkv::launch_slot_mapping(block_tables, max_blocks_per_seq, seq_lens,
                                            cu_new_lens, num_seqs, num_tokens, block_size,
                                            num_blocks, slot_mapping, err_word, as_stream(stream)));
}

pkv_status pkv_kv_write(const void* k, const void* v, const int64_t* slot_mapping,
                        int32_t num_tokens, void* k_pool, void* v_pool, const pkv_pool_desc* pool,
                        int32_t* err_word, void* stream) {
  PKV_NVTX_RANGE("pkv_kv_write");
  PoolShape shape;
  pkv_status st = check_pool(pool, &shape);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_pool || !v_pool) return PKV_ERR_NULL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool))
    return PKV_ERR_ALIGN;
  return from_cuda(pkv::launch_kv_write(k, v, slot_mapping, num_tokens, k_pool, v_pool, shape,
                                        err_word, as_stream(stream)));
}

pkv_status pkv_copy_blocks(void* k_pool, void* v_pool, const pkv_pool_desc* pool,
                          const int32_t* block_pairs, int32_t num_pairs, int32_t* err_word,
                          void* stream) {
  PKV_NVTX_RANGE("pkv_copy_blocks");
  PoolShape shape;
  pkv_status st = check_pool(pool, &shape);
  if (st != PKV_OK) return st;
  if (num_pairs < 0) return PKV_ERR_SHAPE;
  if (num_pairs == 0) return PKV_OK;
  if (!k_pool || !v_pool || !block_pairs) return PKV_ERR_NULL;
  if (!aligned16(k_pool) || !aligned16(v_pool)) return PKV_ERR_ALIGN;
  return from_cuda(pkv::launch_copy_blocks(k_pool, v_pool, shape, block_pairs, num_pairs,
                                           err_word, as_stream(stream)));
}

pkv_status pkv_kv_gather(const void* k_pool, const void* v_pool, const pkv_pool_desc* pool,
                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* seq_lens, const int32_t* cu_seq_lens, int32_t num_seqs,
                         int32_t total_tokens, void* k_out, void* v_out, int32_t* err_word,
                         void* stream) {
  PKV_NVTX_RANGE("pkv_kv_gather");
  PoolShape shape;
  pkv_status st = check_pool(pool, &shape);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || total_tokens < 0 || max_blocks_per_seq < 0) return PKV_ERR_SHAPE;
  if (total_tokens == 0) return PKV_OK;
  if (num_seqs == 0 || max_blocks_per_seq == 0) return PKV_ERR_SHAPE;
  if (!k_pool || !v_pool || !block_tables || !seq_lens || !cu_seq_lens || !k_out || !v_out)
    return PKV_ERR_NULL;
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_out) || !aligned16(v_out))
    return PKV_ERR_ALIGN;
  return from_cuda(pkv::launch_kv_gather(k_pool, v_pool, shape, block_tables, max_blocks_per_seq,
                                         seq_lens, cu_seq_lens, num_seqs, total_tokens, k_out,
                                         v_out, err_word, as_stream(stream)));
}

size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t n_heads, int32_t head_dim,
                                  int32_t max_seq_len, int32_t max_ctas,
                                  int32_t block_size) {
  (void)block_size;
  if (num_seqs < 0) num_seqs = 0;
  if (n_heads < 1) n_heads = 1;
  if (head_dim < 1) head_dim = 1;
  return pkv::decode_workspace_bytes(num_seqs, n_heads, head_dim, max_seq_len, max_ctas, 0);
}

size_t pkv_decode_shared_prefix_workspace_bytes(int32_t num_seqs, int32_t n_heads,
                                                int32_t head_dim, int32_t max_seq_len,
                                                int32_t shared_prefix_blocks, int32_t max_ctas,
                                                int32_t block_size) {
  (void)block_size;
  if (num_seqs < 0) num_seqs = 0;
  if (n_heads < 1) n_heads = 1;
  if (head_dim < 1) head_dim = 1;
  if (shared_prefix_blocks < 0) shared_prefix_blocks = 0;
  return pkv::decode_workspace_bytes(num_seqs, n_heads, head_dim, max_seq_len, max_ctas,
                                     shared_prefix_blocks);
}

namespace {

// Shared body of the decode entry points; k_new / v_new null: plain
// decode; prefix_blocks > 0: the leading table entries are shared.
pkv_status decode_entry(const void* q, const void* k_new, const void* v_new, int32_t num_seqs,
                        int32_t n_heads, const void* k_pool, const void* v_pool,
                        const pkv_pool_desc* pool, const int32_t* block_tables,
                        int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t max_seq_len,
                        int32_t prefix_blocks, float scale, int32_t max_ctas, void* out,
                        void* workspace, size_t workspace_bytes, int32_t* err_word,
                        void* stream, int32_t plan_mode = pkv::kPlanInCall) {
  PoolShape shape;
  pkv_status st = pkv::check_decode(q, num_seqs, n_heads, k_pool, v_pool, pool, block_tables,
                                    max_blocks_per_seq, seq_lens, max_seq_len, scale, max_ctas,
                                    out, &shape);
  if (st != PKV_OK) return st;
  if (num_seqs == 0) return PKV_OK;
  if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_NULL;
  if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PKV_ERR_ALIGN;
  if (prefix_blocks < 0 || prefix_blocks > max_blocks_per_seq) return PKV_ERR_RANGE;
  if (!workspace) return PKV_ERR_WORKSPACE;
  if (workspace_bytes < pkv::decode_workspace_bytes(num_seqs, n_heads, shape.head_dim,
                                                    max_seq_len, max_ctas, prefix_blocks))
    return PKV_ERR_WORKSPACE;
  if (!aligned16(workspace)) return PKV_ERR_ALIGN;
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
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.k_new = k_new;
  a.v_new = v_new;
  a.prefix_blocks = prefix_blocks;
  a.decode_plan = plan_mode;
  a.err = err_word;
  return from_cuda(pkv::launch_decode(a, as_stream(stream)));
}

}  // namespace

pkv_status pkv_paged_attention_decode(const void* q, int32_t num_seqs, int32_t n_heads,
                                      const void* k_pool, const void* v_pool,
                                      const pkv_pool_desc* pool, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                      int32_t max_seq_len, float scale, int32_t max_ctas,
                                      void* out, void* workspace, size_t workspace_bytes,
                                      int32_t* err_word, void* stream) {
  PKV_NVTX_RANGE("pkv_paged_attention_decode");
  return decode_entry(q, nullptr, nullptr, num_seqs, n_heads, k_pool, v_pool, pool, block_tables,
                      max_blocks_per_seq, seq_lens, max_seq_len, 0, scale, max_ctas, out,
                      workspace, workspace_bytes, err_word, stream);
}

pkv_status pkv_paged_attention_decode_shared_prefix(
    const void* q, int32_t num_seqs, int32_t n_heads, const void* k_pool, const void* v_pool,
    const pkv_pool_desc* pool, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* seq_lens, int32_t max_seq_len, int32_t shared_prefix_blocks, float scale,
    int32_t max_ctas, void* out, void* workspace, size_t workspace_bytes, int32_t* err_word,
    void* stream) {
  PKV_NVTX_RANGE("pkv_paged_attention_decode_shared_prefix");
  return decode_entry(q, nullptr, nullptr, num_seqs, n_heads, k_pool, v_pool, pool, block_tables,
                      max_blocks_per_seq, seq_lens, max_seq_len, shared_prefix_blocks, scale,
                      max_ctas, out, workspace, workspace_bytes, err_word, stream);
}

pkv_status pkv_paged_attention_decode_append(
    const void* q, const void* k_new, const void* v_new, int32_t num_seqs, int32_t n_heads,
    void* k_pool, void* v_pool, const pkv_pool_desc* pool, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t max_seq_len, float scale,
    int32_t max_ctas, void* out, void* workspace, size_t workspace_bytes, int32_t* err_word,
    void* stream) {
  PKV_NVTX_RANGE("pkv_paged_attention_decode_append");
  if (num_seqs > 0 && (k_new == nullptr || v_new == nullptr)) return PKV_ERR_NULL;
  return decode_entry(q, k_new, v_new, num_seqs, n_heads, k_pool, v_pool, pool, block_tables,
                      max_blocks_per_seq, seq_lens, max_seq_len, 0, scale, max_ctas, out,
                      workspace, workspace_bytes, err_word, stream);
}

pkv_status pkv_decode_plan(int32_t num_seqs, int32_t n_heads, const pkv_pool_desc* pool,
                           int32_t max_blocks_per_seq, const int32_t* seq_lens,
                           int32_t max_seq_len, int32_t shared_prefix_blocks, int32_t max_ctas,
                           void* workspace, size_t workspace_bytes, int32_t* err_word,
                           void* stream) {
  PKV_NVTX_RANGE("pkv_decode_plan");
  PoolShape shape;
  pkv_status st = check_pool(pool, &shape);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || n_heads <= 0 || max_blocks_per_seq < 0 || max_seq_len < 0)
    return PKV_ERR_SHAPE;
  if (n_heads % shape.n_kv != 0) return PKV_ERR_SHAPE;
  if (max_ctas < 0) return PKV_ERR_RANGE;
  if (shared_prefix_blocks < 0 || shared_prefix_blocks > max_blocks_per_seq) return PKV_ERR_RANGE;
  if (!pkv::decode_supported(shape, n_heads)) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!seq_lens) return PKV_ERR_NULL;
  if (max_blocks_per_seq == 0 && max_seq_len > 0) return PKV_ERR_SHAPE;
  if ((int64_t)max_seq_len > (int64_t)max_blocks_per_seq * shape.block_size) return PKV_ERR_SHAPE;
  if (!workspace) return PKV_ERR_WORKSPACE;
  if (workspace_bytes < pkv::decode_workspace_bytes(num_seqs, n_heads, shape.head_dim,
                                                    max_seq_len, max_ctas, shared_prefix_blocks))
    return PKV_ERR_WORKSPACE;
  if (!aligned16(workspace)) return PKV_ERR_ALIGN;
  pkv::AttnArgs a{};
  a.seq_lens = seq_lens;
  a.num_seqs = num_seqs;
  a.n_heads = n_heads;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_seq_len = max_seq_len;
  a.max_q_len = 1;
  a.total_q = num_seqs;
  a.pool = shape;
  a.scale = 1.f;
  a.max_ctas = max_ctas;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.prefix_blocks = shared_prefix_blocks;
  a.decode_plan = pkv::kPlanOnly;
  a.err = err_word;
  return from_cuda(pkv::launch_decode(a, as_stream(stream)));
}

pkv_status pkv_paged_attention_decode_planned(
    const void* q, const void* k_new, const void* v_new, int32_t num_seqs, int32_t n_heads,
    void* k_pool, void* v_pool, const pkv_pool_desc* pool, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t max_seq_len,
    int32_t shared_prefix_blocks, float scale, int32_t max_ctas, void* out, void* workspace,
    size_t workspace_bytes, int32_t* err_word, void* stream) {
  PKV_NVTX_RANGE("pkv_paged_attention_decode_planned");
  return decode_entry(q, k_new, v_new, num_seqs, n_heads, k_pool, v_pool, pool, block_tables,
                      max_blocks_per_seq, seq_lens, max_seq_len, shared_prefix_blocks, scale,
                      max_ctas, out, workspace, workspace_bytes, err_word, stream,
                      pkv::kPlanned);
}

size_t pkv_prefill_workspace_bytes(int32_t, int32_t, int32_t, int32_t, int32_t) { return 0; }

pkv_status pkv_paged_attention_prefill(const void* q, const int32_t* cu_q_lens, int32_t num_seqs,
                                       int32_t total_q, int32_t max_q_len, int32_t n_heads,
                                       const void* k_pool, const void* v_pool,
                                       const pkv_pool_desc* pool, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                       int32_t max_seq_len, float scale, void* out,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t* err_word, void* stream) {
  PKV_NVTX_RANGE("pkv_paged_attention_prefill");
  (void)workspace;
  (void)workspace_bytes;
  PoolShape shape;
  pkv_status st = check_attention(q, num_seqs, n_heads, k_pool, v_pool, pool, block_tables,
                                  max_blocks_per_seq, seq_lens, max_seq_len, scale, out, &shape);
  if (st != PKV_OK) return st;
  if (total_q < 0 || max_q_len < 0) return PKV_ERR_SHAPE;
  if (!pkv::prefill_supported(shape, n_heads)) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_q == 0) return PKV_OK;
  if (!cu_q_lens) return PKV_ERR_NULL;
  if (max_q_len == 0 || max_q_len > total_q || max_q_len > max_seq_len) return PKV_ERR_SHAPE;
  pkv::AttnArgs a{};
  a.q = q;
  a.out = out;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.cu_q_lens = cu_q_lens;
  a.num_seqs = num_seqs;
  a.n_heads = n_heads;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_seq_len = max_seq_len;
  a.max_q_len = max_q_len;
  a.total_q = total_q;
  a.pool = shape;
  a.scale = scale;
  a.err = err_word;
  return from_cuda(pkv::launch_prefill(a, as_stream(stream)));
}

pkv_status pkv_selftest_bounded_wait(int32_t polls, int32_t* err_word, void* stream) {
  PKV_NVTX_RANGE("pkv_selftest_bounded_wait");
  if (polls < 1) return PKV_ERR_RANGE;
  if (!err_word) return PKV_ERR_NULL;
  return from_cuda(
      pkv::launch_bounded_wait_selftest(static_cast<uint32_t>(polls), err_word, as_stream(stream)));
}

}  // extern "C"
