// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05,
// TMEM accumulators, TMA-staged operands) for bf16 pools.
//
// What is computed ("Build a Mini vLLM" section 4, prefill: causal
// attention after the chunk's K/V is written): query i of a chunk of c
// queries at the end of an L-token sequence attends keys 0 .. L - c + i of
// its KV head, read in place through the block table.
//
// One CTA (one per SM) owns two 128-row tiles, A and B, of one (sequence,
// KV head): each row is one (query, query head) pair, floor(128 / rep)
// queries x the rep query heads that share the KV head (the last 128 mod
// rep rows idle), so one K/V tile feeds every head of the GQA group and
// both tiles.  Keys go in tiles of 128 (eight
// 16-token blocks).
//
//  warp 8    TMA producer for Q_A and Q_B (once; 64-column halves, 128-byte
//            swizzle) and K: per key tile one 16-row box per block and half
//            into a three-stage ring, so K runs two tiles ahead of the MMAs;
//  warp 10   TMA producer for V into a two-stage ring.
//  warp 9    allocates all 512 TMEM columns (S_A, S_B, O_A, O_B) and one
//            lane issues the MMAs in ping-pong order:
//               S_A = Q_A K_j^T, S_B = Q_B K_j^T, then for each tile once its
//               softmax is done: O_X += P_X V_j and at once S_X = Q_X K_{j+1}^T,
//            so the tensor core works on one tile while the other tile's
//            softmax runs.  P_X is read from TMEM (it overwrites S_X as bf16),
//            V MN-major from shared memory.
//  warps 0-3 softmax of tile A, warps 4-7 of tile B: thread r owns TMEM lane
//            r (one row), loads its 128 scores, masks causally, keeps a
//            running max in log2 units and rescales O only when the max grows
//            by more than 2^8, writes P as bf16, and in the epilogue
//            normalises O and stores the row.
//
// Value rows past the sequence end inside the last key tile are zeroed in
// shared memory before P V reads them, so garbage in unused pool slots
// cannot reach the output.  Every wait is bounded; on a timeout the kernel
// flags PKV_DEVERR_TIMEOUT, drains its copies and MMAs, frees its TMEM and
// returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "device.cuh"
#include "host_cache.h"
#include "launch.h"
#include "tcgen05.cuh"
#include "tma_host.h"

namespace pkv {

namespace {

constexpr int kRows = 128;       // MMA rows per tile
constexpr int kTileKeys = 128;   // keys per S tile
constexpr int kBlk = 16;         // tokens per pool block
constexpr int kBlocksPerTile = kTileKeys / kBlk;
constexpr int kProducerWarp = 8;   // Q and K
constexpr int kMmaWarp = 9;
constexpr int kVProducerWarp = 10;  // V
constexpr int kThreads = 11 * 32;
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.f;  // rescale O only when the max grows past 2^8
constexpr uint32_t kTmemCols = 512;  // S_A [0,128) S_B [128,256) O_A [256,..) O_B [384,..)

struct TcParams {
  const int32_t* bt;
  const int32_t* seq_lens;
  const int32_t* cu_q;
  __nv_bfloat16* out;
  int32_t* err;
  int B, n_heads, n_kv, rep, W, num_blocks, max_len, total_q, q_per_tile;
  int ordered;  // 1: heaviest-first slot order (see the kernel), 0: natural grid
  float scale_log2;
};

template <int HD>
struct Layout {
  static constexpr int NH = HD / 64;                    // 128-byte column halves
  static constexpr int Q_HALF = kRows * 128;            // 16 KB
  static constexpr int KV_HALF = kTileKeys * 128;       // 16 KB
  static constexpr int Q_TILE = NH * Q_HALF;
  static constexpr int KV_TILE = NH * KV_HALF;
  static constexpr int K_OFF = 2 * Q_TILE;               // K stage s at K_OFF + s * KV_TILE
  static constexpr int V_OFF = K_OFF + kKStages * KV_TILE;
  static constexpr int BAR_OFF = V_OFF + kVStages * KV_TILE;
  static constexpr int BYTES = BAR_OFF + 256;
  // + 1 KB alignment slack; at least 120 KB so only one CTA fits per SM (it
  // takes all 512 TMEM columns)
  static constexpr int REQUEST = (BYTES + 1024) > 120 * 1024 ? (BYTES + 1024) : 120 * 1024;
};

__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, TcParams p) {
  using Lay = Layout<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  // Work order.  CTAs are dispatched in blockIdx order (x fastest).  With
  // a batch of at most blockDim.x sequences (p.ordered), x numbers the
  // (sequence, KV head, tile pair) triples: sequences by descending work
  // (visible keys of the chunk, c (2L - c + 1) / 2), each sequence's KV
  // heads in turn, and within those the pairs from the last (most keys)
  // down: heavy CTAs start first, the pairs of one (sequence, KV head) run
  // together and share its history in L2, and no CTA is spent on pairs past
  // a short chunk.  Otherwise z is the sequence, y the KV head and x the
  // pair, in the natural order.  The work values are staged in the (still
  // unused) V stages.
  __shared__ int order_s, pair_s, head_s;
  int g = blockIdx.y;
  int b = blockIdx.z, pair = blockIdx.x;
  if (p.ordered) {
    const int t = threadIdx.x;
    int64_t* work_s = reinterpret_cast<int64_t*>(smem + Layout<HD>::V_OFF);
    int* seq_s = reinterpret_cast<int*>(work_s + p.B);   // [B] sequence of each rank
    int* pairs_s = seq_s + p.B;                         // [B] pairs of each rank
    const int qpp = 2 * p.q_per_tile;                   // queries per pair
    int64_t wt = 0;
    int pt = 0;
    if (t < p.B) {
      const int64_t cs = __ldg(p.cu_q + t + 1) - __ldg(p.cu_q + t);
      const int64_t Ls = min(__ldg(p.seq_lens + t), p.max_len);
      wt = cs * (2 * Ls - cs + 1);
      pt = cs > 0 ? static_cast<int>((cs + qpp - 1) / qpp) : 0;
      work_s[t] = wt;
    }
    if (t == 0) order_s = -1;
    __syncthreads();
    int rank = 0;
    if (t < p.B) {
      for (int s = 0; s < p.B; ++s) {
        const int64_t ws = work_s[s];
        rank += (ws > wt) || (ws == wt && s < t);
      }
      seq_s[rank] = t;
      pairs_s[rank] = pt;
    }
    __syncthreads();
    if (t < p.B) {  // rank t's first slot: the (head, pair) slots of the heavier ranks
      int first = 0;
      for (int r = 0; r < t; ++r) first += pairs_s[r];
      const int64_t x = blockIdx.x;
      const int64_t lo = int64_t(first) * p.n_kv, n = int64_t(pairs_s[t]) * p.n_kv;
      if (x >= lo && x < lo + n) {
        const int off = static_cast<int>(x - lo);
        order_s = seq_s[t];
        head_s = off / pairs_s[t];
        pair_s = pairs_s[t] - 1 - (off - (off / pairs_s[t]) * pairs_s[t]);  // last pair first
      }
      fence_proxy_async_smem();  // before the V stages are filled by TMA
    }
    __syncthreads();
    if (order_s < 0) return;  // slot past the last pair
    b = order_s;
    g = head_s;
    pair = pair_s;
  }
  const int q0 = __ldg(p.cu_q + b);
  const int c = __ldg(p.cu_q + b + 1) - q0;
  const int i0 = pair * 2 * p.q_per_tile;  // first query of tile A
  if (i0 >= c) return;  // idle CTA: leave before any barrier or TMEM use
  if (q0 < 0 || q0 + c > p.total_q) {
    if (threadIdx.x == 0 && i0 == 0 && g == 0) report(p.err, PKV_DEVERR_LENGTH);
    return;
  }
  int L = __ldg(p.seq_lens + b);
  if (threadIdx.x == 0 && i0 == 0 && g == 0) {
    if (L < c || L < 0) report(p.err, PKV_DEVERR_LENGTH);
    else if (L > p.max_len)
      report(p.err, L > p.W * kBlk ? PKV_DEVERR_TABLE_WIDTH : PKV_DEVERR_LENGTH);
  }
  if (L > p.max_len) L = p.max_len;
  if (L < c) return;
  const int i_end = min(c, i0 + 2 * p.q_per_tile);
  const int n_tiles = (L - c + i_end - 1) / kTileKeys + 1;
  const int n_blocks_seq = (L + kBlk - 1) / kBlk;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::BAR_OFF);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [3] per K stage
  uint64_t* k_empty = bars + 4;   // [3]
  uint64_t* v_full = bars + 7;    // [2] per V stage
  uint64_t* v_empty = bars + 9;   // [2]
  uint64_t* s_full = bars + 11;   // [2] per tile A/B
  uint64_t* p_ready = bars + 13;  // [2] per tile A/B
  uint64_t* o_done = bars + 15;   // [2] per tile A/B
  uint64_t* drain = bars + 17;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 18);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(k_full + i, 1);
      mbar_init(k_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(v_full + i, 1);
      mbar_init(v_empty + i, 1);
      mbar_init(s_full + i, 1);
      mbar_init(p_ready + i, kRows);
      mbar_init(o_done + i, 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  auto q_tile = [&](int x) { return smem + x * Lay::Q_TILE; };
  auto k_st = [&](int j) { return smem + Lay::K_OFF + (j % kKStages) * Lay::KV_TILE; };
  auto v_st = [&](int j) { return smem + Lay::V_OFF + (j % kVStages) * Lay::KV_TILE; };
  auto s_tm = [&](int x) { return tmem + uint32_t(x) * kTileKeys; };
  auto o_tm = [&](int x) { return tmem + 256u + uint32_t(x) * 128u; };

  if (warp == kProducerWarp || warp == kVProducerWarp) {
    // ---------------------------------------------------------- producers
    const bool is_k = warp == kProducerWarp;
    const int nst = is_k ? kKStages : kVStages;
    uint64_t* full = is_k ? k_full : v_full;
    uint64_t* empty = is_k ? k_empty : v_empty;
    const CUtensorMap* map = is_k ? &tk : &tv;
    if (is_k && lane == 0) {
      // each Q tile holds q_per_tile queries x rep heads (all 128 rows when
      // rep divides 128)
      mbar_arrive_expect_tx(q_full, 2 * Lay::NH * (p.q_per_tile * p.rep) * 128);
      for (int x = 0; x < 2; ++x)
        for (int h = 0; h < Lay::NH; ++h)
          tc::tma_load_3d(q_tile(x) + h * Lay::Q_HALF, &tq, h * 64, g * p.rep,
                          q0 + i0 + x * p.q_per_tile, q_full);
    }
    const int32_t* row = p.bt + int64_t(b) * p.W;
    int issued = 0;
    int ids = 0;  // lane l holds the id of block (j / 4) * 32 + l
    for (int j = 0; j < n_tiles; ++j) {
      if (*abort_flag) break;
      const int st = j % nst;
      const uint32_t use = j / nst;
      if ((j & 3) == 0) {
        const int jb32 = j * kBlocksPerTile + lane;
        ids = jb32 < n_blocks_seq ? __ldg(row + jb32) : 0;
      }
      const int jb = j * kBlocksPerTile + lane;  // lanes 0-7: the tile's eight blocks
      const int blk_l = __shfl_sync(0xffffffffu, ids, ((j & 3) * kBlocksPerTile + lane) & 31);
      int blk = 0;
      bool load = lane < kBlocksPerTile && jb < n_blocks_seq;
      if (load) {
        blk = blk_l;
        if (blk < 0 || blk >= p.num_blocks) {
          if (is_k) report(p.err, PKV_DEVERR_BLOCK_ID);
          load = false;
        }
      }
      const uint32_t nload = __popc(__ballot_sync(0xffffffffu, load));
      if (use > 0 && !wait_all(empty + st, (use - 1) & 1)) {
        if (lane == 0) {
          report(p.err, PKV_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(full + st, nload * Lay::NH * kBlk * 128);
      __syncwarp();
      if (load) {
        uint8_t* dst = is_k ? k_st(j) : v_st(j);
        for (int h = 0; h < Lay::NH; ++h)
          tc::tma_load_3d(dst + h * Lay::KV_HALF + lane * kBlk * 128, map, h * 64, g, blk * kBlk,
                          full + st);
      }
      ++issued;
    }
    if (*abort_flag) {  // let copies in flight land before the CTA exits
      for (int j = max(0, issued - nst); j < issued; ++j) mbar_wait(full + j % nst, (j / nst) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(kRows, kTileKeys, false, false);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(kRows, HD, false, true);
      auto issue_qk = [&](int x, int j) {
        const uint32_t q_addr = smem_addr(q_tile(x));
        const uint32_t k_addr = smem_addr(k_st(j));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off_q = (kk >> 2) * Lay::Q_HALF + (kk & 3) * 32;
          const uint32_t off_k = (kk >> 2) * Lay::KV_HALF + (kk & 3) * 32;
          tc::mma_ss(s_tm(x), tc::sw128_desc(q_addr + off_q, 16, 1024),
                     tc::sw128_desc(k_addr + off_k, 16, 1024), idesc_qk, kk > 0);
        }
        tc::commit(s_full + x);
      };
      auto issue_pv = [&](int x, int j) {
        const uint32_t v_addr = smem_addr(v_st(j));
#pragma unroll
        for (int kk = 0; kk < kTileKeys / 16; ++kk) {
          // 16 keys = two 8-row groups of the V tile; P: 16 bf16 = 8 columns
          tc::mma_ts(o_tm(x), s_tm(x) + kk * 8,
                     tc::sw128_desc(v_addr + kk * 2048, Lay::KV_HALF, 1024), idesc_pv,
                     j > 0 || kk > 0);
        }
        tc::commit(o_done + x);
      };
      bool ok = mbar_wait(q_full, 0) && mbar_wait(k_full, 0);
      if (ok) {
        tc::fence_after_sync();
        issue_qk(0, 0);
        issue_qk(1, 0);
        tc::commit(k_empty);  // K_0 is no longer read
      }
      for (int j = 0; j < n_tiles && ok; ++j) {
        const bool more = j + 1 < n_tiles;
        const int kn = (j + 1) % kKStages;
        for (int x = 0; x < 2 && ok; ++x) {
          if (!(ok = mbar_wait(p_ready + x, j & 1))) break;
          if (x == 0 && !(ok = mbar_wait(v_full + (j % kVStages), (j / kVStages) & 1))) break;
          if (x == 0 && more && !(ok = mbar_wait(k_full + kn, ((j + 1) / kKStages) & 1))) break;
          tc::fence_after_sync();
          issue_pv(x, j);
          if (x == 1) tc::commit(v_empty + (j % kVStages));  // V_j is no longer read
          if (more) issue_qk(x, j + 1);
          if (x == 1 && more) tc::commit(k_empty + kn);      // K_{j+1} is no longer read
        }
      }
      if (!ok) {
        report(p.err, PKV_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      // every MMA issued above has finished before TMEM is released
      tc::commit(drain);
      mbar_wait(drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    const int x = warp >> 2;                   // tile A (warps 0-3) or B (warps 4-7)
    const int r = threadIdx.x - x * kRows;     // TMEM lane = row of the tile
    const int qi = i0 + x * p.q_per_tile + r / p.rep;
    const int hh = r - (r / p.rep) * p.rep;
    const bool active = r < p.q_per_tile * p.rep && qi < c;  // rows past the last full query are idle
    const int last = active ? L - c + qi : -1;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float m_used = -INFINITY, l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!(ok = wait_all(s_full + x, j & 1))) break;
      tc::fence_after_sync();
      const uint32_t s_addr = s_tm(x) + lane_base;
      uint32_t sr[kTileKeys];
#pragma unroll
      for (int ch = 0; ch < kTileKeys / 32; ++ch)
        tc::tmem_ld32(s_addr + ch * 32, *reinterpret_cast<uint32_t(*)[32]>(sr + ch * 32));
      tc::tmem_wait_ld();
      const int pos0 = j * kTileKeys;
      if (pos0 + kTileKeys - 1 > last) {  // tile crosses this row's causal limit
#pragma unroll
        for (int k = 0; k < kTileKeys; ++k)
          if (pos0 + k > last) sr[k] = __float_as_uint(-INFINITY);
      }
      // max on raw scores (scale > 0); scale and shift fold into one packed FMA
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < kTileKeys; ++k) mx = fmaxf(mx, __uint_as_float(sr[k]));
      const float m_new = fmaxf(m_used, mx * p.scale_log2);
      const bool grow = m_new > m_used + kRescaleLog2;
      const float alpha = grow ? fast_exp2(m_used - m_new) : 1.f;
      if (grow) m_used = m_new;
      const float mref = (m_used == -INFINITY) ? 0.f : m_used;
      const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
      const float2 nm2 = make_float2(-mref, -mref);
      float2 acc = make_float2(0.f, 0.f);
      // P overwrites the first half of S_X in TMEM, 16 columns per 32 scores;
      // the scores are already in registers
#pragma unroll
      for (int ch = 0; ch < kTileKeys / 32; ++ch) {
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int e = ch * 32 + 2 * k;
          const float2 t2 = __ffma2_rn(
              make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sc2, nm2);
          const float2 pe = make_float2(fast_exp2(t2.x), fast_exp2(t2.y));
          acc = __fadd2_rn(acc, pe);
          const __nv_bfloat162 pb = __floats2bfloat162_rn(pe.x, pe.y);
          pk[k] = *reinterpret_cast<const uint32_t*>(&pb);
        }
        tc::tmem_st16(s_addr + ch * 16, pk);
      }
      l_sum = l_sum * alpha + (acc.x + acc.y);
      if (j > 0) {
        // P V of the previous tile must be done before O is rescaled (and
        // this keeps the o_done phases in step)
        if (!(ok = wait_all(o_done + x, (j - 1) & 1))) break;
        tc::fence_after_sync();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
          for (int ch = 0; ch < HD / 32; ++ch) {
            uint32_t ov[32];
            tc::tmem_ld32(o_tm(x) + lane_base + ch * 32, ov);
            tc::tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const float2 o2 = __fmul2_rn(
                  make_float2(__uint_as_float(ov[2 * k]), __uint_as_float(ov[2 * k + 1])), a2);
              ov[2 * k] = __float_as_uint(o2.x);
              ov[2 * k + 1] = __float_as_uint(o2.y);
            }
            tc::tmem_st32(o_tm(x) + lane_base + ch * 32, ov);
          }
        }
      }
      tc::tmem_wait_st();
      if (x == 0 && pos0 + kTileKeys > L) {
        // value rows at or past the sequence end: zero them (whole 128-byte
        // rows, so the swizzle does not matter) before P V reads them; tile
        // A's P V is the first reader of this V tile
        if (!(ok = wait_all(v_full + (j % kVStages), (j / kVStages) & 1))) break;
        const int first = L - pos0;  // >= 1
        const int chunks = (kTileKeys - first) * Lay::NH * 8;
        uint8_t* vt = v_st(j);
        for (int idx = r; idx < chunks; idx += kRows) {
          const int rowi = first + idx / (Lay::NH * 8);
          const int h = (idx / 8) % Lay::NH;
          const int chk = idx % 8;
          *reinterpret_cast<uint4*>(vt + h * Lay::KV_HALF + rowi * 128 + chk * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tc::fence_before_sync();
      mbar_arrive(p_ready + x);
    }
    if (ok) ok = wait_all(o_done + x, (n_tiles - 1) & 1);
    if (ok) {
      tc::fence_after_sync();
      const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
      __nv_bfloat16* orow = p.out + (int64_t(q0 + qi) * p.n_heads + g * p.rep + hh) * HD;
#pragma unroll 1
      for (int ch = 0; ch < HD / 32; ++ch) {
        uint32_t ov[32];
        tc::tmem_ld32(o_tm(x) + lane_base + ch * 32, ov);
        tc::tmem_wait_ld();
        if (active) {
          uint32_t pkd[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const __nv_bfloat162 v2 = __floats2bfloat162_rn(__uint_as_float(ov[2 * k]) * inv,
                                                            __uint_as_float(ov[2 * k + 1]) * inv);
            pkd[k] = *reinterpret_cast<const uint32_t*>(&v2);
          }
          uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            dst[k] = make_uint4(pkd[4 * k], pkd[4 * k + 1], pkd[4 * k + 2], pkd[4 * k + 3]);
        }
      }
    } else if (lane == 0) {
      report(p.err, PKV_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }
  }
  // ------------------------------------------------------------ teardown
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------ host side

// 3-D bf16 tensor (dim0 contiguous) with a 128-byte-swizzled box.
bool encode_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1,
               uint32_t b2) {
  const uint64_t dims[3] = {d0, d1, d2};
  const uint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const uint32_t box[3] = {b0, b1, b2};
  return encode_bf16_sw128(map, base, 3, dims, strides, box);
}

template <int HD>
cudaError_t run_tc(const AttnArgs& a, cudaStream_t stream) {
  using Lay = Layout<HD>;
  const PoolShape& pool = a.pool;
  const int rep = a.n_heads / pool.n_kv;
  TcParams p{};
  p.bt = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.cu_q = a.cu_q_lens;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.err = a.err;
  p.B = a.num_seqs;
  p.n_heads = a.n_heads;
  p.n_kv = pool.n_kv;
  p.rep = rep;
  p.W = a.max_blocks_per_seq;
  p.num_blocks = pool.num_blocks;
  p.max_len = min(a.max_seq_len, a.max_blocks_per_seq * kBlk);
  p.total_q = a.total_q;
  p.q_per_tile = kRows / rep;
  p.scale_log2 = a.scale * kLog2e;
  CUtensorMap tq, tk, tv;
  const uint64_t slots = uint64_t(pool.num_blocks) * pool.block_size;
  if (!encode_3d(&tq, a.q, HD, a.n_heads, a.total_q, uint64_t(HD) * 2,
                 uint64_t(a.n_heads) * HD * 2, 64, rep, kRows / rep) ||
      !encode_3d(&tk, a.k_pool, HD, pool.n_kv, slots, uint64_t(HD) * 2,
                 uint64_t(pool.n_kv) * HD * 2, 64, 1, kBlk) ||
      !encode_3d(&tv, a.v_pool, HD, pool.n_kv, slots, uint64_t(HD) * 2,
                 uint64_t(pool.n_kv) * HD * 2, 64, 1, kBlk))
    return cudaErrorInvalidValue;
  auto kern = prefill_tc_kernel<HD>;
  static KernelSetup setup;
  const cudaError_t e = kernel_setup(setup, kern, Lay::REQUEST, kThreads, nullptr);
  if (e != cudaSuccess) return e;
  const int qpp = 2 * p.q_per_tile;
  p.ordered = a.num_seqs <= kThreads;
  // ordered: one slot per (sequence, KV head, pair); the pairs number at
  // most total_q / qpp + one partial pair per sequence
  const int64_t n_slots = (int64_t(a.total_q) + qpp - 1) / qpp + a.num_seqs;
  dim3 grid = p.ordered ? dim3(static_cast<unsigned>(n_slots * pool.n_kv), 1, 1)
                        : dim3((a.max_q_len + qpp - 1) / qpp, pool.n_kv, a.num_seqs);
  kern<<<grid, kThreads, Lay::REQUEST, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(const PoolShape& pool, int32_t n_heads) {
  if (pool.dtype != PKV_BF16 || pool.block_size != kBlk) return false;
  if (pool.head_dim != 64 && pool.head_dim != 128) return false;
  if (pool.n_kv <= 0 || n_heads % pool.n_kv != 0) return false;
  const int rep = n_heads / pool.n_kv;
  return rep >= 1 && rep <= 16;  // a tile holds 128 / rep queries of all rep heads
}

cudaError_t launch_prefill_tc(const AttnArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.max_q_len == 0) return cudaSuccess;
  return a.pool.head_dim == 64 ? run_tc<64>(a, stream) : run_tc<128>(a, stream);
}

}  // namespace pkv
