// Paged attention over the block pool, included by the decode and prefill
// translation units: decode (one query per sequence, split over the whole machine and merged by log-sum-exp weights) and
// chunked prefill (a causal query chunk over paged history).
//
// What is computed ("Build a Mini vLLM" section 3, paged_attention, and
// section 4, prefill / decode_step):  for a query row of head h the output
// is softmax_j(scale * q . K_j) V_j over the keys j the row may see, with
// K_j, V_j read from block table[j / 16], offset j % 16, of KV head
// h / (n_heads / n_kv) ("nano-vLLM", How it works: query heads grouped onto
// their shared K/V head).  Softmax is evaluated online (running maximum,
// rescaled running sum) in fp32; scores are kept in log2 units
// (scale * log2(e) folded into one multiply) so exp2 can be used.
//
// GB300 design.
//  * Data movement: a producer warp copies each 16-token block's K and V
//    rows for the CTA's KV heads into a shared-memory ring with bulk
//    asynchronous copies (cp.async.bulk, the TMA engine), one copy per
//    token row (HG heads x head_dim contiguous elements, up to 1 KB), with
//    completion counted on an mbarrier per stage.  Rows past a sequence's
//    length are zero-filled instead of copied, so pool slots past the
//    length are never read.  Token rows are padded by 16 bytes in shared
//    memory so the MMA fragment loads are bank-conflict free.
//  * Math: bf16 pools use warp-level tensor-core MMA (m16n8k16, fp32
//    accumulate) with the GQA group's query heads as the 16 MMA rows, so
//    one K/V tile serves every head of the group (the group-8 shapes need
//    8 multiply-adds per KV byte, more than the CUDA cores issue at HBM
//    rate).  fp32 pools use a CUDA-core path with fp32 FMAs.
//  * Decode work balance: a persistent grid sized to the SMs divides the
//    total work - every (sequence, KV-head group, 16-token block) unit - into
//    equal contiguous ranges, one per CTA (stream-K style).  A sequence
//    whose blocks fall in one CTA's range is finished there; one that spans
//    several CTAs leaves a partial (normalised output, max, exp-sum) per
//    CTA, which a merge kernel combines.  Split points depend only on
//    logical block positions and lengths, never on physical block ids, so
//    results are bit-identical under any placement or sharing of blocks.
//  * Every mbarrier wait is bounded; a wait that runs out sets
//    PKV_DEVERR_TIMEOUT, and the producer drains its copies before exit.
#pragma once

#include <cuda_runtime.h>
#include <math.h>

#include <algorithm>

#include <type_traits>

#include "device.cuh"
#include "host_cache.h"
#include "launch.h"
#include "tcgen05.cuh"
#include "tma_host.h"

namespace pkv {
namespace attn {

constexpr int kBS = 16;          // tokens per block handled by these kernels
constexpr int kMaxRep = 16;      // query heads per KV head (MMA rows)
constexpr int kBarrierBytes = 1024;
constexpr int kMaxStages = 32;
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ rows

// Per-warp softmax state over up to 16 query rows, tensor-core version
// (bf16).  Thread `lane` owns rows g = lane/4 and g + 8 of every m16n8
// accumulator tile and the columns 2*(lane%4) + {0,1} of it.
template <int HD>
struct MmaRows {
  static_assert(HD % 16 == 0, "head_dim must be a multiple of 16");
  uint32_t qa[HD / 16][4];
  float o[HD / 8][4];
  float m[2], l[2];
  int last[2];  // kNoQuery: the row has no query (it computes garbage, never stored)
  int slot[2];  // with several sequences' rows in the tile: the sequence of each row
  static constexpr int kNoQuery = INT_MIN;

  // Rows r hold sequence r / rep (see block_sw's `only`).
  __device__ __forceinline__ void set_row_slots(int rep) {
    const int g = (threadIdx.x & 31) >> 2;
    slot[0] = g / rep;
    slot[1] = (g + 8) / rep;
  }

  // q_row(r) -> pointer to row r's query (nullptr = inactive row),
  // last_key(r) -> last key position the row may see.
  template <typename QRow, typename LastKey>
  __device__ __forceinline__ void begin(QRow q_row, LastKey last_key) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __nv_bfloat16* qp = q_row(g + 8 * h);
      last[h] = qp ? last_key(g + 8 * h) : kNoQuery;
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        uint32_t lo = 0, hi = 0;
        if (qp) {
          lo = *reinterpret_cast<const uint32_t*>(qp + kk * 16 + 2 * c);
          hi = *reinterpret_cast<const uint32_t*>(qp + kk * 16 + 8 + 2 * c);
        }
        qa[kk][h] = lo;      // a0 (row g) / a1 (row g+8): k = 2c, 2c+1
        qa[kk][2 + h] = hi;  // a2 (row g) / a3 (row g+8): k = 2c+8, 2c+9
      }
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  }

  // Continue from a partial result instead of from nothing (call after
  // begin): part_row(r) -> the row's normalised output (fp32, nullptr =
  // inactive row), ml_row(r) -> its max (log2 units) and exp-sum.
  template <typename PartRow, typename MlRow>
  __device__ __forceinline__ void seed(PartRow part_row, MlRow ml_row) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float* pp = part_row(g + 8 * h);
      if (!pp) continue;
      const float* ml = ml_row(g + 8 * h);
      const float lsum = ml[1];
      m[h] = ml[0];
      l[h] = c == 0 ? lsum : 0.f;  // the four lanes of a row are summed at the end
#pragma unroll
      for (int i = 0; i < HD / 8; ++i) {
        const float2 x = *reinterpret_cast<const float2*>(pp + i * 8 + 2 * c);
        o[i][2 * h] = x.x * lsum;
        o[i][2 * h + 1] = x.y * lsum;
      }
    }
  }

  // One 16-token block.  k_tile / v_tile point at token 0 of this warp's KV
  // head; consecutive tokens are `stride` bytes apart.  j0 = position of
  // token 0 of the block.
  __device__ __forceinline__ void block(const uint8_t* k_tile, const uint8_t* v_tile, int stride,
                                        int j0, float scale_log2) {
    const int lane = threadIdx.x & 31;
    const int mi = lane >> 3, ri = lane & 7;
    const uint8_t* kaddr = k_tile + ((mi >> 1) * 8 + ri) * stride + (mi & 1) * 16;
    const uint8_t* vaddr = v_tile + ((mi & 1) * 8 + ri) * stride + (mi >> 1) * 16;
    block_from([&](int kk) { return kaddr + kk * 32; }, [&](int dp) { return vaddr + dp * 32; },
               j0, scale_log2, last);
  }

  // One 16-token block from TMA tiles in the 128-byte-swizzled layout: rows
  // of 64 head dims (128 bytes), row (h * HD/64 + d / 64) * 16 + t holding
  // token t, dims [d, d + 64) of the group's head h; within a row the
  // 16-byte piece c sits at position c ^ (row % 8).  `head` is this warp's
  // head within the group.
  // `only` >= 0: the block belongs to sequence `only` of the tile's rows
  // (set_row_slots): the other rows see none of it.
  __device__ __forceinline__ void block_sw(const uint8_t* k_tile, const uint8_t* v_tile, int head,
                                           int j0, float scale_log2, int only = -1) {
    const int lane = threadIdx.x & 31;
    const int mi = lane >> 3, ri = lane & 7;
    const int hrow = head * (HD / 64) * kBS;
    const uint8_t* kaddr = k_tile + (hrow + (mi >> 1) * 8 + ri) * 128;
    const uint8_t* vaddr = v_tile + (hrow + (mi & 1) * 8 + ri) * 128;
    const int kx = (mi & 1) ^ ri, vx = (mi >> 1) ^ ri;
    const int lim[2] = {only < 0 || slot[0] == only ? last[0] : -1,
                        only < 0 || slot[1] == only ? last[1] : -1};
    block_from([&](int kk) { return kaddr + (kk >> 2) * (kBS * 128) + ((((kk & 3) * 2) ^ kx) << 4); },
               [&](int dp) { return vaddr + (dp >> 2) * (kBS * 128) + ((((dp & 3) * 2) ^ vx) << 4); },
               j0, scale_log2, lim);
  }

  // kaddr(kk): this lane's ldmatrix row address for the K matrices of dims
  // [16 kk, 16 kk + 16) (lane / 8 = matrix: tokens 0-7 | 8-15 x dims lo |
  // hi); vaddr(dp): the same for V, matrices tokens 0-7 | 8-15 (fast) x
  // dims lo | hi.
  template <typename KAddr, typename VAddr>
  __device__ __forceinline__ void block_from(KAddr kaddr, VAddr vaddr, int j0, float scale_log2,
                                             const int (&lim)[2]) {
    const int lane = threadIdx.x & 31;
    const int c = lane & 3;
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    // S = Q K^T: the four 8x8 matrices are (tokens 0-7 | 8-15) x (dims lo | hi).
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      uint32_t kb[4];
      ldsm_x4(kb, kaddr(kk));
      mma_bf16_16816(s[0], qa[kk], kb[0], kb[1]);
      mma_bf16_16816(s[1], qa[kk], kb[2], kb[3]);
    }
    // causal / length mask: only a block that crosses some live row's last
    // key (warp-uniform test) masks element by element
    const int first_cut = min(last[0] == kNoQuery ? INT_MAX : lim[0],
                              last[1] == kNoQuery ? INT_MAX : lim[1]);
    if (!__all_sync(0xffffffffu, j0 + kBS - 1 <= first_cut)) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (j0 + nt * 8 + 2 * c + (e & 1) > lim[e >> 1]) s[nt][e] = -INFINITY;
    }
    // online softmax in log2 units: the raw maximum times the (positive)
    // scale is the maximum of the scaled scores
    float mx[2] = {fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1])),
                   fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]))};
    float alpha[2], mref[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      const float mn = fmaxf(m[h], mx[h] * scale_log2);
      mref[h] = (mn == -INFINITY) ? 0.f : mn;  // a row with nothing visible yet
      alpha[h] = fast_exp2(m[h] - mref[h]);
      m[h] = mn;
    }
    uint32_t pa[4];
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float p0 = fast_exp2(fmaf(s[nt][2 * h], scale_log2, -mref[h]));
        const float p1 = fast_exp2(fmaf(s[nt][2 * h + 1], scale_log2, -mref[h]));
        const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
        const float2 pr = __bfloat1622float2(pb);
        rs[h] += pr.x + pr.y;  // the sum uses the same rounded weights as P V
        pa[nt * 2 + h] = *reinterpret_cast<const uint32_t*>(&pb);
      }
#pragma unroll
    for (int h = 0; h < 2; ++h) l[h] = l[h] * alpha[h] + rs[h];
    // the outputs are rescaled only when some live row's maximum moved
    // (alpha 1 elsewhere: skipping the product changes no bit)
    if (__any_sync(0xffffffffu, (last[0] != kNoQuery && alpha[0] != 1.f) ||
                                    (last[1] != kNoQuery && alpha[1] != 1.f))) {
#pragma unroll
      for (int i = 0; i < HD / 8; ++i) {
        o[i][0] *= alpha[0];
        o[i][1] *= alpha[0];
        o[i][2] *= alpha[1];
        o[i][3] *= alpha[1];
      }
    }
    // O += P V: matrices (tokens 0-7 | 8-15) x (dims lo | hi), transposed.
#pragma unroll
    for (int dp = 0; dp < HD / 16; ++dp) {
      uint32_t vb[4];
      ldsm_x4_trans(vb, vaddr(dp));
      mma_bf16_16816(o[2 * dp], pa, vb[0], vb[1]);
      mma_bf16_16816(o[2 * dp + 1], pa, vb[2], vb[3]);
    }
  }

  __device__ __forceinline__ void reduce_sums() {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
    }
  }

  // Final output of every active row: out_row(r) -> T* (nullptr = skip).
  template <typename OutRow>
  __device__ __forceinline__ void store(OutRow out_row) {
    reduce_sums();
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      __nv_bfloat16* op = out_row(g + 8 * h);
      if (!op) continue;
      const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
#pragma unroll
      for (int i = 0; i < HD / 8; ++i) {
        *reinterpret_cast<__nv_bfloat162*>(op + i * 8 + 2 * c) =
            __floats2bfloat162_rn(o[i][2 * h] * inv, o[i][2 * h + 1] * inv);
      }
    }
  }

  // Partial result of every active row: normalised output (fp32), max
  // (log2 units) and exp-sum.  part_row(r) -> float* (nullptr = skip),
  // ml_row(r) -> float* of two floats.
  template <typename PartRow, typename MlRow>
  __device__ __forceinline__ void store_partial(PartRow part_row, MlRow ml_row) {
    reduce_sums();
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float* pp = part_row(g + 8 * h);
      if (!pp) continue;
      const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
#pragma unroll
      for (int i = 0; i < HD / 8; ++i)
        *reinterpret_cast<float2*>(pp + i * 8 + 2 * c) =
            make_float2(o[i][2 * h] * inv, o[i][2 * h + 1] * inv);
      if (c == 0) {
        float* ml = ml_row(g + 8 * h);
        ml[0] = m[h];
        ml[1] = l[h];
      }
    }
  }
};

// CUDA-core version (any element type).  Half-warp hw = lane/16 owns rows
// hw, hw+2, ...; within a half-warp lane t = lane%16 owns token t of a
// block for scores and head dims t, t+16, ... for the output.  The warp's
// query rows (fp32) and block weights live in shared scratch.
template <typename T, int HD, int MAXR>
struct SimtRows {
  static_assert(HD % 16 == 0, "head_dim must be a multiple of 16");
  static constexpr int RPH = MAXR / 2;  // rows per half-warp
  static constexpr int SCRATCH_FLOATS = MAXR * HD + MAXR * kBS;
  float o[RPH][HD / 16];
  float m[RPH], l[RPH];
  int last[RPH];
  float* qs;  // [MAXR][HD]
  float* ps;  // [MAXR][16]

  __device__ __forceinline__ void bind(float* scratch) {
    qs = scratch;
    ps = scratch + MAXR * HD;
  }

  template <typename QRow, typename LastKey>
  __device__ __forceinline__ void begin(QRow q_row, LastKey last_key) {
    const int lane = threadIdx.x & 31;
    __syncwarp();
    for (int i = lane; i < MAXR * HD; i += 32) {
      const T* qp = q_row(i / HD);
      qs[i] = qp ? Elem<T>::to_f(qp[i % HD]) : 0.f;
    }
    const int hw = lane >> 4;
#pragma unroll
    for (int k = 0; k < RPH; ++k) {
      const int r = hw + 2 * k;
      last[k] = q_row(r) ? last_key(r) : -1;
      m[k] = -INFINITY;
      l[k] = 0.f;
#pragma unroll
      for (int i = 0; i < HD / 16; ++i) o[k][i] = 0.f;
    }
    __syncwarp();
  }

  // Continue from a partial result (see MmaRows::seed).
  template <typename PartRow, typename MlRow>
  __device__ __forceinline__ void seed(PartRow part_row, MlRow ml_row) {
    const int lane = threadIdx.x & 31;
    const int t = lane & 15, hw = lane >> 4;
#pragma unroll
    for (int k = 0; k < RPH; ++k) {
      const float* pp = part_row(hw + 2 * k);
      if (!pp) continue;
      const float* ml = ml_row(hw + 2 * k);
      m[k] = ml[0];
      l[k] = ml[1];
#pragma unroll
      for (int i = 0; i < HD / 16; ++i) o[k][i] = pp[t + 16 * i] * ml[1];
    }
  }

  __device__ __forceinline__ void block(const uint8_t* k_tile, const uint8_t* v_tile, int stride,
                                        int j0, float scale_log2) {
    const int lane = threadIdx.x & 31;
    const int t = lane & 15, hw = lane >> 4;
    const unsigned half_mask = 0xffffffffu;
    const T* krow = reinterpret_cast<const T*>(k_tile + t * stride);
    const int pos = j0 + t;
#pragma unroll
    for (int k = 0; k < RPH; ++k) {
      const int r = hw + 2 * k;
      float s = 0.f;
      const float* q = qs + r * HD;
#pragma unroll 8
      for (int d = 0; d < HD; ++d) s = fmaf(q[d], Elem<T>::to_f(krow[d]), s);
      s = (pos <= last[k]) ? s * scale_log2 : -INFINITY;
      float mx = s;
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(half_mask, mx, off));
      const float mn = fmaxf(m[k], mx);
      const float mref = (mn == -INFINITY) ? 0.f : mn;
      const float alpha = fast_exp2(m[k] - mref);
      m[k] = mn;
      const float p = fast_exp2(s - mref);
      float sum = p;
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) sum += __shfl_xor_sync(half_mask, sum, off);
      l[k] = l[k] * alpha + sum;
#pragma unroll
      for (int i = 0; i < HD / 16; ++i) o[k][i] *= alpha;
      ps[r * kBS + t] = p;
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < RPH; ++k) {
      const int r = hw + 2 * k;
      const float* p = ps + r * kBS;
#pragma unroll
      for (int i = 0; i < HD / 16; ++i) {
        const int d = t + 16 * i;
        float acc = 0.f;
#pragma unroll
        for (int tt = 0; tt < kBS; ++tt)
          acc = fmaf(p[tt], Elem<T>::to_f(reinterpret_cast<const T*>(v_tile + tt * stride)[d]), acc);
        o[k][i] += acc;
      }
    }
    __syncwarp();
  }

  template <typename OutRow>
  __device__ __forceinline__ void store(OutRow out_row) {
    const int lane = threadIdx.x & 31;
    const int t = lane & 15, hw = lane >> 4;
#pragma unroll
    for (int k = 0; k < RPH; ++k) {
      T* op = out_row(hw + 2 * k);
      if (!op) continue;
      const float inv = l[k] > 0.f ? 1.f / l[k] : 0.f;
#pragma unroll
      for (int i = 0; i < HD / 16; ++i) op[t + 16 * i] = Elem<T>::from_f(o[k][i] * inv);
    }
  }

  template <typename PartRow, typename MlRow>
  __device__ __forceinline__ void store_partial(PartRow part_row, MlRow ml_row) {
    const int lane = threadIdx.x & 31;
    const int t = lane & 15, hw = lane >> 4;
#pragma unroll
    for (int k = 0; k < RPH; ++k) {
      const int r = hw + 2 * k;
      float* pp = part_row(r);
      if (!pp) continue;
      const float inv = l[k] > 0.f ? 1.f / l[k] : 0.f;
#pragma unroll
      for (int i = 0; i < HD / 16; ++i) pp[t + 16 * i] = o[k][i] * inv;
      if (t == 0) {
        float* ml = ml_row(r);
        ml[0] = m[k];
        ml[1] = l[k];
      }
    }
  }
};

template <typename T, int HD, int MAXR, bool MMA>
struct RowsOf {
  using type = SimtRows<T, HD, MAXR>;
  static constexpr int kScratch = SimtRows<T, HD, MAXR>::SCRATCH_FLOATS;
};
template <int HD, int MAXR>
struct RowsOf<__nv_bfloat16, HD, MAXR, true> {
  using type = MmaRows<HD>;
  static constexpr int kScratch = 0;
};

// ------------------------------------------------------------ pipeline

struct Ring {
  uint64_t* full;   // [nstages] producer -> consumers (1 arrival + bytes)
  uint64_t* empty;  // [nstages] consumers -> producer (one arrival per consumer warp)
  volatile int* abort_flag;
  uint8_t* stages;
  int nstages, stage_bytes, tile_bytes, row_stride, row_bytes;

  __device__ __forceinline__ uint8_t* k_tile(int st) const { return stages + st * stage_bytes; }
  __device__ __forceinline__ uint8_t* v_tile(int st) const {
    return stages + st * stage_bytes + tile_bytes;
  }
};

__device__ __forceinline__ Ring make_ring(uint8_t* smem, int nstages, int row_bytes) {
  Ring r;
  r.full = reinterpret_cast<uint64_t*>(smem);
  r.empty = r.full + kMaxStages;
  r.abort_flag = reinterpret_cast<volatile int*>(r.empty + kMaxStages);
  r.stages = smem + kBarrierBytes;
  r.nstages = nstages;
  r.row_bytes = row_bytes;
  r.row_stride = row_bytes + 16;
  r.tile_bytes = kBS * r.row_stride;
  r.stage_bytes = 2 * r.tile_bytes;
  return r;
}

// Ring of TMA tiles: per stage a K tile and a V tile of tile_bytes each,
// starting on 1024-byte boundaries (the period of the 128-byte swizzle).
// Needs 1024 bytes of slack after the barriers.
__device__ __forceinline__ Ring make_tile_ring(uint8_t* smem, int nstages, int tile_bytes) {
  Ring r;
  r.full = reinterpret_cast<uint64_t*>(smem);
  r.empty = r.full + kMaxStages;
  r.abort_flag = reinterpret_cast<volatile int*>(r.empty + kMaxStages);
  uint8_t* base = smem + kBarrierBytes;
  r.stages = base + ((1024u - (smem_addr(base) & 1023u)) & 1023u);
  r.nstages = nstages;
  r.row_bytes = 0;
  r.row_stride = 0;
  r.tile_bytes = tile_bytes;
  r.stage_bytes = 2 * tile_bytes;
  return r;
}

__device__ __forceinline__ void ring_init(const Ring& r, int consumer_warps) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < r.nstages; ++i) {
      mbar_init(r.full + i, 1);
      mbar_init(r.empty + i, consumer_warps);
    }
    *r.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
}

// Producer side, executed by all 32 lanes of the producer warp: fill the
// next stage with rows [0, valid) of block `blk` (lane l < 16: K row l,
// lane l >= 16: V row l-16), zero rows [valid, 16).  `k_src`/`v_src` point
// at the first element of this CTA's heads in token row 0 of the block
// (ignored when valid == 0).  Row `new_row` (if in [0, valid)) is taken
// from `k_new_src`/`v_new_src` instead.  Returns false if the wait timed
// out.
__device__ __forceinline__ bool ring_fill(const Ring& r, uint32_t it, const uint8_t* k_src,
                                          const uint8_t* v_src, int64_t src_row_pitch, int valid,
                                          int32_t* err, int new_row = -1,
                                          const uint8_t* k_new_src = nullptr,
                                          const uint8_t* v_new_src = nullptr) {
  const int lane = threadIdx.x & 31;
  const int st = static_cast<int>(it % r.nstages);
  const uint32_t use = it / r.nstages;
  if (use > 0 && !mbar_wait(r.empty + st, (use - 1) & 1)) {
    if (lane == 0) report(err, PKV_DEVERR_TIMEOUT);
    return false;
  }
  const int row = lane & 15;
  const bool is_v = lane >= 16;
  uint8_t* dst = (is_v ? r.v_tile(st) : r.k_tile(st)) + row * r.row_stride;
  if (row >= valid) {
    for (int off = 0; off < r.row_bytes; off += 16)
      *reinterpret_cast<uint4*>(dst + off) = make_uint4(0, 0, 0, 0);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive_expect_tx(r.full + st, static_cast<uint32_t>(2 * valid * r.row_bytes));
  if (row < valid) {
    fence_proxy_async_smem();
    const uint8_t* src = row == new_row ? (is_v ? v_new_src : k_new_src)
                                        : (is_v ? v_src : k_src) + row * src_row_pitch;
    bulk_copy_g2s(dst, src, static_cast<uint32_t>(r.row_bytes), r.full + st);
  }
  return true;
}

// Producer side of a tile ring, one lane: wait for stage `it` to be free,
// then load the K and V boxes at pool slot `slot` (a block's first token),
// heads [head0, head0 + group) into it.  A slot past the pool's end reads
// zeros.  `policy` (nonzero) is an L2 cache policy for the copied lines.
// Returns false if the wait timed out.
__device__ __forceinline__ bool tile_fill(const Ring& r, uint32_t it, const CUtensorMap* tm_k,
                                          const CUtensorMap* tm_v, int slot, int head0,
                                          int32_t* err, uint64_t policy = 0) {
  const int st = static_cast<int>(it % r.nstages);
  const uint32_t use = it / r.nstages;
  if (use > 0 && !mbar_wait(r.empty + st, (use - 1) & 1)) {
    report(err, PKV_DEVERR_TIMEOUT);
    return false;
  }
  mbar_arrive_expect_tx(r.full + st, static_cast<uint32_t>(r.stage_bytes));
  if (policy != 0) {
    tc::tma_load_4d_hint(r.k_tile(st), tm_k, 0, slot, 0, head0, r.full + st, policy);
    tc::tma_load_4d_hint(r.v_tile(st), tm_v, 0, slot, 0, head0, r.full + st, policy);
  } else {
    tc::tma_load_4d(r.k_tile(st), tm_k, 0, slot, 0, head0, r.full + st);
    tc::tma_load_4d(r.v_tile(st), tm_v, 0, slot, 0, head0, r.full + st);
  }
  return true;
}

// This lane's HD / 16 bytes of the bf16 rows k_new[row_elem ..] and
// v_new[row_elem ..] (HD elements each).
template <int HD>
__device__ __forceinline__ void new_row_piece(const uint8_t* k_new, const uint8_t* v_new,
                                              int64_t row_elem, uint32_t (&kn)[2],
                                              uint32_t (&vn)[2]) {
  const int lane = threadIdx.x & 31;
  const int64_t off = row_elem * 2 + lane * (HD / 16);
  if constexpr (HD / 16 == 8) {
    const uint2 k = __ldg(reinterpret_cast<const uint2*>(k_new + off));
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(v_new + off));
    kn[0] = k.x, kn[1] = k.y, vn[0] = v.x, vn[1] = v.y;
  } else {
    static_assert(HD / 16 == 4, "tile path: head_dim 64 or 128");
    kn[0] = __ldg(reinterpret_cast<const uint32_t*>(k_new + off));
    vn[0] = __ldg(reinterpret_cast<const uint32_t*>(v_new + off));
  }
}

// One warp, in its head `head` of a K / V tile pair (layout of
// MmaRows::block_sw) holding a sequence's last block with `valid` tokens:
// zero the V rows [valid, 16) and, if `fresh`, store the new token's row
// (row valid - 1) from this lane's pieces.
template <int HD>
__device__ __forceinline__ void tile_fix(uint8_t* kt, uint8_t* vt, int head, int valid, bool fresh,
                                         const uint32_t (&kn)[2], const uint32_t (&vn)[2]) {
  constexpr int NH = HD / 64;
  const int lane = threadIdx.x & 31;
  const int hrow = head * NH * kBS;
  const int nz = kBS - valid;
  for (int i = lane; i < NH * nz * 8; i += 32) {
    const int half = i / (nz * 8), rem = i - half * nz * 8;
    *reinterpret_cast<uint4*>(vt + (hrow + half * kBS + valid + (rem >> 3)) * 128 + (rem & 7) * 16) =
        make_uint4(0u, 0u, 0u, 0u);
  }
  if (fresh) {
    const int t = valid - 1;
    const int o = lane * (HD / 16);  // byte of the row
    const int half = o >> 7, ob = o & 127;
    const int off = (hrow + half * kBS + t) * 128 + (((ob >> 4) ^ (t & 7)) << 4) + (ob & 15);
    if constexpr (HD / 16 == 8) {
      *reinterpret_cast<uint2*>(kt + off) = make_uint2(kn[0], kn[1]);
      *reinterpret_cast<uint2*>(vt + off) = make_uint2(vn[0], vn[1]);
    } else {
      *reinterpret_cast<uint32_t*>(kt + off) = kn[0];
      *reinterpret_cast<uint32_t*>(vt + off) = vn[0];
    }
  }
  __syncwarp();
}

// Producer after an abort: wait (bounded) for every stage it may still
// have copies in flight to, so no copy lands after the CTA exits.
__device__ __forceinline__ void ring_drain(const Ring& r, uint32_t issued) {
  const uint32_t first = issued > static_cast<uint32_t>(r.nstages) ? issued - r.nstages : 0;
  for (uint32_t it = first; it < issued; ++it)
    mbar_wait(r.full + (it % r.nstages), (it / r.nstages) & 1);
}

// Consumer side: wait for stage `it`'s tile.  False if the producer gave up
// (abort flag, looked at only while the tile is not there yet) or the wait
// timed out (reported).
__device__ __forceinline__ bool ring_wait_full(const Ring& r, uint32_t it, int32_t* err) {
  const int st = static_cast<int>(it % r.nstages);
  const uint32_t parity = (it / r.nstages) & 1;
  if (mbar_try_wait(r.full + st, parity)) return true;
  for (uint32_t i = 0; i < kMaxPolls; ++i) {
    if (*r.abort_flag) return false;
    if (mbar_try_wait(r.full + st, parity)) return true;
  }
  if ((threadIdx.x & 31) == 0) report(err, PKV_DEVERR_TIMEOUT);
  return false;
}

__device__ __forceinline__ void ring_release(const Ring& r, uint32_t it) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(r.empty + (it % r.nstages));
}

// ------------------------------------------------------------- decode

struct DecodeParams {
  const void* q;
  void* out;
  const uint8_t* k_pool;
  const uint8_t* v_pool;
  const uint8_t* k_new;  // append: this step's K/V per sequence [B, n_kv, HD], else null
  const uint8_t* v_new;
  const int32_t* bt;
  const int32_t* seq_lens;
  int32_t* err;
  int32_t* cu_units;  // [B+1] units (16-token blocks x head groups) before each sequence
  int4* starts;       // [grid] each CTA's first segment: (sequence, head group, block, -)
  int4* splits;       // [grid] per CTA: the split group it merges (sequence, head group,
                      // first CTA, last CTA), sequence = -1 if none
  int32_t* total_units;  // one int: units of the whole batch
  float* ws_o;        // [2 * grid][HG * rep][HD] partial outputs
  float* ws_ml;       // [2 * grid][HG * rep][2] partial max (log2 units) and exp-sum
  int B, n_heads, n_kv, rep, hg_size, n_groups, W, num_blocks, max_len, max_seq_len, head_dim;
  int elem_bytes, nstages, grid;
  // shared prefix: every sequence's first prefix_blocks table entries are
  // the same blocks; the prefix kernel attends over them in prefix_chunks
  // runs of prefix_bpc blocks and leaves per-row partials in pre_o /
  // pre_ml, and units here cover only the blocks after the prefix (0: no
  // shared prefix)
  int prefix_blocks, prefix_chunks, prefix_bpc;
  int prefix_seed_run;  // run slot holding the combined prefix partials
  float* pre_o;   // [chunks][B][n_heads][HD] normalised prefix outputs
  float* pre_ml;  // [chunks][B][n_heads][2] prefix max (log2 units) and exp-sum
  int plan_in_kernel;  // 1: each CTA scans the lengths itself (no plan kernel)
  // 1 (plan kernel): compute the plan only, for later calls: write cu_units,
  // zero no output, let no dependent start before it has finished
  int plan_only;
  // 1 (main kernel): the plan is in the workspace from a finished plan-only
  // launch, so it and the tables are read before the dependency wait
  int planned;
  // cluster decode: CTAs per cluster (0: stream-K path), sequences per
  // cluster (their rows per warp: cluster_seqs * rep), and the byte offset
  // of the partial results in shared memory
  int cluster, cluster_seqs, part_off;
  // warps of 16 query rows that attend a shared prefix: the consumer warps
  // of the wide pass, the prompt warps of the fused launch; and (wide pass)
  // 1 if each prefix tile is read by one cluster only (its lines may leave
  // L2 first)
  int wide_mt, wide_evict;
  // fused shared prefix (stream-K kernel): CTA c < prompt_items also
  // attends item c = ((chunk * n_kv) + KV head) * prompt_runs + run: run
  // `run` (prompt_bpr blocks of row 0's table) for the prompt_seqs
  // sequences of `chunk`, prompt warp w carrying the rows of sequences
  // w * (16 / rep) ..; each leaves a partial per row in run slot `run`.
  // Every group's blocks after the prefix leave partials too (a whole one
  // in run slot prompt_runs) and the prefix merge kernel combines them.
  int prompt_items, prompt_runs, prompt_bpr, prompt_seqs;
  // fused shared prefix, per (sequence, KV-head group), from the plan: the
  // first and last CTA whose ranges hold the group's blocks after the
  // prefix and the first CTA's partial slot (c0 = -1: none)
  int4* gparts;
  float scale_log2;
};

// Exclusive prefix sum of `local` over the CTA's threads in thread order;
// every thread calls it.  warp_tot: 32 ints of shared memory.
__device__ __forceinline__ int cta_exclusive_scan(int local, int* warp_tot) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int t = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += y;
    }
    warp_tot[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  return incl - local + (wid > 0 ? warp_tot[wid - 1] : 0);
}

// Length used for sequence b: seq_lens[b] clamped to [0, max_len]
// (max_len = min(max_seq_len, table width * 16)).
__device__ __forceinline__ int used_len(const DecodeParams& p, int b) {
  const int L = __ldg(p.seq_lens + b);
  return L < 0 ? 0 : (L > p.max_len ? p.max_len : L);
}

// Largest b with cu[b] <= u (cu nondecreasing, u < cu[B]).
__device__ __forceinline__ int seq_of_unit(const int32_t* cu, int B, int u) {
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= u) lo = mid; else hi = mid;
  }
  return lo;
}

// First unit of CTA c's range when U units are split evenly over G CTAs
// (32-bit division when the product fits).
__device__ __forceinline__ int range_begin(int c, int U, int G) {
  const uint64_t n = uint64_t(uint32_t(c)) * uint32_t(U);
  if (n <= 0xffffffffull) return static_cast<int>(uint32_t(n) / uint32_t(G));
  return static_cast<int>(n / uint64_t(G));
}

// Let the programmatic dependent launch start its prologue.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until the preceding kernel has finished and its writes are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// A plan kept in the workspace (by a plan-only launch) was made for this
// grid, batch and shared prefix.
__device__ __forceinline__ bool plan_matches(const DecodeParams& p, int G) {
  return __ldcg(p.total_units + 1) == G && __ldcg(p.total_units + 2) == p.B &&
         __ldcg(p.total_units + 3) == p.prefix_blocks;
}

// Plan for batches too large for the main kernel's own scan: one CTA
// computes the exclusive scan of units per sequence, each CTA's first
// segment and the batch total, zeroes outputs of empty sequences and
// reports bad lengths once.
constexpr int kPlanSmemSeqs = 8191;
// Batches up to this size are planned by every main-kernel CTA itself.
constexpr int kKernelPlanSeqs = 2048;

// Blocks of a sequence of L tokens that this kernel walks (those after the
// shared prefix).
__device__ __forceinline__ int walked_blocks(const DecodeParams& p, int L) {
  const int n = (L + kBS - 1) / kBS - p.prefix_blocks;
  return n > 0 ? n : 0;
}

// Units (16-token blocks x head groups) of sequence b.
__device__ __forceinline__ int units_of(const DecodeParams& p, int b) {
  return p.n_groups * walked_blocks(p, used_len(p, b));
}

__device__ __forceinline__ void check_length(const DecodeParams& p, int b) {
  const int L = __ldg(p.seq_lens + b);
  if (L < 0 || L > p.max_seq_len) report(p.err, PKV_DEVERR_LENGTH);
  else if (L > p.W * kBS) report(p.err, PKV_DEVERR_TABLE_WIDTH);
}

// The split group CTA c merges.  CTA c's range starts at block j of head
// group grp of sequence b (nblk blocks per group).  If j > 0 the group is
// split, and c merges it when c is the first non-empty CTA to start inside
// it.  Entry: (b, grp | flags, first CTA | last CTA << 16, first unit of
// the group); b = -1 when c merges nothing.  Flags: kSplitC0Tail (the
// first CTA's part is the last segment of its range, not its first) and
// kSplitDense (every CTA has a non-empty range, U >= G).
constexpr int kSplitC0Tail = 1 << 16;
constexpr int kSplitDense = 1 << 17;

__device__ __forceinline__ int4 split_entry(int c, int G, int U, int b, int grp, int j,
                                            int nblk) {
  if (j == 0) return make_int4(-1, 0, 0, 0);
  const int a = range_begin(c, U, G) - j;  // the group's first unit
  int lo = 0, hi = c;  // owner of unit a: largest c' with range_begin(c') <= a
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (range_begin(mid, U, G) <= a) lo = mid; else hi = mid;
  }
  const int c0 = lo;
  int first = c0 + 1;  // CTAs between c0 and c with an empty range start nowhere
  while (range_begin(first + 1, U, G) == range_begin(first, U, G)) ++first;
  if (first != c) return make_int4(-1, 0, 0, 0);
  const int e = a + nblk - 1;  // owner of the group's last unit
  lo = c;
  hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (range_begin(mid, U, G) <= e) lo = mid; else hi = mid;
  }
  const int flags = (range_begin(c0, U, G) != a ? kSplitC0Tail : 0) | (U >= G ? kSplitDense : 0);
  return make_int4(b, grp | flags, c0 | (lo << 16), a);
}

// Zero the output rows of empty sequences b = first, first + stride, ...;
// the CTA's warps share them.  empty(b) tells whether b has no tokens.
template <typename T, int HD, typename Empty>
__device__ __forceinline__ void zero_empty(const DecodeParams& p, int first, int stride,
                                           Empty empty) {
  T* out = static_cast<T*>(p.out);
  const int row_elems = p.n_heads * HD;
  const int lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  for (int b = first + int(threadIdx.x >> 5) * stride; b < p.B; b += nw * stride) {
    if (!empty(b)) continue;
    for (int i = lane; i < row_elems; i += 32) out[int64_t(b) * row_elems + i] = Elem<T>::from_f(0.f);
  }
}

template <typename T, int HD>
__global__ void __launch_bounds__(1024) decode_plan_kernel(DecodeParams p) {
  if (!p.plan_only) pdl_launch_dependents();
  __shared__ int warp_tot[32];
  __shared__ int cu_s[kPlanSmemSeqs + 1];
  const bool in_smem = p.B <= kPlanSmemSeqs;
  int* cu = in_smem ? cu_s : p.cu_units;
  const int tid = threadIdx.x;
  const int chunk = (p.B + blockDim.x - 1) / blockDim.x;
  const int b0 = tid * chunk;
  const int b1 = min(p.B, b0 + chunk);
  int local = 0;
  for (int b = b0; b < b1; ++b) {
    check_length(p, b);
    local += units_of(p, b);
  }
  int run = cta_exclusive_scan(local, warp_tot);
  for (int b = b0; b < b1; ++b) {
    cu[b] = run;
    run += units_of(p, b);
  }
  if (tid == blockDim.x - 1) {
    cu[p.B] = run;
    *p.total_units = run;
    if (p.plan_only) {  // what the plan was made for, checked by the calls using it
      p.total_units[1] = p.grid;
      p.total_units[2] = p.B;
      p.total_units[3] = p.prefix_blocks;
    } else {
      p.total_units[1] = -1;  // a call planning for itself replaces any kept plan
    }
  }
  __syncthreads();  // the prefix is complete (same CTA: visible after the barrier)
  const int U = cu[p.B];
  for (int c = tid; c < p.grid; c += blockDim.x) {
    const int r0 = range_begin(c, U, p.grid);
    int4 st = make_int4(0, 0, 0, 0);
    int4 sp = make_int4(-1, 0, 0, 0);
    if (r0 < range_begin(c + 1, U, p.grid)) {
      const int b = seq_of_unit(cu, p.B, r0);
      const int nblk = walked_blocks(p, used_len(p, b));
      const int grp = (r0 - cu[b]) / nblk;
      st = make_int4(b, grp, (r0 - cu[b]) - grp * nblk, 0);
      sp = split_entry(c, p.grid, U, b, grp, st.z, nblk);
    }
    p.starts[c] = st;
    // a plan kept for later calls also fixes which split group each merge
    // CTA merges, so those calls' merge CTAs can read it before they wait
    if (p.plan_only) p.splits[c] = sp;
  }
  if (p.prompt_items > 0) {
    // fused shared prefix: where each (sequence, group)'s blocks after the
    // prefix went, for the prefix merge
    auto owner = [&](int u) {  // largest c with range_begin(c) <= u
      int lo = 0, hi = p.grid;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (range_begin(mid, U, p.grid) <= u) lo = mid; else hi = mid;
      }
      return lo;
    };
    for (int i = tid; i < p.B * p.n_groups; i += blockDim.x) {
      const int b = i / p.n_groups, grp = i - (i / p.n_groups) * p.n_groups;
      const int nblk = (cu[b + 1] - cu[b]) / p.n_groups;
      int4 gp = make_int4(-1, -1, 0, 0);
      if (nblk > 0) {
        const int u0 = cu[b] + grp * nblk;
        const int c0 = owner(u0);
        gp = make_int4(c0, owner(u0 + nblk - 1), range_begin(c0, U, p.grid) == u0 ? 2 * c0 : 2 * c0 + 1, 0);
      }
      p.gparts[i] = gp;
    }
  }
  if (p.plan_only || p.prompt_items > 0) {  // kept for later calls / the prefix merge
    if (in_smem)
      for (int b = tid; b <= p.B; b += blockDim.x) p.cu_units[b] = cu[b];
  } else if (p.prefix_blocks == 0) {  // with a prefix, the prefix kernel writes them
    zero_empty<T, HD>(p, 0, 1, [&](int b) { return used_len(p, b) == 0; });
  }
}

// Walks this CTA's contiguous range of units segment by segment: a segment
// is the run of units of one (sequence, head group) inside the range.
// j counts the walked blocks of the group (block prefix_blocks + j of the
// table); nblk is how many there are.
struct Cursor {
  int b, grp, j, L, nblk;

  __device__ __forceinline__ void load(const DecodeParams& p, int4 st) {
    b = st.x;
    grp = st.y;
    j = st.z;
    L = used_len(p, b);
    nblk = walked_blocks(p, L);
  }
  // advance past n units of the current group
  __device__ __forceinline__ void advance(const DecodeParams& p, int n) {
    j += n;
    if (j < nblk) return;
    j = 0;
    if (++grp < p.n_groups) return;
    grp = 0;
    do {
      if (++b >= p.B) {  // past the last unit: never used
        nblk = 1;
        return;
      }
      L = used_len(p, b);
      nblk = walked_blocks(p, L);
    } while (nblk == 0);
  }
};

// Merge of split groups: out = sum_c w_c o_c / sum_c w_c over the CTAs c
// that computed parts of one (sequence, head group), w_c = exp2(m_c - M) l_c.
// Thread t owns J float4 pieces of the group's rows x head_dim outputs and
// loads each part's pieces and the (max, exp-sum) of their rows straight
// from L2 (the main kernel wrote them moments before and marks its K/V
// stream to leave L2 first), 8 / J parts at a time with every load in
// flight together, folding them in with a running maximum: any number of
// parts in a few dependent round trips, no staging, no barrier.
constexpr int kMergeThreads = 256;
constexpr int kMergeMaxVec = 8;  // float4 per thread: rows * head_dim <= 8192 = 256 x 8 x 4

// Largest decode CTA of an instantiation: one producer warp plus one warp
// per KV head of the group (at most 8 heads, at most 1 KB of row data).
template <typename T, int HD>
constexpr int decode_max_threads() {
  return ((1024 / (HD * int(sizeof(T))) < 8 ? 1024 / (HD * int(sizeof(T))) : 8) + 1) * 32;
}

// The decode body; tm_k / tm_v are the pools' tile maps (tensor-core path)
// or null (CUDA-core path).
template <typename T, int HD, int MAXR, bool MMA, bool PROMPT = false>
__device__ __forceinline__ void decode_body(const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                            const DecodeParams& p) {
  extern __shared__ __align__(128) uint8_t smem[];
  using Rows = typename RowsOf<T, HD, MAXR, MMA>::type;
  const int consumers = p.hg_size;
  const int row_bytes = p.hg_size * HD * p.elem_bytes;
  // tensor-core path: whole-block TMA tiles; CUDA-core path: a copy per row
  Ring ring = MMA ? make_tile_ring(smem, p.nstages, kBS * row_bytes)
                  : make_ring(smem, p.nstages, row_bytes);
  if (PROMPT && threadIdx.x == 0) mbar_init(reinterpret_cast<uint64_t*>(smem + 768), 1);  // pbar
  ring_init(ring, consumers);  // (its barrier also publishes pbar's init)
  // inputs written by the preceding kernel (the plan, when there is one);
  // a planned call waits after reading its plan and first table entries
  if (!p.planned) pdl_wait();
  pdl_launch_dependents();  // the merge kernel may be scheduled (it waits for this grid)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;
  int U;
  int4 st = make_int4(0, 0, 0, 0);
  if (p.plan_in_kernel) {
    // Scan the units per sequence in the (still unused) ring stages.
    int* cu_s = reinterpret_cast<int*>(ring.stages);  // [B + 1]
    int* warp_tot = cu_s + p.B + 1;                    // [32]
    const int nt = blockDim.x;
    for (int b = threadIdx.x; b < p.B; b += nt) {
      if (blockIdx.x == 0) check_length(p, b);
      cu_s[b] = units_of(p, b);
    }
    __syncthreads();
    const int chunk = (p.B + nt - 1) / nt;
    const int b0 = min(p.B, int(threadIdx.x) * chunk);
    const int b1 = min(p.B, b0 + chunk);
    int local = 0;
    for (int b = b0; b < b1; ++b) local += cu_s[b];
    int run = cta_exclusive_scan(local, warp_tot);
    for (int b = b0; b < b1; ++b) {
      const int n = cu_s[b];
      cu_s[b] = run;
      run += n;
    }
    if (threadIdx.x == nt - 1) cu_s[p.B] = run;
    __syncthreads();
    U = cu_s[p.B];
    const int r0 = range_begin(blockIdx.x, U, G);
    if (r0 < range_begin(blockIdx.x + 1, U, G)) {
      const int b = seq_of_unit(cu_s, p.B, r0);
      const int nblk = walked_blocks(p, used_len(p, b));
      const int grp = (r0 - cu_s[b]) / nblk;
      st = make_int4(b, grp, (r0 - cu_s[b]) - grp * nblk, 0);
    }
    if (p.prefix_blocks == 0)  // with a prefix, the prefix kernel writes them
      zero_empty<T, HD>(p, blockIdx.x, G, [&](int b) { return cu_s[b + 1] == cu_s[b]; });
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      p.total_units[0] = U;
      p.total_units[1] = -1;  // a call planning for itself replaces any kept plan
    }
    fence_proxy_async_smem();  // the scan's stores come before the ring's copies
    __syncthreads();
  } else {
    U = __ldcg(p.total_units);
    if (p.planned && !plan_matches(p, G)) {  // nothing of the stale plan is used
      if (blockIdx.x == 0 && threadIdx.x == 0) report(p.err, PKV_DEVERR_PLAN);
      return;
    }
    st = __ldcg(p.starts + blockIdx.x);
  }
  const int r0 = range_begin(blockIdx.x, U, G);
  const int r1 = range_begin(blockIdx.x + 1, U, G);
  const int64_t token_pitch = int64_t(p.n_kv) * HD * p.elem_bytes;  // bytes per pool slot
  const int rows_per_group = p.hg_size * p.rep;
  Cursor cur;
  if (r0 < r1) cur.load(p, st);
  // planned call: the producer's first table entries are loaded before the
  // wait (the plan's contract: lengths and tables unchanged since the plan),
  // and on the tile path its first blocks too: up to a ring's worth of the
  // first segment, never the sequence's last block (the only block a decode
  // step writes), so their bytes stream in while the preceding kernel ends
  // fused shared prefix: this CTA's prompt item (item_nb blocks of one KV
  // head), held in its own buffer after the ring and attended by the
  // prompt warps (warps consumers + 1 ..) while the consumers stream the
  // blocks after the prefix
  [[maybe_unused]] int item_run = 0, item_head = 0, item_s0 = 0, item_j0 = 0, item_nb = 0;
  [[maybe_unused]] uint8_t* pbuf = ring.stages + p.nstages * ring.stage_bytes;  // K tiles, then V tiles
  [[maybe_unused]] uint64_t* pbar = reinterpret_cast<uint64_t*>(smem + 768);   // past the ring's barriers
  if constexpr (PROMPT) {
    if (static_cast<int>(blockIdx.x) < p.prompt_items) {
      const int c = blockIdx.x;
      item_run = c % p.prompt_runs;
      item_head = (c / p.prompt_runs) % p.n_kv;
      item_s0 = c / (p.prompt_runs * p.n_kv) * p.prompt_seqs;
      item_j0 = item_run * p.prompt_bpr;
      item_nb = max(0, min(p.prompt_bpr, p.prefix_blocks - item_j0));
      // The prefix blocks are never written by a decode step, so their
      // loads go out before the dependency wait.  One head of a block is 16
      // rows of HD * 2 bytes a token pitch apart, only 2-4 KB: the whole
      // run is requested at once (16-byte copies by every producer lane,
      // into the 128-byte-swizzled tile layout) so that enough bytes are in
      // flight, and published on pbar once landed.
      if (warp == consumers) {
        const int id = lane < item_nb ? __ldg(p.bt + item_j0 + lane) : 0;  // row 0's table
        constexpr int kChunks = kBS * HD * 2 / 16;  // 16-byte pieces of one head of a block
        const int64_t pitch = int64_t(p.n_kv) * HD * 2;
        for (int i = 0; i < item_nb; ++i) {
          const int b_id = __shfl_sync(0xffffffffu, id, i);
          const bool bad = b_id < 0 || b_id >= p.num_blocks;
          if (bad && lane == 0) report(p.err, PKV_DEVERR_BLOCK_ID);
          const int64_t off = int64_t(bad ? 0 : b_id) * kBS * pitch + int64_t(item_head) * HD * 2;
          uint8_t* kt = pbuf + i * (kBS * HD * 2);
          uint8_t* vt = pbuf + (p.prompt_bpr + i) * (kBS * HD * 2);
          for (int x = lane; x < kChunks; x += 32) {
            // piece x: token t, 16-byte column cx of the head's row
            const int t = x / (HD / 8), cx = x - t * (HD / 8);
            const int row = (cx >> 3) * kBS + t;  // (64-dim half, token)
            const int dst = row * 128 + (((cx & 7) ^ (row & 7)) << 4);
            const int64_t src = off + int64_t(t) * pitch + cx * 16;
            if (bad) {  // as the zeros a bad id reads elsewhere
              *reinterpret_cast<uint4*>(kt + dst) = make_uint4(0u, 0u, 0u, 0u);
              *reinterpret_cast<uint4*>(vt + dst) = make_uint4(0u, 0u, 0u, 0u);
            } else {
              cp_async_16(kt + dst, p.k_pool + src);
              cp_async_16(vt + dst, p.v_pool + src);
            }
          }
        }
      }
    }
  }
  // the prompt buffer is published once its copies have landed: after the
  // first blocks after the prefix are requested (planned call) or at once
  // (the dependency wait came first)
  [[maybe_unused]] auto publish_prompt = [&]() {
    if constexpr (PROMPT) {
      if (item_nb > 0 && warp == consumers) {
        cp_async_wait_all();
        __syncwarp();
        if (lane == 0) mbar_arrive(pbar);
      }
    }
  };
  if (!p.planned) publish_prompt();
  int pre_id = 0, early = 0;
  bool pre = false;
  if (p.planned) {
    if (warp == consumers && r0 < r1) {
      const int n0 = min(r1 - r0, cur.nblk - cur.j);
      pre_id = lane < n0 ? __ldg(p.bt + int64_t(cur.b) * p.W + p.prefix_blocks + cur.j + lane) : 0;
      pre = true;
      if constexpr (MMA) {
        const uint64_t pol = tc::l2_evict_first_policy();
        const int lim = min(min(n0, 32), min(p.nstages, cur.nblk - 1 - cur.j));
        for (; early < lim; ++early) {
          const int blk = __shfl_sync(0xffffffffu, pre_id, early);
          if (blk < 0 || blk >= p.num_blocks) break;  // the main loop reports it
          if (lane == 0)  // stage `early` is unused yet: no wait
            tile_fill(ring, static_cast<uint32_t>(early), tm_k, tm_v, blk * kBS,
                      cur.grp * p.hg_size, p.err, pol);
        }
      }
    }
    publish_prompt();
    pdl_wait();
    if (p.prefix_blocks == 0)
      zero_empty<T, HD>(p, blockIdx.x, G,
                        [&](int b) { return __ldcg(p.cu_units + b + 1) == __ldcg(p.cu_units + b); });
  }

  if (warp == consumers) {
    // ------------------------------------------------------ producer
    // each K/V block is read once per call: its lines leave L2 first
    const uint64_t pol = MMA ? tc::l2_evict_first_policy() : 0;
    uint32_t it = static_cast<uint32_t>(early);  // blocks already issued before the wait
    int skip = early;
    bool ok = true;
    for (int u = r0; u < r1 && ok;) {
      const int n = min(r1 - u, cur.nblk - cur.j);
      const int32_t* row = p.bt + int64_t(cur.b) * p.W;
      const int64_t head_off = int64_t(cur.grp) * p.hg_size * HD * p.elem_bytes;
      for (int jj = 0; jj < n && ok; jj += 32) {
        int id = pre ? pre_id : (jj + lane < n) ? __ldg(row + p.prefix_blocks + cur.j + jj + lane) : 0;
        pre = false;
        const int n_here = min(32, n - jj);
        const int k0 = skip;
        skip = 0;
        for (int k = k0; k < n_here; ++k) {
          if (*ring.abort_flag) { ok = false; break; }
          const int blk = __shfl_sync(0xffffffffu, id, k);
          const int j = p.prefix_blocks + cur.j + jj + k;  // table index
          int valid = min(kBS, cur.L - j * kBS);
          if (blk < 0 || blk >= p.num_blocks) {
            if (lane == 0) report(p.err, PKV_DEVERR_BLOCK_ID);
            valid = 0;
          }
          const int64_t off = int64_t(valid > 0 ? blk : 0) * kBS * token_pitch + head_off;
          // append: the step's token is the last of the sequence; its row
          // comes from k_new / v_new, which this CTA also stores to the pool
          const bool fresh = p.k_new != nullptr && j == p.prefix_blocks + cur.nblk - 1 && valid > 0 &&
                             __ldg(p.seq_lens + cur.b) == cur.L;  // not a clamped bad length
          const int new_row = fresh ? cur.L - 1 - j * kBS : -1;
          const int64_t new_off = int64_t(cur.b) * p.n_kv * HD * p.elem_bytes + head_off;
          bool filled;
          if constexpr (MMA) {
            // one lane loads the block's K and V boxes (a bad id reads the
            // zeros past the pool's end); the consumers put the new row in
            filled = lane == 0 ? tile_fill(ring, it, tm_k, tm_v,
                                           valid > 0 ? blk * kBS : p.num_blocks * kBS,
                                           cur.grp * p.hg_size, p.err, pol)
                               : true;
            filled = __shfl_sync(0xffffffffu, filled, 0);
          } else {
            filled = ring_fill(ring, it, p.k_pool + off, p.v_pool + off, token_pitch, valid, p.err,
                               new_row, p.k_new + new_off, p.v_new + new_off);
          }
          if (!filled) {
            *ring.abort_flag = 1;
            ok = false;
            break;
          }
          ++it;
          if (fresh) {
            const int nvec = row_bytes / 16;  // 16-byte pieces of this group's row
            const int64_t dst = off + int64_t(new_row) * token_pitch;
            for (int i = lane; i < 2 * nvec; i += 32) {
              const bool is_v = i >= nvec;
              const int64_t o = int64_t(is_v ? i - nvec : i) * 16;
              const uint4 x = __ldg(reinterpret_cast<const uint4*>((is_v ? p.v_new : p.k_new) +
                                                                   new_off + o));
              *reinterpret_cast<uint4*>(const_cast<uint8_t*>(is_v ? p.v_pool : p.k_pool) + dst +
                                        o) = x;
            }
          }
        }
      }
      u += n;
      cur.advance(p, n);
    }
    if (!ok) ring_drain(ring, it);
    // the split group this CTA merges (read by the merge kernel; a planned
    // call's plan already holds it)
    if (lane == 0 && !p.planned) {
      p.splits[blockIdx.x] = r0 < r1 ? split_entry(blockIdx.x, G, U, st.x, st.y, st.z,
                                                   walked_blocks(p, used_len(p, st.x)))
                                     : make_int4(-1, 0, 0, 0);
    }
  } else if (warp < consumers) {
    // ------------------------------------------------------ consumers
    Rows rows;
    if constexpr (!MMA) {
      float* scratch = reinterpret_cast<float*>(ring.stages + p.nstages * ring.stage_bytes);
      rows.bind(scratch + warp * RowsOf<T, HD, MAXR, MMA>::kScratch);
    }
    uint32_t it = 0;
    bool ok = true;
    const T* q = static_cast<const T*>(p.q);
    T* out = static_cast<T*>(p.out);
    for (int u = r0; u < r1 && ok;) {
      const int n = min(r1 - u, cur.nblk - cur.j);
      const int b = cur.b;
      const int kv_head = cur.grp * p.hg_size + warp;
      const int head0 = kv_head * p.rep;
      const int last = cur.L - 1;
      rows.begin(
          [&](int r) -> const T* {
            return r < p.rep ? q + (int64_t(b) * p.n_heads + head0 + r) * HD : nullptr;
          },
          [&](int) { return last; });
      if (!PROMPT && p.prefix_blocks > 0 && cur.j == 0) {
        // the group's first walked block: continue from the shared prefix
        const int64_t prow = int64_t(p.prefix_seed_run) * p.B * p.n_heads +
                             int64_t(b) * p.n_heads + head0;
        rows.seed([&](int r) -> const float* { return r < p.rep ? p.pre_o + (prow + r) * HD : nullptr; },
                  [&](int r) -> const float* { return p.pre_ml + (prow + r) * 2; });
      }
      // tile path, append: this lane's piece of the new token's K / V row
      // for this warp's head (the pool's copy is written by the producer)
      const bool has_last = cur.j + n == cur.nblk;
      bool fresh = false;
      uint32_t kn[2] = {0u, 0u}, vn[2] = {0u, 0u};
      if constexpr (MMA) {
        if (has_last && p.k_new != nullptr && __ldg(p.seq_lens + b) == cur.L) {
          const int blk = __ldg(p.bt + int64_t(b) * p.W + p.prefix_blocks + cur.nblk - 1);
          fresh = blk >= 0 && blk < p.num_blocks;
          if (fresh) new_row_piece<HD>(p.k_new, p.v_new, (int64_t(b) * p.n_kv + kv_head) * HD, kn, vn);
        }
      }
      for (int k = 0; k < n; ++k) {
        if (!ring_wait_full(ring, it, p.err)) {
          *ring.abort_flag = 1;
          ok = false;
          break;
        }
        const int st = static_cast<int>(it % ring.nstages);
        const int j0 = (p.prefix_blocks + cur.j + k) * kBS;
        if constexpr (MMA) {
          uint8_t* kt = ring.k_tile(st);
          uint8_t* vt = ring.v_tile(st);
          // the sequence's last block: rows past its end hold whatever the
          // pool slots hold, so zero them in V (K's are masked), and put in
          // the new token's row
          const bool fix = has_last && k == n - 1 && (cur.L - j0 < kBS || fresh);
          if (fix) tile_fix<HD>(kt, vt, warp, cur.L - j0, fresh, kn, vn);
          rows.block_sw(kt, vt, warp, j0, p.scale_log2);
          if (fix) fence_proxy_async_smem();  // before the stage's next TMA writes
        } else {
          const int hoff = warp * HD * p.elem_bytes;
          rows.block(ring.k_tile(st) + hoff, ring.v_tile(st) + hoff, ring.row_stride, j0,
                     p.scale_log2);
        }
        ring_release(ring, it);
        ++it;
      }
      if (!ok) break;
      const bool whole = (cur.j == 0) && (n == cur.nblk);
      if (PROMPT && whole) {
        // fused shared prefix: the prefix merge kernel adds the prompt runs
        const int64_t prow = int64_t(p.prompt_runs) * p.B * p.n_heads + int64_t(b) * p.n_heads + head0;
        rows.store_partial(
            [&](int r) -> float* { return r < p.rep ? p.pre_o + (prow + r) * HD : nullptr; },
            [&](int r) -> float* { return p.pre_ml + (prow + r) * 2; });
      } else if (whole) {
        rows.store([&](int r) -> T* {
          return r < p.rep ? out + (int64_t(b) * p.n_heads + head0 + r) * HD : nullptr;
        });
      } else {
        // partial result of a group split over several CTAs
        const int slot = 2 * blockIdx.x + (u == r0 ? 0 : 1);
        const int64_t base_row = int64_t(slot) * rows_per_group + warp * p.rep;
        rows.store_partial(
            [&](int r) -> float* { return r < p.rep ? p.ws_o + (base_row + r) * HD : nullptr; },
            [&](int r) -> float* { return p.ws_ml + (base_row + r) * 2; });
      }
      u += n;
      cur.advance(p, n);
    }
  } else if (PROMPT && warp > consumers && warp <= consumers + p.wide_mt && item_nb > 0) {
    // ------------------------------------------------------ prompt warps
    // warp consumers + 1 + w carries sequences item_s0 + w spm .. (row r:
    // query head r % rep of the KV head item_head); keys past a row's own
    // length are masked, and V rows past every chunk sequence's reach
    // (which may hold anything) are zeroed by each reading warp alike
    // before its P V
    if constexpr (PROMPT) {
      const int w = warp - consumers - 1;
      const int spm = kMaxRep / p.rep;
      const int pre_len = p.prefix_blocks * kBS;
      const int nseq = min(p.prompt_seqs, p.B - item_s0);
      int vis = 0;
      for (int t = lane; t < nseq; t += 32) vis = max(vis, min(used_len(p, item_s0 + t), pre_len));
      vis = static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<unsigned>(vis)));
      const int sw = item_s0 + w * spm;  // this warp's first sequence
      const int nrow = min(spm, max(0, p.B - sw)) * p.rep;
      if (nrow > 0) {
        const T* q = static_cast<const T*>(p.q);
        Rows rows;
        rows.begin(
            [&](int r) -> const T* {
              return r < nrow ? q + (int64_t(sw + r / p.rep) * p.n_heads + item_head * p.rep + r % p.rep) * HD
                              : nullptr;
            },
            [&](int r) { return min(used_len(p, sw + r / p.rep), pre_len) - 1; });
        if (!mbar_wait(pbar, 0)) {
          if (lane == 0) report(p.err, PKV_DEVERR_TIMEOUT);
        } else {
          const uint32_t none[2] = {0u, 0u};
          for (int i = 0; i < item_nb; ++i) {
            const int jpos = (item_j0 + i) * kBS;
            if (jpos >= vis) break;  // no chunk sequence reaches it
            uint8_t* kt = pbuf + i * (kBS * HD * 2);
            uint8_t* vt = pbuf + (p.prompt_bpr + i) * (kBS * HD * 2);
            if (vis - jpos < kBS) tile_fix<HD>(kt, vt, 0, vis - jpos, false, none, none);
            rows.block_sw(kt, vt, 0, jpos, p.scale_log2);
          }
        }
        const int64_t prow = int64_t(item_run) * p.B * p.n_heads;
        rows.store_partial(
            [&](int r) -> float* {
              return r < nrow ? p.pre_o + (prow + int64_t(sw + r / p.rep) * p.n_heads +
                                           item_head * p.rep + r % p.rep) * HD
                              : nullptr;
            },
            [&](int r) -> float* {
              return p.pre_ml + (prow + int64_t(sw + r / p.rep) * p.n_heads + item_head * p.rep +
                                 r % p.rep) * 2;
            });
      }
    }
  }
}

// Tensor-core path (bf16, head_dim 64 / 128): whole blocks as TMA tiles.
// The head_dim-64 kernel gets up to 112 registers (two 288-thread CTAs per
// SM), enough to keep it free of spills.
template <typename T, int HD>
__global__ void __launch_bounds__(decode_max_threads<T, HD>()) __maxnreg__(HD == 64 ? 112 : 224)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  DecodeParams p) {
  decode_body<T, HD, 16, true>(&tm_k, &tm_v, p);
}

// Tensor-core path with a shared prefix attended in the same launch: in
// the first prompt_items CTAs a second set of warps (wide_mt prompt warps)
// takes one run of the prefix for a chunk of sequences at one KV head
// while the consumers walk the CTA's range of the blocks after the prefix;
// all results are partials for decode_prefix_merge_kernel.
// Warps of the fused shared-prefix CTA: the consumers (one per KV head of
// the group, hg), the producer and up to hg prompt warps, within what the
// register file gives each of the four schedulers (at most 16 warps at 112
// registers for head_dim 64, 12 at 168 for head_dim 128).
template <int HD>
constexpr int fused_max_warps() {
  return HD == 64 ? 16 : 12;
}
inline int fused_prompt_warps(int hg, int max_warps) { return std::max(0, std::min(hg, max_warps - hg - 1)); }

template <typename T, int HD>
constexpr int fused_max_threads() {
  return (decode_max_threads<T, HD>() / 32 +
          (decode_max_threads<T, HD>() / 32 - 1 < fused_max_warps<HD>() - decode_max_threads<T, HD>() / 32
               ? decode_max_threads<T, HD>() / 32 - 1
               : fused_max_warps<HD>() - decode_max_threads<T, HD>() / 32)) * 32;
}

template <typename T, int HD>
__global__ void __launch_bounds__(fused_max_threads<T, HD>()) __maxnreg__(HD == 64 ? 112 : 224)
    decode_fused_prefix_kernel(const __grid_constant__ CUtensorMap tm_k,
                               const __grid_constant__ CUtensorMap tm_v, DecodeParams p) {
  decode_body<T, HD, 16, true, true>(&tm_k, &tm_v, p);
}

// CUDA-core path: a bulk copy per token row into a padded ring.
template <typename T, int HD, int MAXR>
__global__ void __launch_bounds__(decode_max_threads<T, HD>()) decode_rows_kernel(DecodeParams p) {
  decode_body<T, HD, MAXR, false>(nullptr, nullptr, p);
}

// ------------------------------------------------------- cluster decode
//
// Latency-bound batches (few, short sequences, where the stream-K split
// would leave each CTA a handful of blocks and the merge launch would cost
// as much as the reads) and shared prompt prefixes: one thread-block
// cluster of C CTAs per chunk of `spc` sequences and KV-head group.  The
// chunk's rows share one tensor-core tile (spc * rep <= 16 rows: row r is
// query head r % rep of sequence r / rep).  The cluster's block list is
// the shared prefix's blocks (every chunk row attends; keys past a row's
// own length are masked), then, sequence by sequence, each sequence's
// blocks after the prefix (only that sequence's rows attend): the prefix
// is read once per chunk instead of once per sequence.  Without a prefix
// and with one sequence per cluster this is plain split decode.  CTA r
// walks list positions [r n / C, (r + 1) n / C) (split points depend only
// on the lengths, C and spc, so placement and sharing of blocks change no
// bit), leaves its normalised partial (output rows, max, exp-sum) in its
// own shared memory, and after a cluster barrier the C CTAs combine the
// partials through distributed shared memory, each CTA a slice of the
// output elements, with log-sum-exp weights.  A second barrier keeps every
// CTA's shared memory alive until its peers have read it.  Every thread of
// the cluster reaches both barriers (waits in the loops are bounded; an
// aborted CTA still leaves a partial).  Nothing goes through global memory
// but the inputs and the output: no workspace, no merge launch.
constexpr int kMaxCluster = 8;
constexpr int kMaxChunk = 16;  // sequences per cluster (tile rows at one query head per KV head)

// Shared-memory bytes of the cluster kernel's partials and staged new rows
// beyond its ring: spc * rep rows per consumer warp.  Kept small so that
// the next call's CTAs fit beside the running ones (programmatic launch
// lets them enter early and set up while this call finishes).
inline size_t cluster_extra_bytes(int hg, int rep, int hd, int elem_bytes, int spc, bool append) {
  const size_t rows = size_t(hg) * spc * rep;
  return rows * hd * 4 + (rows * 2 * 4 + 15) / 16 * 16 +  // outputs; (max, sum) pairs, padded
         (append ? size_t(spc) * 2 * hg * hd * elem_bytes : 0);  // staged step rows
}

// Plain split decode of latency-bound batches (no shared prefix): one
// cluster per (sequence, KV-head group), as above with spc = 1; a leaner
// body than the prefix one below (no list, no staging), so that the next
// call's CTAs fit beside it and the set-up stays one round trip.
template <typename T, int HD, int MAXR, bool MMA>
__device__ __forceinline__ void decode_cluster_body(const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                                    const DecodeParams& p) {
  extern __shared__ __align__(128) uint8_t smem[];
  using Rows = typename RowsOf<T, HD, MAXR, MMA>::type;
  const int consumers = p.hg_size;
  const int row_bytes = p.hg_size * HD * p.elem_bytes;
  Ring ring = MMA ? make_tile_ring(smem, p.nstages, kBS * row_bytes)
                  : make_ring(smem, p.nstages, row_bytes);
  ring_init(ring, consumers);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = p.cluster;
  const int rank = static_cast<int>(cluster_ctarank());
  const int seg = static_cast<int>(blockIdx.x) / C;  // (sequence, head group)
  const int b = seg / p.n_groups;
  const int grp = seg - b * p.n_groups;
  const int rows_per_group = p.hg_size * p.rep;
  float* part_o = reinterpret_cast<float*>(smem + p.part_off);  // [rows_per_group][HD]
  float* part_ml = part_o + rows_per_group * HD;                // [rows_per_group][2]

  // A planned call checks the kept plan (written by a finished launch) before
  // anything else; every CTA of the cluster reads the same record, so all of
  // them leave here together, before any cluster barrier.  Its lengths and
  // tables are unchanged since the plan, so they are read in the same round
  // trip; a call planning for itself reads them after the dependency wait.
  if (!p.planned) pdl_wait();  // lengths and tables may come from the preceding kernel
  const bool plan_ok = !p.planned || plan_matches(p, p.grid);
  const int L = used_len(p, b);
  // the producer holds the table row's first 64 entries (this path's
  // sequences have at most 64 blocks; entries past the length are not used)
  int ids[2] = {0, 0};
  if (warp == consumers) {
    const int32_t* trow = p.bt + int64_t(b) * p.W;
    if (lane < p.W) ids[0] = __ldg(trow + lane);
    if (lane + 32 < p.W) ids[1] = __ldg(trow + lane + 32);
  }
  if (!plan_ok) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(p.err, PKV_DEVERR_PLAN);
    return;
  }
  pdl_launch_dependents();
  if (!p.planned && blockIdx.x == 0 && threadIdx.x == 0)
    p.total_units[1] = -1;  // a call planning for itself replaces any kept plan

  const int nblk = (L + kBS - 1) / kBS;
  const int j0 = static_cast<int>(int64_t(rank) * nblk / C);
  const int j1 = static_cast<int>(int64_t(rank + 1) * nblk / C);
  if (!p.planned && rank == 0 && grp == 0 && threadIdx.x == 0) check_length(p, b);
  const int64_t token_pitch = int64_t(p.n_kv) * HD * p.elem_bytes;
  const int64_t head_off = int64_t(grp) * p.hg_size * HD * p.elem_bytes;
  // append: the CTA holding the sequence's last block stores and uses the
  // step's row (not for a length clamped from a bad value)
  const bool append = p.k_new != nullptr && j1 == nblk && j1 > j0 && __ldg(p.seq_lens + b) == L;

  if (warp == consumers) {
    // ------------------------------------------------------ producer
    // A planned call loads its first blocks before the kernel launched just
    // before it has finished (up to a ring's worth, never the sequence's
    // last block, the only one a decode step writes), then waits.
    bool waited = !p.planned;
    const uint64_t pol = MMA ? tc::l2_evict_first_policy() : 0;  // K/V read once
    uint32_t it = 0;
    bool ok = true;
    {
      for (int j = j0; j < j1 && ok; ++j) {
        const int jj = j & ~31, k = j & 31;  // the entry sits in lane k of ids[jj / 32]
        if (!waited && (!MMA || it >= static_cast<uint32_t>(p.nstages) || j == nblk - 1)) {
          pdl_wait();
          waited = true;
        }
        if (*ring.abort_flag) { ok = false; break; }
        const int blk = __shfl_sync(0xffffffffu, ids[jj >> 5], k);
        int valid = min(kBS, L - j * kBS);
        if (blk < 0 || blk >= p.num_blocks) {
          if (lane == 0) report(p.err, PKV_DEVERR_BLOCK_ID);
          valid = 0;
        }
        const int64_t off = int64_t(valid > 0 ? blk : 0) * kBS * token_pitch + head_off;
        const bool fresh = append && j == nblk - 1 && valid > 0;
        const int new_row = fresh ? L - 1 - j * kBS : -1;
        const int64_t new_off = int64_t(b) * p.n_kv * HD * p.elem_bytes + head_off;
        bool filled;
        if constexpr (MMA) {
          filled = lane == 0 ? tile_fill(ring, it, tm_k, tm_v,
                                         valid > 0 ? blk * kBS : p.num_blocks * kBS,
                                         grp * p.hg_size, p.err, pol)
                             : true;
          filled = __shfl_sync(0xffffffffu, filled, 0);
        } else {
          filled = ring_fill(ring, it, p.k_pool + off, p.v_pool + off, token_pitch, valid, p.err,
                             new_row, p.k_new + new_off, p.v_new + new_off);
        }
        if (!filled) {
          *ring.abort_flag = 1;
          ok = false;
          break;
        }
        ++it;
        if (fresh) {  // the pool's copy of the step's row (this group's heads)
          const int nvec = row_bytes / 16;
          const int64_t dst = off + int64_t(new_row) * token_pitch;
          for (int i = lane; i < 2 * nvec; i += 32) {
            const bool is_v = i >= nvec;
            const int64_t o = int64_t(is_v ? i - nvec : i) * 16;
            const uint4 x = __ldg(reinterpret_cast<const uint4*>((is_v ? p.v_new : p.k_new) +
                                                                 new_off + o));
            *reinterpret_cast<uint4*>(const_cast<uint8_t*>(is_v ? p.v_pool : p.k_pool) + dst + o) = x;
          }
        }
      }
    }
    if (!ok) ring_drain(ring, it);
  } else if (warp < consumers) {
    // ------------------------------------------------------ consumers
    Rows rows;
    if constexpr (!MMA) {
      float* scratch = reinterpret_cast<float*>(ring.stages + p.nstages * ring.stage_bytes);
      rows.bind(scratch + warp * RowsOf<T, HD, MAXR, MMA>::kScratch);
    }
    if (p.planned) pdl_wait();  // the queries may come from the preceding kernel
    const T* q = static_cast<const T*>(p.q);
    const int kv_head = grp * p.hg_size + warp;
    const int head0 = kv_head * p.rep;
    const int last = L - 1;
    rows.begin(
        [&](int r) -> const T* {
          return r < p.rep ? q + (int64_t(b) * p.n_heads + head0 + r) * HD : nullptr;
        },
        [&](int) { return last; });
    bool fresh = false;
    uint32_t kn[2] = {0u, 0u}, vn[2] = {0u, 0u};
    if constexpr (MMA) {
      if (append) {
        const int blk = __ldg(p.bt + int64_t(b) * p.W + nblk - 1);
        fresh = blk >= 0 && blk < p.num_blocks;
        if (fresh) new_row_piece<HD>(p.k_new, p.v_new, (int64_t(b) * p.n_kv + kv_head) * HD, kn, vn);
      }
    }
    uint32_t it = 0;
    for (int j = j0; j < j1; ++j, ++it) {
      if (!ring_wait_full(ring, it, p.err)) {
        *ring.abort_flag = 1;
        break;
      }
      const int st = static_cast<int>(it % ring.nstages);
      const int jpos = j * kBS;
      if constexpr (MMA) {
        uint8_t* kt = ring.k_tile(st);
        uint8_t* vt = ring.v_tile(st);
        const bool fix = j == nblk - 1 && (L - jpos < kBS || fresh);
        if (fix) tile_fix<HD>(kt, vt, warp, L - jpos, fresh, kn, vn);
        rows.block_sw(kt, vt, warp, jpos, p.scale_log2);
        if (fix) fence_proxy_async_smem();
      } else {
        const int hoff = warp * HD * p.elem_bytes;
        rows.block(ring.k_tile(st) + hoff, ring.v_tile(st) + hoff, ring.row_stride, jpos,
                   p.scale_log2);
      }
      ring_release(ring, it);
    }
    // this CTA's part (also after an abort, so the barrier below is reached)
    rows.store_partial(
        [&](int r) -> float* { return r < p.rep ? part_o + (warp * p.rep + r) * HD : nullptr; },
        [&](int r) -> float* { return part_ml + (warp * p.rep + r) * 2; });
  }

  cluster_sync();  // every CTA's partial is in its shared memory
  // CTA `rank` combines elements [rank E / C, (rank + 1) E / C) of the
  // group's rows x head_dim outputs from the C partials
  const int E = rows_per_group * HD;
  const int e0 = rank * E / C, e1 = (rank + 1) * E / C;
  T* out = static_cast<T*>(p.out) + (int64_t(b) * p.n_heads + int64_t(grp) * rows_per_group) * HD;
  for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += static_cast<int>(blockDim.x)) {
    const int r = e / HD;
    float2 ml[kMaxCluster];
    float oc[kMaxCluster];
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {  // every peer's values in one round trip
      ml[c] = make_float2(-INFINITY, 0.f);
      oc[c] = 0.f;
      if (c < C) {
        ml[c] = ld_cluster_f32x2(cluster_map(part_ml + r * 2, c));
        oc[c] = ld_cluster_f32(cluster_map(part_o + e, c));
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c)
      if (ml[c].y > 0.f) M = fmaxf(M, ml[c].x);  // a part that saw no key has no weight
    float acc = 0.f, den = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {
      if (ml[c].y > 0.f) {
        const float w = fast_exp2(ml[c].x - M) * ml[c].y;
        den += w;
        acc = fmaf(w, oc[c], acc);
      }
    }
    out[e] = Elem<T>::from_f(den > 0.f ? acc * (1.f / den) : 0.f);
  }
  cluster_sync();  // the peers have read this CTA's partials
}

template <typename T, int HD, int MAXR, bool MMA>
__device__ __forceinline__ void decode_cluster_prefix_body(const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                                    const DecodeParams& p) {
  extern __shared__ __align__(128) uint8_t smem[];
  using Rows = typename RowsOf<T, HD, MAXR, MMA>::type;
  const int consumers = p.hg_size;
  const int row_bytes = p.hg_size * HD * p.elem_bytes;  // the group's heads of one token
  Ring ring = MMA ? make_tile_ring(smem, p.nstages, kBS * row_bytes)
                  : make_ring(smem, p.nstages, row_bytes);
  uint64_t* fresh_bar = reinterpret_cast<uint64_t*>(smem + 768);  // past the ring's barriers
  if (threadIdx.x == 0) mbar_init(fresh_bar, 1);
  ring_init(ring, consumers);  // (its barrier also publishes fresh_bar's init)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = p.cluster;
  const int rank = static_cast<int>(cluster_ctarank());
  const int seg = static_cast<int>(blockIdx.x) / C;  // (chunk of sequences, head group)
  const int chunk = seg / p.n_groups;
  const int grp = seg - chunk * p.n_groups;
  const int spc = p.cluster_seqs;
  const int s0 = chunk * spc;
  const int ns = min(spc, p.B - s0);  // sequences of this chunk
  const int P = p.prefix_blocks;
  const bool plain = spc == 1 && P == 0;
  const int PR = spc * p.rep;  // partial rows per consumer warp (<= R)
  float* part_o = reinterpret_cast<float*>(smem + p.part_off);  // [consumers][PR][HD]
  float* part_ml = part_o + consumers * PR * HD;                // [consumers][PR][2]
  // staged step rows [spc][K|V][row_bytes]: bulk-copy destinations, so on a
  // 16-byte boundary after the (max, sum) pairs
  uint8_t* fresh = reinterpret_cast<uint8_t*>(part_ml) + (consumers * PR * 2 * 4 + 15) / 16 * 16;
  __shared__ int len_s[kMaxChunk];      // used length of each chunk sequence
  __shared__ int cum_s[kMaxChunk + 1];  // list position where each sequence's own blocks start
  __shared__ int app_s[kMaxChunk];      // 1: the sequence's step row is appended (k_new given,
                                        // a length not clamped, the token past the prefix)
  __shared__ int fresh_s[kMaxChunk];    // set by the producer with the sequence's last tile:
                                        // 1 if its step row goes into that tile

  // A planned call checks the kept plan (written by a finished launch) before
  // anything else; every CTA of the cluster reads the same record, so all of
  // them leave here together, before any cluster barrier.  Its lengths and
  // tables are unchanged since the plan, so they are read in the same round
  // trip; a call planning for itself reads them after the dependency wait.
  if (!p.planned) pdl_wait();  // lengths and tables may come from the preceding kernel
  const bool plan_ok = !p.planned || plan_matches(p, p.grid);
  if (threadIdx.x < kMaxChunk) {
    const int t = threadIdx.x;
    const int raw = t < ns ? __ldg(p.seq_lens + s0 + t) : 0;
    const int L = raw < 0 ? 0 : (raw > p.max_len ? p.max_len : raw);  // as used_len
    len_s[t] = L;
    app_s[t] = p.k_new != nullptr && raw == L && L > P * kBS;
    fresh_s[t] = 0;
    // bad lengths (as check_length; a planned call's plan reported them),
    // once, by the group-0 CTAs of rank 0
    if (t < ns && !p.planned && grp == 0 && cluster_ctarank() == 0) {
      if (raw < 0 || raw > p.max_seq_len) report(p.err, PKV_DEVERR_LENGTH);
      else if (raw > p.W * kBS) report(p.err, PKV_DEVERR_TABLE_WIDTH);
    }
    // with append, a new token inside the shared prefix would land in a
    // block other sequences read: not written, reported
    if (t < ns && p.k_new != nullptr && P > 0 && L > 0 && L <= P * kBS && grp == 0 &&
        cluster_ctarank() == 0)
      report(p.err, PKV_DEVERR_PREFIX);
  }
  // plain split decode: the producer holds the table row's first 64 entries
  // (this path's sequences have at most 64 blocks; entries past the length
  // are not used), loaded with the length
  int ids_pre[2] = {0, 0};
  if (plain && warp == consumers) {
    const int32_t* trow = p.bt + int64_t(s0) * p.W;
    if (lane < p.W) ids_pre[0] = __ldg(trow + lane);
    if (lane + 32 < p.W) ids_pre[1] = __ldg(trow + lane + 32);
  }
  __syncthreads();
  if (!plan_ok) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(p.err, PKV_DEVERR_PLAN);
    return;
  }
  pdl_launch_dependents();
  if (!p.planned && blockIdx.x == 0 && threadIdx.x == 0)
    p.total_units[1] = -1;  // a call planning for itself replaces any kept plan
  // the list: prefix positions [0, Pe) (as far as any chunk sequence sees),
  // then sequence s's own blocks from cum_s[s]
  int vis = 0;  // positions of the prefix some chunk sequence sees
  for (int s = 0; s < ns; ++s) vis = max(vis, min(len_s[s], P * kBS));
  const int Pe = (vis + kBS - 1) / kBS;
  if (threadIdx.x == 0) {
    int c = Pe;
    for (int s = 0; s < ns; ++s) {
      cum_s[s] = c;
      c += max(0, (len_s[s] + kBS - 1) / kBS - P);
    }
    cum_s[ns] = c;
  }
  __syncthreads();
  const int n = cum_s[ns];
  const int j0 = static_cast<int>(int64_t(rank) * n / C);
  const int j1 = static_cast<int>(int64_t(rank + 1) * n / C);
  const int64_t token_pitch = int64_t(p.n_kv) * HD * p.elem_bytes;
  const int64_t head_off = int64_t(grp) * p.hg_size * HD * p.elem_bytes;
  // list position -> (chunk sequence or -1 for the prefix, table index)
  auto locate = [&](int t, int& sq, int& j) {
    if (t < Pe) {
      sq = -1;
      j = t;
    } else {
      sq = 0;
      while (sq + 1 < ns && cum_s[sq + 1] <= t) ++sq;
      j = P + (t - cum_s[sq]);
    }
  };
  // append: sequence s's step row is stored and used by the CTA holding its
  // last block (a length clamped from a bad value, or a token inside the
  // shared prefix, gets none)
  auto appends = [&](int sq) { return app_s[sq] != 0; };

  if (warp == consumers) {
    // ------------------------------------------------------ producer
    // A planned call loads its first blocks before the kernel launched just
    // before it has finished (up to a ring's worth, never a sequence's last
    // block, the only one a decode step writes), then waits.
    bool waited = !p.planned;
    const uint64_t pol = MMA ? tc::l2_evict_first_policy() : 0;  // K/V read once
    // The step rows this CTA's tiles need (tile path, append), staged once
    // for the consumers to patch into the tiles.  k_new / v_new may come
    // from the preceding kernel: staged right after the dependency wait.
    // (with one sequence per cluster the consumers load the row themselves)
    const bool stage = MMA && p.k_new != nullptr && spc > 1;
    auto stage_fresh = [&]() {
      if (lane != 0) return;
      uint32_t bytes = 0;
      for (int sq = 0; sq < ns; ++sq) {
        const int last_t = cum_s[sq + 1] - 1;
        if (cum_s[sq + 1] > cum_s[sq] && last_t >= j0 && last_t < j1 && appends(sq)) bytes += 2 * row_bytes;
      }
      mbar_arrive_expect_tx(fresh_bar, bytes);
      for (int sq = 0; sq < ns; ++sq) {
        const int last_t = cum_s[sq + 1] - 1;
        if (cum_s[sq + 1] > cum_s[sq] && last_t >= j0 && last_t < j1 && appends(sq)) {
          const int64_t src = int64_t(s0 + sq) * p.n_kv * HD * p.elem_bytes + head_off;
          bulk_copy_g2s(fresh + (2 * sq) * row_bytes, p.k_new + src, row_bytes, fresh_bar);
          bulk_copy_g2s(fresh + (2 * sq + 1) * row_bytes, p.v_new + src, row_bytes, fresh_bar);
        }
      }
    };
    if (stage && waited) stage_fresh();
    uint32_t it = 0;
    bool ok = true;
    for (int t0 = j0; t0 < j1 && ok; t0 += 32) {
      int my_s = -1, my_j = 0, my_id = 0;
      if (t0 + lane < j1) {
        locate(t0 + lane, my_s, my_j);
        if (!plain) my_id = __ldg(p.bt + int64_t(my_s < 0 ? 0 : s0 + my_s) * p.W + my_j);
      }
      const int n_here = min(32, j1 - t0);
      for (int k = 0; k < n_here && ok; ++k) {
        const int t = t0 + k;
        const int sq = __shfl_sync(0xffffffffu, my_s, k);
        const int j = __shfl_sync(0xffffffffu, my_j, k);
        const int blk = plain ? __shfl_sync(0xffffffffu, ids_pre[t >> 5], t & 31)
                              : __shfl_sync(0xffffffffu, my_id, k);
        const int L = sq < 0 ? vis : len_s[sq];
        const bool last_blk = sq >= 0 && t == cum_s[sq + 1] - 1;
        if (!waited && (!MMA || it >= static_cast<uint32_t>(p.nstages) || last_blk)) {
          pdl_wait();
          waited = true;
          if (stage) stage_fresh();
        }
        if (*ring.abort_flag) { ok = false; break; }
        int valid = min(kBS, L - j * kBS);
        if (blk < 0 || blk >= p.num_blocks) {
          if (lane == 0) report(p.err, PKV_DEVERR_BLOCK_ID);
          valid = 0;
        }
        const int64_t off = int64_t(valid > 0 ? blk : 0) * kBS * token_pitch + head_off;
        const bool fresh_row = last_blk && valid > 0 && appends(sq);
        const int new_row = fresh_row ? L - 1 - j * kBS : -1;
        // for the consumers, published by the tile's arrival (release / acquire)
        if (last_blk && lane == 0) fresh_s[sq] = fresh_row ? 1 : 0;
        const int64_t new_off = int64_t(s0 + (sq < 0 ? 0 : sq)) * p.n_kv * HD * p.elem_bytes + head_off;
        bool filled;
        if constexpr (MMA) {
          // prefix blocks are read by every chunk's cluster: no evict-first
          filled = lane == 0 ? tile_fill(ring, it, tm_k, tm_v,
                                         valid > 0 ? blk * kBS : p.num_blocks * kBS,
                                         grp * p.hg_size, p.err, sq < 0 ? 0 : pol)
                             : true;
          filled = __shfl_sync(0xffffffffu, filled, 0);
        } else {
          filled = ring_fill(ring, it, p.k_pool + off, p.v_pool + off, token_pitch, valid, p.err,
                             new_row, p.k_new + new_off, p.v_new + new_off);
        }
        if (!filled) {
          *ring.abort_flag = 1;
          ok = false;
          break;
        }
        ++it;
        if (fresh_row) {  // the pool's copy of the step's row (this group's heads)
          const int nvec = row_bytes / 16;
          const int64_t dst = off + int64_t(new_row) * token_pitch;
          for (int i = lane; i < 2 * nvec; i += 32) {
            const bool is_v = i >= nvec;
            const int64_t o = int64_t(is_v ? i - nvec : i) * 16;
            const uint4 x = __ldg(reinterpret_cast<const uint4*>((is_v ? p.v_new : p.k_new) +
                                                                 new_off + o));
            *reinterpret_cast<uint4*>(const_cast<uint8_t*>(is_v ? p.v_pool : p.k_pool) + dst + o) = x;
          }
        }
      }
    }
    if (!ok) ring_drain(ring, it);
    if (stage) {
      if (!waited) {  // every block was loaded early: stage now (nothing here needs it)
        pdl_wait();
        waited = true;
        stage_fresh();
      }
      if (lane == 0) mbar_wait(fresh_bar, 0);  // staged rows land before the CTA can exit
    }
    // the prefix blocks this CTA read: every chunk sequence that reaches one
    // must name it where row 0 does (checked off the loading path)
    const int pe1 = min(j1, Pe);
    for (int idx = lane; idx < ns * max(0, pe1 - j0); idx += 32) {
      const int sq = idx / (pe1 - j0), j = j0 + idx - sq * (pe1 - j0);
      if (len_s[sq] > j * kBS && __ldg(p.bt + int64_t(s0 + sq) * p.W + j) != __ldg(p.bt + j))
        report(p.err, PKV_DEVERR_PREFIX);
    }
  } else if (warp < consumers) {
    // ------------------------------------------------------ consumers
    Rows rows;
    if constexpr (MMA) rows.set_row_slots(p.rep);
    if constexpr (!MMA) {
      float* scratch = reinterpret_cast<float*>(ring.stages + p.nstages * ring.stage_bytes);
      rows.bind(scratch + warp * RowsOf<T, HD, MAXR, MMA>::kScratch);
    }
    if (p.planned) pdl_wait();  // the queries may come from the preceding kernel
    const T* q = static_cast<const T*>(p.q);
    const int kv_head = grp * p.hg_size + warp;
    const int head0 = kv_head * p.rep;
    const int nrows = ns * p.rep;
    rows.begin(
        [&](int r) -> const T* {
          return r < nrows ? q + (int64_t(s0 + r / p.rep) * p.n_heads + head0 + r % p.rep) * HD
                           : nullptr;
        },
        [&](int r) { return len_s[r / p.rep] - 1; });
    // one sequence per cluster: its step row, loaded with the queries when
    // this CTA holds the sequence's last block (used if the producer finds
    // that block's id valid)
    uint32_t kn1[2] = {0u, 0u}, vn1[2] = {0u, 0u};
    if constexpr (MMA) {
      if (spc == 1 && app_s[0] && j1 == n && n > cum_s[0])
        new_row_piece<HD>(p.k_new, p.v_new, (int64_t(s0) * p.n_kv + kv_head) * HD, kn1, vn1);
    }
    bool fresh_ready = false;
    uint32_t it = 0;
    for (int t = j0; t < j1; ++t, ++it) {
      if (!ring_wait_full(ring, it, p.err)) {
        *ring.abort_flag = 1;
        break;
      }
      int sq, j;
      locate(t, sq, j);
      const int st = static_cast<int>(it % ring.nstages);
      const int jpos = j * kBS;
      if constexpr (MMA) {
        uint8_t* kt = ring.k_tile(st);
        uint8_t* vt = ring.v_tile(st);
        const int L = sq < 0 ? vis : len_s[sq];
        const bool last_blk = sq >= 0 && t == cum_s[sq + 1] - 1;
        bool fresh_row = false;
        uint32_t kn[2] = {0u, 0u}, vn[2] = {0u, 0u};
        if (last_blk && appends(sq)) {
          fresh_row = fresh_s[sq] != 0;  // the producer found a valid block id
          if (fresh_row && spc == 1) {
            kn[0] = kn1[0], kn[1] = kn1[1], vn[0] = vn1[0], vn[1] = vn1[1];
          } else if (fresh_row) {
            if (!fresh_ready && !mbar_wait(fresh_bar, 0)) {
              if (lane == 0) report(p.err, PKV_DEVERR_TIMEOUT);
              *ring.abort_flag = 1;
              break;
            }
            fresh_ready = true;
            const uint8_t* fk = fresh + (2 * sq) * row_bytes + warp * HD * 2 + lane * (HD / 16);
            if constexpr (HD / 16 == 8) {
              const uint2 a = *reinterpret_cast<const uint2*>(fk);
              const uint2 c = *reinterpret_cast<const uint2*>(fk + row_bytes);
              kn[0] = a.x, kn[1] = a.y, vn[0] = c.x, vn[1] = c.y;
            } else {
              kn[0] = *reinterpret_cast<const uint32_t*>(fk);
              vn[0] = *reinterpret_cast<const uint32_t*>(fk + row_bytes);
            }
          }
        }
        const bool fix = (L - jpos < kBS) || fresh_row;
        if (fix) tile_fix<HD>(kt, vt, warp, min(kBS, L - jpos), fresh_row, kn, vn);
        rows.block_sw(kt, vt, warp, jpos, p.scale_log2, sq);
        if (fix) fence_proxy_async_smem();
      } else {
        // plain split decode only (a shared prefix takes the tile path)
        const int hoff = warp * HD * p.elem_bytes;
        rows.block(ring.k_tile(st) + hoff, ring.v_tile(st) + hoff, ring.row_stride, jpos,
                   p.scale_log2);
      }
      ring_release(ring, it);
    }
    // this CTA's part (also after an abort, so the barrier below is reached)
    rows.store_partial(
        [&](int r) -> float* { return r < nrows ? part_o + (warp * PR + r) * HD : nullptr; },
        [&](int r) -> float* { return part_ml + (warp * PR + r) * 2; });
  }

  cluster_sync();  // every CTA's partial is in its shared memory
  // CTA `rank` combines elements [rank E / C, (rank + 1) E / C) of the
  // chunk's active rows x head_dim outputs (warp-major) from the C partials
  const int nrows = ns * p.rep;
  const int E = consumers * nrows * HD;
  const int e0 = static_cast<int>(int64_t(rank) * E / C), e1 = static_cast<int>(int64_t(rank + 1) * E / C);
  T* out = static_cast<T*>(p.out);
  for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += static_cast<int>(blockDim.x)) {
    const int w = e / (nrows * HD);
    const int rem = e - w * nrows * HD;
    const int r = rem / HD, d = rem - (rem / HD) * HD;
    const int prow = w * PR + r;
    float2 ml[kMaxCluster];
    float oc[kMaxCluster];
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {  // every peer's values in one round trip
      ml[c] = make_float2(-INFINITY, 0.f);
      oc[c] = 0.f;
      if (c < C) {
        ml[c] = ld_cluster_f32x2(cluster_map(part_ml + prow * 2, c));
        oc[c] = ld_cluster_f32(cluster_map(part_o + prow * HD + d, c));
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c)
      if (ml[c].y > 0.f) M = fmaxf(M, ml[c].x);  // a part that saw no key has no weight
    float acc = 0.f, den = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {
      if (ml[c].y > 0.f) {
        const float wgt = fast_exp2(ml[c].x - M) * ml[c].y;
        den += wgt;
        acc = fmaf(wgt, oc[c], acc);
      }
    }
    const int64_t orow = int64_t(s0 + r / p.rep) * p.n_heads + (grp * p.hg_size + w) * p.rep + r % p.rep;
    out[orow * HD + d] = Elem<T>::from_f(den > 0.f ? acc * (1.f / den) : 0.f);
  }
  cluster_sync();  // the peers have read this CTA's partials
}

template <typename T, int HD>
__global__ void __launch_bounds__(decode_max_threads<T, HD>()) __maxnreg__(HD == 64 ? 112 : 224)
    decode_cluster_kernel(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, DecodeParams p) {
  decode_cluster_body<T, HD, 16, true>(&tm_k, &tm_v, p);
}

template <typename T, int HD, int MAXR>
__global__ void __launch_bounds__(decode_max_threads<T, HD>())
    decode_cluster_rows_kernel(DecodeParams p) {
  decode_cluster_body<T, HD, MAXR, false>(nullptr, nullptr, p);
}

template <typename T, int HD>
__global__ void __launch_bounds__(decode_max_threads<T, HD>()) __maxnreg__(HD == 64 ? 112 : 224)
    decode_cluster_prefix_kernel(const __grid_constant__ CUtensorMap tm_k,
                                 const __grid_constant__ CUtensorMap tm_v, DecodeParams p) {
  decode_cluster_prefix_body<T, HD, 16, true>(&tm_k, &tm_v, p);
}

// ------------------------------------------------- wide shared prefix
//
// A long prompt common to many sequences: every sequence's rows attend to
// all of its blocks, so each block is read once per KV head for a chunk of
// up to 16 tiles of rows (64 sequences at 4 query heads per KV head)
// instead of once per tile.  One cluster of K CTAs per (KV head, chunk of
// sequences); CTA r walks run r of the prefix, blocks [r P / K, (r+1) P / K)
// of row 0's table, one KV head per TMA tile (16 tokens x head_dim), each
// tile used by every consumer warp.  Warp w carries the rows of sequences
// s0 + w spm .. s0 + (w+1) spm - 1 (spm = 16 / rep; row i = query head
// i % rep of sequence i / rep), keys past a row's own length masked.  After
// a cluster barrier the K partials of each row are combined through
// distributed shared memory, each CTA a slice of the rows x head_dim
// elements: a sequence that ends inside the prefix gets its output, any
// other sequence a normalised partial (output, max, exp-sum) in run slot
// prefix_seed_run, from which the main kernel goes on over its own blocks.
// A second barrier keeps each CTA's partials alive until its peers have
// read them.
constexpr int kWideMaxSeqs = 256;  // sequences of one chunk: 16 tiles x 16 rows at one head

template <int HD>
constexpr int wide_max_warps() {
  return HD == 64 ? 16 : 8;  // 112 / 224 registers per thread: 544 / 288 threads per CTA
}

template <typename T, int HD>
__global__ void __launch_bounds__((wide_max_warps<HD>() + 1) * 32) __maxnreg__(HD == 64 ? 112 : 224)
    decode_prefix_wide_kernel(const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v, DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int len_s[kWideMaxSeqs];  // used length of each chunk sequence
  __shared__ int vis_s;                // prefix positions some chunk sequence sees
  const int mt = p.wide_mt;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = p.cluster;
  const int rank = static_cast<int>(cluster_ctarank());
  const int seg = static_cast<int>(blockIdx.x) / K;  // (chunk of sequences, KV head)
  const int head = seg % p.n_kv;
  const int s0 = (seg / p.n_kv) * p.cluster_seqs;
  const int ns = min(p.cluster_seqs, p.B - s0);
  const int spm = kMaxRep / p.rep;  // sequences per warp
  const int P = p.prefix_blocks;
  const int pre_len = P * kBS;
  const int j0 = static_cast<int>(int64_t(rank) * P / K);
  const int jr = static_cast<int>(int64_t(rank + 1) * P / K);  // this CTA's run: [j0, jr)
  float* part_o = reinterpret_cast<float*>(smem + p.part_off);  // [mt][16][HD]
  float* part_ml = part_o + mt * 16 * HD;                        // [mt][16][2]

  // A planned call reads its plan record, the lengths and the run's table
  // entries (unchanged since the plan) before the dependency wait, all in
  // one round trip; every CTA of the cluster sees the same record, so all
  // leave together on a mismatch.
  if (!p.planned) pdl_wait();
  int id0 = 0;  // producer: the first 32 table entries of the run (row 0's)
  if (warp == mt && j0 + lane < jr) id0 = __ldg(p.bt + j0 + lane);
  const bool plan_ok = !p.planned || plan_matches(p, p.grid);
  int my_vis = 0;
  for (int t = threadIdx.x; t < ns; t += blockDim.x) {
    const int L = used_len(p, s0 + t);
    len_s[t] = L;
    my_vis = max(my_vis, min(L, pre_len));
  }
  if (threadIdx.x == 0) vis_s = 0;
  Ring ring = make_tile_ring(smem, p.nstages, kBS * HD * 2);  // one head: 16 tokens x HD bf16
  ring_init(ring, mt);  // (its barrier publishes vis_s = 0 and the lengths)
  my_vis = static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<unsigned>(my_vis)));
  if (lane == 0 && my_vis > 0) atomicMax(&vis_s, my_vis);
  __syncthreads();
  if (!plan_ok) return;  // reported by the main kernel
  const int vis = vis_s;
  const int j1 = min(jr, (vis + kBS - 1) / kBS);

  if (warp == mt) {
    // ------------------------------------------------------ producer
    // The prefix blocks are never written by a decode step (a token that
    // would land in one is refused), so a planned call loads them before
    // the preceding kernel has finished.
    const uint64_t pol = p.wide_evict ? tc::l2_evict_first_policy() : 0;
    uint32_t it = 0;
    bool ok = true;
    for (int jb = j0; jb < j1 && ok; jb += 32) {
      const int id = jb == j0 ? id0 : jb + lane < j1 ? __ldg(p.bt + jb + lane) : 0;  // row 0's table
      for (int k = 0; k < min(32, j1 - jb); ++k) {
        if (*ring.abort_flag) { ok = false; break; }
        const int blk = __shfl_sync(0xffffffffu, id, k);
        const bool bad = blk < 0 || blk >= p.num_blocks;
        if (bad && lane == 0) report(p.err, PKV_DEVERR_BLOCK_ID);
        // a bad id reads the zeros past the pool's end
        bool filled = lane == 0 ? tile_fill(ring, it, &tm_k, &tm_v, bad ? p.num_blocks * kBS : blk * kBS,
                                            head, p.err, pol)
                                : true;
        filled = __shfl_sync(0xffffffffu, filled, 0);
        if (!filled) {
          *ring.abort_flag = 1;
          ok = false;
          break;
        }
        ++it;
      }
    }
    if (!ok) ring_drain(ring, it);
    // every chunk sequence that reaches one of this run's blocks must name
    // it where row 0 does (checked once, by the head-0 clusters)
    if (head == 0 && j1 > j0) {
      const int nj = j1 - j0;
      for (int idx = lane; idx < ns * nj; idx += 32) {
        const int t = idx / nj, j = j0 + idx - t * nj;
        if (len_s[t] > j * kBS && __ldg(p.bt + int64_t(s0 + t) * p.W + j) != __ldg(p.bt + j))
          report(p.err, PKV_DEVERR_PREFIX);
      }
    }
  } else if (warp < mt) {
    // ------------------------------------------------------ consumers
    if (p.planned) pdl_wait();  // the queries may come from the preceding kernel
    MmaRows<HD> rows;
    const int sw = warp * spm;  // this warp's first chunk sequence
    const T* q = static_cast<const T*>(p.q);
    rows.begin(
        [&](int r) -> const T* {
          const int t = sw + r / p.rep;
          return r < spm * p.rep && t < ns
                     ? q + (int64_t(s0 + t) * p.n_heads + head * p.rep + r % p.rep) * HD
                     : nullptr;
        },
        [&](int r) { return min(len_s[sw + r / p.rep], pre_len) - 1; });
    const bool active = sw < ns;
    const uint32_t none[2] = {0u, 0u};
    uint32_t it = 0;
    for (int j = j0; j < j1; ++j, ++it) {
      // every warp takes every tile (the stage is free once all have)
      if (!ring_wait_full(ring, it, p.err)) {
        *ring.abort_flag = 1;
        break;
      }
      const int st = static_cast<int>(it % ring.nstages);
      if (active) {
        // slots past every chunk sequence's reach may hold anything: each
        // reading warp zeroes those V rows itself (the others write the
        // same zeros) before its P V
        const bool fix = vis - j * kBS < kBS;
        if (fix) tile_fix<HD>(ring.k_tile(st), ring.v_tile(st), 0, vis - j * kBS, false, none, none);
        rows.block_sw(ring.k_tile(st), ring.v_tile(st), 0, j * kBS, p.scale_log2);
        if (fix) fence_proxy_async_smem();  // before the stage's next TMA writes
      }
      ring_release(ring, it);
    }
    rows.store_partial([&](int r) -> float* { return part_o + (warp * 16 + r) * HD; },
                       [&](int r) -> float* { return part_ml + (warp * 16 + r) * 2; });
  }
  pdl_launch_dependents();  // after this CTA's wait: the main kernel may be scheduled

  cluster_sync();  // every CTA's partial is in its shared memory
  // CTA `rank` combines pieces [rank E / K, (rank + 1) E / K) of four
  // elements of the chunk's rows x head_dim (row i: query head i % rep of
  // sequence i / rep), every peer's values loaded in one round trip
  constexpr int V4 = HD / 4;
  const int E = ns * p.rep * V4;
  const int e0 = static_cast<int>(int64_t(rank) * E / K);
  const int e1 = static_cast<int>(int64_t(rank + 1) * E / K);
  T* out = static_cast<T*>(p.out);
  const int64_t seed = int64_t(p.prefix_seed_run) * p.B * p.n_heads;
  for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += static_cast<int>(blockDim.x)) {
    const int i = e / V4, d = (e - (e / V4) * V4) * 4;
    const int t = i / p.rep, r = i - (i / p.rep) * p.rep;
    const int prow = (t / spm) * 16 + (t - (t / spm) * spm) * p.rep + r;
    float2 ml[kMaxCluster];
    float4 oc[kMaxCluster];
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {
      ml[c] = make_float2(-INFINITY, 0.f);
      oc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c < K) {
        ml[c] = ld_cluster_f32x2(cluster_map(part_ml + prow * 2, c));
        oc[c] = ld_cluster_f32x4(cluster_map(part_o + prow * HD + d, c));
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c)
      if (ml[c].y > 0.f) M = fmaxf(M, ml[c].x);  // a run that saw no key has no weight
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {
      if (ml[c].y > 0.f) {
        const float w = fast_exp2(ml[c].x - M) * ml[c].y;
        den += w;
        acc = make_float4(fmaf(w, oc[c].x, acc.x), fmaf(w, oc[c].y, acc.y), fmaf(w, oc[c].z, acc.z),
                          fmaf(w, oc[c].w, acc.w));
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const float4 v = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    const int L = len_s[t];
    const int64_t orow = int64_t(s0 + t) * p.n_heads + head * p.rep + r;
    if (L <= pre_len) {
      T* o = out + orow * HD + d;
      o[0] = Elem<T>::from_f(v.x);
      o[1] = Elem<T>::from_f(v.y);
      o[2] = Elem<T>::from_f(v.z);
      o[3] = Elem<T>::from_f(v.w);
      // with append, this sequence's token would belong in a shared block
      // (other sequences read it): not written, reported
      if (p.k_new != nullptr && L > 0 && head == 0 && r == 0 && d == 0) report(p.err, PKV_DEVERR_PREFIX);
    } else {
      *reinterpret_cast<float4*>(p.pre_o + (seed + orow) * HD + d) = v;
      if (d == 0) *reinterpret_cast<float2*>(p.pre_ml + (seed + orow) * 2) = make_float2(M, den);
    }
  }
  cluster_sync();  // the peers have read this CTA's partials
}

// Shared-prefix attention: the first prefix_blocks table entries are the
// same blocks for every sequence (a common prompt), so they are read once
// for a whole chunk of sequences instead of once per sequence.  The prefix
// is cut into prefix_chunks runs of prefix_bpc blocks.  CTA (head group g,
// key run kc; sequences s0 ..): a producer warp streams run kc's blocks
// (row 0's table, the group's heads of each token, as in the main kernel)
// through the shared-memory ring; consumer warp w (KV head g*hg + w) packs
// the query rows of several sequences into one set of rows (sequence
// s0 + r / rep, query head r % rep), all of which see the same keys, and
// leaves a normalised partial per row and run.  The main kernel combines a
// sequence's runs when it starts the sequence's first walked block; a
// sequence wholly inside the prefix gets its output from the main kernel's
// end.  Consumer warp 0 also checks that each sequence's table starts with
// row 0's blocks in this run.
template <typename T, int HD, int MAXR, bool MMA>
__global__ void __launch_bounds__(decode_max_threads<T, HD>())
    decode_prefix_kernel(const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  using Rows = typename RowsOf<T, HD, MAXR, MMA>::type;
  constexpr int R = MMA ? 16 : MAXR;  // rows one warp carries
  const int consumers = p.hg_size;
  const int row_bytes = p.hg_size * HD * p.elem_bytes;
  // tensor-core path: whole-block TMA tiles (as the main kernel); the maps
  // are unused on the CUDA-core path
  Ring ring = MMA ? make_tile_ring(smem, p.nstages, kBS * row_bytes)
                  : make_ring(smem, p.nstages, row_bytes);
  ring_init(ring, consumers);
  pdl_wait();  // inputs written by the preceding kernel
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = p.prefix_chunks;
  const int g = blockIdx.x / K, kc = blockIdx.x - (blockIdx.x / K) * K;
  const int j0 = kc * p.prefix_bpc;
  const int j1 = min(p.prefix_blocks, j0 + p.prefix_bpc);
  const int pre_len = p.prefix_blocks * kBS;
  const int spc = R / p.rep;  // sequences per CTA
  const int s0 = blockIdx.y * spc;
  const int64_t token_pitch = int64_t(p.n_kv) * HD * p.elem_bytes;
  const int64_t head_off = int64_t(g) * p.hg_size * HD * p.elem_bytes;
  if (warp == consumers) {
    // ------------------------------------------------------ producer
    uint32_t it = 0;
    bool ok = true;
    for (int jb = j0; jb < j1 && ok; jb += 32) {
      const int id = jb + lane < j1 ? __ldg(p.bt + jb + lane) : 0;  // row 0's table
      for (int k = 0; k < min(32, j1 - jb); ++k) {
        if (*ring.abort_flag) { ok = false; break; }
        const int blk = __shfl_sync(0xffffffffu, id, k);
        int valid = kBS;
        if (blk < 0 || blk >= p.num_blocks) {
          if (lane == 0) report(p.err, PKV_DEVERR_BLOCK_ID);
          valid = 0;
        }
        const int64_t off = int64_t(valid > 0 ? blk : 0) * kBS * token_pitch + head_off;
        bool filled;
        if constexpr (MMA) {  // a bad id reads the zeros past the pool's end
          filled = lane == 0 ? tile_fill(ring, it, &tm_k, &tm_v,
                                         valid > 0 ? blk * kBS : p.num_blocks * kBS,
                                         g * p.hg_size, p.err)
                             : true;
          filled = __shfl_sync(0xffffffffu, filled, 0);
        } else {
          filled = ring_fill(ring, it, p.k_pool + off, p.v_pool + off, token_pitch, valid, p.err);
        }
        if (!filled) {
          *ring.abort_flag = 1;
          ok = false;
          break;
        }
        ++it;
      }
    }
    if (!ok) ring_drain(ring, it);
    return;
  }
  if (warp > consumers) return;
  // ------------------------------------------------------ consumers
  if (warp == 0) {
    for (int s = 0; s < spc && s0 + s < p.B; ++s) {
      const int b = s0 + s;
      const int vis = min(used_len(p, b), pre_len);
      for (int j = j0 + lane; j < min(j1, (vis + kBS - 1) / kBS); j += 32)
        if (__ldg(p.bt + int64_t(b) * p.W + j) != __ldg(p.bt + j)) report(p.err, PKV_DEVERR_PREFIX);
    }
  }
  Rows rows;
  if constexpr (!MMA) {
    float* scratch = reinterpret_cast<float*>(ring.stages + p.nstages * ring.stage_bytes);
    rows.bind(scratch + warp * RowsOf<T, HD, MAXR, MMA>::kScratch);
  }
  const T* q = static_cast<const T*>(p.q);
  const int head0 = (g * p.hg_size + warp) * p.rep;  // first query head of this KV head
  auto seq_of = [&](int r) { return s0 + r / p.rep; };
  auto active = [&](int r) { return r < spc * p.rep && seq_of(r) < p.B; };
  auto row_of = [&](int r) { return int64_t(seq_of(r)) * p.n_heads + head0 + r % p.rep; };
  rows.begin([&](int r) -> const T* { return active(r) ? q + row_of(r) * HD : nullptr; },
             [&](int r) { return active(r) ? min(used_len(p, seq_of(r)), pre_len) - 1 : -1; });
  const int hoff = warp * HD * p.elem_bytes;
  for (uint32_t it = 0; it < static_cast<uint32_t>(j1 - j0); ++it) {
    if (!ring_wait_full(ring, it, p.err)) {
      *ring.abort_flag = 1;
      return;
    }
    const int st = static_cast<int>(it % ring.nstages);
    if constexpr (MMA)
      rows.block_sw(ring.k_tile(st), ring.v_tile(st), warp, (j0 + static_cast<int>(it)) * kBS,
                    p.scale_log2);
    else
      rows.block(ring.k_tile(st) + hoff, ring.v_tile(st) + hoff, ring.row_stride,
                 (j0 + static_cast<int>(it)) * kBS, p.scale_log2);
    ring_release(ring, it);
  }
  const int64_t part = int64_t(kc) * p.B * p.n_heads;  // run kc's rows
  rows.store_partial(
      [&](int r) -> float* { return active(r) ? p.pre_o + (part + row_of(r)) * HD : nullptr; },
      [&](int r) -> float* { return p.pre_ml + (part + row_of(r)) * 2; });
}

// Combine the prefix runs of every (sequence, query head) row with
// log-sum-exp weights: one thread per 4 output dims of a row.  Rows of a
// sequence that lies wholly inside the prefix (length 0 included) get the
// final output; the others a normalised partial in run slot prefix_chunks,
// which the main kernel continues from.
constexpr int kMaxPrefixRuns = 16;

template <typename T, int HD>
__global__ void __launch_bounds__(256) decode_prefix_combine_kernel(DecodeParams p) {
  pdl_wait();  // the prefix runs
  pdl_launch_dependents();
  constexpr int V = HD / 4;
  const int64_t rows = int64_t(p.B) * p.n_heads;
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= rows * V) return;
  const int64_t row = i / V;
  const int e = static_cast<int>(i - row * V) * 4;
  const int K = p.prefix_chunks;
  // every run's max / sum and partial output are loaded before any is used,
  // so the loads are all in flight at once
  float2 ml[kMaxPrefixRuns];
  float4 o[kMaxPrefixRuns];
#pragma unroll
  for (int k = 0; k < kMaxPrefixRuns; ++k) {
    ml[k] = k < K ? __ldcg(reinterpret_cast<const float2*>(p.pre_ml + (k * rows + row) * 2))
                  : make_float2(-INFINITY, 0.f);
    o[k] = k < K ? __ldcg(reinterpret_cast<const float4*>(p.pre_o + (k * rows + row) * HD + e))
                 : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < kMaxPrefixRuns; ++k)
    if (ml[k].y > 0.f) M = fmaxf(M, ml[k].x);  // a run that saw no key has no weight
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxPrefixRuns; ++k) {
    const float w = ml[k].y > 0.f ? fast_exp2(ml[k].x - M) * ml[k].y : 0.f;
    den += w;
    acc = make_float4(fmaf(w, o[k].x, acc.x), fmaf(w, o[k].y, acc.y), fmaf(w, o[k].z, acc.z),
                      fmaf(w, o[k].w, acc.w));
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  const int b = static_cast<int>(row / p.n_heads);
  if (used_len(p, b) <= p.prefix_blocks * kBS) {
    // with append, this sequence's new token would belong in a shared block
    // (other sequences read it): not written, reported
    if (p.k_new != nullptr && used_len(p, b) > 0 && i % (int64_t(p.n_heads) * V) == 0)
      report(p.err, PKV_DEVERR_PREFIX);
    T* out = static_cast<T*>(p.out) + row * HD + e;
    out[0] = Elem<T>::from_f(acc.x * inv);
    out[1] = Elem<T>::from_f(acc.y * inv);
    out[2] = Elem<T>::from_f(acc.z * inv);
    out[3] = Elem<T>::from_f(acc.w * inv);
  } else {
    *reinterpret_cast<float4*>(p.pre_o + (K * rows + row) * HD + e) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (e == 0) *reinterpret_cast<float2*>(p.pre_ml + (K * rows + row) * 2) = make_float2(M, den);
  }
}

// ------------------------------------------------------------ prefill

struct PrefillParams {
  const void* q;
  void* out;
  const uint8_t* k_pool;
  const uint8_t* v_pool;
  const int32_t* bt;
  const int32_t* seq_lens;
  const int32_t* cu_q;
  int32_t* err;
  int B, n_heads, n_kv, rep, W, num_blocks, max_len, queries_per_warp, consumer_warps, total_q;
  int elem_bytes, nstages;
  float scale_log2;
};

// CTA = (query tile, KV head, sequence).  Consumer warps each own
// `queries_per_warp` consecutive queries x all `rep` heads of the group
// (rows r -> query r / rep, head r % rep); the ring holds the KV head's
// rows of each block up to the tile's last visible key.
template <typename T, int HD, int MAXR, bool MMA>
__global__ void __launch_bounds__(288) prefill_kernel(PrefillParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  using Rows = typename RowsOf<T, HD, MAXR, MMA>::type;
  const int b = blockIdx.z;
  const int g = blockIdx.y;
  const int q0 = __ldg(p.cu_q + b);
  const int c = __ldg(p.cu_q + b + 1) - q0;
  const int tile_q = p.consumer_warps * p.queries_per_warp;
  const int i0 = blockIdx.x * tile_q;
  if (i0 >= c) return;  // whole CTA idle: exit before touching barriers
  if (q0 < 0 || q0 + c > p.total_q) {  // offsets disagree with the query count
    if (threadIdx.x == 0 && blockIdx.x == 0 && g == 0) report(p.err, PKV_DEVERR_LENGTH);
    return;
  }
  int L = __ldg(p.seq_lens + b);
  if (threadIdx.x == 0 && blockIdx.x == 0 && g == 0) {
    if (L < c || L < 0) report(p.err, PKV_DEVERR_LENGTH);
    else if (L > p.max_len) report(p.err, L > p.W * kBS ? PKV_DEVERR_TABLE_WIDTH : PKV_DEVERR_LENGTH);
  }
  if (L > p.max_len) L = p.max_len;
  if (L < c) return;  // inconsistent chunk: reported above, nothing computed
  const int i_end = min(c, i0 + tile_q);
  const int last_needed = L - c + i_end - 1;  // last key any row of the tile sees
  const int n_blocks = last_needed / kBS + 1;

  const int row_bytes = HD * p.elem_bytes;
  Ring ring = make_ring(smem, p.nstages, row_bytes);
  ring_init(ring, p.consumer_warps);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t token_pitch = int64_t(p.n_kv) * HD * p.elem_bytes;

  if (warp == p.consumer_warps) {
    const int32_t* row = p.bt + int64_t(b) * p.W;
    const int64_t head_off = int64_t(g) * HD * p.elem_bytes;
    uint32_t it = 0;
    bool ok = true;
    for (int jj = 0; jj < n_blocks && ok; jj += 32) {
      int id = (jj + lane < n_blocks) ? __ldg(row + jj + lane) : 0;
      const int n_here = min(32, n_blocks - jj);
      for (int k = 0; k < n_here; ++k) {
        if (*ring.abort_flag) { ok = false; break; }
        const int blk = __shfl_sync(0xffffffffu, id, k);
        const int j = jj + k;
        int valid = min(kBS, L - j * kBS);
        if (blk < 0 || blk >= p.num_blocks) {
          if (lane == 0) report(p.err, PKV_DEVERR_BLOCK_ID);
          valid = 0;
        }
        const int64_t off = int64_t(valid > 0 ? blk : 0) * kBS * token_pitch + head_off;
        if (!ring_fill(ring, it, p.k_pool + off, p.v_pool + off, token_pitch, valid, p.err)) {
          *ring.abort_flag = 1;
          ok = false;
          break;
        }
        ++it;
      }
    }
    if (!ok) ring_drain(ring, it);
  } else if (warp < p.consumer_warps) {
    Rows rows;
    if constexpr (!MMA) {
      float* scratch = reinterpret_cast<float*>(ring.stages + p.nstages * ring.stage_bytes);
      rows.bind(scratch + warp * RowsOf<T, HD, MAXR, MMA>::kScratch);
    }
    const T* q = static_cast<const T*>(p.q);
    const int qw = i0 + warp * p.queries_per_warp;  // first query of this warp
    const int nrows = p.queries_per_warp * p.rep;
    auto query_of = [&](int r) { return qw + r / p.rep; };
    rows.begin(
        [&](int r) -> const T* {
          if (r >= nrows || query_of(r) >= c) return nullptr;
          return q + (int64_t(q0 + query_of(r)) * p.n_heads + g * p.rep + r % p.rep) * HD;
        },
        [&](int r) { return L - c + query_of(r); });
    // this warp's last visible key (its rows beyond it are masked anyway)
    const int my_last = L - c + min(c, qw + p.queries_per_warp) - 1;
    for (int k = 0; k < n_blocks; ++k) {
      if (!ring_wait_full(ring, k, p.err)) {
        *ring.abort_flag = 1;
        return;
      }
      if (qw < c && k * kBS <= my_last) {
        const int st = k % ring.nstages;
        rows.block(ring.k_tile(st), ring.v_tile(st), ring.row_stride, k * kBS, p.scale_log2);
      }
      ring_release(ring, k);
    }
    T* out = static_cast<T*>(p.out);
    rows.store([&](int r) -> T* {
      if (r >= nrows || query_of(r) >= c) return nullptr;
      return out + (int64_t(q0 + query_of(r)) * p.n_heads + g * p.rep + r % p.rep) * HD;
    });
  }
}

// ------------------------------------------------------------ host side

inline bool use_mma(const PoolShape& pool) { return pool.dtype == PKV_BF16 && (pool.head_dim == 64 || pool.head_dim == 128); }

// Heads per CTA for decode: the largest divisor of n_kv, at most 8, whose
// rows (heads x head_dim elements) fit in 1 KB.
inline int decode_group(const PoolShape& pool) {
  const int per_head = pool.head_dim * pool.elem_bytes();
  int best = 1;
  for (int h = 1; h <= 8 && h <= pool.n_kv; ++h)
    if (pool.n_kv % h == 0 && h * per_head <= 1024) best = h;
  return best;
}

inline int stages_for(int stage_bytes, int scratch_bytes, int target_bytes) {
  int ns = (target_bytes - kBarrierBytes - scratch_bytes) / stage_bytes;
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns < 2) ns = 2;
  return ns;
}

// Merge of the split groups, one CTA per main-kernel CTA: CTA c merges the
// group main-kernel CTA c recorded, if any.  Launched as a programmatic
// dependent of the main kernel.  J = float4 pieces per thread.
template <typename T, int HD, int J>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(DecodeParams p) {
  constexpr int NB = kMergeMaxVec / J;  // parts per batch
  pdl_launch_dependents();  // the next kernel's prologue may overlap this merge
  // the split group to merge: from the plan of a planned call (written by a
  // finished plan launch, so read before the wait: a CTA with nothing to
  // merge leaves at once), else written by the main kernel
  int4 sp = make_int4(-1, 0, 0, 0);
  if (p.planned) {
    if (!plan_matches(p, p.grid)) return;  // reported by the main kernel
    sp = __ldcg(p.splits + blockIdx.x);
    if (sp.x < 0) return;
  }
  pdl_wait();  // the main kernel's partials (and split entries)
  if (!p.planned) sp = __ldcg(p.splits + blockIdx.x);
  if (sp.x < 0) return;
  const int t = threadIdx.x;
  const int rows = p.hg_size * p.rep;
  const int E = rows * HD;  // elements of one part
  const int grp = sp.y & 0xffff;
  const bool c0_tail = (sp.y & kSplitC0Tail) != 0;
  const bool dense = (sp.y & kSplitDense) != 0;
  const int U = dense ? 0 : __ldcg(p.total_units);  // only sparse grids look at range starts
  const int G = p.grid;
  const int c0 = sp.z & 0xffff, c1 = static_cast<int>(static_cast<uint32_t>(sp.z) >> 16);
  float4 acc[J];
  float M[J], den[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    M[j] = -INFINITY;
    den[j] = 0.f;
  }
  for (int cs = c0; cs <= c1; cs += NB) {
    // the parts of CTAs cs .. cs + NB - 1 (those whose range is not empty);
    // c0 holds the group's first units at the end of its range unless its
    // range starts at the group (then they are its first segment)
    int slot[NB];
    bool has[NB];
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      const int c = cs + k;
      has[k] = c <= c1 && (dense || range_begin(c + 1, U, G) > range_begin(c, U, G));
      slot[k] = (c == c0 && c0_tail) ? 2 * c + 1 : 2 * c;
    }
    float4 o[J][NB];
    float2 ml[J][NB];
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int e = (t + j * kMergeThreads) * 4;
#pragma unroll
      for (int k = 0; k < NB; ++k) {
        if (has[k] && e < E) {
          o[j][k] = __ldcg(reinterpret_cast<const float4*>(p.ws_o + int64_t(slot[k]) * E + e));
          ml[j][k] = __ldcg(reinterpret_cast<const float2*>(
              p.ws_ml + (int64_t(slot[k]) * rows + e / HD) * 2));
        } else {
          o[j][k] = make_float4(0.f, 0.f, 0.f, 0.f);
          ml[j][k] = make_float2(-INFINITY, 0.f);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
#pragma unroll
      for (int k = 0; k < NB; ++k) {
        if (ml[j][k].y > 0.f) {  // a part that saw no key has no weight
          const float Mn = fmaxf(M[j], ml[j][k].x);
          const float a = fast_exp2(M[j] - Mn);
          const float w = fast_exp2(ml[j][k].x - Mn) * ml[j][k].y;
          acc[j] = make_float4(fmaf(w, o[j][k].x, acc[j].x * a), fmaf(w, o[j][k].y, acc[j].y * a),
                               fmaf(w, o[j][k].z, acc[j].z * a), fmaf(w, o[j][k].w, acc[j].w * a));
          den[j] = fmaf(den[j], a, w);
          M[j] = Mn;
        }
      }
    }
  }
  T* out = static_cast<T*>(p.out) + (int64_t(sp.x) * p.n_heads + grp * rows) * HD;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int e = (t + j * kMergeThreads) * 4;
    if (e < E) {
      const float inv = den[j] > 0.f ? 1.f / den[j] : 0.f;
      const float4 v = make_float4(acc[j].x * inv, acc[j].y * inv, acc[j].z * inv, acc[j].w * inv);
      if constexpr (std::is_same<T, float>::value) {
        *reinterpret_cast<float4*>(out + e) = v;
      } else {  // four bf16 in one 8-byte store
        *reinterpret_cast<uint2*>(out + e) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
      }
    }
  }
}

// Merge of the fused shared-prefix call: per (sequence, KV-head group),
// the prompt runs' partials of the group's rows (run slots 0 ..
// prompt_runs - 1) and, for a sequence that goes past the prefix, the
// partial(s) of its own blocks (run slot prompt_runs when one CTA walked
// them all, else the split parts of the CTAs whose ranges hold them), with
// log-sum-exp weights.  One thread per four outputs, kPrefixMergeThreads
// per CTA (a group's rows take one or more CTAs); where the parts are comes
// from the plan, so all loads go out together.  It also reports a
// table that leaves row 0's prefix blocks where the sequence reaches them,
// and with append a sequence whose new token would land in a shared block.
constexpr int kPrefixMergeThreads = 128;

template <typename T, int HD>
__global__ void __launch_bounds__(kPrefixMergeThreads) decode_prefix_merge_kernel(DecodeParams p) {
  pdl_launch_dependents();
  if (p.planned && !plan_matches(p, p.grid)) return;  // reported by the main kernel
  const int rows = p.hg_size * p.rep;
  const int slices = (rows * HD / 4 + kPrefixMergeThreads - 1) / kPrefixMergeThreads;
  const int gs = static_cast<int>(blockIdx.x) / slices;
  const int slice = static_cast<int>(blockIdx.x) - gs * slices;
  const int b = gs / p.n_groups, grp = gs - (gs / p.n_groups) * p.n_groups;
  const int t = threadIdx.x;
  const int L = used_len(p, b);  // lengths and tables are inputs: read before the wait
  const int P = p.prefix_blocks;
  if (grp == 0 && slice == 0) {
    const int reach = min(P, (L + kBS - 1) / kBS);
    for (int j = t; j < reach; j += kPrefixMergeThreads)
      if (__ldg(p.bt + int64_t(b) * p.W + j) != __ldg(p.bt + j)) report(p.err, PKV_DEVERR_PREFIX);
    if (t == 0 && p.k_new != nullptr && L > 0 && L <= P * kBS) report(p.err, PKV_DEVERR_PREFIX);
  }
  const int E = rows * HD;
  const int e = (slice * kPrefixMergeThreads + t) * 4;  // this thread's four outputs
  if (e >= E) return;
  const int64_t row = int64_t(b) * p.n_heads + grp * rows + e / HD;  // output row
  const int d = e % HD;
  const int64_t run_rows = int64_t(p.B) * p.n_heads;
  // where the group's own blocks went: part of a plan kept for this call
  // (read before the wait), else written by the preceding plan launch
  int4 gp = p.planned ? __ldcg(p.gparts + gs) : make_int4(-1, -1, 0, 0);
  int U = p.planned ? __ldcg(p.total_units) : 0;
  pdl_wait();  // the main kernel's partials
  if (!p.planned) {
    gp = __ldcg(p.gparts + gs);
    U = __ldcg(p.total_units);
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float M = -INFINITY, den = 0.f;
  auto fold = [&](float4 o, float2 ml) {
    if (ml.y > 0.f) {  // a part that saw no key has no weight
      const float Mn = fmaxf(M, ml.x);
      const float a = fast_exp2(M - Mn);
      const float w = fast_exp2(ml.x - Mn) * ml.y;
      acc = make_float4(fmaf(w, o.x, acc.x * a), fmaf(w, o.y, acc.y * a), fmaf(w, o.z, acc.z * a),
                        fmaf(w, o.w, acc.w * a));
      den = fmaf(den, a, w);
      M = Mn;
    }
  };
  // every load goes out before the first is used: each prompt run's piece,
  // then the part of the group's own blocks (one CTA walked them all: run
  // slot prompt_runs) or the first kParts split parts (an empty range's
  // slot is skipped)
  float4 po[kMaxPrefixRuns];
  float2 pml[kMaxPrefixRuns];
#pragma unroll
  for (int k = 0; k < kMaxPrefixRuns; ++k) {
    if (k < p.prompt_runs) {
      po[k] = __ldcg(reinterpret_cast<const float4*>(p.pre_o + (k * run_rows + row) * HD + d));
      pml[k] = __ldcg(reinterpret_cast<const float2*>(p.pre_ml + (k * run_rows + row) * 2));
    } else {
      po[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      pml[k] = make_float2(-INFINITY, 0.f);
    }
  }
  constexpr int kParts = 8;
  const int G = p.grid;
  const int pr = e / HD;  // row within the group
  const int c0 = gp.x, c1 = gp.y;
  auto load_parts = [&](int cs, float4 (&o)[kParts], float2 (&ml)[kParts]) {
#pragma unroll
    for (int k = 0; k < kParts; ++k) {
      const int c = cs + k;
      bool has = c0 >= 0 && c <= c1;
      int64_t orow = 0, mrow = 0;
      const float* ob = p.ws_o;
      const float* mb = p.ws_ml;
      if (has && c0 == c1) {  // the whole part, in run slot prompt_runs
        orow = (int64_t(p.prompt_runs) * run_rows + row) * HD + d;
        mrow = (int64_t(p.prompt_runs) * run_rows + row) * 2;
        ob = p.pre_o;
        mb = p.pre_ml;
      } else if (has) {
        has = c == c0 || range_begin(c + 1, U, G) > range_begin(c, U, G);
        const int slot = c == c0 ? gp.z : 2 * c;
        orow = int64_t(slot) * E + e;
        mrow = (int64_t(slot) * rows + pr) * 2;
      }
      o[k] = has ? __ldcg(reinterpret_cast<const float4*>(ob + orow)) : make_float4(0.f, 0.f, 0.f, 0.f);
      ml[k] = has ? __ldcg(reinterpret_cast<const float2*>(mb + mrow)) : make_float2(-INFINITY, 0.f);
    }
  };
  {
    float4 o[kParts];
    float2 ml[kParts];
    load_parts(c0, o, ml);
#pragma unroll
    for (int k = 0; k < kMaxPrefixRuns; ++k) fold(po[k], pml[k]);
#pragma unroll
    for (int k = 0; k < kParts; ++k) fold(o[k], ml[k]);
  }
  for (int cs = c0 + kParts; c0 >= 0 && cs <= c1; cs += kParts) {  // long split groups
    float4 o[kParts];
    float2 ml[kParts];
    load_parts(cs, o, ml);
#pragma unroll
    for (int k = 0; k < kParts; ++k) fold(o[k], ml[k]);
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  const float4 v = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  T* out = static_cast<T*>(p.out) + row * HD + d;
  if constexpr (std::is_same<T, float>::value) {
    *reinterpret_cast<float4*>(out) = v;
  } else {  // four bf16 in one 8-byte store
    *reinterpret_cast<uint2*>(out) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  }
}

// Launch the merge with the fewest float4 pieces per thread that covers a
// part of rows x HD elements (more parts per batch for small parts).
template <typename T, int HD>
cudaError_t launch_merge(cudaLaunchConfig_t cfg, const DecodeParams& p) {
  const int pieces = (p.hg_size * p.rep * HD / 4 + kMergeThreads - 1) / kMergeThreads;
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  if (pieces <= 1) return cudaLaunchKernelEx(&cfg, decode_merge_kernel<T, HD, 1>, p);
  if (pieces <= 2) return cudaLaunchKernelEx(&cfg, decode_merge_kernel<T, HD, 2>, p);
  if (pieces <= 4) return cudaLaunchKernelEx(&cfg, decode_merge_kernel<T, HD, 4>, p);
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel<T, HD, 8>, p);
}

// Runs the shared prefix is cut into for the prefix kernel: enough CTAs
// (head groups x sequence chunks x runs) to fill about two per SM, at most
// kMaxPrefixRuns runs and at most 1,024 run-rows per query head (which
// bounds the partials' workspace), at least one block per run.  *bpc =
// blocks per run.  One more slot holds the combined partials.
inline int max_prefix_runs(int num_seqs, int prefix_blocks) {
  const int k = 1024 / (num_seqs > 0 ? num_seqs : 1);
  return std::max(1, std::min({kMaxPrefixRuns, prefix_blocks, std::max(1, k)}));
}
inline int prefix_slots(int runs) { return runs > 0 ? runs + 1 : 0; }

inline int prefix_runs(int num_seqs, int n_groups, int seqs_per_cta, int prefix_blocks, int* bpc) {
  const int base = n_groups * ((num_seqs + seqs_per_cta - 1) / seqs_per_cta);
  int k = (2 * sm_count() + base - 1) / base;
  k = std::max(1, std::min(k, max_prefix_runs(num_seqs, prefix_blocks)));
  *bpc = (prefix_blocks + k - 1) / k;
  return (prefix_blocks + *bpc - 1) / *bpc;
}

// Decode workspace layout: cu_units [B+1] | starts [G] | splits [G] |
// total units | partial max/sum [2G][rows][2] | partial outputs
// [2G][rows][HD] | with a shared prefix: prefix partial outputs
// [runs][B][n_heads][HD] and max/sum [runs][B][n_heads][2]; each region
// 256-byte aligned.
struct DecodeWs {
  size_t cu, starts, splits, total_units, ml, o, pre_o, pre_ml, gparts, total;
  // prefix_heads: runs x n_heads with a shared prefix (its partials
  // follow), else 0; prefix_groups: KV-head groups per sequence with a
  // shared prefix (where each group's parts are, for the prefix merge)
  DecodeWs(int num_seqs, size_t G, size_t rows_per_group, int head_dim, int prefix_heads = 0,
           int prefix_groups = 0) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    cu = 0;
    starts = up(size_t(num_seqs + 1) * 4);
    splits = starts + up(G * 16);
    total_units = splits + up(G * 16);
    ml = total_units + 256;
    o = ml + up(2 * G * rows_per_group * 2 * 4);
    pre_o = o + up(2 * G * rows_per_group * size_t(head_dim) * 4);
    pre_ml = pre_o + up(size_t(num_seqs) * prefix_heads * head_dim * 4);
    gparts = pre_ml + up(size_t(num_seqs) * prefix_heads * 2 * 4);
    total = gparts + size_t(num_seqs) * prefix_groups * 16;
  }
};

template <typename T, int HD, int MAXR, bool MMA>
struct DecodeLaunch {
  static constexpr int kRowsPerWarp = MMA ? 16 : MAXR;  // query rows one consumer warp carries
  static size_t scratch_bytes(int warps) {
    return MMA ? 0 : size_t(warps) * RowsOf<T, HD, MAXR, MMA>::kScratch * sizeof(float);
  }
  // Bytes of one ring stage: padded rows (CUDA-core path, and the shared
  // prefix kernel, which shares the launch shape) or TMA tiles.
  static int stage_bytes(int hg, int elem_bytes, bool tiles) {
    const int row_bytes = hg * HD * elem_bytes;
    return tiles ? 2 * kBS * row_bytes : 2 * kBS * (row_bytes + 16);
  }
  // Ring depth: the tile path keeps five 32 KB stages per CTA at one CTA
  // per SM (160 KB in flight per SM; measured against 3, 4 and 6 stages on
  // the 1B, 7B and 70B shapes, five was best or tied on each, and a deeper
  // ring also holds more of a planned call's early loads); the CUDA-core
  // path keeps about 110 KB.
  static size_t smem_bytes(int hg, int elem_bytes, int* nstages) {
    const int padded = stage_bytes(hg, elem_bytes, false);
    const size_t scratch = scratch_bytes(hg);
    *nstages = stages_for(padded, static_cast<int>(scratch), (MMA ? 180 : 110) * 1024);
    return smem_for(hg, elem_bytes, *nstages);
  }
  // Shared memory of a ring of `nstages` stages (plus the CUDA-core rows'
  // scratch; the tile ring needs 1024 bytes of alignment slack after the
  // barriers).
  static size_t smem_for(int hg, int elem_bytes, int nstages) {
    size_t bytes = kBarrierBytes + size_t(nstages) * stage_bytes(hg, elem_bytes, false) +
                   scratch_bytes(hg);
    if (MMA)
      bytes = std::max(bytes, kBarrierBytes + 1024 + size_t(nstages) * stage_bytes(hg, elem_bytes, true));
    return bytes;
  }
  static auto main_kernel() {
    if constexpr (MMA)
      return decode_kernel<T, HD>;
    else
      return decode_rows_kernel<T, HD, MAXR>;
  }
  static auto cluster_kernel() {
    if constexpr (MMA)
      return decode_cluster_kernel<T, HD>;
    else
      return decode_cluster_rows_kernel<T, HD, MAXR>;
  }
  // the shared-prefix cluster kernel (tile path only; the CUDA-core path
  // never selects it)
  static auto cluster_prefix_kernel() {
    if constexpr (MMA)
      return decode_cluster_prefix_kernel<T, HD>;
    else
      return decode_cluster_rows_kernel<T, HD, MAXR>;  // unused
  }
  // Shape of the cluster path for a call (C = 0: the stream-K path).  Only
  // calls that leave the grid to the library (max_ctas 0) qualify.
  //  * No shared prefix: one sequence per cluster, when the longest
  //    sequence is at most 64 blocks and the clusters fit in two waves of
  //    the stream-K grid: batches too small to keep the machine streaming,
  //    whose time is latency (a block's round trip, the merge launch)
  //    rather than bytes.  About 4 blocks per CTA, at most 8 CTAs.
  //  * A shared prefix (tile path): the prefix is read once per chunk of
  //    spc sequences; spc (up to a tile's 16 rows) and C are chosen for the
  //    fewest blocks on the busiest CTA times the waves of clusters.
  // The ring holds a CTA's blocks (2 to nstages_max stages).
  struct ClusterShape {
    int C = 0, spc = 1, stages = 0;
    size_t smem = 0;
  };
  // The cluster kernel is opted into nearly the most dynamic shared memory
  // a CTA may have (227 KB, less 1 KB for its static shared variables), once
  // per device; each launch uses what its shape needs.
  static constexpr int kClusterSmemMax = 226 * 1024;
  static cudaError_t cluster_kernel_setup(bool prefix, int threads) {
    static KernelSetup setup, prefix_setup;
    return prefix ? kernel_setup(prefix_setup, cluster_prefix_kernel(), kClusterSmemMax, threads,
                                 nullptr)
                  : kernel_setup(setup, cluster_kernel(), kClusterSmemMax, threads, nullptr);
  }
  static ClusterShape cluster_shape(const AttnArgs& a, int hg, int wave, int nstages_max) {
    ClusterShape best;
    if (a.max_ctas != 0) return best;
    const int P = a.prefix_blocks;
    if (P > 0 && !MMA) return best;
    const int nmax = (min(a.max_seq_len, a.max_blocks_per_seq * kBS) + kBS - 1) / kBS;
    const int rep = a.n_heads / a.pool.n_kv;
    const int groups = a.pool.n_kv / hg;
    const int eb = a.pool.elem_bytes();
    const bool staged = MMA && a.k_new != nullptr && P > 0;  // the prefix kernel stages step rows
    const int threads = (hg + 1) * 32;
    auto shape_for = [&](int C, int spc, int per) {
      ClusterShape c;
      c.C = C;
      c.spc = spc;
      c.stages = std::max(2, std::min(nstages_max, per));
      for (;; --c.stages) {
        c.smem = (smem_for(hg, eb, c.stages) + 15) / 16 * 16 +
                 cluster_extra_bytes(hg, rep, HD, eb, spc, staged);
        if (c.smem <= 220 * 1024 || c.stages == 2) break;
      }
      return c;
    };
    if (P == 0) {
      if (nmax > 8 * kMaxCluster) return best;
      const int C = std::max(1, std::min(kMaxCluster, (nmax + 3) / 4));
      const int64_t ctas = int64_t(a.num_seqs) * groups * C;
      if (ctas > 2 * int64_t(wave)) return best;
      return shape_for(C, 1, (nmax + C - 1) / C);
    }
    // shared prefix: every (spc, C), costed as the busiest CTA's blocks
    // times the waves of clusters the device holds at once
    static ClusterOccupancy occ;
    if (cluster_kernel_setup(true, threads) != cudaSuccess) {
      cudaGetLastError();
      return best;
    }
    int64_t best_cost = -1;
    for (int spc = 1; spc <= std::min(kRowsPerWarp / rep, kMaxChunk); ++spc) {
      const int64_t clusters = int64_t((a.num_seqs + spc - 1) / spc) * groups;
      const int list = P + spc * std::max(0, nmax - P);
      for (int C = 1; C <= kMaxCluster; ++C) {
        const int per = (list + C - 1) / C;
        const ClusterShape c = shape_for(C, spc, per);
        if (c.smem > kClusterSmemMax) continue;
        const int at_once = max_active_clusters(occ, cluster_prefix_kernel(), C,
                                                static_cast<int>(c.smem), threads);
        if (at_once <= 0) continue;
        const int64_t cost = (clusters + at_once - 1) / at_once * per;
        if (best_cost < 0 || cost < best_cost) {
          best_cost = cost;
          best = c;
        }
      }
    }
    return best;
  }
  // Shape of the wide shared-prefix pass (K = 0: not used): K CTAs per
  // cluster (runs of the prefix), mt consumer warps of 16 rows, `seqs`
  // sequences per chunk, `chunks` chunks, a ring of `stages` one-head tiles.
  // Chosen (tile path, grid left to the library) when the prefix bytes it
  // saves against the cluster path (which reads the prefix once per chunk
  // of at most a tile's rows) exceed about what its two extra launches and
  // its partials cost, 16 MB of reads; K for the fewest prefix blocks per
  // CTA times the waves of clusters the device holds at once.
  struct WideShape {
    int K = 0, mt = 0, seqs = 0, chunks = 0, stages = 0;
    size_t part_off = 0, smem = 0;
  };
  static constexpr int kWideSmemMax = 200 * 1024;
  static cudaError_t wide_setup(int threads) {
    static KernelSetup setup;
    return kernel_setup(setup, decode_prefix_wide_kernel<T, HD>, kWideSmemMax, threads, nullptr);
  }
  static WideShape wide_shape(const AttnArgs& a, const ClusterShape& cs) {
    WideShape w;
    if constexpr (MMA) {
      const int P = a.prefix_blocks;
      if (a.max_ctas != 0 || P == 0 || a.num_seqs <= 0) return w;
      const int rep = a.n_heads / a.pool.n_kv;
      const int spm = kMaxRep / rep;
      const int mt_max = std::min(wide_max_warps<HD>(), (a.num_seqs + spm - 1) / spm);
      const int64_t prefix_bytes = int64_t(P) * kBS * a.pool.n_kv * HD * 2 * 2;
      const int64_t cluster_reads =
          (a.num_seqs + (cs.C > 0 ? cs.spc : spm) - 1) / (cs.C > 0 ? cs.spc : spm);
      const int64_t min_reads = (a.num_seqs + mt_max * spm - 1) / (mt_max * spm);
      if ((cluster_reads - min_reads) * prefix_bytes < (int64_t(16) << 20)) return w;
      static ClusterOccupancy occ;
      const int sms = sm_count();
      double best = -1.0;
      // candidates: 16-row tiles per CTA (mt_max, half, quarter) x runs;
      // cost = waves x blocks per CTA x a block's time on one SM for mt
      // warps (measured: 4, 2 and 1 warps per scheduler take about 218,
      // 301 and 450 cycles per warp-block) x CTAs sharing an SM
      for (int mt = mt_max; mt >= 1; mt = mt > 1 ? std::max(1, mt / 2) : 0) {
        const int threads = (mt + 1) * 32;
        if (wide_setup(threads) != cudaSuccess) {
          cudaGetLastError();
          return WideShape{};
        }
        const int seqs = mt * spm;
        const int chunks = (a.num_seqs + seqs - 1) / seqs;
        const int per_sched = (mt + 3) / 4;
        const double warp_block = per_sched >= 4 ? 218.0 : per_sched == 3 ? 250.0 : per_sched == 2 ? 301.0 : 450.0;
        const double cta_block = warp_block * per_sched;
        const int64_t clusters = int64_t(chunks) * a.pool.n_kv;
        for (int K = 1; K <= std::min(kMaxCluster, P); ++K) {
          const int per = (P + K - 1) / K;
          const int stages = std::max(2, std::min(16, per));
          const size_t part_off =
              (kBarrierBytes + 1024 + size_t(stages) * 2 * kBS * HD * 2 + 15) / 16 * 16;
          const size_t smem = part_off + size_t(mt) * 16 * (HD + 2) * 4;
          if (smem > size_t(kWideSmemMax)) continue;
          const int at_once = max_active_clusters(occ, decode_prefix_wide_kernel<T, HD>, K,
                                                  static_cast<int>(smem), threads);
          if (at_once <= 0) continue;
          const int64_t waves = (clusters + at_once - 1) / at_once;
          const int64_t in_wave = std::min<int64_t>(clusters, at_once) * K;
          const double cost = double(waves) * per * cta_block *
                              std::max(1.0, double(in_wave) / std::max(1, sms));
          if (best < 0 || cost < best) {
            best = cost;
            w.K = K, w.mt = mt, w.seqs = seqs, w.chunks = chunks, w.stages = stages;
            w.part_off = part_off, w.smem = smem;
          }
        }
        if (mt == 1) break;
      }
    }
    return w;
  }
  // Shape of the fused shared-prefix call (R = 0: not used): the tile path
  // with the grid left to the library, when the prefix bytes it saves
  // against the cluster path exceed 16 MB of reads (a function of the
  // sizes only, so that a plan and the calls using it agree).  A chunk is the rows of
  // one tile per consumer warp (hg * 16 / rep sequences); the prefix is cut
  // into R runs of bpr blocks so that every (chunk, KV head, run) item has
  // its own CTA, a run fits in the ring beside at least one stage of the
  // blocks after the prefix (hg one-head blocks per stage) and R run slots
  // plus one fit in the workspace's prefix partials (max_runs + 1 slots).
  struct FusedShape {
    int R = 0, bpr = 0, seqs = 0, chunks = 0, pw = 0;
    size_t smem = 0;
  };
  static FusedShape fused_shape(const AttnArgs& a, int hg, int G, int nstages, int max_runs) {
    FusedShape f;
    const int P = a.prefix_blocks;
    if (!MMA || a.max_ctas != 0 || P == 0 || a.num_seqs <= 0) return f;
    const int rep = a.n_heads / a.pool.n_kv;
    const int spm = kMaxRep / rep;
    const int pw = fused_prompt_warps(hg, fused_max_warps<HD>());
    if (pw < 1) return f;
    const int seqs = pw * spm;
    const int chunks = (a.num_seqs + seqs - 1) / seqs;
    // (the cluster path reads the prefix once per chunk of at most a tile's
    // spm sequences; the plan and every call using it decide alike)
    const int64_t prefix_bytes = int64_t(P) * kBS * a.pool.n_kv * HD * 2 * 2;
    const int64_t cluster_reads = (a.num_seqs + spm - 1) / spm;
    if ((cluster_reads - chunks) * prefix_bytes < (int64_t(16) << 20)) return f;
    const int64_t per_run = int64_t(a.pool.n_kv) * chunks;
    int R = static_cast<int>(std::min<int64_t>({int64_t(max_runs), G / per_run, int64_t(P)}));
    if (R < 1) return f;
    const int bpr = (P + R - 1) / R;
    R = (P + bpr - 1) / bpr;
    // the ring, then the run's K and V tiles (one head each)
    const size_t smem = smem_for(hg, a.pool.elem_bytes(), nstages) + size_t(bpr) * 2 * kBS * HD * 2;
    if (bpr > 32 || smem > size_t(kClusterSmemMax)) return f;
    f.R = R, f.bpr = bpr, f.seqs = seqs, f.chunks = chunks, f.smem = smem, f.pw = pw;
    return f;
  }
  // Persistent grid: every SM filled with as many CTAs as fit, capped by
  // max_ctas; *wave (optional) = the uncapped full wave.
  static cudaError_t grid(const AttnArgs& a, int hg, int* G, size_t* smem, int* nstages,
                          int* wave = nullptr) {
    *smem = smem_bytes(hg, a.pool.elem_bytes(), nstages);
    static KernelSetup setup;
    int per_sm = 0;
    const cudaError_t e = kernel_setup(setup, main_kernel(),
                                       static_cast<int>(*smem), (hg + 1) * 32, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    *G = sm_count() * per_sm;
    if (wave) *wave = *G;
    if (a.max_ctas > 0 && a.max_ctas < *G) *G = a.max_ctas;
    // no more CTAs than the batch can have units (a small batch would
    // otherwise leave most ranges empty and its split groups spread thin)
    const int64_t max_units = int64_t(a.num_seqs) * (a.pool.n_kv / hg) *
                              ((min(a.max_seq_len, a.max_blocks_per_seq * kBS) + kBS - 1) / kBS);
    if (max_units < *G) *G = static_cast<int>(std::max<int64_t>(1, max_units));
    return cudaSuccess;
  }
  static cudaError_t run(const AttnArgs& a, int hg, cudaStream_t stream) {
    const PoolShape& pool = a.pool;
    DecodeParams p{};
    p.q = a.q;
    p.out = a.out;
    p.k_pool = static_cast<const uint8_t*>(a.k_pool);
    p.v_pool = static_cast<const uint8_t*>(a.v_pool);
    p.bt = a.block_tables;
    p.seq_lens = a.seq_lens;
    p.k_new = static_cast<const uint8_t*>(a.k_new);
    p.v_new = static_cast<const uint8_t*>(a.v_new);
    p.err = a.err;
    p.B = a.num_seqs;
    p.n_heads = a.n_heads;
    p.n_kv = pool.n_kv;
    p.rep = a.n_heads / pool.n_kv;
    p.hg_size = hg;
    p.n_groups = pool.n_kv / hg;
    p.W = a.max_blocks_per_seq;
    p.num_blocks = pool.num_blocks;
    p.max_len = min(a.max_seq_len, a.max_blocks_per_seq * kBS);
    p.max_seq_len = a.max_seq_len;
    p.head_dim = HD;
    p.elem_bytes = pool.elem_bytes();
    p.scale_log2 = a.scale * kLog2e;
    int G = 0, wave = 0;
    size_t smem = 0;
    cudaError_t e = grid(a, hg, &G, &smem, &p.nstages, &wave);
    if (e != cudaSuccess) return e;
    if (G > 65535) return cudaErrorInvalidValue;  // split entries pack CTA indices in 16 bits
    p.grid = G;
    p.prefix_blocks = a.prefix_blocks;
    p.prefix_chunks = 0;
    if (p.prefix_blocks > 0)
      p.prefix_chunks = prefix_runs(p.B, p.n_groups, kRowsPerWarp / p.rep, p.prefix_blocks,
                                    &p.prefix_bpc);
    p.prefix_seed_run = p.prefix_chunks;
    const DecodeWs L(a.num_seqs, G, size_t(hg) * p.rep, HD,
                     prefix_slots(p.prefix_chunks) * a.n_heads, p.prefix_blocks > 0 ? p.n_groups : 0);
    if (L.total > a.workspace_bytes) return cudaErrorInvalidValue;
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    p.cu_units = reinterpret_cast<int32_t*>(ws + L.cu);
    p.starts = reinterpret_cast<int4*>(ws + L.starts);
    p.splits = reinterpret_cast<int4*>(ws + L.splits);
    p.total_units = reinterpret_cast<int32_t*>(ws + L.total_units);
    p.ws_ml = reinterpret_cast<float*>(ws + L.ml);
    p.ws_o = reinterpret_cast<float*>(ws + L.o);
    p.pre_o = reinterpret_cast<float*>(ws + L.pre_o);
    p.pre_ml = reinterpret_cast<float*>(ws + L.pre_ml);
    p.gparts = reinterpret_cast<int4*>(ws + L.gparts);
    // the launch shape (a plan made for later calls records what the fused
    // shared-prefix merge needs)
    const ClusterShape cs = cluster_shape(a, hg, wave, p.nstages);
    const FusedShape fused = p.prefix_blocks > 0
                                 ? fused_shape(a, hg, G, p.nstages, p.prefix_chunks)
                                 : FusedShape{};
    if (fused.R > 0) {
      p.prompt_runs = fused.R;
      p.prompt_bpr = fused.bpr;
      p.prompt_seqs = fused.seqs;
      p.prompt_items = fused.R * pool.n_kv * fused.chunks;
      p.wide_mt = fused.pw;
    }
    if (a.decode_plan == kPlanOnly) {  // the plan alone, kept in the workspace
      p.plan_only = 1;
      p.out = nullptr;
      decode_plan_kernel<T, HD><<<1, 1024, 0, stream>>>(p);
      return cudaGetLastError();
    }
    // tensor-core path: the pools as 4-D tensors (64 dims, slot, 64-dim half,
    // KV head) read in boxes of one block's 16 slots x the group's heads
    CUtensorMap tm_k{}, tm_v{};
    if constexpr (MMA) {
      const uint64_t slots = uint64_t(pool.num_blocks) * kBS;
      if (slots >= (uint64_t(1) << 31)) return cudaErrorInvalidValue;  // 32-bit box coordinates
      const uint64_t dims[4] = {64, slots, HD / 64, uint64_t(pool.n_kv)};
      const uint64_t strides[3] = {uint64_t(pool.n_kv) * HD * 2, 128, uint64_t(HD) * 2};
      const uint32_t box[4] = {64, kBS, HD / 64, static_cast<uint32_t>(hg)};
      if (!encode_bf16_sw128(&tm_k, a.k_pool, 4, dims, strides, box) ||
          !encode_bf16_sw128(&tm_v, a.v_pool, 4, dims, strides, box))
        return cudaErrorInvalidValue;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    p.planned = a.decode_plan == kPlanned;
    if (fused.R > 0) {
      // a long prefix shared by many sequences: one launch attends both the
      // prefix (runs x chunks x KV heads, one per CTA) and each sequence's
      // own blocks (stream-K), the prefix merge combines them
      if constexpr (MMA) {
        p.plan_in_kernel = 0;
        if (!p.planned) {
          decode_plan_kernel<T, HD><<<1, 1024, 0, stream>>>(p);
          if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        static KernelSetup fused_setup;
        e = kernel_setup(fused_setup, decode_fused_prefix_kernel<T, HD>, static_cast<int>(fused.smem),
                         (hg + 1 + fused.pw) * 32, nullptr);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t fcfg = {};
        fcfg.gridDim = dim3(G);
        fcfg.blockDim = dim3((hg + 1 + fused.pw) * 32);
        fcfg.dynamicSmemBytes = fused.smem;
        fcfg.stream = stream;
        fcfg.attrs = attr;
        fcfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&fcfg, decode_fused_prefix_kernel<T, HD>, tm_k, tm_v, p);
        if (e != cudaSuccess) return e;
        const int slices = (hg * p.rep * HD / 4 + kPrefixMergeThreads - 1) / kPrefixMergeThreads;
        fcfg.gridDim = dim3(static_cast<unsigned>(int64_t(p.B) * p.n_groups * slices));
        fcfg.blockDim = dim3(kPrefixMergeThreads);
        fcfg.dynamicSmemBytes = 0;
        e = cudaLaunchKernelEx(&fcfg, decode_prefix_merge_kernel<T, HD>, p);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
      }
    }
    const WideShape wide = p.prefix_blocks > 0 ? wide_shape(a, cs) : WideShape{};
    if (cs.C > 0 && wide.K == 0) {
      // latency-bound batch, or a shared prefix: one cluster of C CTAs per
      // (chunk of spc sequences, head group), partials combined in
      // distributed shared memory
      const int C = cs.C;
      p.cluster = C;
      p.cluster_seqs = cs.spc;
      p.nstages = cs.stages;
      p.part_off = static_cast<int>((smem_for(hg, p.elem_bytes, cs.stages) + 15) / 16 * 16);
      e = cluster_kernel_setup(p.prefix_blocks > 0, (hg + 1) * 32);
      if (e != cudaSuccess) return e;
      cudaLaunchAttribute cattr[2];
      cattr[0] = attr[0];
      cattr[1].id = cudaLaunchAttributeClusterDimension;
      cattr[1].val.clusterDim.x = static_cast<unsigned>(C);
      cattr[1].val.clusterDim.y = 1;
      cattr[1].val.clusterDim.z = 1;
      cudaLaunchConfig_t ccfg = {};
      const int64_t chunks = (int64_t(p.B) + cs.spc - 1) / cs.spc;
      ccfg.gridDim = dim3(static_cast<unsigned>(chunks * p.n_groups * C));
      ccfg.blockDim = dim3((hg + 1) * 32);
      ccfg.dynamicSmemBytes = cs.smem;
      ccfg.stream = stream;
      ccfg.attrs = cattr;
      ccfg.numAttrs = 2;
      if constexpr (MMA) {
        if (p.prefix_blocks > 0)
          e = cudaLaunchKernelEx(&ccfg, decode_cluster_prefix_kernel<T, HD>, tm_k, tm_v, p);
        else
          e = cudaLaunchKernelEx(&ccfg, decode_cluster_kernel<T, HD>, tm_k, tm_v, p);
      } else {
        e = cudaLaunchKernelEx(&ccfg, decode_cluster_rows_kernel<T, HD, MAXR>, p);
      }
      if (e != cudaSuccess) return e;
      return cudaGetLastError();
    }
    if (wide.K > 0) {
      // a long prefix shared by many sequences: one pass per KV head and
      // chunk of up to 16 tiles of rows, its runs combined in the cluster;
      // the seed is run slot 0
      if constexpr (MMA) {
        DecodeParams pw = p;
        pw.cluster = wide.K;
        pw.cluster_seqs = wide.seqs;
        pw.wide_mt = wide.mt;
        pw.wide_evict = wide.chunks == 1;
        pw.nstages = wide.stages;
        pw.part_off = static_cast<int>(wide.part_off);
        pw.prefix_seed_run = 0;
        CUtensorMap wk{}, wv{};
        const uint64_t dims[4] = {64, uint64_t(pool.num_blocks) * kBS, HD / 64, uint64_t(pool.n_kv)};
        const uint64_t strides[3] = {uint64_t(pool.n_kv) * HD * 2, 128, uint64_t(HD) * 2};
        const uint32_t box[4] = {64, kBS, HD / 64, 1};
        if (!encode_bf16_sw128(&wk, a.k_pool, 4, dims, strides, box) ||
            !encode_bf16_sw128(&wv, a.v_pool, 4, dims, strides, box))
          return cudaErrorInvalidValue;
        cudaLaunchAttribute wattr[2];
        wattr[0] = attr[0];
        wattr[1].id = cudaLaunchAttributeClusterDimension;
        wattr[1].val.clusterDim.x = static_cast<unsigned>(wide.K);
        wattr[1].val.clusterDim.y = 1;
        wattr[1].val.clusterDim.z = 1;
        cudaLaunchConfig_t wcfg = {};
        wcfg.gridDim = dim3(static_cast<unsigned>(int64_t(wide.chunks) * pool.n_kv * wide.K));
        wcfg.blockDim = dim3((wide.mt + 1) * 32);
        wcfg.dynamicSmemBytes = wide.smem;
        wcfg.stream = stream;
        wcfg.attrs = wattr;
        wcfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&wcfg, decode_prefix_wide_kernel<T, HD>, wk, wv, pw);
        if (e != cudaSuccess) return e;
        p.prefix_seed_run = 0;
      }
    } else if (p.prefix_blocks > 0) {
      // the shared prefix: runs of its blocks, each read once per head group
      // for a chunk of sequences (same ring and shared memory as below)
      static KernelSetup prefix_setup;
      e = kernel_setup(prefix_setup, decode_prefix_kernel<T, HD, MAXR, MMA>,
                       static_cast<int>(smem), (hg + 1) * 32, nullptr);
      if (e != cudaSuccess) return e;
      const int spc = kRowsPerWarp / p.rep;
      cudaLaunchConfig_t pcfg = {};
      pcfg.gridDim = dim3(p.n_groups * p.prefix_chunks, (p.B + spc - 1) / spc);
      pcfg.blockDim = dim3((hg + 1) * 32);
      pcfg.dynamicSmemBytes = smem;
      pcfg.stream = stream;
      pcfg.attrs = attr;
      pcfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&pcfg, decode_prefix_kernel<T, HD, MAXR, MMA>, tm_k, tm_v, p);
      if (e != cudaSuccess) return e;
      const int64_t threads = int64_t(p.B) * p.n_heads * (HD / 4);
      pcfg.gridDim = dim3(static_cast<unsigned>((threads + 255) / 256));
      pcfg.blockDim = dim3(256);
      pcfg.dynamicSmemBytes = 0;
      e = cudaLaunchKernelEx(&pcfg, decode_prefix_combine_kernel<T, HD>, p);
      if (e != cudaSuccess) return e;
    }
    // small batches: every CTA scans the lengths in its ring stages (unless
    // the plan is already in the workspace)
    const size_t ring_bytes = size_t(p.nstages) * stage_bytes(hg, p.elem_bytes, MMA);
    p.plan_in_kernel = !p.planned && a.num_seqs <= kKernelPlanSeqs &&
                       size_t(a.num_seqs + 1 + 32) * 4 <= ring_bytes;
    if (!p.plan_in_kernel && !p.planned) {
      decode_plan_kernel<T, HD><<<1, 1024, 0, stream>>>(p);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // the main kernel may start while the preceding kernel runs: it waits
    // for that kernel's results (griddepcontrol.wait) after its prologue
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3((hg + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if constexpr (MMA)
      e = cudaLaunchKernelEx(&cfg, decode_kernel<T, HD>, tm_k, tm_v, p);
    else
      e = cudaLaunchKernelEx(&cfg, decode_rows_kernel<T, HD, MAXR>, p);
    if (e != cudaSuccess) return e;
    // split groups: one small CTA per main-kernel boundary, most exit at once
    cfg.gridDim = dim3(G);
    e = launch_merge<T, HD>(cfg, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
};

// Exact workspace of the grid DecodeLaunch::run would launch for these
// arguments.
template <typename T, int HD, int MAXR, bool MMA>
size_t decode_exact_workspace(const AttnArgs& a, int hg) {
  int G = 0, nstages = 0;
  size_t smem = 0;
  if (DecodeLaunch<T, HD, MAXR, MMA>::grid(a, hg, &G, &smem, &nstages) != cudaSuccess) return 0;
  int runs = 0, bpc = 0;
  if (a.prefix_blocks > 0)
    runs = prefix_runs(a.num_seqs, a.pool.n_kv / hg,
                       DecodeLaunch<T, HD, MAXR, MMA>::kRowsPerWarp / (a.n_heads / a.pool.n_kv),
                       a.prefix_blocks, &bpc);
  return DecodeWs(a.num_seqs, G, size_t(hg) * (a.n_heads / a.pool.n_kv), HD,
                  prefix_slots(runs) * a.n_heads, a.prefix_blocks > 0 ? a.pool.n_kv / hg : 0)
      .total;
}

template <typename T, int HD, int MAXR, bool MMA>
struct PrefillLaunch {
  static cudaError_t run(const AttnArgs& a, cudaStream_t stream) {
    const PoolShape& pool = a.pool;
    PrefillParams p{};
    p.q = a.q;
    p.out = a.out;
    p.k_pool = static_cast<const uint8_t*>(a.k_pool);
    p.v_pool = static_cast<const uint8_t*>(a.v_pool);
    p.bt = a.block_tables;
    p.seq_lens = a.seq_lens;
    p.cu_q = a.cu_q_lens;
    p.err = a.err;
    p.B = a.num_seqs;
    p.n_heads = a.n_heads;
    p.n_kv = pool.n_kv;
    p.rep = a.n_heads / pool.n_kv;
    p.W = a.max_blocks_per_seq;
    p.num_blocks = pool.num_blocks;
    p.max_len = min(a.max_seq_len, a.max_blocks_per_seq * kBS);
    p.total_q = a.total_q;
    p.elem_bytes = pool.elem_bytes();
    p.scale_log2 = a.scale * kLog2e;
    p.consumer_warps = 8;
    p.queries_per_warp = MMA ? (kMaxRep / p.rep) : 1;
    const int row_bytes = HD * p.elem_bytes;
    const int stage_bytes = 2 * kBS * (row_bytes + 16);
    const size_t scratch =
        MMA ? 0 : size_t(p.consumer_warps) * RowsOf<T, HD, MAXR, MMA>::kScratch * sizeof(float);
    p.nstages = stages_for(stage_bytes, static_cast<int>(scratch), 100 * 1024);
    const size_t smem = kBarrierBytes + size_t(p.nstages) * stage_bytes + scratch;
    auto kern = prefill_kernel<T, HD, MAXR, MMA>;
    static KernelSetup setup;
    cudaError_t e = kernel_setup(setup, kern, static_cast<int>(smem),
                                 (p.consumer_warps + 1) * 32, nullptr);
    if (e != cudaSuccess) return e;
    const int tile_q = p.consumer_warps * p.queries_per_warp;
    const int tiles = (a.max_q_len + tile_q - 1) / tile_q;
    if (tiles == 0 || a.num_seqs == 0) return cudaSuccess;
    dim3 grid(tiles, pool.n_kv, a.num_seqs);
    kern<<<grid, (p.consumer_warps + 1) * 32, smem, stream>>>(p);
    return cudaGetLastError();
  }
};

template <template <typename, int, int, bool> class Launch, typename T, int HD>
cudaError_t by_rep_simt(int rep, const AttnArgs& a, cudaStream_t s, int hg) {
  if constexpr (std::is_same<Launch<T, HD, 4, false>, DecodeLaunch<T, HD, 4, false>>::value) {
    if (rep <= 4) return DecodeLaunch<T, HD, 4, false>::run(a, hg, s);
    return DecodeLaunch<T, HD, 16, false>::run(a, hg, s);
  } else {
    if (rep <= 4) return PrefillLaunch<T, HD, 4, false>::run(a, s);
    return PrefillLaunch<T, HD, 16, false>::run(a, s);
  }
}

inline bool simt_head_dim(int hd) { return hd == 16 || hd == 32 || hd == 64 || hd == 128; }


// Decode paths compiled in their own translation units so the kernels build
// in parallel: decode_mma64.cu (tensor cores, bf16 head_dim 64),
// decode_simt.cu (CUDA cores, fp32 head_dim 64 / 128) and
// decode_simt_narrow.cu (CUDA cores, head_dim 16 / 32 of either type);
// decode.cu holds the head_dim-128 tensor-core path and the dispatch.  Each
// launches, or sizes the workspace of, one decode for its pool type.
cudaError_t launch_decode_mma64(const AttnArgs& a, int hg, cudaStream_t s);
size_t exact_workspace_mma64(const AttnArgs& a, int hg);
cudaError_t launch_decode_simt_wide(const AttnArgs& a, int hg, cudaStream_t s);
size_t exact_workspace_simt_wide(const AttnArgs& a, int hg);
cudaError_t launch_decode_simt_narrow(const AttnArgs& a, int hg, cudaStream_t s);
size_t exact_workspace_simt_narrow(const AttnArgs& a, int hg);

}  // namespace attn
}  // namespace pkv
