// Tiered GQA decode attention: split-K flash-decoding over a cache whose
// cells [0, N) are in VRAM and [N, L) in pinned host memory (or a VRAM
// staging copy of them).  llama.cpp PR "tiered KV cache (--kv-vram-cells)":
// the arithmetic does not depend on where a cell lives, so a tiered cache
// gives output bit-identical to an all-VRAM one.
//
// Work decomposition.  The cells of a sequence are cut into fixed chunks
// (a multiple of 32 cells, a function of max_ctx, batch and the SM count
// only).  Each chunk yields one unnormalised partial (m, l, acc) per query
// head; a second kernel folds the chunks of a head in a fixed order.  Which
// CTA computes a chunk never changes a bit of its partial, so the grid is
// persistent (one CTA per SM, chunks dealt round-robin) and the tier split
// only decides how a chunk's rows reach shared memory:
//   * a chunk wholly in device memory streams through a ring of 32-cell
//     tiles (two stages for q8_0 rows, up to three for 16-bit rows) filled
//     with cp.async (16-byte copies, L1 bypassed);
//   * a chunk with host-resident rows is filled tile by tile with 16-byte
//     loads through the host mapping, every thread keeping 8 in flight.
//
// Per tile, each warp computes, for one kv head and G of its query heads
// (all of them, or an equal share when fewer than 8 kv heads leave room for
// more warps), the scores of the tile's 32 cells, an online softmax in the
// log2 domain, and P*V:
//   * QK: lane = (quarter or eighth of the head dims, cell).  The lane's
//     query slice lives in registers for the whole chunk; each pass takes CPP
//     cells, and the LPC partial dot products of a cell are added by a
//     transposing butterfly, after which lane c holds the G scores of cell c.
//     fp16/bf16 caches: the slice as 16-bit pairs, products fp16 x fp16 (or
//     bf16 x bf16) into an fp32 accumulator (exact products, fp32 sums).
//     q8_0 caches: the slice is rounded once per chunk to 16-bit integers
//     n = round(q / s), s = max|q| / 32767 over the lane's dims of the head,
//     so that |q - s n| <= s / 2; the block's 32 int8 values then meet them
//     in exact integer dot products (dp2a: two int16 x int8 products per
//     instruction, int32 sums), and the block scale d times s scales the
//     integer sum once.  dp2a issues at the same multiply-add rate as fp32
//     FMA, twice that of the mixed fp16-operand FMA, and reads the int8
//     bytes as they are stored (no conversion).
//   * softmax: per-head tile maxima by warp butterflies; the running maximum
//     moves only when a tile exceeds it by more than 2^8 (all p stay <= 256);
//     l is kept per lane and summed once per chunk.
//   * PV: lane owns D/32 dims of every head; V is converted to fp32 (q8_0:
//     exact d * x) and accumulated with packed f32x2 FMAs, weights (p, p)
//     read from shared memory.
// launch_d is instantiated per K/V dtype, head_dim and mode in the
// decode_k_*.cu units; the dispatch over group shapes is decode_dispatch.cuh.
#pragma once
#include <cuda_fp16.h>
#include <math.h>

#include "kvo_internal.cuh"

namespace kvo {
namespace dec {

constexpr int kTile = 32;                 // cells per tile
constexpr int kMaxStages = 3;
constexpr int kSmemLimit = 232448;        // dynamic shared memory per CTA (sm_103a opt-in)

// Shared-memory pitch of a cell row: rows stay 16-byte aligned and an odd
// number of 16-byte units apart, so 16-byte reads of consecutive rows by
// 8 lanes hit distinct banks.
__host__ __device__ constexpr int64_t row_pitch(int64_t rb) { return (rb % 32 == 0) ? rb + 16 : rb; }

template <int KVT, int G, int D>
struct Shape {
  static constexpr int LPC = (G * D / 8 <= 96) ? 4 : 8;   // lanes per cell in QK
  static constexpr int CPP = 32 / LPC;                    // cells per QK pass
  static constexpr int NP = kTile / CPP;                  // QK passes per tile
  static constexpr int DL = D / LPC;                      // head dims per lane in QK
  static constexpr int QW = DL / 2;                       // query pair words per head
  static constexpr int DV = D / 32;                       // head dims per lane in PV
  static constexpr int NB = D / 32;                       // q8_0 blocks per head
  static constexpr int HB = KVT == KVO_Q8_0 ? NB * 34 : 2 * D;   // bytes of one head in a row
};

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// lo(a) * lo(b) + c and hi(a) * hi(b) + c for 16-bit float pairs (fp16, or
// bf16 for a bf16 cache), fp32 accumulator.
template <int KVT>
__device__ __forceinline__ float mfma_lo(uint32_t a, uint32_t b, float c) {
  float r;
  if constexpr (KVT == KVO_BF16)
    asm("{.reg .b16 a0,a1,b0,b1;\n mov.b32 {a0,a1}, %1;\n mov.b32 {b0,b1}, %2;\n"
        " fma.rn.f32.bf16 %0, a0, b0, %3;}" : "=f"(r) : "r"(a), "r"(b), "f"(c));
  else
    asm("{.reg .b16 a0,a1,b0,b1;\n mov.b32 {a0,a1}, %1;\n mov.b32 {b0,b1}, %2;\n"
        " fma.rn.f32.f16 %0, a0, b0, %3;}" : "=f"(r) : "r"(a), "r"(b), "f"(c));
  return r;
}
template <int KVT>
__device__ __forceinline__ float mfma_hi(uint32_t a, uint32_t b, float c) {
  float r;
  if constexpr (KVT == KVO_BF16)
    asm("{.reg .b16 a0,a1,b0,b1;\n mov.b32 {a0,a1}, %1;\n mov.b32 {b0,b1}, %2;\n"
        " fma.rn.f32.bf16 %0, a1, b1, %3;}" : "=f"(r) : "r"(a), "r"(b), "f"(c));
  else
    asm("{.reg .b16 a0,a1,b0,b1;\n mov.b32 {a0,a1}, %1;\n mov.b32 {b0,b1}, %2;\n"
        " fma.rn.f32.f16 %0, a1, b1, %3;}" : "=f"(r) : "r"(a), "r"(b), "f"(c));
  return r;
}

// c + a.lo16 * b.byte0 + a.hi16 * b.byte1 (lo) or b.byte2 / b.byte3 (hi),
// signed, exact in int32.
__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.lo.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.hi.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Packed fp32 pairs.
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float &a, float &b) {
  asm("mov.b64 {%0,%1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fsub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ float h2f(uint16_t b, int dt) {
  if (dt == KVO_BF16) return __uint_as_float((uint32_t)b << 16);
  return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Four int8 values (one word) -> two packed fp32 pairs, exact (int8 -> fp32
// conversions of the sign-extended bytes).
__device__ __forceinline__ void i8x4_to_f32x2(uint32_t w, uint64_t &p01, uint64_t &p23) {
  p01 = pk2(__int2float_rn((int)(int8_t)(w & 0xffu)), __int2float_rn((int)(int8_t)((w >> 8) & 0xffu)));
  p23 = pk2(__int2float_rn((int)(int8_t)((w >> 16) & 0xffu)), __int2float_rn((int)(int8_t)(w >> 24)));
}

// ---------------------------------------------------------------- tile fill

// floor(n / d) for a divisor d >= 2 fixed per launch: m = ceil(2^32 / d)
// gives the exact quotient for every n < 2^32 / d.
struct FastDiv {
  uint32_t d, m;
};
__host__ __device__ inline FastDiv make_fastdiv(uint32_t d) {
  return FastDiv{d, (uint32_t)((0x100000000ull + d - 1) / d)};
}
__device__ __forceinline__ uint32_t fdiv(uint32_t n, FastDiv f) { return __umulhi(n, f.m); }

// Source of 16-byte chunk ch of K or V row j of sequence b.
__device__ __forceinline__ const int4 *row_src(const DecodeArgs &a, int b, int64_t j, bool is_v) {
  const uint8_t *p;
  if (j < a.n_vram) p = (is_v ? a.v_lo : a.k_lo) + (b * a.lo_seq_stride_rows + j) * a.row_bytes;
  else p = (is_v ? a.v_hi : a.k_hi) + (b * a.hi_seq_stride_rows + (j - a.n_vram)) * a.row_bytes;
  return (const int4 *)p;
}

// Cell rows [c0, c0 + n) of sequence b, K and V, into one stage: asynchronous
// 16-byte copies, all in flight at once (device-resident rows only).  A tile
// within one tier (the usual case) walks its chunks from one base pointer
// per plane with incremental (row, chunk) indices; a tile that straddles the
// VRAM/tail boundary takes each row's tier.
__device__ __forceinline__ void fill_async(const DecodeArgs &a, int b, int64_t c0, int n,
                                           uint8_t *sk, uint8_t *sv, int64_t pitch, FastDiv cpr) {
  const int cprd = (int)cpr.d;
  const int total = n * cprd;
  const int T = blockDim.x;
  if (c0 + n <= a.n_vram || c0 >= a.n_vram) {
    // The tile's rows are contiguous in global memory: chunk i is 16 i bytes
    // from the first row; in shared memory it is r (pitch - row_bytes) further.
    const uint32_t pad = (uint32_t)(pitch - a.row_bytes);
    const uint8_t *kp = (const uint8_t *)row_src(a, b, c0, false) + threadIdx.x * 16;
    const uint8_t *vp = (const uint8_t *)row_src(a, b, c0, true) + threadIdx.x * 16;
    const int r0 = (int)fdiv((uint32_t)threadIdx.x, cpr);
    int ch = (int)threadIdx.x - r0 * cprd;
    const int dr = (int)fdiv((uint32_t)T, cpr), dch = T - dr * cprd;
    uint32_t so = (uint32_t)(threadIdx.x * 16 + r0 * pad);
    const uint32_t sk0 = smem_addr(sk), sv0 = smem_addr(sv), step = (uint32_t)(T * 16 + dr * pad);
    for (int i = threadIdx.x; i < total; i += T) {
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sk0 + so), "l"(kp) : "memory");
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sv0 + so), "l"(vp) : "memory");
      kp += T * 16;
      vp += T * 16;
      so += step;
      ch += dch;
      if (ch >= cprd) {
        ch -= cprd;
        so += pad;
      }
    }
    return;
  }
  for (int i = threadIdx.x; i < 2 * total; i += T) {
    const bool is_v = i >= total;
    const int k = is_v ? i - total : i;
    const int r = (int)fdiv((uint32_t)k, cpr), ch = k - r * cprd;
    const uint32_t dst = smem_addr((is_v ? sv : sk) + r * pitch + ch * 16);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
                 "l"(row_src(a, b, c0 + r, is_v) + ch)
                 : "memory");
  }
}

// The same rows with plain 16-byte loads (any device-accessible memory),
// eight per thread in flight.
__device__ __forceinline__ void fill_sync(const DecodeArgs &a, int b, int64_t c0, int n,
                                          uint8_t *sk, uint8_t *sv, int64_t pitch, FastDiv cpr) {
  const int cprd = (int)cpr.d;
  const int total = n * cprd;
  const int nthr = blockDim.x;
  constexpr int kBatch = 8;
  if (c0 + n <= a.n_vram || c0 >= a.n_vram) {
    // one tier: K and V chunk i together, kBatch / 2 chunk pairs in flight,
    // (row, chunk) indices advanced incrementally as in fill_async
    constexpr int kPairs = kBatch / 2;
    const int64_t rb = a.row_bytes;
    const uint8_t *kb = (const uint8_t *)row_src(a, b, c0, false), *vb = (const uint8_t *)row_src(a, b, c0, true);
    int r = (int)fdiv((uint32_t)threadIdx.x, cpr), ch = (int)threadIdx.x - r * cprd;
    const int dr = (int)fdiv((uint32_t)nthr, cpr), dch = nthr - dr * cprd;
    for (int i0 = threadIdx.x; i0 < total; i0 += kPairs * nthr) {
      int4 kv[kPairs], vv[kPairs];
      uint32_t so[kPairs];
#pragma unroll
      for (int u = 0; u < kPairs; ++u) {
        so[u] = (uint32_t)(r * pitch + ch * 16);
        if (i0 + u * nthr < total) {
          const int64_t go = (int64_t)r * rb + ch * 16;
          kv[u] = *(const int4 *)(kb + go);
          vv[u] = *(const int4 *)(vb + go);
        }
        r += dr;
        ch += dch;
        if (ch >= cprd) {
          ch -= cprd;
          ++r;
        }
      }
#pragma unroll
      for (int u = 0; u < kPairs; ++u)
        if (i0 + u * nthr < total) {
          *(int4 *)(sk + so[u]) = kv[u];
          *(int4 *)(sv + so[u]) = vv[u];
        }
    }
    return;
  }
  for (int base = 0; base < 2 * total; base += kBatch * nthr) {
    int4 v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * nthr + (int)threadIdx.x;
      if (i < 2 * total) {
        const bool is_v = i >= total;
        const int k = is_v ? i - total : i;
        const int r = (int)fdiv((uint32_t)k, cpr), ch = k - r * cprd;
        v[u] = row_src(a, b, c0 + r, is_v)[ch];
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * nthr + (int)threadIdx.x;
      if (i < 2 * total) {
        const bool is_v = i >= total;
        const int k = is_v ? i - total : i;
        const int r = (int)fdiv((uint32_t)k, cpr), ch = k - r * cprd;
        *(int4 *)((is_v ? sv : sk) + r * pitch + ch * 16) = v[u];
      }
    }
  }
}

// ---------------------------------------------------------------- sparse rows (selection mode)

// Row of cache position j in selection mode, or null when j is padding
// (outside [win_lo, win_hi)) or its page-table entry is out of range.
__device__ __forceinline__ const uint8_t *sparse_row(const DecodeArgs &a, int64_t j, bool is_v) {
  if (j < a.win_lo || j >= a.win_hi) return nullptr;
  if (a.sparse_staged) return (is_v ? a.v_lo : a.k_lo) + (j - a.win_lo) * a.row_bytes;
  const int64_t page = a.block_table[j / a.page_size];
  if (page < 0 || page >= a.n_pages_total) return nullptr;
  return (is_v ? a.v_hi : a.k_hi) + (page * a.page_size + j % a.page_size) * a.row_bytes;
}

// The n (<= 32) slots of a tile, K and V, into one stage; lane r of every
// warp holds slot r's cache position in jl (one coalesced load per warp, made
// ahead of time by the caller).  Warp w takes slots w, w + warps, ...; a
// padding slot gets a zero V row (its weight is 0 and must meet finite
// values).  Async: 16-byte cp.async copies (device-resident arena); else
// 16-byte loads through the mapping.
template <bool ASYNC>
__device__ __forceinline__ void fill_sparse(const DecodeArgs &a, int32_t jl, int n, uint8_t *sk,
                                            uint8_t *sv, int64_t pitch) {
  const int warps = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cpr = (int)(a.row_bytes >> 4);
  for (int r = warp; r < n; r += warps) {    // warp-uniform; r < n <= 32
    const int64_t j = __shfl_sync(0xffffffffu, jl, r);
    const int4 *ks = (const int4 *)sparse_row(a, j, false);
    const int4 *vs = (const int4 *)sparse_row(a, j, true);
    if (!ks && lane == 0 && j >= a.win_lo && j < a.win_hi) atomicOr(a.err, kErrPageTable);
    uint8_t *kd = sk + r * pitch, *vd = sv + r * pitch;
    for (int ch = lane; ch < cpr; ch += 32) {
      if (!ks) {
        *(int4 *)(vd + ch * 16) = make_int4(0, 0, 0, 0);
      } else if constexpr (ASYNC) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(kd + ch * 16)), "l"(ks + ch)
                     : "memory");
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(vd + ch * 16)), "l"(vs + ch)
                     : "memory");
      } else {
        const int4 kx = ks[ch], vx = vs[ch];
        *(int4 *)(kd + ch * 16) = kx;
        *(int4 *)(vd + ch * 16) = vx;
      }
    }
  }
}

// ---------------------------------------------------------------- per-warp state

template <int KVT, int G, int D>
struct WarpState {
  using S = Shape<KVT, G, D>;
  uint32_t q[G][S::QW];      // this lane's query slice, 16-bit pairs (q8_0: int16 pairs)
  float qs[G];               // q8_0: s * scale_log2, the slice's integer step times the score scale
  uint64_t acc[G][S::DV / 2];// PV accumulators, fp32 pairs
  float m[G], l[G];          // running max (log2 units) and this lane's share of l
};

// ---------------------------------------------------------------- QK

// Partial dot products of this lane's dims for cell row `row` (kv head g).
template <int KVT, int G, int D>
__device__ __forceinline__ void qk_cell(const WarpState<KVT, G, D> &ws, const uint8_t *row, int g,
                                        int qq, float scale_log2, float *part) {
  using S = Shape<KVT, G, D>;
  if constexpr (KVT == KVO_Q8_0) {
    constexpr int DL = S::DL;                            // 16 or 32 values of one block
    const int blk = (qq * DL) / 32, wo = (qq * DL) % 32;
    const int o = (g * S::NB + blk) * 34;                // block start in the row
    const float d = __half2float(__ushort_as_half(*(const uint16_t *)(row + o)));
    const int vb = o + 2 + wo;                           // first value byte (even)
    const uint32_t *wp = (const uint32_t *)(row + (vb & ~3));
    const uint32_t sh = (uint32_t)(vb & 3) * 8;          // 0 or 16
    uint32_t w[DL / 4 + 1];
#pragma unroll
    for (int i = 0; i <= DL / 4; ++i) w[i] = wp[i];
    int acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0;
#pragma unroll
    for (int i = 0; i < DL / 4; ++i) {
      const uint32_t x = __funnelshift_r(w[i], w[i + 1], sh);   // values 4i .. 4i+3
#pragma unroll
      for (int h = 0; h < G; ++h) {
        acc[h] = dp2a_lo(ws.q[h][2 * i], x, acc[h]);
        acc[h] = dp2a_hi(ws.q[h][2 * i + 1], x, acc[h]);
      }
    }
    // explicit roundings (never contracted into FMAs): the same bits whatever
    // code the compiler generates around them
#pragma unroll
    for (int h = 0; h < G; ++h) part[h] = __fmul_rn(__fmul_rn(d, ws.qs[h]), __int2float_rn(acc[h]));
  } else {
    const uint4 *kp = (const uint4 *)(row + g * S::HB + qq * S::DL * 2);
    float sb[G], sc[G];                                  // two chains per head
#pragma unroll
    for (int h = 0; h < G; ++h) sb[h] = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) sc[h] = 0.f;
#pragma unroll
    for (int i = 0; i < S::DL / 8; ++i) {
      const uint4 k = kp[i];
      const uint32_t kw[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int h = 0; h < G; ++h) {
          sb[h] = mfma_lo<KVT>(ws.q[h][4 * i + e], kw[e], sb[h]);
          sc[h] = mfma_hi<KVT>(ws.q[h][4 * i + e], kw[e], sc[h]);
        }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) part[h] = __fmul_rn(__fadd_rn(sb[h], sc[h]), scale_log2);
  }
}

// Scores of the tile's 32 cells: lane c ends with the G scores of cell c
// (meaningful for c < n only: a pass whose cells all lie past n is skipped).
template <int KVT, int G, int D>
__device__ __forceinline__ void qk_tile(const WarpState<KVT, G, D> &ws, const uint8_t *sk,
                                        int64_t pitch, int g, int lane, float scale_log2, int n,
                                        float *s) {
  using S = Shape<KVT, G, D>;
  const int qq = lane / S::CPP, cl = lane % S::CPP;
  float v[S::NP][G];
#pragma unroll
  for (int ps = 0; ps < S::NP; ++ps) {
    if (ps == 0 || ps * S::CPP < n) {        // warp-uniform
      qk_cell<KVT, G, D>(ws, sk + (int64_t)(cl + S::CPP * ps) * pitch, g, qq, scale_log2, v[ps]);
    } else {
#pragma unroll
      for (int h = 0; h < G; ++h) v[ps][h] = 0.f;
    }
  }
  // Transposing butterfly: stage k pairs passes that differ in bit k and
  // keeps the one whose bit k equals bit k of qq, adding the partner lane's
  // (lane ^ (CPP << k)) other half.  After log2(LPC) stages the remaining
  // pass is qq, i.e. cell cl + CPP * qq = lane.
#pragma unroll
  for (int k = 0, n = S::NP; n > 1; ++k, n >>= 1) {
    const bool hi = (qq >> k) & 1;
#pragma unroll
    for (int i = 0; i < n / 2; ++i)
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mine = hi ? v[2 * i + 1][h] : v[2 * i][h];
        const float other = hi ? v[2 * i][h] : v[2 * i + 1][h];
        v[i][h] = __fadd_rn(mine, __shfl_xor_sync(0xffffffffu, other, S::CPP << k));
      }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) s[h] = v[0][h];
}

// ---------------------------------------------------------------- PV

// This lane's D/32 dims of V for cell row `row` (kv head g), as fp32 pairs.
template <int KVT, int G, int D>
__device__ __forceinline__ void v_cell(const uint8_t *row, int g, int lane, uint64_t *vp) {
  using S = Shape<KVT, G, D>;
  constexpr int DV = S::DV;
  if constexpr (KVT == KVO_Q8_0) {
    const int blk = (DV * lane) / 32, wo = (DV * lane) % 32;
    const int o = (g * S::NB + blk) * 34;
    const float d = __half2float(__ushort_as_half(*(const uint16_t *)(row + o)));
    const uint64_t dd = pk2(d, d);
    const int vb = o + 2 + wo;                           // even
    if constexpr (DV == 4) {
      const uint32_t *wp = (const uint32_t *)(row + (vb & ~3));
      const uint32_t x = __funnelshift_r(wp[0], wp[1], (uint32_t)(vb & 3) * 8);
      uint64_t p01, p23;
      i8x4_to_f32x2(x, p01, p23);
      vp[0] = fmul2(p01, dd);
      vp[1] = fmul2(p23, dd);
    } else {
      const uint32_t x = *(const uint16_t *)(row + vb);
      uint64_t p01, p23;
      i8x4_to_f32x2(x, p01, p23);
      vp[0] = fmul2(p01, dd);
    }
  } else {
    const uint8_t *hp = row + g * S::HB + lane * DV * 2;
    if constexpr (DV == 4) {
      const uint2 u = *(const uint2 *)hp;
      vp[0] = pk2(h2f(u.x & 0xffff, KVT), h2f(u.x >> 16, KVT));
      vp[1] = pk2(h2f(u.y & 0xffff, KVT), h2f(u.y >> 16, KVT));
    } else {
      const uint32_t u = *(const uint32_t *)hp;
      vp[0] = pk2(h2f(u & 0xffff, KVT), h2f(u >> 16, KVT));
    }
  }
}

// ---------------------------------------------------------------- kernel

// Up to 16 warps when a warp holds at most two query heads (few registers),
// else up to 8.
template <int G>
constexpr int max_decode_threads() { return G <= 2 ? 512 : 256; }

// SP: selection mode (QSA sparse rows): cell k of work row b is cache
// position a.indices[b * a.max_ctx + k], padding masked out.
template <int KVT, int QT, int G, int D, bool SP>
__global__ void __launch_bounds__(max_decode_threads<G>(), 1)
decode_split_kernel(const DecodeArgs a, int n_stages) {
  using S = Shape<KVT, G, D>;
  extern __shared__ __align__(16) uint8_t smem[];
  // Warp w serves kv head g = w / wph and its query heads h0 .. h0 + G - 1
  // (G = heads per warp; wph warps share a kv head when the group allows).
  const int w_id = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wph = a.group / G;
  const int g = w_id / wph, h0 = g * a.group + (w_id % wph) * G;
  const int64_t pitch = row_pitch(a.row_bytes);
  const int64_t stage_bytes = 2 * kTile * pitch;
  // weights (p, p) of the tile: [cell][GP], GP = G rounded up to even so
  // that every cell's entries start on a 16-byte boundary
  constexpr int GP = (G + 1) & ~1;
  uint64_t *pbuf = (uint64_t *)(smem + n_stages * stage_bytes) + (size_t)w_id * kTile * GP;
  // Rows prefetched into shared memory (selection mode, staged, one stage,
  // one chunk per row): two slots, each a row's query [Hq][D] and running
  // state; slot n % 2 holds the n-th row this CTA works on, tagged with it.
  const bool pre = SP && a.pre_rows && n_stages == 1;
  const int64_t q_bytes = (int64_t)a.n_q_heads * D * 2;
  const int64_t rs_bytes = (int64_t)a.n_q_heads * (D + 2) * 4;
  uint8_t *pre_base = smem + n_stages * stage_bytes + (size_t)(blockDim.x >> 5) * kTile * GP * sizeof(uint64_t);
  int pre_tag[2] = {-1, -1};
  const float *pre_rs = nullptr;             // running state of the current row in shared memory
  const uint16_t *pre_q = nullptr;           // query of the current row in shared memory
  const int qq = lane / S::CPP;
  const int64_t n_items = (int64_t)a.batch * a.n_splits;
  const FastDiv cpr = make_fastdiv((uint32_t)(a.row_bytes >> 4));   // 16-byte chunks per row

  const int64_t w_end = a.item_hi < 0 ? n_items : a.item_hi;

  // Work item w = (chunk w / batch, row or sequence w % batch); nt = 0 for a
  // chunk beyond the context (never combined).
  struct Item {
    int64_t w, cs, ce, sel0;
    int chunk, b, nt;
  };
  auto item_at = [&](int64_t w) {
    Item it;
    it.w = w;
    it.nt = 0;
    it.cs = it.ce = it.sel0 = 0;
    it.chunk = it.b = 0;
    if (w >= w_end) return it;
    const int c = (int)(w / a.batch);
    it.chunk = a.interleave ? ((c & 1) ? a.n_splits - 1 - (c >> 1) : (c >> 1)) : c;
    it.b = (int)(w % a.batch);
    int64_t ctx;
    if constexpr (SP) {                      // selection mode: the row's slots sel0 .. sel0 + ctx
      ctx = a.max_ctx;
      if (a.offs) {
        const int32_t *ob = a.offs + (int64_t)it.b * a.offs_stride + a.bucket;
        it.sel0 = ob[0];
        ctx = ob[1] - ob[0];
      }
    } else {
      ctx = a.ctx_len[it.b] < a.max_ctx ? a.ctx_len[it.b] : a.max_ctx;
    }
    it.cs = (int64_t)it.chunk * a.split_cells;
    it.ce = it.cs + a.split_cells < ctx ? it.cs + a.split_cells : ctx;
    if (it.cs < it.ce) it.nt = (int)((it.ce - it.cs + kTile - 1) / kTile);
    return it;
  };
  // One chunk per row (selection mode, staged): fold the chunk's (m, l, acc)
  // straight into the row's running state (the per-bucket fold of the
  // ExLlamaV3 qsa-kv-offload patch, in log2 units), or finish the row:
  //   m' = max(m, m_b); alpha = 2^(m - m') (0 if m = -inf); beta = 2^(m_b - m') (0 if m_b = -inf)
  //   acc = alpha acc + beta acc_b; l = alpha l + beta l_b
  // This warp alone owns the (row, head) pairs it folds.
  // rs: a shared-memory copy of the row's running state ([Hq][D] acc, then
  // [Hq][2] (m, l)), or null to read it from global memory.
  auto fold = [&](const Item &it, int h, float m_b, float l_b, const float *acc_b, const float *rs) {
    const size_t oi = (size_t)it.b * a.n_q_heads + h0 + h;
    const float *ra_in = rs ? rs + (size_t)(h0 + h) * D + lane * S::DV : a.run_acc + oi * D + lane * S::DV;
    const float *ml_in = rs ? rs + (size_t)a.n_q_heads * D + (size_t)(h0 + h) * 2 : a.run_ml + oi * 2;
    float m_run = -INFINITY, l_run = 0.f;
    if (!a.init) {
      m_run = ml_in[0];
      l_run = ml_in[1];
    }
    const float m_new = fmaxf(m_run, m_b);
    const float alpha = m_run == -INFINITY ? 0.f : exp2f(m_run - m_new);
    const float beta = m_b == -INFINITY ? 0.f : exp2f(m_b - m_new);
    const float l_new = alpha * l_run + beta * l_b;
    float *ra = a.run_acc + oi * D + lane * S::DV;
    float *o = a.out + oi * D + lane * S::DV;
#pragma unroll
    for (int i = 0; i < S::DV; ++i) {
      const float acc_new = alpha * (a.init ? 0.f : ra_in[i]) + beta * acc_b[i];
      if (a.finalize) o[i] = acc_new / fmaxf(l_new, 1e-30f);
      else ra[i] = acc_new;
    }
    __syncwarp();                            // every lane has read run_ml
    if (!a.finalize && lane == 0) {
      a.run_ml[oi * 2] = m_new;
      a.run_ml[oi * 2 + 1] = l_new;
    }
  };
  // A row with no picks in this bucket: the running state only needs to be
  // started (first bucket) or finished (last bucket).
  auto fold_empty = [&](const Item &it) {
    if (!(a.init || a.finalize)) return;
    float z[S::DV];
#pragma unroll
    for (int i = 0; i < S::DV; ++i) z[i] = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) fold(it, h, -INFINITY, 0.f, z, nullptr);
  };

  // First non-empty item at or after w (stride gridDim.x); fold_empties: the
  // skipped items of a launch that folds in the split kernel are folded here.
  auto next_item = [&](int64_t w, bool fold_empties) {
    Item it = item_at(w);
    while (it.w < w_end && it.nt == 0) {
      if (SP && fold_empties && a.fold_in_split) fold_empty(it);
      it = item_at(it.w + gridDim.x);
    }
    return it;
  };
  // Selection mode: lane r's cache position for slot r of tile t of `it`
  // (meaningless past the tile's end or past the launch's items).
  auto picks = [&](const Item &it, int t) -> int32_t {
    if constexpr (SP) {
      const int64_t t0 = it.cs + (int64_t)t * kTile;
      if (it.w < w_end && t0 + lane < it.ce) return a.indices[(int64_t)it.b * a.max_ctx + it.sel0 + t0 + lane];
    }
    return -1;
  };
  // Device-resident rows: asynchronous copies into a ring stage (jl: picks()).
  auto issue = [&](const Item &it, int t, uint8_t *st, int32_t jl) {
    const int64_t t0 = it.cs + (int64_t)t * kTile;
    const int n = (int)(it.ce - t0 < kTile ? it.ce - t0 : kTile);
    if constexpr (SP) fill_sparse<true>(a, jl, n, st, st + kTile * pitch, pitch);
    else fill_async(a, it.b, t0, n, st, st + kTile * pitch, pitch, cpr);
  };

  WarpState<KVT, G, D> ws;
  auto init_item = [&](const Item &it) {
    // query slice of each of the warp's heads: dims [qq*DL, qq*DL + DL)
    const uint16_t *qsrc = (pre_q ? pre_q : (const uint16_t *)a.q + (size_t)it.b * a.n_q_heads * D) + (size_t)h0 * D;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const uint4 *qp = (const uint4 *)(qsrc + (size_t)h * D + qq * S::DL);
#pragma unroll
      for (int i = 0; i < S::DL / 8; ++i) {
        const uint4 u = qp[i];
        ws.q[h][4 * i] = u.x; ws.q[h][4 * i + 1] = u.y;
        ws.q[h][4 * i + 2] = u.z; ws.q[h][4 * i + 3] = u.w;
      }
      if constexpr (KVT == KVO_Q8_0) {
        // round the slice to 16-bit integers: step s = max|q| / 32767
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < S::QW; ++i)
          amax = fmaxf(amax, fmaxf(fabsf(h2f(ws.q[h][i] & 0xffff, QT)), fabsf(h2f(ws.q[h][i] >> 16, QT))));
        const float inv = amax > 0.f ? __fdiv_rn(32767.f, amax) : 0.f;
#pragma unroll
        for (int i = 0; i < S::QW; ++i) {
          const float x0 = h2f(ws.q[h][i] & 0xffff, QT), x1 = h2f(ws.q[h][i] >> 16, QT);
          const int n0 = max(-32767, min(32767, __float2int_rn(__fmul_rn(x0, inv))));
          const int n1 = max(-32767, min(32767, __float2int_rn(__fmul_rn(x1, inv))));
          ws.q[h][i] = ((uint32_t)n0 & 0xffffu) | ((uint32_t)n1 << 16);
        }
        ws.qs[h] = __fmul_rn(__fdiv_rn(amax, 32767.f), a.scale_log2);
      }
      ws.m[h] = -INFINITY;
      ws.l[h] = 0.f;
#pragma unroll
      for (int i = 0; i < S::DV / 2; ++i) ws.acc[h][i] = 0ull;
    }
  };

  // One tile of item `it` (tile t, K rows at sk, V rows at sv): scores of
  // cell `lane` and the online softmax (weights to pbuf), then P*V.
  auto compute_qk = [&](const Item &it, int t, const uint8_t *sk) {
    const int64_t t0 = it.cs + (int64_t)t * kTile;
    const int n = (int)(it.ce - t0 < kTile ? it.ce - t0 : kTile);
    float s[G];
    qk_tile<KVT, G, D>(ws, sk, pitch, g, lane, a.scale_log2, n, s);
    bool valid = lane < n;
    if constexpr (SP)                        // staged picks are grouped inside the window already
      if (!a.offs) valid = valid && sparse_row(a, a.indices[(int64_t)it.b * a.max_ctx + it.sel0 + t0 + lane], false);
    // tile maxima of all G heads: one butterfly with the heads interleaved, so
    // that the G shuffle chains overlap instead of running one after another
    float sv[G], tmax[G];
#pragma unroll
    for (int h = 0; h < G; ++h) tmax[h] = sv[h] = valid ? s[h] : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int h = 0; h < G; ++h) tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], o));
#pragma unroll
    for (int h = 0; h < G; ++h) {
      if (tmax[h] > ws.m[h] + 8.f) {         // warp-uniform: move the reference
        const float alpha = exp2f(__fsub_rn(ws.m[h], tmax[h]));
        const uint64_t aa = pk2(alpha, alpha);
        ws.l[h] = __fmul_rn(ws.l[h], alpha);
#pragma unroll
        for (int i = 0; i < S::DV / 2; ++i) ws.acc[h][i] = fmul2(ws.acc[h][i], aa);
        ws.m[h] = tmax[h];
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float p = valid ? exp2f(__fsub_rn(sv[h], ws.m[h])) : 0.f;
      ws.l[h] = __fadd_rn(ws.l[h], p);
      pbuf[lane * GP + h] = pk2(p, p);
    }
    __syncwarp();
  };
  auto pv_cell = [&](const uint8_t *sv, int c) {
      uint64_t vp[S::DV / 2];
      v_cell<KVT, G, D>(sv + (int64_t)c * pitch, g, lane, vp);
      const uint64_t *pc = pbuf + c * GP;
      uint64_t pp[G];
#pragma unroll
      for (int h = 0; h + 1 < G; h += 2) {
        const ulonglong2 u = *(const ulonglong2 *)(pc + h);   // h and GP even: 16-byte aligned
        pp[h] = u.x; pp[h + 1] = u.y;
      }
      if constexpr (G & 1) pp[G - 1] = pc[G - 1];
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int i = 0; i < S::DV / 2; ++i) ws.acc[h][i] = ffma2(pp[h], vp[i], ws.acc[h][i]);
  };
  auto compute_pv = [&](const Item &it, int t, const uint8_t *sv) {
    const int64_t t0 = it.cs + (int64_t)t * kTile;
    const int n = (int)(it.ce - t0 < kTile ? it.ce - t0 : kTile);
    if (n == kTile) {                        // full tile: unrolled, so that the next cells'
#pragma unroll 8                             // shared-memory reads overlap this cell's FMAs
      for (int c = 0; c < kTile; ++c) pv_cell(sv, c);
    } else {
      for (int c = 0; c < n; ++c) pv_cell(sv, c);
    }
    __syncwarp();                            // pbuf reads done before the next tile's writes
  };
  auto compute_tile = [&](const Item &it, int t, const uint8_t *st) {
    compute_qk(it, t, st);
    compute_pv(it, t, st + kTile * pitch);
  };

  // Partial of an item: acc (this lane's dims), m, l.
  auto write_partial = [&](const Item &it) {
    float lsums[G];                          // the G butterflies interleaved (same sums per head)
#pragma unroll
    for (int h = 0; h < G; ++h) lsums[h] = ws.l[h];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int h = 0; h < G; ++h) lsums[h] += __shfl_xor_sync(0xffffffffu, lsums[h], o);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float lsum = lsums[h];
      if (SP && a.fold_in_split) {
        float x[S::DV];
#pragma unroll
        for (int i = 0; i < S::DV / 2; ++i) upk2(ws.acc[h][i], x[2 * i], x[2 * i + 1]);
        fold(it, h, ws.m[h], lsum, x, pre_rs);
        continue;
      }
      const int qh = h0 + h;
      const size_t pi = ((size_t)it.b * a.n_splits + it.chunk) * a.n_q_heads + qh;
      float *pa = a.part_acc + pi * D + lane * S::DV;
      if constexpr (S::DV == 4) {
        float x0, x1, x2, x3;
        upk2(ws.acc[h][0], x0, x1);
        upk2(ws.acc[h][1], x2, x3);
        *(float4 *)pa = make_float4(x0, x1, x2, x3);
      } else {
        float x0, x1;
        upk2(ws.acc[h][0], x0, x1);
        *(float2 *)pa = make_float2(x0, x1);
      }
      if (lane == 0) {
        a.part_ml[pi * 2] = ws.m[h];
        a.part_ml[pi * 2 + 1] = lsum;
      }
    }
  };

  if (SP && a.all_ring) {
    // Every row of the launch is device-resident: one continuous ring over all
    // of this CTA's (item, tile) pairs, so the next item's first tiles are in
    // flight while the current one finishes.  fi/ft: the next tile to fill;
    // ci/ct: the tile being computed.  With a single stage (wide rows) each
    // tile is copied asynchronously and waited for before its compute.
    // fj: the picks of tile (fi, ft), loaded one tile ahead so that their
    // latency hides behind a tile's compute.
    Item ci = next_item(a.item_lo + blockIdx.x, true), fi = ci;
    int ft = 0, ct = 0;
    if (ci.w >= w_end) return;
    auto advance = [&](Item &it, int &t) {
      if (++t == it.nt) {
        it = next_item(it.w + gridDim.x, false);
        t = 0;
      }
    };
    int32_t fj = picks(fi, ft);
    // Prefetch of row n (the raw item w, which holds row w % batch) into
    // slot n % 2, committed with the next tile copy.
    int64_t n_pre = 0, n_cur = 0;
    auto prefetch_row = [&](int64_t w) {
      const int slot = (int)(n_pre++ & 1);
      if (w >= w_end) return;
      const int b = (int)(w % a.batch);
      uint8_t *dq = pre_base + slot * (q_bytes + rs_bytes);
      const uint8_t *sq = (const uint8_t *)a.q + (size_t)b * q_bytes;
      for (int64_t i = threadIdx.x; i < q_bytes / 16; i += blockDim.x)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dq + i * 16)), "l"(sq + i * 16)
                     : "memory");
      if (!a.init) {
        uint8_t *dr = dq + q_bytes;
        const uint8_t *sa = (const uint8_t *)(a.run_acc + (size_t)b * a.n_q_heads * D);
        const uint8_t *sm = (const uint8_t *)(a.run_ml + (size_t)b * a.n_q_heads * 2);
        const int64_t na = (int64_t)a.n_q_heads * D * 4 / 16, nm = (int64_t)a.n_q_heads * 8 / 16;
        for (int64_t i = threadIdx.x; i < na + nm; i += blockDim.x) {
          const uint8_t *src = i < na ? sa + i * 16 : sm + (i - na) * 16;
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dr + i * 16)), "l"(src)
                       : "memory");
        }
      }
      pre_tag[slot] = b;
    };
    // Row n_cur is the current item: use its slot when the prefetch was for it.
    auto take_row = [&](const Item &it) {
      const int slot = (int)(n_cur++ & 1);
      const bool hit = pre && pre_tag[slot] == it.b;
      uint8_t *base = pre_base + slot * (q_bytes + rs_bytes);
      pre_q = hit ? (const uint16_t *)base : nullptr;
      pre_rs = hit && !a.init ? (const float *)(base + q_bytes) : nullptr;
    };
    if (pre) prefetch_row(ci.w);
    for (int s = 0; s < n_stages - 1; ++s) {
      if (fi.w < w_end) {
        issue(fi, ft, smem + s * stage_bytes, fj);
        advance(fi, ft);
        fj = picks(fi, ft);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
    if (!pre) init_item(ci);
    bool fresh = true;                       // the first tile of ci comes next
    for (int64_t k = 0;; ++k) {
      if (n_stages == 1) {
        __syncthreads();                     // tile k-1 fully consumed
        if (pre && fresh) prefetch_row(ci.w + gridDim.x);   // its slot's last row is done
        issue(fi, ft, smem, fj);
        advance(fi, ft);
        fj = picks(fi, ft);
        asm volatile("cp.async.commit_group;" ::: "memory");
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();                     // tile k (and any prefetch) landed
        if (pre && fresh) {
          take_row(ci);
          init_item(ci);
        }
        fresh = false;
      } else {
        if (n_stages == 3) asm volatile("cp.async.wait_group 1;" ::: "memory");
        else asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();                     // tile k landed; tile k-1 fully consumed
        if (fi.w < w_end) {
          issue(fi, ft, smem + ((k + n_stages - 1) % n_stages) * stage_bytes, fj);
          advance(fi, ft);
          fj = picks(fi, ft);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
      }
      compute_tile(ci, ct, smem + (k % n_stages) * stage_bytes);
      if (ct + 1 == ci.nt) {
        write_partial(ci);
        ci = next_item(ci.w + gridDim.x, true);
        ct = 0;
        if (ci.w >= w_end) break;
        if (pre) fresh = true;
        else init_item(ci);
      } else {
        ++ct;
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    return;
  }

  // Items one at a time: a device-resident item streams through the ring, an
  // item with host-resident rows is filled tile by tile.
  for (int64_t w = a.item_lo + blockIdx.x; w < w_end; w += gridDim.x) {
    const Item it = item_at(w);
    if (it.nt == 0) {
      if (SP && a.fold_in_split) fold_empty(it);
      continue;
    }
    init_item(it);
    const bool dev = SP ? a.sparse_staged != 0 : (it.ce <= a.n_vram || a.hi_device);
    const bool ring = n_stages >= 2 && dev;
    __syncthreads();                         // smem of the previous item fully consumed
    if (ring) {
      for (int t = 0; t < n_stages - 1; ++t) {
        if (t < it.nt) issue(it, t, smem + t * stage_bytes, picks(it, t));
        asm volatile("cp.async.commit_group;" ::: "memory");
      }
    }
    for (int t = 0; t < it.nt; ++t) {
      uint8_t *st;
      if (ring) {
        if (n_stages == 3) asm volatile("cp.async.wait_group 1;" ::: "memory");
        else asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();                     // tile t landed; tile t-1 fully consumed
        const int tn = t + n_stages - 1;
        if (tn < it.nt) issue(it, tn, smem + (tn % n_stages) * stage_bytes, picks(it, tn));
        asm volatile("cp.async.commit_group;" ::: "memory");
        st = smem + (t % n_stages) * stage_bytes;
      } else {
        if (t > 0) __syncthreads();          // previous tile fully consumed
        st = smem;
        if (dev) {                           // one stage: copy asynchronously, then wait
          issue(it, t, st, picks(it, t));
          asm volatile("cp.async.commit_group;" ::: "memory");
          asm volatile("cp.async.wait_group 0;" ::: "memory");
        } else {
          const int64_t t0 = it.cs + (int64_t)t * kTile;
          const int n = (int)(it.ce - t0 < kTile ? it.ce - t0 : kTile);
          if constexpr (SP) fill_sparse<false>(a, picks(it, t), n, st, st + kTile * pitch, pitch);
          else fill_sync(a, it.b, t0, n, st, st + kTile * pitch, pitch, cpr);
        }
        __syncthreads();
      }
      compute_tile(it, t, st);
    }
    if (ring) asm volatile("cp.async.wait_group 0;" ::: "memory");
    write_partial(it);
  }
}

// Fold the chunks of one (sequence, q head): weights 2^(m_s - M) with M the
// maximum over chunks, out = acc / max(l, 1e-30).  Warp w sums the chunks
// s = w, w + 32, w + 64, ... in ascending order and the 32 warp sums are
// added in warp order: a fixed reduction tree, so the result depends on the
// partials only (never on timing, the tier split or staging).  32 warps
// (against 8: 189 -> 181 us for 184,320 cells, 304 chunks per head) spread
// a head's partial loads over more warps.
constexpr int kCombineWarps = 32;

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
decode_combine_kernel(const DecodeArgs a) {
  // Launched as a programmatic dependent of the split kernel: wait here until
  // that grid has finished and its partials are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int DPL = D / 32;
  __shared__ float red[kCombineWarps][D];
  __shared__ float red_l[kCombineWarps];
  __shared__ float red_m[kCombineWarps];
  const int h = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int64_t ctx;
  if (a.offs) {                              // selection mode, staged: this bucket's picks
    const int32_t *ob = a.offs + (int64_t)b * a.offs_stride + a.bucket;
    ctx = ob[1] - ob[0];
  } else {
    ctx = !a.ctx_len ? a.max_ctx : (a.ctx_len[b] < a.max_ctx ? a.ctx_len[b] : a.max_ctx);
  }
  const int ns = ctx > 0 ? (int)((ctx + a.split_cells - 1) / a.split_cells) : 0;
  const size_t base = (size_t)b * a.n_splits * a.n_q_heads + h;
  float M = -INFINITY;
  for (int s = threadIdx.x; s < ns; s += kCombineWarps * 32)
    M = fmaxf(M, a.part_ml[(base + (size_t)s * a.n_q_heads) * 2]);
  M = warp_max(M);
  if (lane == 0) red_m[warp] = M;
  __syncthreads();
  M = red_m[0];
#pragma unroll
  for (int w = 1; w < kCombineWarps; ++w) M = fmaxf(M, red_m[w]);
  float l = 0.f, acc[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
#pragma unroll 4
  for (int s = warp; s < ns; s += kCombineWarps) {
    const size_t pi = base + (size_t)s * a.n_q_heads;
    const float ms = a.part_ml[pi * 2];
    const float w = ms == -INFINITY ? 0.f : exp2f(ms - M);     // a chunk with nothing selected
    l = fmaf(w, a.part_ml[pi * 2 + 1], l);
    const float *pa = a.part_acc + pi * D + lane * DPL;
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = fmaf(w, pa[i], acc[i]);
  }
#pragma unroll
  for (int i = 0; i < DPL; ++i) red[warp][lane * DPL + i] = acc[i];
  if (lane == 0) red_l[warp] = l;
  __syncthreads();
  const size_t oi = (size_t)b * a.n_q_heads + h;
  if (!a.run_acc) {
    for (int d = threadIdx.x; d < D; d += kCombineWarps * 32) {
      float sl = 0.f, sa = 0.f;
#pragma unroll
      for (int w = 0; w < kCombineWarps; ++w) {
        sl += red_l[w];
        sa += red[w][d];
      }
      a.out[oi * D + d] = sa / fmaxf(sl, 1e-30f);
    }
    return;
  }
  // Fold this launch's (M, l, acc) into the running state (ExLlamaV3
  // qsa-kv-offload patch, the per-bucket fold), in log2 units:
  //   m' = max(m, M); alpha = 2^(m - m') (0 if m = -inf); beta = 2^(M - m') (0 if M = -inf)
  //   acc = alpha acc + beta acc_b; l = alpha l + beta l_b
  float sl = 0.f;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) sl += red_l[w];
  float m_run = -INFINITY, l_run = 0.f;
  if (!a.init) {
    m_run = a.run_ml[oi * 2];
    l_run = a.run_ml[oi * 2 + 1];
  }
  const float m_new = fmaxf(m_run, M);
  const float alpha = m_run == -INFINITY ? 0.f : exp2f(m_run - m_new);
  const float beta = M == -INFINITY ? 0.f : exp2f(M - m_new);
  const float l_new = alpha * l_run + beta * sl;
  for (int d = threadIdx.x; d < D; d += kCombineWarps * 32) {
    float sa = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) sa += red[w][d];
    const float acc_run = a.init ? 0.f : a.run_acc[oi * D + d];
    const float acc_new = alpha * acc_run + beta * sa;
    if (a.finalize) a.out[oi * D + d] = acc_new / fmaxf(l_new, 1e-30f);
    else a.run_acc[oi * D + d] = acc_new;
  }
  if (!a.finalize && threadIdx.x == 0) {
    a.run_ml[oi * 2] = m_new;
    a.run_ml[oi * 2 + 1] = l_new;
  }
}

// The same fold for launches with few chunks (<= kSmallCombineChunks): one
// warp per (row, q head), chunks folded in ascending order, lane l owning
// dims [l * D/32, (l + 1) * D/32).  Many small (row, head) items (the sparse
// rows) then cost one warp each instead of one CTA.
constexpr int kSmallCombineChunks = 4;

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
decode_combine_small_kernel(const DecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");   // as in decode_combine_kernel
  constexpr int DPL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t item = (int64_t)blockIdx.x * kCombineWarps + warp;
  if (item >= (int64_t)a.batch * a.n_q_heads) return;
  const int b = (int)(item / a.n_q_heads), h = (int)(item % a.n_q_heads);
  int64_t ctx;
  if (a.offs) {
    const int32_t *ob = a.offs + (int64_t)b * a.offs_stride + a.bucket;
    ctx = ob[1] - ob[0];
  } else {
    ctx = !a.ctx_len ? a.max_ctx : (a.ctx_len[b] < a.max_ctx ? a.ctx_len[b] : a.max_ctx);
  }
  const int ns = ctx > 0 ? (int)((ctx + a.split_cells - 1) / a.split_cells) : 0;
  const size_t base = (size_t)b * a.n_splits * a.n_q_heads + h;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, a.part_ml[(base + (size_t)s * a.n_q_heads) * 2]);
  float l = 0.f, acc[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
  for (int s = 0; s < ns; ++s) {
    const size_t pi = base + (size_t)s * a.n_q_heads;
    const float ms = a.part_ml[pi * 2];
    const float w = ms == -INFINITY ? 0.f : exp2f(ms - M);
    l = fmaf(w, a.part_ml[pi * 2 + 1], l);
    const float *pa = a.part_acc + pi * D + lane * DPL;
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = fmaf(w, pa[i], acc[i]);
  }
  const size_t oi = (size_t)b * a.n_q_heads + h;
  float *o = a.out + oi * D + lane * DPL;
  if (!a.run_acc) {
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[i] = acc[i] / fmaxf(l, 1e-30f);
    return;
  }
  float m_run = -INFINITY, l_run = 0.f;
  if (!a.init) {
    m_run = a.run_ml[oi * 2];
    l_run = a.run_ml[oi * 2 + 1];
  }
  const float m_new = fmaxf(m_run, M);
  const float alpha = m_run == -INFINITY ? 0.f : exp2f(m_run - m_new);
  const float beta = M == -INFINITY ? 0.f : exp2f(M - m_new);
  const float l_new = alpha * l_run + beta * l;
  float *ra = a.run_acc + oi * D + lane * DPL;
#pragma unroll
  for (int i = 0; i < DPL; ++i) {
    const float acc_new = alpha * (a.init ? 0.f : ra[i]) + beta * acc[i];
    if (a.finalize) o[i] = acc_new / fmaxf(l_new, 1e-30f);
    else ra[i] = acc_new;
  }
  if (!a.finalize && lane == 0) {
    a.run_ml[oi * 2] = m_new;
    a.run_ml[oi * 2 + 1] = l_new;
  }
}

// Shared memory of the split kernel for n_stages ring stages.
inline size_t split_smem_bytes(const DecodeArgs &a, int g_per_warp, int n_stages) {
  const int warps = a.n_kv_heads * (a.group / g_per_warp);
  const int gp = (g_per_warp + 1) & ~1;
  return (size_t)n_stages * 2 * kTile * row_pitch(a.row_bytes) + (size_t)warps * kTile * gp * sizeof(uint64_t);
}

template <int KVT, int QT, int G, int D, bool SP>
cudaError_t launch_d(const DecodeArgs &a0, cudaStream_t st) {
  DecodeArgs a = a0;
  // q8_0 rows: two stages (measured faster than three, e.g. 165 -> 151 us for
  // 96,256 cells with 94,208 in VRAM); 16-bit rows: as many as fit, up to three
  int n_stages = KVT == KVO_Q8_0 ? 2 : kMaxStages;
  while (n_stages > 1 && split_smem_bytes(a, G, n_stages) > (size_t)kSmemLimit) --n_stages;
  size_t smem = split_smem_bytes(a, G, n_stages);
  // one stage, one chunk per row: prefetch rows' query and running state
  const size_t pre = 2 * ((size_t)a.n_q_heads * D * 2 + (size_t)a.n_q_heads * (D + 2) * 4);
  a.pre_rows = SP && a.all_ring && a.fold_in_split && a.n_splits == 1 && n_stages == 1 &&
               a.n_q_heads % 2 == 0 && smem + pre <= (size_t)kSmemLimit;
  if (a.pre_rows) smem += pre;
  if (smem > (size_t)kSmemLimit) return cudaErrorInvalidConfiguration;
  auto k = decode_split_kernel<KVT, QT, G, D, SP>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (a.phase != 2) {
    const int64_t items = (a.item_hi < 0 ? (int64_t)a.batch * a.n_splits : a.item_hi) - a.item_lo;
    const int64_t cap = a.grid_cap > 0 && a.grid_cap < num_sms() ? a.grid_cap : num_sms();
    const int64_t grid = items < cap ? items : cap;
    if (grid > 0) k<<<(unsigned)grid, 32 * a.n_kv_heads * (a.group / G), smem, st>>>(a, n_stages);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.phase == 1) return cudaSuccess;
  // The combine is a programmatic dependent launch: it is set up while the
  // split kernel runs and starts as its CTAs exit, then waits on the device
  // (griddepcontrol.wait) for the whole grid, which hides the launch gap.
  // (A trigger at the split kernel's start slowed the multi-item decodes.)
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kCombineWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.n_splits <= kSmallCombineChunks) {
    const int64_t items = (int64_t)a.batch * a.n_q_heads;
    cfg.gridDim = dim3((unsigned)((items + kCombineWarps - 1) / kCombineWarps));
    return cudaLaunchKernelEx(&cfg, decode_combine_small_kernel<D>, a);
  }
  cfg.gridDim = dim3(a.n_q_heads, a.batch);
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, a);
}

}  // namespace dec
}  // namespace kvo
