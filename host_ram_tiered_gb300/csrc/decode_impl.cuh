// Tiered GQA decode attention: split-K flash-decoding over a cache whose
// cells [0, N) are in VRAM and [N, L) in pinned host memory (or a VRAM
// staging copy of them).  llama.cpp PR "tiered KV cache (--kv-vram-cells)":
// the arithmetic does not depend on where a cell lives, so a tiered cache
// gives output bit-identical to an all-VRAM one.
//
// One CTA = one fixed cell range (split) of one sequence, one warp per kv
// head (n_kv_heads warps).  A tile of 32 cell rows (all kv heads, 16-byte
// chunks, coalesced across the CTA) is copied into shared memory from
// whichever tier holds each cell, rows padded so that lane-per-row reads hit
// distinct banks.  Scores: lane c owns cell c of the tile and computes its
// G dot products against the warp's query heads, which sit in shared memory
// pre-scaled by scale*log2(e) (for q8_0 the block scale multiplies each
// 32-value partial; d * q is exact in fp32).  Online softmax in the log2
// domain with warp-wide max / sum (fixed butterflies).  P*V: lane l owns head
// dims [l*D/32, (l+1)*D/32) and walks the tile's cells in order with the
// weights broadcast from shared memory.  Each CTA writes an unnormalised
// partial (m, l, acc); a second kernel folds the splits of a head in a fixed
// order.  Instantiated per K/V dtype in decode_<dtype>.cu.
#pragma once
#include <cuda_fp16.h>
#include <math.h>

#include "kvo_internal.cuh"

namespace kvo {
namespace dec {


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

__device__ __forceinline__ float h2f(uint16_t b, int dt) {
  if (dt == KVO_BF16) return __uint_as_float((uint32_t)b << 16);
  return __half2float(__ushort_as_half(b));
}

// Four int8 values packed in a word -> four exact floats without the
// conversion pipe: x ^ 0x80 is x + 128 as an unsigned byte; placed in the low
// mantissa byte of 2^23 it reads as 2^23 + x + 128, and subtracting
// 2^23 + 128 leaves x (all steps exact in fp32).
__device__ __forceinline__ void i8x4_to_f32(uint32_t w, float *f) {
  const uint32_t u = w ^ 0x80808080u;
  f[0] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540)) - 8388736.f;
  f[1] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541)) - 8388736.f;
  f[2] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542)) - 8388736.f;
  f[3] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543)) - 8388736.f;
}

// Four int8 values at a 2-byte aligned shared-memory address.
__device__ __forceinline__ uint32_t ld_i8x4(const uint8_t *p) {
  return __byte_perm(*(const uint16_t *)p, *(const uint16_t *)(p + 2), 0x5410);
}

// Read this lane's DPL dims of kv head g from a cell row held in shared memory.
template <int KVT, int D>
__device__ __forceinline__ void lane_dims(const uint8_t *row, int g, int lane, float *x) {
  constexpr int DPL = D / 32;
  if constexpr (KVT == KVO_Q8_0) {
    constexpr int NB = D / 32;                       // blocks per head
    constexpr int LPB = 32 / DPL;                    // lanes per block
    const uint8_t *blk = row + (g * NB + lane / LPB) * 34;
    const float d = __half2float(__ushort_as_half(*(const uint16_t *)blk));
    const uint8_t *qs = blk + 2 + (lane % LPB) * DPL;  // 2-byte aligned
    float f[4];
    if constexpr (DPL == 4) i8x4_to_f32(ld_i8x4(qs), f);
    else i8x4_to_f32(*(const uint16_t *)qs, f);
#pragma unroll
    for (int i = 0; i < DPL; ++i) x[i] = d * f[i];
  } else {
    const uint16_t *h = (const uint16_t *)(row + g * D * 2) + lane * DPL;
    if constexpr (DPL == 4) {
      const uint2 u = *(const uint2 *)h;
      x[0] = h2f(u.x & 0xffff, KVT); x[1] = h2f(u.x >> 16, KVT);
      x[2] = h2f(u.y & 0xffff, KVT); x[3] = h2f(u.y >> 16, KVT);
    } else {
      const uint32_t u = *(const uint32_t *)h;
      x[0] = h2f(u & 0xffff, KVT); x[1] = h2f(u >> 16, KVT);
    }
  }
}

constexpr int kTile = 32;                             // cells per tile (one per lane)

// Shared-memory pitch of a cell row: 16 bytes of padding, so 16-byte rows
// stay aligned and lane-per-row reads spread over the banks.
template <int KVT>
__host__ __device__ constexpr int64_t row_pitch(int64_t rb) {
  return rb + 16;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Tile of cell rows [c0, c0 + n) of sequence b (K and V) that lies wholly in
// device memory: every 16-byte chunk is an asynchronous copy (cp.async,
// bypassing L1), all in flight at once; V rows n..kTile-1 are zero-filled.
template <int KVT>
__device__ __forceinline__ void load_tile_async(const DecodeArgs &a, int b, int64_t c0, int n,
                                                uint8_t *sk, uint8_t *sv) {
  const int64_t rb = a.row_bytes;
  const int64_t pitch = row_pitch<KVT>(rb);
  const int cpr = (int)(rb >> 4);
  const int total = kTile * cpr;
  for (int i = threadIdx.x; i < 2 * total; i += blockDim.x) {
    const bool is_v = i >= total;
    const int k = is_v ? i - total : i;
    const int r = k / cpr, ch = k - r * cpr;
    const int64_t j = c0 + (r < n ? r : 0);
    const uint8_t *src;
    if (j < a.n_vram) src = (is_v ? a.v_lo : a.k_lo) + (b * a.lo_seq_stride_rows + j) * rb;
    else src = (is_v ? a.v_hi : a.k_hi) + (b * a.hi_seq_stride_rows + (j - a.n_vram)) * rb;
    const uint32_t dst = smem_addr((is_v ? sv : sk) + r * pitch + ch * 16);
    const uint32_t bytes = r < n ? 16u : 0u;            // 0: zero-fill, nothing read
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst),
                 "l"((const int4 *)src + ch), "r"(bytes)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// Copy cell rows [c0, c0 + n) of sequence b (K and V) into shared memory;
// V rows n..kTile-1 are zeroed (their weights are 0 and must meet finite
// values).
template <int KVT>
__device__ __forceinline__ void load_tile(const DecodeArgs &a, int b, int64_t c0, int n,
                                          uint8_t *sk, uint8_t *sv) {
  const int64_t rb = a.row_bytes;
  const int64_t pitch = row_pitch<KVT>(rb);
  const int cpr = (int)(rb >> 4);                    // 16-byte chunks per row
  const int total = kTile * cpr;                     // per tensor, full tile
  const int nthr = blockDim.x;
  constexpr int kBatch = 8;
  for (int base = 0; base < 2 * total; base += kBatch * nthr) {
    int4 v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * nthr + (int)threadIdx.x;
      v[u] = make_int4(0, 0, 0, 0);
      if (i < 2 * total) {
        const bool is_v = i >= total;
        const int k = is_v ? i - total : i;
        const int r = k / cpr, ch = k - r * cpr;
        if (r < n) {
          const int64_t j = c0 + r;
          const uint8_t *src;
          if (j < a.n_vram) src = (is_v ? a.v_lo : a.k_lo) + (b * a.lo_seq_stride_rows + j) * rb;
          else src = (is_v ? a.v_hi : a.k_hi) + (b * a.hi_seq_stride_rows + (j - a.n_vram)) * rb;
          v[u] = *((const int4 *)src + ch);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * nthr + (int)threadIdx.x;
      if (i < 2 * total) {
        const bool is_v = i >= total;
        const int k = is_v ? i - total : i;
        const int r = k / cpr, ch = k - r * cpr;
        *(int4 *)((is_v ? sv : sk) + r * pitch + ch * 16) = v[u];
      }
    }
  }
}

// Dot products of one cell's kv head g (row in shared memory) with the G
// query heads (qs: [G][D] fp32, pre-scaled), into s[G].
template <int KVT, int G, int D>
__device__ __forceinline__ void cell_scores(const uint8_t *row, int g, const float *qs, float *s) {
#pragma unroll
  for (int h = 0; h < G; ++h) s[h] = 0.f;
  if constexpr (KVT == KVO_Q8_0) {
    constexpr int NB = D / 32;
#pragma unroll
    for (int bk = 0; bk < NB; ++bk) {
      const uint8_t *blk = row + (g * NB + bk) * 34;
      const float d = __half2float(__ushort_as_half(*(const uint16_t *)blk));
      float sb[G];
#pragma unroll
      for (int h = 0; h < G; ++h) sb[h] = 0.f;
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        float kf[4];
        i8x4_to_f32(ld_i8x4(blk + 2 + i), kf);
        const float k0 = kf[0], k1 = kf[1], k2 = kf[2], k3 = kf[3];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 q = *(const float4 *)(qs + h * D + bk * 32 + i);
          sb[h] = fmaf(q.x, k0, sb[h]);
          sb[h] = fmaf(q.y, k1, sb[h]);
          sb[h] = fmaf(q.z, k2, sb[h]);
          sb[h] = fmaf(q.w, k3, sb[h]);
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) s[h] = fmaf(d, sb[h], s[h]);
    }
  } else {
    const uint8_t *hrow = row + g * D * 2;
#pragma unroll 4
    for (int dc = 0; dc < D / 8; ++dc) {
      const uint4 u = *(const uint4 *)(hrow + dc * 16);
      float k[8];
      k[0] = h2f(u.x & 0xffff, KVT); k[1] = h2f(u.x >> 16, KVT);
      k[2] = h2f(u.y & 0xffff, KVT); k[3] = h2f(u.y >> 16, KVT);
      k[4] = h2f(u.z & 0xffff, KVT); k[5] = h2f(u.z >> 16, KVT);
      k[6] = h2f(u.w & 0xffff, KVT); k[7] = h2f(u.w >> 16, KVT);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float4 q0 = *(const float4 *)(qs + h * D + dc * 8);
        const float4 q1 = *(const float4 *)(qs + h * D + dc * 8 + 4);
        float t = s[h];
        t = fmaf(q0.x, k[0], t); t = fmaf(q0.y, k[1], t);
        t = fmaf(q0.z, k[2], t); t = fmaf(q0.w, k[3], t);
        t = fmaf(q1.x, k[4], t); t = fmaf(q1.y, k[5], t);
        t = fmaf(q1.z, k[6], t); t = fmaf(q1.w, k[7], t);
        s[h] = t;
      }
    }
  }
}

template <int KVT, int QT, int G, int D>
__global__ void __launch_bounds__(256)
decode_split_kernel(const DecodeArgs a) {
  constexpr int DPL = D / 32;
  extern __shared__ __align__(16) uint8_t smem[];
  const int split = blockIdx.x, b = blockIdx.y;
  const int g = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t ctx = a.ctx_len[b] < a.max_ctx ? a.ctx_len[b] : a.max_ctx;
  const int64_t cs = (int64_t)split * a.split_cells;
  const int64_t ce = cs + a.split_cells < ctx ? cs + a.split_cells : ctx;
  if (cs >= ce) return;                               // split beyond the context: never combined
  const int64_t pitch = row_pitch<KVT>(a.row_bytes);
  float *qs_all = (float *)smem;                                    // [Hq][D]
  float *ps_all = qs_all + (size_t)a.n_q_heads * D;                 // [Hkv][G][kTile]
  uint8_t *sk = (uint8_t *)(ps_all + (size_t)a.n_kv_heads * G * kTile);
  uint8_t *sv = sk + (size_t)kTile * pitch;
  float *qs = qs_all + (size_t)g * G * D;
  float *ps = ps_all + (size_t)g * G * kTile;
  // Cells wholly in device memory are fetched with asynchronous copies;
  // host-mapped cells with plain 16-byte loads.  Same bytes either way.
  const bool dev_split = ce <= a.n_vram || a.hi_device;

  // query heads of this sequence, pre-scaled, into shared memory
  for (int i = threadIdx.x; i < a.n_q_heads * D; i += blockDim.x)
    qs_all[i] = h2f(((const uint16_t *)a.q)[(size_t)b * a.n_q_heads * D + i], QT) * a.scale_log2;

  float acc[G][DPL], m[G], l[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[h][i] = 0.f;
    m[h] = -INFINITY;
    l[h] = 0.f;
  }

  for (int64_t t0 = cs; t0 < ce; t0 += kTile) {
    const int n = ce - t0 < kTile ? (int)(ce - t0) : kTile;
    __syncthreads();                                  // previous tile fully consumed
    if (dev_split) load_tile_async<KVT>(a, b, t0, n, sk, sv);
    else load_tile<KVT>(a, b, t0, n, sk, sv);
    __syncthreads();
    float sc[G];
    cell_scores<KVT, G, D>(sk + (size_t)lane * pitch, g, qs, sc);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float sv_h = lane < n ? sc[h] : -INFINITY;
      const float m_new = fmaxf(m[h], warp_max(sv_h));
      const float alpha = exp2f(m[h] - m_new);
      const float p = lane < n ? exp2f(sv_h - m_new) : 0.f;
      l[h] = l[h] * alpha + warp_sum(p);
#pragma unroll
      for (int i = 0; i < DPL; ++i) acc[h][i] *= alpha;
      m[h] = m_new;
      ps[h * kTile + lane] = p;
    }
    __syncwarp();
    for (int c = 0; c < kTile; c += 4) {
      if (c >= n) break;
      float4 p4[G];
#pragma unroll
      for (int h = 0; h < G; ++h) p4[h] = *(const float4 *)(ps + h * kTile + c);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float vd[DPL];
        lane_dims<KVT, D>(sv + (size_t)(c + cc) * pitch, g, lane, vd);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float pc = cc == 0 ? p4[h].x : cc == 1 ? p4[h].y : cc == 2 ? p4[h].z : p4[h].w;
#pragma unroll
          for (int i = 0; i < DPL; ++i) acc[h][i] = fmaf(pc, vd[i], acc[h][i]);
        }
      }
    }
  }

#pragma unroll
  for (int h = 0; h < G; ++h) {
    const int qh = g * G + h;
    const size_t pi = ((size_t)b * a.n_splits + split) * a.n_q_heads + qh;
    float *pa = a.part_acc + pi * D + lane * DPL;
#pragma unroll
    for (int i = 0; i < DPL; ++i) pa[i] = acc[h][i];
    if (lane == 0) {
      a.part_ml[pi * 2] = m[h];
      a.part_ml[pi * 2 + 1] = l[h];
    }
  }
}

// Fold the splits of one (sequence, q head): weights 2^(m_s - M) with M the
// maximum over splits, out = acc / max(l, 1e-30).  Warp w sums the splits
// s = w, w + 8, w + 16, ... in ascending order and the 8 warp sums are added
// in warp order: a fixed reduction tree, so the result depends on the
// partials only (never on timing, the tier split or staging).
constexpr int kCombineWarps = 8;

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
decode_combine_kernel(const DecodeArgs a) {
  constexpr int DPL = D / 32;
  __shared__ float red[kCombineWarps][D];
  __shared__ float red_l[kCombineWarps];
  __shared__ float red_m[kCombineWarps];
  const int h = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t ctx = a.ctx_len[b] < a.max_ctx ? a.ctx_len[b] : a.max_ctx;
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
    const float w = exp2f(a.part_ml[pi * 2] - M);
    l = fmaf(w, a.part_ml[pi * 2 + 1], l);
    const float *pa = a.part_acc + pi * D + lane * DPL;
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = fmaf(w, pa[i], acc[i]);
  }
#pragma unroll
  for (int i = 0; i < DPL; ++i) red[warp][lane * DPL + i] = acc[i];
  if (lane == 0) red_l[warp] = l;
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += kCombineWarps * 32) {
    float sl = 0.f, sa = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) {
      sl += red_l[w];
      sa += red[w][d];
    }
    a.out[((size_t)b * a.n_q_heads + h) * D + d] = sa / fmaxf(sl, 1e-30f);
  }
}

template <int KVT, int QT, int G, int D>
cudaError_t launch_d(const DecodeArgs &a, cudaStream_t st) {
  const size_t smem = (size_t)a.n_q_heads * D * 4 + (size_t)a.n_kv_heads * G * kTile * 4 +
                      (size_t)2 * kTile * row_pitch<KVT>(a.row_bytes);
  auto k = decode_split_kernel<KVT, QT, G, D>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_splits, a.batch);
  k<<<grid, 32 * a.n_kv_heads, smem, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<D><<<dim3(a.n_q_heads, a.batch), kCombineWarps * 32, 0, st>>>(a);
  return cudaGetLastError();
}

template <int KVT, int QT, int G>
cudaError_t launch_g(const DecodeArgs &a, cudaStream_t st) {
  if (a.head_dim == 128) return launch_d<KVT, QT, G, 128>(a, st);
  return launch_d<KVT, QT, G, 64>(a, st);
}

template <int KVT, int QT>
cudaError_t launch_q(const DecodeArgs &a, cudaStream_t st) {
  switch (a.group) {
    case 1: return launch_g<KVT, QT, 1>(a, st);
    case 2: return launch_g<KVT, QT, 2>(a, st);
    case 3: return launch_g<KVT, QT, 3>(a, st);
    case 4: return launch_g<KVT, QT, 4>(a, st);
    case 5: return launch_g<KVT, QT, 5>(a, st);
    case 6: return launch_g<KVT, QT, 6>(a, st);
    case 7: return launch_g<KVT, QT, 7>(a, st);
    default: return launch_g<KVT, QT, 8>(a, st);
  }
}

template <int KVT>
cudaError_t launch_kv(const DecodeArgs &a, cudaStream_t st) {
  if (a.q_dtype == KVO_BF16) return launch_q<KVT, KVO_BF16>(a, st);
  return launch_q<KVT, KVO_F16>(a, st);
}

}  // namespace dec
}  // namespace kvo
