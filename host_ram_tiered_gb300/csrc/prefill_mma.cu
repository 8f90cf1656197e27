// Tiered causal chunked-prefill attention, one launch = (row block) x (cell
// range): QK^T and PV on the tensor cores with warp-level mma.sync
// (m16n8k16, bf16/f16 in, fp32 accumulate), online softmax in fp32, and the
// running (m, l, acc) of earlier launches folded in (ExLlamaV3
// qsa-kv-offload patch, the fold of a bucket's partial into the running
// softmax: m' = max(m, m_b), rescale both sides by 2^(m - m')).
//
// GQA packing: the 64 MMA rows of a CTA are 64/G query positions x the G
// query heads of one kv head, so one K/V tile serves the whole group.
// Cells j < n_vram come from k_lo/v_lo, cells j >= n_vram from
// k_hi/v_hi (row j - hi_origin): the VRAM head, the host tail (direct) or an
// arena bucket (staged).
#include <cuda_fp16.h>
#include <math.h>

#include "kvo_internal.cuh"

namespace kvo {

namespace {

constexpr int BM = 64;        // MMA rows per CTA (4 warps x 16)
constexpr int BN = 64;        // cells per K/V tile
constexpr int HD = 128;       // head_dim
constexpr int kThreads = 128;
constexpr int kRowBytes = HD * 2;                // 256 B per head row
constexpr int kTileBytes = BN * kRowBytes;       // 16 KiB

// Swizzled byte offset of 16-byte chunk c of row r in a [rows][256 B] tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * kRowBytes + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <int DT>
__device__ __forceinline__ void mma16816(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
  if constexpr (DT == KVO_BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

template <int DT>
__device__ __forceinline__ float2 unpack2(uint32_t u) {
  if constexpr (DT == KVO_BF16) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
  } else {
    __half2 h = *reinterpret_cast<__half2 *>(&u);
    return __half22float2(h);
  }
}

template <int DT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  if constexpr (DT == KVO_BF16) {
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  }
  return r;
}

// 16-byte chunk i (0..1023) of the K or V tile: row i / 16, chunk i % 16.
__device__ __forceinline__ const int4 *tile_src(const PrefillArgs &a, bool is_v, int64_t j, int g,
                                                int ch) {
  const uint8_t *base;
  if (j < a.n_vram) base = (is_v ? a.v_lo : a.k_lo) + j * a.row_bytes;
  else base = (is_v ? a.v_hi : a.k_hi) + (j - a.hi_origin) * a.row_bytes;
  return (const int4 *)(base + g * kRowBytes) + ch;
}

template <int DT, int G>
__global__ void __launch_bounds__(kThreads)
prefill_mma_kernel(const PrefillArgs a) {
  constexpr int PB = BM / G;                         // query positions per CTA
  __shared__ __align__(128) uint8_t sq[BM * kRowBytes];
  __shared__ __align__(128) uint8_t sk[kTileBytes];
  __shared__ __align__(128) uint8_t sv[kTileBytes];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y;
  const int i0 = blockIdx.x * PB;                    // first query row of the CTA (launch-local)
  const int n_pos = a.rows - i0 < PB ? a.rows - i0 : PB;

  // ---- Q tile: MMA row r = position (r / G) x head (g*G + r % G)
  for (int i = tid; i < BM * 16; i += kThreads) {
    const int r = i >> 4, ch = i & 15;
    const int pi = r / G, hh = r % G;
    int4 v = make_int4(0, 0, 0, 0);
    if (pi < n_pos)
      v = *((const int4 *)(a.q + ((size_t)(i0 + pi) * a.n_q_heads + g * G + hh) * HD) + ch);
    *(int4 *)(sq + swz(r, ch)) = v;
  }

  // Rows owned by this thread: r_lo = warp*16 + lane/4 and r_hi = r_lo + 8.
  const int r_lo = warp * 16 + (lane >> 2), r_hi = r_lo + 8;
  const int pi_lo = r_lo / G, pi_hi = r_hi / G;
  const bool ok_lo = pi_lo < n_pos, ok_hi = pi_hi < n_pos;
  const int64_t pos_lo = a.pos0 + i0 + pi_lo, pos_hi = a.pos0 + i0 + pi_hi;
  const size_t row_lo = (size_t)(i0 + pi_lo) * a.n_q_heads + g * G + r_lo % G;   // (row, head) index
  const size_t row_hi = (size_t)(i0 + pi_hi) * a.n_q_heads + g * G + r_hi % G;

  float o[16][4];
  float m_lo, m_hi, l_lo, l_hi;
  if (a.init) {
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    m_lo = m_hi = -INFINITY;
    l_lo = l_hi = 0.f;
  } else {
    const int cc = (lane & 3) * 2;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      float2 x = ok_lo ? *(const float2 *)(a.acc + row_lo * HD + n * 8 + cc) : make_float2(0.f, 0.f);
      float2 y = ok_hi ? *(const float2 *)(a.acc + row_hi * HD + n * 8 + cc) : make_float2(0.f, 0.f);
      o[n][0] = x.x; o[n][1] = x.y; o[n][2] = y.x; o[n][3] = y.y;
    }
    m_lo = ok_lo ? a.ml[row_lo * 2] : -INFINITY;
    l_lo = ok_lo ? a.ml[row_lo * 2 + 1] : 0.f;
    m_hi = ok_hi ? a.ml[row_hi * 2] : -INFINITY;
    l_hi = ok_hi ? a.ml[row_hi * 2 + 1] : 0.f;
  }

  __syncthreads();
  // Q fragments for the whole loop (8 k-steps of 16 dims).
  uint32_t qf[8][4];
  {
    const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int ch = ks * 2 + (lane >> 4);
      ldsm_x4(smem_u32(sq + swz(r, ch)), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
    }
  }

  // Cells this CTA can see end at its last position.
  const int64_t cta_last_pos = a.pos0 + i0 + (n_pos > 0 ? n_pos - 1 : 0);
  int64_t c_end = a.c1 < cta_last_pos + 1 ? a.c1 : cta_last_pos + 1;
  if (n_pos <= 0) c_end = a.c0;
  const int64_t cta_first_pos = a.pos0 + i0;

  for (int64_t t0 = a.c0; t0 < c_end; t0 += BN) {
    __syncthreads();                                  // previous tile consumed
    {
      int4 v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = u * kThreads + tid;             // 0..2047: K chunks then V chunks
        const bool is_v = i >= 1024;
        const int k = i & 1023, r = k >> 4, ch = k & 15;
        const int64_t j = t0 + r;
        v[u] = j < c_end ? *tile_src(a, is_v, j, g, ch) : make_int4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = u * kThreads + tid;
        const bool is_v = i >= 1024;
        const int k = i & 1023, r = k >> 4, ch = k & 15;
        *(int4 *)((is_v ? sv : sk) + swz(r, ch)) = v[u];
      }
    }
    __syncthreads();

    // ---- S = Q K^T (16 x 64 per warp)
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {               // pairs of 8-cell n-tiles
        uint32_t b0, b1, b2, b3;
        const int r = np * 16 + (lane & 7) + (lane >> 4) * 8;
        const int ch = ks * 2 + ((lane >> 3) & 1);
        ldsm_x4(smem_u32(sk + swz(r, ch)), b0, b1, b2, b3);
        mma16816<DT>(s[np * 2], qf[ks], b0, b1);
        mma16816<DT>(s[np * 2 + 1], qf[ks], b2, b3);
      }
    }

    // ---- scale, mask, online softmax (log2 domain)
    const bool need_mask = (t0 + BN > c_end) || (t0 + BN - 1 > cta_first_pos);
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int64_t j = t0 + n * 8 + (lane & 3) * 2 + e;
        float x0 = s[n][e] * a.scale_log2, x1 = s[n][2 + e] * a.scale_log2;
        if (need_mask) {
          if (!ok_lo || j >= c_end || j > pos_lo) x0 = -INFINITY;
          if (!ok_hi || j >= c_end || j > pos_hi) x1 = -INFINITY;
        }
        s[n][e] = x0; s[n][2 + e] = x1;
        mx_lo = fmaxf(mx_lo, x0); mx_hi = fmaxf(mx_hi, x1);
      }
    }
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float ref_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
    const float ref_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
    const float al_lo = exp2f(m_lo - ref_lo), al_hi = exp2f(m_hi - ref_hi);
    float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      s[n][0] = exp2f(s[n][0] - ref_lo); s[n][1] = exp2f(s[n][1] - ref_lo);
      s[n][2] = exp2f(s[n][2] - ref_hi); s[n][3] = exp2f(s[n][3] - ref_hi);
      sum_lo += s[n][0] + s[n][1];
      sum_hi += s[n][2] + s[n][3];
    }
    sum_lo += __shfl_xor_sync(0xffffffffu, sum_lo, 1);
    sum_lo += __shfl_xor_sync(0xffffffffu, sum_lo, 2);
    sum_hi += __shfl_xor_sync(0xffffffffu, sum_hi, 1);
    sum_hi += __shfl_xor_sync(0xffffffffu, sum_hi, 2);
    l_lo = l_lo * al_lo + sum_lo;
    l_hi = l_hi * al_hi + sum_hi;
    m_lo = mn_lo; m_hi = mn_hi;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      o[n][0] *= al_lo; o[n][1] *= al_lo;
      o[n][2] *= al_hi; o[n][3] *= al_hi;
    }

    // ---- O += P V  (P as A fragments straight from the S accumulators).
    // P is carried as a pair hi + lo of the input type (lo = the rounding
    // residual of hi), so the product keeps ~16 bits of P instead of 8.
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {                  // 16 cells per k-step
      uint32_t pa[4], pl[4];
      pa[0] = pack2<DT>(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack2<DT>(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack2<DT>(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack2<DT>(s[2 * kk + 1][2], s[2 * kk + 1][3]);
      {
        float2 h;
        h = unpack2<DT>(pa[0]); pl[0] = pack2<DT>(s[2 * kk][0] - h.x, s[2 * kk][1] - h.y);
        h = unpack2<DT>(pa[1]); pl[1] = pack2<DT>(s[2 * kk][2] - h.x, s[2 * kk][3] - h.y);
        h = unpack2<DT>(pa[2]); pl[2] = pack2<DT>(s[2 * kk + 1][0] - h.x, s[2 * kk + 1][1] - h.y);
        h = unpack2<DT>(pa[3]); pl[3] = pack2<DT>(s[2 * kk + 1][2] - h.x, s[2 * kk + 1][3] - h.y);
      }
#pragma unroll
      for (int np = 0; np < 8; ++np) {               // pairs of 8-dim n-tiles
        uint32_t b0, b1, b2, b3;
        const int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int ch = np * 2 + (lane >> 4);
        ldsm_x4_t(smem_u32(sv + swz(r, ch)), b0, b1, b2, b3);
        mma16816<DT>(o[np * 2], pa, b0, b1);
        mma16816<DT>(o[np * 2 + 1], pa, b2, b3);
        mma16816<DT>(o[np * 2], pl, b0, b1);
        mma16816<DT>(o[np * 2 + 1], pl, b2, b3);
      }
    }
  }

  // ---- write back: running state, or the normalised output
  const int cc = (lane & 3) * 2;
  if (a.finalize) {
    const float inv_lo = 1.f / fmaxf(l_lo, 1e-30f), inv_hi = 1.f / fmaxf(l_hi, 1e-30f);
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      if (ok_lo) *(float2 *)(a.acc + row_lo * HD + n * 8 + cc) = make_float2(o[n][0] * inv_lo, o[n][1] * inv_lo);
      if (ok_hi) *(float2 *)(a.acc + row_hi * HD + n * 8 + cc) = make_float2(o[n][2] * inv_hi, o[n][3] * inv_hi);
    }
  } else {
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      if (ok_lo) *(float2 *)(a.acc + row_lo * HD + n * 8 + cc) = make_float2(o[n][0], o[n][1]);
      if (ok_hi) *(float2 *)(a.acc + row_hi * HD + n * 8 + cc) = make_float2(o[n][2], o[n][3]);
    }
    if ((lane & 3) == 0) {
      if (ok_lo) { a.ml[row_lo * 2] = m_lo; a.ml[row_lo * 2 + 1] = l_lo; }
      if (ok_hi) { a.ml[row_hi * 2] = m_hi; a.ml[row_hi * 2 + 1] = l_hi; }
    }
  }
}

template <int DT, int G>
cudaError_t launch_g(const PrefillArgs &a, cudaStream_t st) {
  constexpr int PB = BM / G;
  dim3 grid((a.rows + PB - 1) / PB, a.n_kv_heads);
  prefill_mma_kernel<DT, G><<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

template <int DT>
cudaError_t launch_dt(const PrefillArgs &a, cudaStream_t st) {
  switch (a.group) {
    case 1: return launch_g<DT, 1>(a, st);
    case 2: return launch_g<DT, 2>(a, st);
    case 4: return launch_g<DT, 4>(a, st);
    default: return launch_g<DT, 8>(a, st);
  }
}

}  // namespace

int launch_prefill(const PrefillArgs &a, cudaStream_t st) {
  cudaError_t e = a.dtype == KVO_BF16 ? launch_dt<KVO_BF16>(a, st) : launch_dt<KVO_F16>(a, st);
  return cuda_status(e, "prefill kernel launch");
}

}  // namespace kvo
