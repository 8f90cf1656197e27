// Write path of the tiered cache: new tokens' K/V rows become cells
// [pos0, pos0 + n_new) of one sequence, each in the tier that holds it (VRAM
// head for cells < N, pinned host tail row j - N beyond), in the cache dtype.
// fp16/bf16 caches take a plain copy; q8_0 caches are quantised on the way
// in, one warp per (token, K|V) row, lane i holding 32-value blocks i and
// i + 32: amax = max|x| (exact), d = amax / 127,
// q = round-half-away-from-zero(x * (1/d)), all in fp32, d stored as fp16.
#include <cuda_fp16.h>

#include "kvo_internal.cuh"

namespace kvo {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float to_f32(uint16_t b, int dt) {
  if (dt == KVO_BF16) return __uint_as_float((uint32_t)b << 16);
  return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ uint8_t *cell_row(const AppendArgs &a, bool is_v, int64_t j) {
  if (j < a.n_vram) return (is_v ? a.v_lo : a.k_lo) + j * a.row_bytes;
  return (is_v ? a.v_hi : a.k_hi) + (j - a.n_vram) * a.row_bytes;
}

// fp16/bf16: one warp per (token, K|V) row copy, 16-byte vectors.
__global__ void __launch_bounds__(kThreads) append_copy_kernel(const AppendArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * kThreads) >> 5;
  const int64_t chunks = a.row_bytes >> 4;
  for (int64_t w = warp; w < 2 * a.n_new; w += n_warps) {
    const bool is_v = w >= a.n_new;
    const int64_t t = is_v ? w - a.n_new : w;
    const int4 *src = (const int4 *)((is_v ? a.v_new : a.k_new) + t * a.row_bytes);
    int4 *dst = (int4 *)cell_row(a, is_v, a.pos0 + t);
    for (int64_t c = lane; c < chunks; c += 32) dst[c] = src[c];
  }
}

// q8_0: one warp per (token, K|V) cell row, lane i quantising blocks i and
// i + 32 of the row (a row has at most 64): its 32 source values arrive in
// four 16-byte loads and their amax is taken in registers.  The 34-byte
// blocks are assembled in the warp's shared row buffer; the finished row
// leaves with 16-byte stores when the row and the tier base allow it (so the
// host tail sees whole-line writes), else with halfword stores.
constexpr int kMaxBlocks = 8 * (256 / 32);                  // 8 heads x 256 dims
constexpr int kMaxRowBytes = kMaxBlocks * 34;

__global__ void __launch_bounds__(kThreads) append_q8_0_kernel(const AppendArgs a) {
  __shared__ __align__(16) uint8_t buf[kThreads / 32][kMaxRowBytes];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * kThreads) >> 5;
  const int nblk = (int)(a.n_kv_heads * (a.head_dim / 32));
  const int64_t rb = a.row_bytes;
  uint8_t *wbuf = buf[wib];
  for (int64_t w = warp; w < 2 * a.n_new; w += n_warps) {
    const bool is_v = w >= a.n_new;
    const int64_t t = is_v ? w - a.n_new : w;
    const uint4 *src = (const uint4 *)((is_v ? a.v_new : a.k_new) + t * nblk * 64);
    uint8_t *row = cell_row(a, is_v, a.pos0 + t);
    for (int hb = lane; hb < nblk; hb += 32) {
      uint4 u[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) u[k] = src[hb * 4 + k];
      float x[32];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t wv[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          x[8 * k + 2 * e] = to_f32((uint16_t)(wv[e] & 0xffffu), a.src_dtype);
          x[8 * k + 2 * e + 1] = to_f32((uint16_t)(wv[e] >> 16), a.src_dtype);
        }
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
      const float d = amax / 127.0f;
      const float id = d != 0.0f ? 1.0f / d : 0.0f;
      // halfword k of the 34-byte block: k = 0 holds d, k >= 1 holds q[2k-2], q[2k-1]
      uint16_t *blk = (uint16_t *)(wbuf + hb * 34);
      blk[0] = __half_as_ushort(__float2half_rn(d));
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int q0 = (int)roundf(x[2 * k] * id), q1 = (int)roundf(x[2 * k + 1] * id);
        blk[1 + k] = (uint16_t)((uint8_t)(int8_t)q0 | ((uint16_t)(uint8_t)(int8_t)q1 << 8));
      }
    }
    __syncwarp();
    if (rb <= kMaxRowBytes && (rb & 15) == 0 && ((uintptr_t)row & 15) == 0) {
      for (int64_t c = lane; c < (rb >> 4); c += 32) ((int4 *)row)[c] = ((const int4 *)wbuf)[c];
    } else {
      for (int64_t c = lane; c < (rb >> 1); c += 32) ((uint16_t *)row)[c] = ((const uint16_t *)wbuf)[c];
    }
    __syncwarp();                                     // buffer free for the next row
  }
}

}  // namespace

int launch_append(const AppendArgs &a, cudaStream_t st) {
  const int64_t rows = 2 * a.n_new;                    // (token, K|V) rows
  const int64_t cap = (int64_t)num_sms() * 8;
  if (a.kv_dtype == KVO_Q8_0) {
    int64_t grid = (rows + (kThreads / 32) - 1) / (kThreads / 32);   // one warp per row
    if (grid > cap) grid = cap;
    append_q8_0_kernel<<<(unsigned)grid, kThreads, 0, st>>>(a);
  } else {
    int64_t grid = (rows + (kThreads / 32) - 1) / (kThreads / 32);   // one warp per row
    if (grid > cap) grid = cap;
    append_copy_kernel<<<(unsigned)grid, kThreads, 0, st>>>(a);
  }
  return cuda_status(cudaGetLastError(), "append kernel launch");
}

}  // namespace kvo
