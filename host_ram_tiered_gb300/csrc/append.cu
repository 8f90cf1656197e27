// Write path of the tiered cache: new tokens' K/V rows become cells
// [pos0, pos0 + n_new) of one sequence, each in the tier that holds it (VRAM
// head for cells < N, pinned host tail row j - N beyond), in the cache dtype.
// fp16/bf16 caches take a plain copy; q8_0 caches are quantised on the way
// in, one CTA per (token, K|V) row, lane i holding value i of each 32-value
// block: amax = max|x| (warp butterfly, exact), d = amax / 127,
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

// q8_0: one CTA per (token, K|V) cell row, warp w quantising the blocks of
// heads w, w + 8, ... into a shared row buffer (lane i = value i of a block;
// lanes 0..16 store the block's 17 halfwords).  The finished row then leaves
// with 16-byte stores when the row and the tier base allow it, so the host
// tail sees whole-line writes.
constexpr int kMaxRowBytes = 8 * (256 / 32) * 34;           // 8 heads x 256 dims

__global__ void __launch_bounds__(kThreads) append_q8_0_kernel(const AppendArgs a) {
  __shared__ __align__(16) uint8_t buf[kMaxRowBytes];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int nb = a.head_dim / 32;
  const int64_t rb = a.row_bytes;
  for (int64_t w = blockIdx.x; w < 2 * a.n_new; w += gridDim.x) {
    const bool is_v = w >= a.n_new;
    const int64_t t = is_v ? w - a.n_new : w;
    const uint16_t *src = (const uint16_t *)(is_v ? a.v_new : a.k_new) + t * a.n_kv_heads * a.head_dim;
    uint8_t *row = cell_row(a, is_v, a.pos0 + t);
    const bool staged = rb <= kMaxRowBytes && (rb & 15) == 0 && ((uintptr_t)row & 15) == 0;
    for (int hb = wib; hb < a.n_kv_heads * nb; hb += kThreads / 32) {   // block hb = head*nb + b
      const float x = to_f32(src[hb * 32 + lane], a.src_dtype);
      float amax = fabsf(x);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float d = amax / 127.0f;
      const float id = d != 0.0f ? 1.0f / d : 0.0f;
      const int q = (int)roundf(x * id);
      // halfword k of the 34-byte block: k = 0 holds d, k >= 1 holds q[2k-2], q[2k-1]
      const int q_prev = __shfl_sync(0xffffffffu, q, (2 * lane - 2) & 31);
      const int q_next = __shfl_sync(0xffffffffu, q, (2 * lane - 1) & 31);
      uint16_t *blk = (uint16_t *)((staged ? buf : row) + hb * 34);
      if (lane == 0) {
        blk[0] = __half_as_ushort(__float2half_rn(d));
      } else if (lane < 17) {
        blk[lane] = (uint16_t)((uint8_t)(int8_t)q_prev | ((uint16_t)(uint8_t)(int8_t)q_next << 8));
      }
    }
    if (staged) {
      __syncthreads();
      for (int64_t c = threadIdx.x; c < (rb >> 4); c += kThreads) ((int4 *)row)[c] = ((const int4 *)buf)[c];
    }
    __syncthreads();                                  // buffer free for the next row
  }
}

}  // namespace

int launch_append(const AppendArgs &a, cudaStream_t st) {
  const int64_t rows = 2 * a.n_new;                    // (token, K|V) rows
  const int64_t cap = (int64_t)num_sms() * 8;
  if (a.kv_dtype == KVO_Q8_0) {
    const int64_t grid = rows < cap ? rows : cap;       // one CTA per row
    append_q8_0_kernel<<<(unsigned)grid, kThreads, 0, st>>>(a);
  } else {
    int64_t grid = (rows + (kThreads / 32) - 1) / (kThreads / 32);   // one warp per row
    if (grid > cap) grid = cap;
    append_copy_kernel<<<(unsigned)grid, kThreads, 0, st>>>(a);
  }
  return cuda_status(cudaGetLastError(), "append kernel launch");
}

}  // namespace kvo
