// Batched block swap and top-k block gather: SM copy kernels that read and
// write pinned host memory through the device mapping (16-byte vectors,
// coalesced across a warp, several loads in flight per lane).
//
// On GB300 the host link (NVLink-C2C) is saturated by SM loads from about
// one CTA of 256 threads per SM, at the same bandwidth as the copy engine,
// while a copy-engine call costs ~2.7 us to issue: for page-sized copies a
// warp-per-descriptor kernel is the fast path.
#include "kvo_internal.cuh"

namespace kvo {

namespace {

constexpr int kSwapThreads = 256;
constexpr int kUnroll = 4;

// Copy `bytes` from s to d with one warp.  16-byte vectors when both
// addresses and the size allow, else 8-, 4- or 1-byte units.
__device__ __forceinline__ void warp_copy(const char *s, char *d, int64_t bytes, int lane) {
  const uintptr_t mis = ((uintptr_t)s | (uintptr_t)d | (uintptr_t)bytes);
  if ((mis & 15) == 0) {
    const int4 *s4 = (const int4 *)s;
    int4 *d4 = (int4 *)d;
    const int64_t n = bytes >> 4;
    int64_t i = lane;
    for (; i + (kUnroll - 1) * 32 < n; i += kUnroll * 32) {
      int4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) v[u] = s4[i + u * 32];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) d4[i + u * 32] = v[u];
    }
    for (; i < n; i += 32) d4[i] = s4[i];
  } else if ((mis & 7) == 0) {
    const int64_t n = bytes >> 3;
    for (int64_t i = lane; i < n; i += 32) ((int2 *)d)[i] = ((const int2 *)s)[i];
  } else if ((mis & 3) == 0) {
    const int64_t n = bytes >> 2;
    for (int64_t i = lane; i < n; i += 32) ((int *)d)[i] = ((const int *)s)[i];
  } else {
    for (int64_t i = lane; i < bytes; i += 32) d[i] = s[i];
  }
}

// Long batches: a warp takes `per_warp` (1..32) consecutive descriptors:
// lane i loads descriptor i (coalesced reads through the mapping instead of
// dependent ones), then the warp copies them one after another, broadcasting
// each by shuffle.  Short batches (parts > 1): each descriptor is cut into
// `parts` pieces of a whole number of 512-byte units and a warp copies one
// piece, so that a few large copies still spread over every SM.  The pieces
// start at multiples of 512 bytes from the descriptor's start, which keeps
// each piece's alignment class (and so its vector width) that of the whole.
constexpr int64_t kPartUnit = 512;

__global__ void __launch_bounds__(kSwapThreads)
swap_kernel(const int64_t *__restrict__ src, const int64_t *__restrict__ dst,
            const int64_t *__restrict__ sizes, int64_t n, int per_warp, int parts) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kSwapThreads + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * kSwapThreads) >> 5;
  if (parts > 1) {
    for (int64_t item = warp; item < n * parts; item += n_warps) {
      const int64_t i = item / parts;
      const int64_t p = item - i * parts;
      const int64_t z = sizes[i];            // every lane reads the same word: one request
      if (z <= 0) continue;
      int64_t piece = (z + parts - 1) / parts;
      piece = (piece + kPartUnit - 1) / kPartUnit * kPartUnit;
      const int64_t b0 = p * piece;
      if (b0 >= z) continue;
      const int64_t b1 = b0 + piece < z ? b0 + piece : z;
      warp_copy((const char *)(uintptr_t)src[i] + b0, (char *)(uintptr_t)dst[i] + b0, b1 - b0, lane);
    }
    return;
  }
  for (int64_t base = warp * per_warp; base < n; base += n_warps * per_warp) {
    const int64_t i = base + lane;
    int64_t s = 0, d = 0, z = 0;
    if (lane < per_warp && i < n) {
      s = src[i];
      d = dst[i];
      z = sizes[i];
    }
    const int cnt = n - base < per_warp ? (int)(n - base) : per_warp;
    for (int k = 0; k < cnt; ++k) {
      const int64_t zk = __shfl_sync(0xffffffffu, z, k);
      const int64_t sk = __shfl_sync(0xffffffffu, s, k);
      const int64_t dk = __shfl_sync(0xffffffffu, d, k);
      if (zk > 0) warp_copy((const char *)(uintptr_t)sk, (char *)(uintptr_t)dk, zk, lane);
    }
  }
}

// Gather: one warp per (plane, seq, kv head, rank) block of block_tokens
// token rows of head_bytes each; source and destination rows are strided by
// n_kv_heads * head_bytes.  Index order of work items: rank fastest, so
// neighbouring warps read neighbouring selections of one (seq, head).
__global__ void __launch_bounds__(kSwapThreads)
gather_kernel(const char *__restrict__ k_plane, const char *__restrict__ v_plane, int64_t n_seq,
              int64_t seq_stride_tokens, int64_t n_kv_heads, int64_t head_bytes,
              int64_t block_tokens, const int32_t *__restrict__ sel, int64_t n_sel,
              char *__restrict__ k_out, char *__restrict__ v_out, uint32_t *err) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kSwapThreads + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * kSwapThreads) >> 5;
  const int64_t per_plane = n_seq * n_kv_heads * n_sel;
  const int64_t n_blocks_plane = seq_stride_tokens / block_tokens;
  const int64_t row_stride = n_kv_heads * head_bytes;        // bytes between token rows
  const int64_t chunks_per_row = head_bytes >> 4;
  const int64_t chunks = block_tokens * chunks_per_row;
  const int64_t out_tokens = n_sel * block_tokens;
  for (int64_t item = warp; item < 2 * per_plane; item += n_warps) {
    const bool is_v = item >= per_plane;
    const int64_t w = is_v ? item - per_plane : item;       // (s, h, r), r fastest
    const int64_t r = w % n_sel;
    const int64_t sh = w / n_sel;
    const int64_t h = sh % n_kv_heads;
    const int64_t s = sh / n_kv_heads;
    const int64_t blk = sel[w];
    if (blk < 0 || blk >= n_blocks_plane) {
      if (lane == 0) atomicOr(err, (uint32_t)kErrGatherSel);
      continue;
    }
    const char *src = (is_v ? v_plane : k_plane) +
                      ((s * seq_stride_tokens + blk * block_tokens) * n_kv_heads + h) * head_bytes;
    char *dst = (is_v ? v_out : k_out) +
                ((s * out_tokens + r * block_tokens) * n_kv_heads + h) * head_bytes;
    int64_t c = lane;
    for (; c + (kUnroll - 1) * 32 < chunks; c += kUnroll * 32) {
      int4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t cc = c + u * 32;
        v[u] = *((const int4 *)(src + (cc / chunks_per_row) * row_stride) + cc % chunks_per_row);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t cc = c + u * 32;
        *((int4 *)(dst + (cc / chunks_per_row) * row_stride) + cc % chunks_per_row) = v[u];
      }
    }
    for (; c < chunks; c += 32)
      *((int4 *)(dst + (c / chunks_per_row) * row_stride) + c % chunks_per_row) =
          *((const int4 *)(src + (c / chunks_per_row) * row_stride) + c % chunks_per_row);
  }
}

__device__ uint32_t g_device_errors;

}  // namespace

uint32_t *device_error_word() {
  static uint32_t *cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cached[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_errors) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    cached[dev] = (uint32_t *)p;
  }
  return cached[dev];
}

cudaError_t launch_swap_sm(const int64_t *src, const int64_t *dst, const int64_t *sizes, int64_t n,
                           int64_t max_size, cudaStream_t st) {
  const int64_t warps_per_cta = kSwapThreads / 32;
  const int64_t max_warps = (int64_t)num_sms() * 8 * warps_per_cta;   // 8 CTAs of 8 warps per SM
  int64_t per_warp = n / max_warps;
  if (per_warp < 1) per_warp = 1;
  if (per_warp > 32) per_warp = 32;
  // Fewer descriptors than warps: cut each into pieces (at most 256).  When
  // the host knows the largest size, pieces are at least 4 KiB, so that small
  // pages do not launch warps with nothing to copy.
  int64_t parts = n < max_warps ? max_warps / n : 1;
  if (max_size >= 0) {
    const int64_t want = (max_size + 4095) / 4096;
    if (parts > want) parts = want > 0 ? want : 1;
  }
  if (parts > 256) parts = 256;
  int64_t grid = parts > 1 ? (n * parts + warps_per_cta - 1) / warps_per_cta
                           : (n + per_warp * warps_per_cta - 1) / (per_warp * warps_per_cta);
  if (grid > max_warps / warps_per_cta) grid = max_warps / warps_per_cta;
  swap_kernel<<<(unsigned)grid, kSwapThreads, 0, st>>>(src, dst, sizes, n, (int)per_warp, (int)parts);
  return cudaGetLastError();
}

cudaError_t launch_gather(const void *k_plane, const void *v_plane, int64_t n_seq,
                          int64_t seq_stride_tokens, int64_t n_kv_heads, int64_t head_bytes,
                          int64_t block_tokens, const int32_t *sel, int64_t n_sel, void *k_out,
                          void *v_out, uint32_t *err, cudaStream_t st) {
  const int64_t items = 2 * n_seq * n_kv_heads * n_sel;
  const int64_t warps_per_cta = kSwapThreads / 32;
  int64_t grid = (items + warps_per_cta - 1) / warps_per_cta;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (grid > cap) grid = cap;
  gather_kernel<<<(unsigned)grid, kSwapThreads, 0, st>>>(
      (const char *)k_plane, (const char *)v_plane, n_seq, seq_stride_tokens, n_kv_heads, head_bytes,
      block_tokens, sel, n_sel, (char *)k_out, (char *)v_out, err);
  return cudaGetLastError();
}

}  // namespace kvo
