// kvo_attn_decode_tiered_noalloc: the tiered decode for callers that cannot
// hand the library a workspace.  The split partials live in a fixed
// file-scope device array instead of caller memory; everything else
// (arguments, layouts, kernels, result within the decode tolerance) is the
// same as kvo_attn_decode_tiered.
#include <cstdio>
#include <mutex>

#include "kvo_internal.cuh"

namespace kvo {

namespace {

// Scratch for the split partials: KVO_NOALLOC_SCRATCH_BYTES on every GPU
// that loads the library, held until the process exits.
__device__ __align__(256) unsigned char g_decode_scratch[KVO_NOALLOC_SCRATCH_BYTES];

// Device address of g_decode_scratch, looked up once per device (with that
// device current) on the first call made on it.  The lookup and the cache
// are guarded by a mutex, so host threads calling at the same time on one
// device do not race; a failed lookup is retried on the next call.  The
// address is never looked up again, so a cudaDeviceReset (which reloads the
// module, and may move the array) leaves the entry point unusable on that
// device for the rest of the process.
void *scratch_address() {
  static std::mutex mu;
  static void *cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    cached[dev] = p;
  }
  return cached[dev];
}

int64_t row_bytes_of(int dt, int64_t hkv, int64_t d) {
  if (dt == KVO_F16 || dt == KVO_BF16) return hkv * d * 2;
  if (dt == KVO_Q8_0) return (d % 32) ? -1 : hkv * (d / 32) * 34;
  return -1;
}

}  // namespace

}  // namespace kvo

using namespace kvo;

extern "C" int kvo_attn_decode_tiered_noalloc(
    const void *q, int q_dtype, int64_t batch, int64_t n_q_heads, int64_t n_kv_heads,
    int64_t head_dim, const void *k_vram, const void *v_vram, int64_t vram_seq_stride_rows,
    const void *k_host, const void *v_host, int64_t host_seq_stride_rows, int kv_dtype,
    const int32_t *ctx_len, int64_t max_ctx, int64_t n_vram_cells, float scale, void *staging_k,
    void *staging_v, float *out, void *stream) {
  clear_error();
  cudaStream_t st = (cudaStream_t)stream;
  const char *fn = "kvo_attn_decode_tiered_noalloc";
  if (batch < 0 || max_ctx < 0 || n_vram_cells < 0 || n_q_heads < 1 || n_kv_heads < 1)
    return fail(KVO_ERR_ARG, "%s: bad size", fn);
  if (batch == 0) return KVO_OK;
  if (q_dtype != KVO_F16 && q_dtype != KVO_BF16)
    return fail(KVO_ERR_UNSUPPORTED, "%s: q dtype must be f16 or bf16", fn);
  if (n_q_heads % n_kv_heads) return fail(KVO_ERR_ARG, "%s: n_q_heads %% n_kv_heads", fn);
  const int64_t group = n_q_heads / n_kv_heads;
  if (group > 8 || n_kv_heads > 8 || (head_dim != 64 && head_dim != 128))
    return fail(KVO_ERR_UNSUPPORTED, "%s: group %lld, kv heads %lld, head_dim %lld", fn,
                (long long)group, (long long)n_kv_heads, (long long)head_dim);
  const int64_t rb = row_bytes_of(kv_dtype, n_kv_heads, head_dim);
  if (rb < 0) return fail(KVO_ERR_UNSUPPORTED, "%s: kv dtype", fn);
  if (q_dtype != (kv_dtype == KVO_BF16 ? KVO_BF16 : KVO_F16))
    return fail(KVO_ERR_UNSUPPORTED, "%s: q dtype must be the cache's 16-bit type (f16 for q8_0)", fn);
  if (rb % 16) return fail(KVO_ERR_ALIGN, "%s: cell row bytes %% 16 != 0", fn);
  if (!out || !q || !ctx_len) return fail(KVO_ERR_ARG, "%s: NULL q/out/ctx_len", fn);
  if (!aligned16(q) || !aligned16(out)) return fail(KVO_ERR_ALIGN, "%s: q/out alignment", fn);

  // Split geometry that fits the scratch: the regular one when its partials
  // fit, else the fewest splits of whole 32-cell tiles that the scratch holds.
  const size_t per_split = (size_t)batch * n_q_heads * (head_dim + 2) * sizeof(float);
  if (per_split > (size_t)KVO_NOALLOC_SCRATCH_BYTES)
    return fail(KVO_ERR_WORKSPACE,
                "%s: batch * n_q_heads * (head_dim + 2) * 4 = %zu bytes exceeds the %d-byte scratch",
                fn, per_split, (int)KVO_NOALLOC_SCRATCH_BYTES);
  int split_cells = 0, n_splits = 0;
  decode_geometry(batch, max_ctx, head_dim, &split_cells, &n_splits);
  const int64_t max_splits = (int64_t)((size_t)KVO_NOALLOC_SCRATCH_BYTES / per_split);   // >= 1
  if (n_splits > max_splits) {
    const int64_t cells = (max_ctx + max_splits - 1) / max_splits;
    split_cells = (int)((cells + 31) / 32 * 32);
    n_splits = (int)((max_ctx + split_cells - 1) / split_cells);
  }

  const int64_t n_lo = n_vram_cells < max_ctx ? n_vram_cells : max_ctx;
  const int64_t n_hi = max_ctx - n_lo;
  if (n_hi > 0 && !k_host && !v_host && k_vram && v_vram) {
    // one range (a VMM tier): the tail continues right after the VRAM cells
    k_host = (const uint8_t *)k_vram + (size_t)n_lo * rb;
    v_host = (const uint8_t *)v_vram + (size_t)n_lo * rb;
    host_seq_stride_rows = vram_seq_stride_rows;
  }
  if (n_lo > 0) {
    if (vram_seq_stride_rows < n_lo) return fail(KVO_ERR_ARG, "%s: vram stride < cells", fn);
    const size_t bytes = (size_t)((batch - 1) * vram_seq_stride_rows + n_lo) * rb;
    if (!aligned16(k_vram) || !aligned16(v_vram)) return fail(KVO_ERR_ALIGN, "%s: vram alignment", fn);
    if (classify(k_vram, bytes) != kDeviceMem || classify(v_vram, bytes) != kDeviceMem)
      return fail(KVO_ERR_NOT_MAPPED, "%s: k_vram/v_vram must be device memory", fn);
  }
  const bool staged = staging_k != nullptr || staging_v != nullptr;
  if (n_hi > 0) {
    if (host_seq_stride_rows < n_hi) return fail(KVO_ERR_ARG, "%s: host stride < tail cells", fn);
    const size_t bytes = (size_t)((batch - 1) * host_seq_stride_rows + n_hi) * rb;
    if (!aligned16(k_host) || !aligned16(v_host)) return fail(KVO_ERR_ALIGN, "%s: host alignment", fn);
    if (!classify(k_host, bytes) || !classify(v_host, bytes))
      return fail(KVO_ERR_NOT_MAPPED, "%s: k_host/v_host not device-accessible", fn);
    if (staged) {
      const size_t sb = (size_t)batch * n_hi * rb;
      if (!staging_k || !staging_v) return fail(KVO_ERR_ARG, "%s: one staging buffer is NULL", fn);
      if (!aligned16(staging_k) || !aligned16(staging_v)) return fail(KVO_ERR_ALIGN, "%s: staging alignment", fn);
      if (classify(staging_k, sb) != kDeviceMem || classify(staging_v, sb) != kDeviceMem)
        return fail(KVO_ERR_NOT_MAPPED, "%s: staging buffers must be device memory", fn);
    }
  }
  float *scratch = (float *)scratch_address();
  if (!scratch) return fail(KVO_ERR_CUDA, "%s: cudaGetSymbolAddress of the scratch array failed", fn);

  DecodeArgs a;
  a.q = q; a.q_dtype = q_dtype;
  a.batch = (int)batch; a.n_q_heads = (int)n_q_heads; a.n_kv_heads = (int)n_kv_heads;
  a.head_dim = (int)head_dim; a.group = (int)group;
  a.k_lo = (const uint8_t *)k_vram; a.v_lo = (const uint8_t *)v_vram;
  a.lo_seq_stride_rows = vram_seq_stride_rows;
  a.k_hi = (const uint8_t *)k_host; a.v_hi = (const uint8_t *)v_host;
  a.hi_seq_stride_rows = host_seq_stride_rows;
  const size_t hi_bytes = n_hi > 0 ? (size_t)((batch - 1) * host_seq_stride_rows + n_hi) * rb : 0;
  a.hi_device = (n_hi > 0 && classify(k_host, hi_bytes) == kDeviceMem && classify(v_host, hi_bytes) == kDeviceMem) ? 1 : 0;
  a.kv_dtype = kv_dtype; a.row_bytes = rb;
  a.ctx_len = ctx_len; a.max_ctx = max_ctx; a.n_vram = n_lo;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = out;
  a.split_cells = split_cells;
  a.n_splits = n_splits;
  // Every partial the combine reads is written by the split kernel of the
  // same call first, so nothing in the scratch needs clearing.
  a.part_acc = scratch;
  a.part_ml = scratch + (size_t)batch * n_splits * n_q_heads * head_dim;

  if (n_hi > 0 && staged)
    return launch_decode_staged(a, k_host, v_host, host_seq_stride_rows, staging_k, staging_v, st);
  // Host rows read directly over more than one wave of CTAs, a quarter of the
  // context or more: deal VRAM and host chunks interleaved, so that the first
  // wave already keeps the host link busy (measured at 184,320 cells with
  // 94,208 in VRAM: 1,056 -> 964 us).  With fewer host rows the plain order
  // measured faster (up to 7 %), and within one wave the order does not matter.
  a.interleave = n_hi > 0 && !a.hi_device && (int64_t)batch * a.n_splits > num_sms() && 4 * n_hi >= max_ctx ? 1 : 0;
  return launch_decode(a, st);
}
