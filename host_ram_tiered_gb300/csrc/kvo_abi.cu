// libkvo C ABI: argument validation and dispatch.  Declarations, argument
// meaning, layout and error behaviour are documented in include/kvo.h.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "kvo_internal.cuh"

namespace kvo {

static thread_local char g_last_error[512];

int fail(int st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

void clear_error() { g_last_error[0] = 0; }

int cuda_status(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return KVO_OK;
  return fail(KVO_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

static int classify_one(const void *p, cudaPointerAttributes *a) {
  if (cudaPointerGetAttributes(a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of an unknown pointer
    return 0;
  }
  if (a->type == cudaMemoryTypeDevice || a->type == cudaMemoryTypeManaged) return kDeviceMem;
  if (a->type == cudaMemoryTypeHost && a->devicePointer == p) return kMappedHost;
  return 0;
}

int classify(const void *p, size_t bytes) {
  if (p == nullptr) return 0;
  const uintptr_t end = (uintptr_t)p + (bytes > 0 ? bytes : 1);
  uintptr_t cur = (uintptr_t)p;
  int kind = 0;
  // Walk the allocations the range spans: each step classifies the byte at
  // `cur` and jumps past the end of the allocation (or VMM tier range) that
  // holds it.  A range spans few allocations; one over 1024 is refused.
  for (int step = 0; cur < end; ++step) {
    if (step == 1024) return 0;
    int k;
    uintptr_t next = 0;
    const int vm = vmm_host_backed((const void *)cur, &next);   // a tier's ranges: known without asking
    if (vm >= 0) {
      k = vm ? kMappedHost : kDeviceMem;
    } else {
      cudaPointerAttributes a;
      k = classify_one((const void *)cur, &a);
      uintptr_t lo = 0;
      if (k && !alloc_range((const void *)cur, &lo, &next)) {
        // the driver gives no range: fall back to the kind of the last byte
        cudaPointerAttributes b;
        const int k2 = classify_one((const void *)(end - 1), &b);
        if (!k2) return 0;
        k = k2 == k ? k : kMappedHost;
        next = end;
      }
    }
    if (!k) return 0;
    kind = kind == 0 || kind == k ? k : kMappedHost;
    if (next <= cur) return 0;
    cur = next;
  }
  return kind;
}

Ring *ring(int which) {
  static Ring rings[3][64];
  int dev = 0;
  if (which < 0 || which > 2 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  Ring &r = rings[which][dev];
  static std::mutex mu;                      // two host threads never create one ring twice
  std::lock_guard<std::mutex> lock(mu);
  if (!r.side) {
    cudaStream_t s = nullptr, s2 = nullptr;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaStreamCreateWithFlags(&s2, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    cudaEvent_t *ev[13] = {&r.fork, &r.join, &r.join2, &r.ready[0], &r.ready[1],
                           &r.freed[0], &r.freed[1], &r.done2[0], &r.done2[1],
                           &r.part[0], &r.part[1], &r.part[2], &r.part[3]};
    for (cudaEvent_t *e : ev)
      if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    r.comp2 = s2;
    r.side = s;
  }
  return &r;
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = v > 0 ? v : 148;
  }
  return cached[dev];
}

}  // namespace kvo

using namespace kvo;

extern "C" {

const char *kvo_status_string(int status) {
  switch (status) {
    case KVO_OK: return "ok";
    case KVO_ERR_ARG: return "invalid argument";
    case KVO_ERR_ALIGN: return "misaligned pointer or size";
    case KVO_ERR_NOT_MAPPED: return "buffer is not device-accessible";
    case KVO_ERR_UNSUPPORTED: return "unsupported combination";
    case KVO_ERR_CUDA: return "CUDA error";
    case KVO_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

const char *kvo_last_error(void) { return g_last_error; }

int kvo_device_errors(uint32_t *bits, int clear) {
  clear_error();
  if (!bits) return fail(KVO_ERR_ARG, "kvo_device_errors: bits is NULL");
  uint32_t *w = device_error_word();
  if (!w) return fail(KVO_ERR_CUDA, "kvo_device_errors: no device error word");
  int st = cuda_status(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  if (st) return st;
  st = cuda_status(cudaMemcpy(bits, w, sizeof(uint32_t), cudaMemcpyDeviceToHost), "cudaMemcpy");
  if (st) return st;
  if (clear) st = cuda_status(cudaMemset(w, 0, sizeof(uint32_t)), "cudaMemset");
  return st;
}

// ---------------------------------------------------------------- a1
int kvo_sub_block_ptrs(const int64_t *block_ids, int64_t n_ids, int64_t blocks_per_chunk,
                       int64_t skip_count, uint64_t base, int64_t row_stride_bytes,
                       int64_t row_bytes, int64_t *out, int64_t n_out) {
  clear_error();
  if (n_ids < 0 || n_out < 0 || row_stride_bytes < 0 || row_bytes < 0)
    return fail(KVO_ERR_ARG, "kvo_sub_block_ptrs: negative size");
  if (blocks_per_chunk < 1) return fail(KVO_ERR_ARG, "kvo_sub_block_ptrs: blocks_per_chunk < 1");
  if (skip_count < 0 || skip_count >= blocks_per_chunk)
    return fail(KVO_ERR_ARG, "kvo_sub_block_ptrs: skip_count %lld not in [0, blocks_per_chunk)",
                (long long)skip_count);
  if (blocks_per_chunk > 1 && row_bytes % blocks_per_chunk != 0)
    return fail(KVO_ERR_ARG, "kvo_sub_block_ptrs: row_bytes %% blocks_per_chunk != 0");
  if (n_out + skip_count > n_ids * blocks_per_chunk)
    return fail(KVO_ERR_ARG, "kvo_sub_block_ptrs: n_out + skip exceeds n_ids * blocks_per_chunk");
  if (n_out == 0) return KVO_OK;
  if (!block_ids || !out) return fail(KVO_ERR_ARG, "kvo_sub_block_ptrs: NULL array");
  const uint64_t stride = (uint64_t)row_stride_bytes;
  if (blocks_per_chunk == 1) {
    for (int64_t i = 0; i < n_out; ++i)
      out[i] = (int64_t)(base + (uint64_t)block_ids[i] * stride);
    return KVO_OK;
  }
  // Walk the flattened grid from (k, j) = divmod(skip, bpc) without a divide
  // per element.
  const uint64_t page = (uint64_t)(row_bytes / blocks_per_chunk);
  int64_t k = 0, j = skip_count;
  uint64_t row = base + (uint64_t)block_ids[0] * stride;
  for (int64_t i = 0; i < n_out; ++i) {
    out[i] = (int64_t)(row + (uint64_t)j * page);
    if (++j == blocks_per_chunk) {
      j = 0;
      if (++k < n_ids) row = base + (uint64_t)block_ids[k] * stride;
    }
  }
  return KVO_OK;
}

// ---------------------------------------------------------------- multi-GPU shards
int kvo_shard_range(int64_t n_units, int64_t world, int64_t rank, int64_t *lo, int64_t *hi) {
  clear_error();
  if (!lo || !hi) return fail(KVO_ERR_ARG, "kvo_shard_range: NULL lo/hi");
  if (n_units < 0 || world < 1 || rank < 0 || rank >= world)
    return fail(KVO_ERR_ARG, "kvo_shard_range: n_units %lld, world %lld, rank %lld", (long long)n_units,
                (long long)world, (long long)rank);
  // floor(n * r / w) without overflow for any n < 2^63 and w < 2^31
  auto cut = [&](int64_t r) {
    return (n_units / world) * r + (n_units % world) * r / world;
  };
  *lo = cut(rank);
  *hi = cut(rank + 1);
  return KVO_OK;
}

// ---------------------------------------------------------------- canonical fragments
int kvo_copy_plan(const int64_t *local_offset, const int64_t *local_stride,
                  const int64_t *canonical_offset, const int64_t *canonical_stride,
                  const int64_t *num_fragments, const int64_t *fragment_size, int64_t n_runs,
                  int gpu_to_cpu, int64_t *frag_src, int64_t *frag_dst, int64_t *frag_sizes,
                  int64_t capacity, int64_t *n_frags) {
  clear_error();
  const char *fn = "kvo_copy_plan";
  if (!n_frags) return fail(KVO_ERR_ARG, "%s: n_frags is NULL", fn);
  *n_frags = 0;
  if (n_runs < 0 || capacity < 0) return fail(KVO_ERR_ARG, "%s: negative size", fn);
  if (n_runs == 0) return KVO_OK;
  if (!local_offset || !local_stride || !canonical_offset || !canonical_stride || !num_fragments ||
      !fragment_size)
    return fail(KVO_ERR_ARG, "%s: NULL run array", fn);
  int64_t total = 0;
  for (int64_t r = 0; r < n_runs; ++r) {
    if (num_fragments[r] < 0 || fragment_size[r] < 0) return fail(KVO_ERR_ARG, "%s: negative run field", fn);
    total += num_fragments[r];
  }
  if (total > capacity) return fail(KVO_ERR_ARG, "%s: %lld fragments exceed capacity %lld", fn,
                                    (long long)total, (long long)capacity);
  if (total > 0 && (!frag_src || !frag_dst || !frag_sizes)) return fail(KVO_ERR_ARG, "%s: NULL output", fn);
  int64_t n = 0;
  for (int64_t r = 0; r < n_runs; ++r) {
    int64_t local = local_offset[r], canon = canonical_offset[r];
    for (int64_t i = 0; i < num_fragments[r]; ++i, ++n) {
      frag_src[n] = gpu_to_cpu ? local : canon;
      frag_dst[n] = gpu_to_cpu ? canon : local;
      frag_sizes[n] = fragment_size[r];
      local += local_stride[r];
      canon += canonical_stride[r];
    }
  }
  *n_frags = n;
  return KVO_OK;
}

int kvo_fragment_ptrs(const int64_t *src_bases, const int64_t *dst_bases, int64_t n_blocks,
                      const int64_t *frag_src, const int64_t *frag_dst, const int64_t *frag_sizes,
                      int64_t n_frags, int64_t *out_src, int64_t *out_dst, int64_t *out_sizes) {
  clear_error();
  const char *fn = "kvo_fragment_ptrs";
  if (n_blocks < 0 || n_frags < 0) return fail(KVO_ERR_ARG, "%s: negative size", fn);
  if (n_blocks == 0 || n_frags == 0) return KVO_OK;
  if (!src_bases || !dst_bases || !frag_src || !frag_dst || !frag_sizes || !out_src || !out_dst || !out_sizes)
    return fail(KVO_ERR_ARG, "%s: NULL array", fn);
  for (int64_t b = 0; b < n_blocks; ++b) {
    const uint64_t sb = (uint64_t)src_bases[b], db = (uint64_t)dst_bases[b];
    int64_t *os = out_src + b * n_frags, *od = out_dst + b * n_frags, *oz = out_sizes + b * n_frags;
    for (int64_t f = 0; f < n_frags; ++f) {
      os[f] = (int64_t)(sb + (uint64_t)frag_src[f]);
      od[f] = (int64_t)(db + (uint64_t)frag_dst[f]);
      oz[f] = frag_sizes[f];
    }
  }
  return KVO_OK;
}

// ---------------------------------------------------------------- a2
int kvo_swap_blocks_batch(const int64_t *src, const int64_t *dst, const int64_t *sizes,
                          int64_t n, uint32_t flags, void *stream) {
  clear_error();
  cudaStream_t st = (cudaStream_t)stream;
  if (n < 0) return fail(KVO_ERR_ARG, "kvo_swap_blocks_batch: n < 0");
  if (n == 0) return KVO_OK;
  if (!src || !dst || !sizes) return fail(KVO_ERR_ARG, "kvo_swap_blocks_batch: NULL descriptor array");
  if ((flags & KVO_SWAP_FORCE_SM) && (flags & KVO_SWAP_FORCE_CE))
    return fail(KVO_ERR_ARG, "kvo_swap_blocks_batch: both FORCE_SM and FORCE_CE");
  const size_t db = (size_t)n * sizeof(int64_t);
  int ks = classify(src, db), kd = classify(dst, db), kz = classify(sizes, db);
  // Mode: SM copies unless the copy engine is forced.  Measured on GB300
  // over 2 KiB - 1 MiB pages, 64 and 2,048 descriptors, both directions: the
  // SM kernel reaches 97-100 % of the pinned-copy peak from 32 KiB x 2,048 /
  // 1 MiB x 64 up and is faster than the copy engine in every cell (one
  // cudaMemcpyAsync per merged run costs ~1.7 us to issue, and the copy
  // engine moves 1 MiB copies at 126-147 GB/s against the SM kernel's 205-211).
  const bool use_ce = (flags & KVO_SWAP_FORCE_CE) != 0;
  if (use_ce) {
    if (ks != kMappedHost || kd != kMappedHost || kz != kMappedHost)
      return fail(KVO_ERR_NOT_MAPPED,
                  "kvo_swap_blocks_batch: copy-engine mode needs pinned host descriptor arrays");
    // Merge runs whose source and destination both continue the previous
    // descriptor: fewer, larger copy-engine calls.
    int64_t i = 0;
    while (i < n) {
      if (sizes[i] < 0) return fail(KVO_ERR_ARG, "kvo_swap_blocks_batch: negative size at %lld", (long long)i);
      int64_t s = src[i], d = dst[i], len = sizes[i];
      int64_t j = i + 1;
      while (j < n && sizes[j] >= 0 && src[j] == s + len && dst[j] == d + len) { len += sizes[j]; ++j; }
      if (len > 0) {
        cudaError_t e = cudaMemcpyAsync((void *)(uintptr_t)d, (const void *)(uintptr_t)s, (size_t)len,
                                        cudaMemcpyDefault, st);
        if (e != cudaSuccess) return cuda_status(e, "cudaMemcpyAsync");
      }
      i = j;
    }
    return KVO_OK;
  }
  if (!ks || !kd || !kz)
    return fail(KVO_ERR_NOT_MAPPED,
                "kvo_swap_blocks_batch: descriptor arrays must be device-accessible (pinned host or device)");
  // A short batch whose sizes the host can read: its largest size lets the
  // kernel cut the copies into pieces no smaller than needed.
  int64_t max_size = -1;
  if (kz == kMappedHost && n <= KVO_SWAP_SHORT_BATCH) {
    max_size = 0;
    for (int64_t i = 0; i < n; ++i) max_size = sizes[i] > max_size ? sizes[i] : max_size;
  }
  return cuda_status(launch_swap_sm(src, dst, sizes, n, max_size, st), "swap kernel launch");
}

// ---------------------------------------------------------------- a3
int kvo_gather_blocks(const void *k_plane, const void *v_plane, int64_t n_seq,
                      int64_t seq_stride_tokens, int64_t n_kv_heads, int64_t head_dim, int dtype,
                      int64_t block_tokens, const int32_t *sel, int64_t n_sel, void *k_out,
                      void *v_out, void *stream) {
  clear_error();
  if (n_seq < 0 || seq_stride_tokens < 0 || n_kv_heads < 1 || head_dim < 1 || block_tokens < 1 ||
      n_sel < 0)
    return fail(KVO_ERR_ARG, "kvo_gather_blocks: bad size");
  if (dtype == KVO_Q8_0) return fail(KVO_ERR_UNSUPPORTED, "kvo_gather_blocks: q8_0 planes");
  if (dtype != KVO_F16 && dtype != KVO_BF16) return fail(KVO_ERR_ARG, "kvo_gather_blocks: dtype");
  if (n_seq == 0 || n_sel == 0) return KVO_OK;
  const int64_t head_bytes = head_dim * 2;
  if (head_bytes % 16) return fail(KVO_ERR_ALIGN, "kvo_gather_blocks: head_dim*2 not a multiple of 16");
  if (!aligned16(k_plane) || !aligned16(v_plane) || !aligned16(k_out) || !aligned16(v_out))
    return fail(KVO_ERR_ALIGN, "kvo_gather_blocks: buffers must be 16-byte aligned");
  const size_t plane_bytes = (size_t)n_seq * seq_stride_tokens * n_kv_heads * head_bytes;
  const size_t out_bytes = (size_t)n_seq * n_sel * block_tokens * n_kv_heads * head_bytes;
  if (!classify(k_plane, plane_bytes) || !classify(v_plane, plane_bytes))
    return fail(KVO_ERR_NOT_MAPPED, "kvo_gather_blocks: planes are not device-accessible");
  if (!classify(k_out, out_bytes) || !classify(v_out, out_bytes))
    return fail(KVO_ERR_NOT_MAPPED, "kvo_gather_blocks: outputs are not device-accessible");
  if (!classify(sel, (size_t)n_seq * n_kv_heads * n_sel * 4))
    return fail(KVO_ERR_NOT_MAPPED, "kvo_gather_blocks: sel is not device-accessible");
  uint32_t *err = device_error_word();
  if (!err) return fail(KVO_ERR_CUDA, "kvo_gather_blocks: device error word unavailable");
  return cuda_status(launch_gather(k_plane, v_plane, n_seq, seq_stride_tokens, n_kv_heads, head_bytes,
                                   block_tokens, sel, n_sel, k_out, v_out, err,
                                   (cudaStream_t)stream),
                     "gather kernel launch");
}

// ---------------------------------------------------------------- a4-a6
size_t kvo_attn_decode_workspace_bytes(int64_t batch, int64_t n_q_heads, int64_t head_dim,
                                       int64_t max_ctx) {
  if (batch < 0 || n_q_heads < 0 || head_dim < 0 || max_ctx < 0) return 0;
  return decode_workspace_bytes(batch, n_q_heads, head_dim, max_ctx);
}

int kvo_attn_decode_launches(int64_t batch, int64_t max_ctx, int64_t head_dim, int64_t n_vram_cells,
                             int staged) {
  if (batch < 0 || max_ctx < 0 || head_dim < 0 || n_vram_cells < 0) return KVO_ERR_ARG;
  if (batch == 0) return 0;
  if (!staged || n_vram_cells >= max_ctx) return 2;
  int sc = 0, ns = 0;
  decode_geometry(batch, max_ctx, head_dim, &sc, &ns);
  const StagedPlan pl = staged_plan(batch, sc, ns, n_vram_cells);
  return (pl.c_v > 0 ? 1 : 0) + pl.parts + 1;
}

static int64_t kv_row_bytes(int dt, int64_t hkv, int64_t d) {
  if (dt == KVO_F16 || dt == KVO_BF16) return hkv * d * 2;
  if (dt == KVO_Q8_0) return (d % 32) ? -1 : hkv * (d / 32) * 34;
  return -1;
}

int kvo_attn_decode_tiered(const void *q, int q_dtype, int64_t batch, int64_t n_q_heads,
                           int64_t n_kv_heads, int64_t head_dim, const void *k_vram,
                           const void *v_vram, int64_t vram_seq_stride_rows, const void *k_host,
                           const void *v_host, int64_t host_seq_stride_rows, int kv_dtype,
                           const int32_t *ctx_len, int64_t max_ctx, int64_t n_vram_cells,
                           float scale, void *staging_k, void *staging_v, float *out,
                           void *workspace, size_t workspace_bytes, void *stream) {
  clear_error();
  cudaStream_t st = (cudaStream_t)stream;
  if (batch < 0 || max_ctx < 0 || n_vram_cells < 0 || n_q_heads < 1 || n_kv_heads < 1)
    return fail(KVO_ERR_ARG, "kvo_attn_decode_tiered: bad size");
  if (batch == 0) return KVO_OK;
  if (q_dtype != KVO_F16 && q_dtype != KVO_BF16)
    return fail(KVO_ERR_UNSUPPORTED, "kvo_attn_decode_tiered: q dtype must be f16 or bf16");
  if (n_q_heads % n_kv_heads) return fail(KVO_ERR_ARG, "kvo_attn_decode_tiered: n_q_heads %% n_kv_heads");
  const int64_t group = n_q_heads / n_kv_heads;
  if (group > 8 || n_kv_heads > 8 || (head_dim != 64 && head_dim != 128))
    return fail(KVO_ERR_UNSUPPORTED, "kvo_attn_decode_tiered: group %lld, kv heads %lld, head_dim %lld",
                (long long)group, (long long)n_kv_heads, (long long)head_dim);
  const int64_t rb = kv_row_bytes(kv_dtype, n_kv_heads, head_dim);
  if (rb < 0) return fail(KVO_ERR_UNSUPPORTED, "kvo_attn_decode_tiered: kv dtype");
  if (q_dtype != (kv_dtype == KVO_BF16 ? KVO_BF16 : KVO_F16))
    return fail(KVO_ERR_UNSUPPORTED, "kvo_attn_decode_tiered: q dtype must be the cache's 16-bit type (f16 for q8_0)");
  if (rb % 16) return fail(KVO_ERR_ALIGN, "kvo_attn_decode_tiered: cell row bytes %% 16 != 0");
  if (!out || !q || !ctx_len) return fail(KVO_ERR_ARG, "kvo_attn_decode_tiered: NULL q/out/ctx_len");
  if (!aligned16(q) || !aligned16(out)) return fail(KVO_ERR_ALIGN, "kvo_attn_decode_tiered: q/out alignment");
  const int64_t n_lo = n_vram_cells < max_ctx ? n_vram_cells : max_ctx;   // rows read from VRAM
  const int64_t n_hi = max_ctx - n_lo;                                     // rows past N
  if (n_hi > 0 && !k_host && !v_host && k_vram && v_vram) {
    // one range (a VMM tier): the tail continues right after the VRAM cells
    k_host = (const uint8_t *)k_vram + (size_t)n_lo * rb;
    v_host = (const uint8_t *)v_vram + (size_t)n_lo * rb;
    host_seq_stride_rows = vram_seq_stride_rows;
  }
  if (n_lo > 0) {
    if (vram_seq_stride_rows < n_lo) return fail(KVO_ERR_ARG, "kvo_attn_decode_tiered: vram stride < cells");
    const size_t bytes = (size_t)((batch - 1) * vram_seq_stride_rows + n_lo) * rb;
    if (!aligned16(k_vram) || !aligned16(v_vram)) return fail(KVO_ERR_ALIGN, "kvo_attn_decode_tiered: vram alignment");
    if (classify(k_vram, bytes) != kDeviceMem || classify(v_vram, bytes) != kDeviceMem)
      return fail(KVO_ERR_NOT_MAPPED, "kvo_attn_decode_tiered: k_vram/v_vram must be device memory");
  }
  const bool staged = staging_k != nullptr || staging_v != nullptr;
  if (n_hi > 0) {
    if (host_seq_stride_rows < n_hi) return fail(KVO_ERR_ARG, "kvo_attn_decode_tiered: host stride < tail cells");
    const size_t bytes = (size_t)((batch - 1) * host_seq_stride_rows + n_hi) * rb;
    if (!aligned16(k_host) || !aligned16(v_host)) return fail(KVO_ERR_ALIGN, "kvo_attn_decode_tiered: host alignment");
    if (!classify(k_host, bytes) || !classify(v_host, bytes))
      return fail(KVO_ERR_NOT_MAPPED, "kvo_attn_decode_tiered: k_host/v_host not device-accessible");
    if (staged) {
      const size_t sb = (size_t)batch * n_hi * rb;
      if (!staging_k || !staging_v) return fail(KVO_ERR_ARG, "kvo_attn_decode_tiered: one staging buffer is NULL");
      if (!aligned16(staging_k) || !aligned16(staging_v)) return fail(KVO_ERR_ALIGN, "kvo_attn_decode_tiered: staging alignment");
      if (classify(staging_k, sb) != kDeviceMem || classify(staging_v, sb) != kDeviceMem)
        return fail(KVO_ERR_NOT_MAPPED, "kvo_attn_decode_tiered: staging buffers must be device memory");
    }
  }
  const size_t need = decode_workspace_bytes(batch, n_q_heads, head_dim, max_ctx);
  if (!workspace || workspace_bytes < need || !aligned16(workspace))
    return fail(KVO_ERR_WORKSPACE, "kvo_attn_decode_tiered: workspace needs %zu bytes", need);

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
  decode_geometry(batch, max_ctx, head_dim, &a.split_cells, &a.n_splits);
  a.part_acc = (float *)workspace;
  a.part_ml = a.part_acc + (size_t)batch * a.n_splits * n_q_heads * head_dim;

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

// ---------------------------------------------------------------- write path
int kvo_append_kv_tiered(const void *k_new, const void *v_new, int src_dtype, int64_t n_new,
                         int64_t pos0, int64_t n_kv_heads, int64_t head_dim, void *k_vram,
                         void *v_vram, void *k_host, void *v_host, int kv_dtype,
                         int64_t n_vram_cells, int64_t capacity_cells, void *stream) {
  clear_error();
  const char *fn = "kvo_append_kv_tiered";
  if (n_new < 0 || pos0 < 0 || n_kv_heads < 1 || head_dim < 1 || n_vram_cells < 0 || capacity_cells < 0)
    return fail(KVO_ERR_ARG, "%s: bad size", fn);
  if (n_new == 0) return KVO_OK;
  if (pos0 + n_new > capacity_cells) return fail(KVO_ERR_ARG, "%s: cells past the capacity", fn);
  if (src_dtype != KVO_F16 && src_dtype != KVO_BF16)
    return fail(KVO_ERR_UNSUPPORTED, "%s: source dtype must be f16 or bf16", fn);
  if (kv_dtype != KVO_Q8_0 && kv_dtype != src_dtype)
    return fail(KVO_ERR_UNSUPPORTED, "%s: a f16/bf16 cache takes its own dtype only", fn);
  if (kv_dtype == KVO_Q8_0 && head_dim % 32)
    return fail(KVO_ERR_UNSUPPORTED, "%s: q8_0 needs head_dim %% 32 == 0", fn);
  if (kv_dtype == KVO_Q8_0 && n_kv_heads * head_dim > 8 * 256)
    return fail(KVO_ERR_UNSUPPORTED, "%s: q8_0 rows of more than 2048 values", fn);
  const int64_t src_row = n_kv_heads * head_dim * 2;
  const int64_t rb = kv_dtype == KVO_Q8_0 ? n_kv_heads * (head_dim / 32) * 34 : src_row;
  if (src_row % 16 || (kv_dtype != KVO_Q8_0 && rb % 16))
    return fail(KVO_ERR_ALIGN, "%s: row bytes %% 16 != 0", fn);
  if (!aligned16(k_new) || !aligned16(v_new)) return fail(KVO_ERR_ALIGN, "%s: source alignment", fn);
  if (!classify(k_new, (size_t)n_new * src_row) || !classify(v_new, (size_t)n_new * src_row))
    return fail(KVO_ERR_NOT_MAPPED, "%s: k_new/v_new not device-accessible", fn);
  const int64_t n_lo = n_vram_cells < capacity_cells ? n_vram_cells : capacity_cells;
  const int64_t end = pos0 + n_new;
  if (pos0 < n_lo) {                                   // touches the VRAM head
    const size_t bytes = (size_t)(end < n_lo ? end : n_lo) * rb;
    if (classify(k_vram, bytes) != kDeviceMem || classify(v_vram, bytes) != kDeviceMem)
      return fail(KVO_ERR_NOT_MAPPED, "%s: k_vram/v_vram must be device memory", fn);
    if (kv_dtype != KVO_Q8_0 && (!aligned16(k_vram) || !aligned16(v_vram)))
      return fail(KVO_ERR_ALIGN, "%s: vram alignment", fn);
    if (kv_dtype == KVO_Q8_0 && (((uintptr_t)k_vram | (uintptr_t)v_vram) & 1))
      return fail(KVO_ERR_ALIGN, "%s: vram alignment", fn);
  }
  if (end > n_lo) {                                    // touches the host tail
    const size_t bytes = (size_t)(end - n_lo) * rb;
    if (!classify(k_host, bytes) || !classify(v_host, bytes))
      return fail(KVO_ERR_NOT_MAPPED, "%s: k_host/v_host not device-accessible", fn);
    if (kv_dtype != KVO_Q8_0 && (!aligned16(k_host) || !aligned16(v_host)))
      return fail(KVO_ERR_ALIGN, "%s: host alignment", fn);
    if (kv_dtype == KVO_Q8_0 && (((uintptr_t)k_host | (uintptr_t)v_host) & 1))
      return fail(KVO_ERR_ALIGN, "%s: host alignment", fn);
  }
  AppendArgs a;
  a.k_new = (const uint8_t *)k_new; a.v_new = (const uint8_t *)v_new;
  a.src_dtype = src_dtype; a.kv_dtype = kv_dtype;
  a.n_new = n_new; a.pos0 = pos0; a.n_kv_heads = n_kv_heads; a.head_dim = head_dim; a.row_bytes = rb;
  a.k_lo = (uint8_t *)k_vram; a.v_lo = (uint8_t *)v_vram;
  a.k_hi = (uint8_t *)k_host; a.v_hi = (uint8_t *)v_host;
  a.n_vram = n_lo;
  return launch_append(a, (cudaStream_t)stream);
}

// ---------------------------------------------------------------- a7-a8
size_t kvo_attn_prefill_workspace_bytes(int64_t rows, int64_t n_q_heads) {
  if (rows < 0 || n_q_heads < 0) return 0;
  return (size_t)rows * n_q_heads * 2 * sizeof(float);
}

int kvo_attn_prefill_tiered(const void *q, int64_t rows, int64_t q_pos0, int64_t n_q_heads,
                            int64_t n_kv_heads, int64_t head_dim, const void *k_vram,
                            const void *v_vram, const void *k_host, const void *v_host,
                            int kv_dtype, int64_t ctx_len, int64_t n_vram_cells, float scale,
                            void *arena, size_t arena_bytes, int64_t rows_per_launch, float *out,
                            void *workspace, size_t workspace_bytes, void *stream) {
  clear_error();
  cudaStream_t st = (cudaStream_t)stream;
  if (rows < 0 || q_pos0 < 0 || ctx_len < 0 || n_vram_cells < 0 || n_q_heads < 1 || n_kv_heads < 1)
    return fail(KVO_ERR_ARG, "kvo_attn_prefill_tiered: bad size");
  if (rows == 0) return KVO_OK;
  if (kv_dtype != KVO_F16 && kv_dtype != KVO_BF16)
    return fail(KVO_ERR_UNSUPPORTED, "kvo_attn_prefill_tiered: kv dtype must be f16 or bf16");
  if (n_q_heads % n_kv_heads) return fail(KVO_ERR_ARG, "kvo_attn_prefill_tiered: n_q_heads %% n_kv_heads");
  const int64_t group = n_q_heads / n_kv_heads;
  if (head_dim != 128 || (group != 1 && group != 2 && group != 4 && group != 8))
    return fail(KVO_ERR_UNSUPPORTED, "kvo_attn_prefill_tiered: head_dim %lld group %lld",
                (long long)head_dim, (long long)group);
  if (rows_per_launch <= 0) rows_per_launch = rows;
  if (!(scale > 0.f) || !(scale < 3.0e38f))
    return fail(KVO_ERR_ARG, "kvo_attn_prefill_tiered: scale must be positive and finite");
  if (!q || !out) return fail(KVO_ERR_ARG, "kvo_attn_prefill_tiered: NULL q/out");
  if (!aligned16(q) || !aligned16(out)) return fail(KVO_ERR_ALIGN, "kvo_attn_prefill_tiered: q/out alignment");
  const int64_t rb = n_kv_heads * head_dim * 2;
  // Cells any row can see: [0, min(ctx_len, q_pos0 + rows)).
  const int64_t c_end = ctx_len < q_pos0 + rows ? ctx_len : q_pos0 + rows;
  const int64_t n_lo = n_vram_cells < c_end ? n_vram_cells : c_end;
  const int64_t n_hi = c_end - n_lo;
  if (n_hi > 0 && !k_host && !v_host && k_vram && v_vram) {
    // one range (a VMM tier): the tail continues right after the VRAM cells
    k_host = (const uint8_t *)k_vram + (size_t)n_vram_cells * rb;
    v_host = (const uint8_t *)v_vram + (size_t)n_vram_cells * rb;
  }
  if (n_lo > 0) {
    if (!aligned16(k_vram) || !aligned16(v_vram)) return fail(KVO_ERR_ALIGN, "kvo_attn_prefill_tiered: vram alignment");
    if (classify(k_vram, (size_t)n_lo * rb) != kDeviceMem || classify(v_vram, (size_t)n_lo * rb) != kDeviceMem)
      return fail(KVO_ERR_NOT_MAPPED, "kvo_attn_prefill_tiered: k_vram/v_vram must be device memory");
  }
  int64_t bucket = 0;
  int n_slots = 0;
  if (n_hi > 0) {
    if (!aligned16(k_host) || !aligned16(v_host)) return fail(KVO_ERR_ALIGN, "kvo_attn_prefill_tiered: host alignment");
    if (!classify(k_host, (size_t)n_hi * rb) || !classify(v_host, (size_t)n_hi * rb))
      return fail(KVO_ERR_NOT_MAPPED, "kvo_attn_prefill_tiered: k_host/v_host not device-accessible");
    if (arena) {
      // Two slots (copy one bucket while scoring the other) when the arena
      // holds at least two cell rows of K and V per slot, else one.
      bucket = (int64_t)(arena_bytes / (4 * (size_t)rb));
      n_slots = 2;
      if (bucket < 1) {
        bucket = (int64_t)(arena_bytes / (2 * (size_t)rb));
        n_slots = 1;
      }
      if (bucket < 1) return fail(KVO_ERR_ARG, "kvo_attn_prefill_tiered: arena holds no cell row");
      if (!aligned16(arena)) return fail(KVO_ERR_ALIGN, "kvo_attn_prefill_tiered: arena alignment");
      if (classify(arena, (size_t)2 * n_slots * bucket * rb) != kDeviceMem)
        return fail(KVO_ERR_NOT_MAPPED, "kvo_attn_prefill_tiered: arena must be device memory");
    }
  }
  const size_t need = kvo_attn_prefill_workspace_bytes(rows, n_q_heads);
  if (!workspace || workspace_bytes < need || !aligned16(workspace))
    return fail(KVO_ERR_WORKSPACE, "kvo_attn_prefill_tiered: workspace needs %zu bytes", need);

  PrefillArgs a;
  memset(&a, 0, sizeof(a));
  a.n_q_heads = (int)n_q_heads; a.n_kv_heads = (int)n_kv_heads; a.head_dim = (int)head_dim;
  a.group = (int)group; a.dtype = kv_dtype; a.row_bytes = rb;
  a.k_lo = (const uint8_t *)k_vram; a.v_lo = (const uint8_t *)v_vram;
  a.n_vram = n_lo;
  a.scale_log2 = scale * 1.4426950408889634f;

  // Segments of the visible cell range, in ascending order: the VRAM head,
  // then either the whole host tail (direct) or its arena buckets (staged).
  struct Seg { int64_t c0, c1; };
  std::vector<Seg> segs;
  if (n_lo > 0) segs.push_back({0, n_lo});
  if (n_hi > 0) {
    if (!arena) segs.push_back({n_lo, c_end});
    else for (int64_t c = n_lo; c < c_end; c += bucket) segs.push_back({c, c + bucket < c_end ? c + bucket : c_end});
  }
  float *ml = (float *)workspace;
  // Staged mode: buckets go through the arena slots on the side stream; the
  // launch streams wait for a slot's copy and release it after their
  // launches.  Row blocks alternate between the caller's stream and comp2.
  const int64_t n_blocks = (rows + rows_per_launch - 1) / rows_per_launch;
  const bool staged = arena && n_hi > 0;
  const bool two = n_blocks > 1;
  Ring *rg = nullptr;
  static std::mutex ring_mu;
  std::unique_lock<std::mutex> lock(ring_mu, std::defer_lock);
  if (staged || two) {
    lock.lock();
    rg = ring(0);
    if (!rg) return fail(KVO_ERR_CUDA, "kvo_attn_prefill_tiered: library streams unavailable");
    int e = cuda_status(cudaEventRecord(rg->fork, st), "cudaEventRecord");
    if (!e && staged) e = cuda_status(cudaStreamWaitEvent(rg->side, rg->fork, 0), "cudaStreamWaitEvent");
    if (!e && two) e = cuda_status(cudaStreamWaitEvent(rg->comp2, rg->fork, 0), "cudaStreamWaitEvent");
    if (e) return e;
  }
  int64_t bi = 0;                                       // bucket index
  for (size_t si = 0; si < segs.size(); ++si) {
    const Seg s = segs[si];
    const bool tail = s.c0 >= n_lo && n_hi > 0;
    const uint8_t *k_slot = nullptr, *v_slot = nullptr;
    int slot = 0;
    if (tail && arena) {
      slot = (int)(bi % n_slots);
      k_slot = (const uint8_t *)arena + (size_t)slot * 2 * bucket * rb;
      v_slot = k_slot + (size_t)bucket * rb;
      const size_t bytes = (size_t)(s.c1 - s.c0) * rb;
      const uint8_t *ks = (const uint8_t *)k_host + (size_t)(s.c0 - n_lo) * rb;
      const uint8_t *vs = (const uint8_t *)v_host + (size_t)(s.c0 - n_lo) * rb;
      int e = KVO_OK;
      // the slot is free once both row blocks' launches of its previous bucket
      // have finished (freed: the caller's stream, done2: the second stream)
      if (bi >= n_slots) e = cuda_status(cudaStreamWaitEvent(rg->side, rg->freed[slot], 0), "cudaStreamWaitEvent");
      if (!e && bi >= n_slots && two) e = cuda_status(cudaStreamWaitEvent(rg->side, rg->done2[slot], 0), "cudaStreamWaitEvent");
      if (!e) e = cuda_status(cudaMemcpyAsync((void *)k_slot, ks, bytes, cudaMemcpyDefault, rg->side), "arena copy K");
      if (!e) e = cuda_status(cudaMemcpyAsync((void *)v_slot, vs, bytes, cudaMemcpyDefault, rg->side), "arena copy V");
      if (!e) e = cuda_status(cudaEventRecord(rg->ready[slot], rg->side), "cudaEventRecord");
      if (!e) e = cuda_status(cudaStreamWaitEvent(st, rg->ready[slot], 0), "cudaStreamWaitEvent");
      if (!e && two) e = cuda_status(cudaStreamWaitEvent(rg->comp2, rg->ready[slot], 0), "cudaStreamWaitEvent");
      if (e) return e;
      a.k_hi = k_slot; a.v_hi = v_slot; a.hi_origin = s.c0;
    } else if (tail) {
      a.k_hi = (const uint8_t *)k_host; a.v_hi = (const uint8_t *)v_host; a.hi_origin = n_lo;
    }
    for (int64_t r0 = 0; r0 < rows; r0 += rows_per_launch) {
      const int64_t r1 = r0 + rows_per_launch < rows ? r0 + rows_per_launch : rows;
      cudaStream_t ls = (two && ((r0 / rows_per_launch) & 1)) ? rg->comp2 : st;
      // Rows of this block see cells < q_pos0 + r1; the segments that can
      // hold such cells are the ones starting before it.
      const int64_t vis_end = q_pos0 + r1;
      if (s.c0 >= vis_end) continue;
      // The last segment this row block sees finalises it.
      bool last = true;
      if (si + 1 < segs.size() && segs[si + 1].c0 < vis_end) last = false;
      a.q = (const uint16_t *)q + (size_t)r0 * n_q_heads * head_dim;
      a.rows = (int)(r1 - r0);
      a.pos0 = q_pos0 + r0;
      a.c0 = s.c0;
      a.c1 = s.c1 < vis_end ? s.c1 : vis_end;
      a.acc = out + (size_t)r0 * n_q_heads * head_dim;
      a.ml = ml + (size_t)r0 * n_q_heads * 2;
      a.init = (si == 0);
      a.finalize = last;
      int e;
      if (!tail) {
        // VRAM head: tensor cores fed by TMA
        a.hi_origin = 0;
        e = launch_prefill_tc(a, k_vram, v_vram, n_lo, ls);
      } else if (arena) {
        // arena bucket: tensor cores fed by TMA
        e = launch_prefill_tc(a, k_slot, v_slot, s.c1 - s.c0, ls);
      } else if ((int64_t)a.rows * group >= 512) {
        // direct, enough query tiles to fill the GPU: the host tail read in
        // place, tensor cores fed by plain loads (one producer warp per CTA)
        e = launch_prefill_tc_host(a, ls);
      } else {
        // direct, few query rows: the tensor-core kernel would run one CTA per
        // kv head, each bound by its one producer warp; the mma.sync kernel's
        // 16-position tiles give 4x the CTAs, each loading with all threads
        e = launch_prefill(a, ls);
      }
      if (e) return e;
    }
    if (tail && arena) {
      int e = KVO_OK;
      if (two) e = cuda_status(cudaEventRecord(rg->done2[slot], rg->comp2), "cudaEventRecord");
      if (!e) e = cuda_status(cudaEventRecord(rg->freed[slot], st), "cudaEventRecord");
      if (e) return e;
      ++bi;
    }
  }
  if (rg) {
    int e = KVO_OK;
    if (staged) {
      e = cuda_status(cudaEventRecord(rg->join, rg->side), "cudaEventRecord");
      if (!e) e = cuda_status(cudaStreamWaitEvent(st, rg->join, 0), "cudaStreamWaitEvent");
    }
    if (!e && two) {
      e = cuda_status(cudaEventRecord(rg->join2, rg->comp2), "cudaEventRecord");
      if (!e) e = cuda_status(cudaStreamWaitEvent(st, rg->join2, 0), "cudaStreamWaitEvent");
    }
    if (e) return e;
  }
  if (segs.empty()) {
    // Nothing visible (ctx_len == 0): the result is 0 by the 1e-30 clamp.
    return cuda_status(cudaMemsetAsync(out, 0, (size_t)rows * n_q_heads * head_dim * sizeof(float), st),
                       "cudaMemsetAsync");
  }
  return KVO_OK;
}

}  // extern "C"
