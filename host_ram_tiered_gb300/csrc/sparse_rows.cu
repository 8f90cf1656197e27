// QSA sparse rows over a paged host-resident cache (ExLlamaV3 patch "QSA KV
// cache host-RAM offload": qsa_sparse_attend_rows and
// qsa_sparse_attend_rows_staged, qsa_staging_worthwhile, copy_page).
//
// Each query row attends to its own list of selected cache positions
// (-1 padded).  Direct mode: the decode split kernel in selection mode reads
// every row's picks through the host mapping.  Staged mode: the page range is
// walked in arena-sized buckets; a bucket's pages are gathered host -> arena
// once, every row block scores its picks in the bucket (grouped by bucket
// once per call), and the bucket's (m, l, acc) is folded into a running state
// -- in the split kernel's epilogue when each row has one chunk, else by the
// combine kernel -- writing out = acc / max(l, 1e-30) after the last bucket.
#include <cstring>
#include <mutex>

#include "decode_dispatch.cuh"

namespace kvo {
namespace dec {
template cudaError_t launch_kv<KVO_F16, true>(const DecodeArgs &a, cudaStream_t st);
template cudaError_t launch_kv<KVO_BF16, true>(const DecodeArgs &a, cudaStream_t st);
}  // namespace dec

namespace {

constexpr int kGatherThreads = 256;
// Staged with two arena slots: the split kernel leaves this many SMs to the
// next bucket's page gather, which runs beside it on the library stream.  A
// split CTA holds a whole SM, so the gather then runs as kGatherSms CTAs of
// kGatherWideThreads threads that each reserve more than half an SM's shared
// memory: one per SM, so whichever kernel starts first, the gather never
// holds more than kGatherSms SMs and the split kernel always finds its own.
// Four SMs of 1024 threads keep a bucket's gather at the link rate behind the
// split kernel (measured per step: 16 SMs 10.5 ms, 8 10.2, 4 9.2, 2 11.4).
constexpr int kGatherSms = 4;
constexpr int kGatherWideThreads = 1024;
constexpr int kGatherWideSmem = 120 * 1024;
constexpr size_t kPartitionSmem = 200 * 1024;   // bucket counters per CTA

// Pages block_table[p0 .. p0 + n) of K and V -> arena slots 0 .. n-1.  Work
// item = (tensor, page, slice): each page is cut into `parts` slices so that
// enough CTAs (and 16-byte loads, 4 per thread) are in flight to fill the
// host link; a CTA loops over items with stride gridDim.x.
__global__ void __launch_bounds__(1024)
page_gather_kernel(const uint8_t *kp, const uint8_t *vp, int64_t page_bytes, const int32_t *bt, int64_t p0,
                   int64_t n, int64_t n_pages_total, uint8_t *ka, uint8_t *va, uint32_t *err, int parts) {
  const int64_t cpp = page_bytes >> 4;
  const int64_t per = (cpp + parts - 1) / parts;    // 16-byte chunks per slice
  for (int64_t item = blockIdx.x; item < 2 * n * parts; item += gridDim.x) {
    const int64_t pg = item / parts;
    const int64_t c_lo = (item % parts) * per, c_hi = c_lo + per < cpp ? c_lo + per : cpp;
    const bool is_v = pg >= n;
    const int64_t i = is_v ? pg - n : pg;
    const int64_t page = bt[p0 + i];
    if (page < 0 || page >= n_pages_total) {
      if (threadIdx.x == 0 && item % parts == 0) atomicOr(err, kErrPageTable);
      continue;
    }
    const int4 *src = (const int4 *)((is_v ? vp : kp) + page * page_bytes);
    int4 *dst = (int4 *)((is_v ? va : ka) + i * page_bytes);
    constexpr int U = 4;
    const int64_t nt = blockDim.x;
    for (int64_t c0 = c_lo + threadIdx.x; c0 < c_hi; c0 += U * nt) {
      int4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t c = c0 + u * nt;
        if (c < c_hi) v[u] = src[c];
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t c = c0 + u * nt;
        if (c < c_hi) dst[c] = v[u];
      }
    }
  }
}

// Staged mode, once per call: the picks of every row grouped by arena bucket
// (bucket = position / (arena_pages * page_size)), padding dropped, order
// kept within a bucket (a stable counting sort, one warp per row): picks of
// row r in bucket k are grouped[r][offs[r][k] .. offs[r][k + 1]).
__global__ void partition_kernel(const int32_t *idx, int64_t rows, int64_t k_pad, int64_t hi,
                                 int64_t bucket_cells, int n_b, int32_t *grouped, int32_t *offs) {
  extern __shared__ int32_t bins[];          // [warps][n_b + 1]
  const int warps = blockDim.x >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * warps + w;
  if (r >= rows) return;                     // whole warp; no block-wide barrier below
  int32_t *cnt = bins + (size_t)w * (n_b + 1);
  for (int i = lane; i <= n_b; i += 32) cnt[i] = 0;
  __syncwarp();
  const int32_t *ir = idx + r * k_pad;
  for (int64_t k = lane; k < k_pad; k += 32) {
    const int64_t j = ir[k];
    if (j >= 0 && j < hi) atomicAdd(&cnt[j / bucket_cells], 1);
  }
  __syncwarp();
  int run = 0;                               // exclusive prefix sum over the bins
  for (int base = 0; base < n_b; base += 32) {
    const int i = base + lane;
    const int c = i < n_b ? cnt[i] : 0;
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (i < n_b) cnt[i] = run + x - c;
    run += __shfl_sync(0xffffffffu, x, 31);
  }
  __syncwarp();
  if (lane == 0) cnt[n_b] = run;
  __syncwarp();
  for (int i = lane; i <= n_b; i += 32) offs[r * (n_b + 1) + i] = cnt[i];
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
  for (int64_t k0 = 0; k0 < k_pad; k0 += 32) {
    const int64_t k = k0 + lane;
    const int64_t j = k < k_pad ? ir[k] : -1;
    const bool ok = j >= 0 && j < hi;
    const int bin = ok ? (int)(j / bucket_cells) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, bin);
    const int rank = __popc(peers & lt);
    if (ok) grouped[r * k_pad + cnt[bin] + rank] = (int32_t)j;
    __syncwarp();
    if (ok && rank == 0) cnt[bin] += __popc(peers);
    __syncwarp();
  }
}

// Chunks of a selection list: one chunk per row when the launch has at least
// as many rows as SMs (nothing left to balance), else the decode geometry.
void sparse_geometry(int64_t rows, int64_t k_pad, int *chunk, int *n_chunks) {
  if (rows >= num_sms()) {
    int64_t c = (k_pad + 31) / 32 * 32;
    if (c < 32) c = 32;
    *chunk = (int)c;
    *n_chunks = 1;
    return;
  }
  decode_geometry(rows, k_pad, 0, chunk, n_chunks);
}

int64_t row_block(int64_t rows, int64_t rows_per_launch) {
  return rows_per_launch < rows ? rows_per_launch : rows;
}

size_t up16(size_t x) { return (x + 15) / 16 * 16; }

// Arena pages per bucket (0: direct).  The page sizes one bucket as half the
// arena each for K and V pages (at most the pages in use); here the arena
// holds two such slots when it can, so that the next bucket's pages arrive
// while the current one is scored: slot pages = arena / (4 page_bytes), or
// arena / (2 page_bytes) with a single slot when two do not fit.
int64_t arena_pages_of(size_t arena_bytes, int64_t page_bytes, int64_t num_pages_used, int *slots) {
  *slots = 0;
  if (arena_bytes == 0 || num_pages_used <= 0 || page_bytes <= 0) return 0;
  int64_t n = (int64_t)(arena_bytes / (4 * (size_t)page_bytes));
  *slots = 2;
  if (n < 1) {
    n = (int64_t)(arena_bytes / (2 * (size_t)page_bytes));
    *slots = 1;
  }
  if (n < 1) *slots = 0;
  return n < num_pages_used ? n : num_pages_used;
}

// Workspace layout: running state (acc, m/l), one row block's chunk
// partials, then for staged mode the grouped picks and their offsets.
struct SparseWs {
  size_t run_acc, run_ml, part, grouped, offs, total;
};
SparseWs sparse_workspace(int64_t rows, int64_t n_q_heads, int64_t head_dim, int64_t k_pad,
                          int64_t rows_per_launch, int64_t n_b) {
  const int64_t rb = row_block(rows, rows_per_launch);
  int chunk = 0, n_chunks = 0;
  sparse_geometry(rb, k_pad, &chunk, &n_chunks);
  SparseWs w;
  w.run_acc = 0;
  w.run_ml = w.run_acc + up16((size_t)rows * n_q_heads * head_dim * 4);
  w.part = w.run_ml + up16((size_t)rows * n_q_heads * 2 * 4);
  w.grouped = w.part + up16((size_t)rb * n_chunks * n_q_heads * (head_dim + 2) * 4);
  w.offs = w.grouped + (n_b > 0 ? up16((size_t)rows * k_pad * 4) : 0);
  w.total = w.offs + (n_b > 0 ? up16((size_t)rows * (n_b + 1) * 4) : 0);
  return w;
}

}  // namespace

cudaError_t launch_page_gather(const void *k_pages, const void *v_pages, int64_t page_bytes,
                               const int32_t *block_table, int64_t p0, int64_t n, int64_t n_pages_total,
                               void *k_arena, void *v_arena, uint32_t *err, bool beside, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t cap = beside ? kGatherSms : (int64_t)num_sms() * 4;
  const int threads = beside ? kGatherWideThreads : kGatherThreads;
  const int smem = beside ? kGatherWideSmem : 0;
  if (beside) {
    const cudaError_t e =
        cudaFuncSetAttribute(page_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGatherWideSmem);
    if (e != cudaSuccess) return e;
  }
  // slices per page: enough items for every CTA, each slice at least 16 KiB
  int64_t parts = (cap + 2 * n - 1) / (2 * n);
  const int64_t max_parts = (page_bytes >> 4) / 1024 > 0 ? (page_bytes >> 4) / 1024 : 1;
  if (parts > max_parts) parts = max_parts;
  if (parts < 1) parts = 1;
  int64_t grid = 2 * n * parts;
  if (grid > cap) grid = cap;
  page_gather_kernel<<<(unsigned)grid, threads, smem, st>>>(
      (const uint8_t *)k_pages, (const uint8_t *)v_pages, page_bytes, block_table, p0, n, n_pages_total,
      (uint8_t *)k_arena, (uint8_t *)v_arena, err, (int)parts);
  return cudaGetLastError();
}

int launch_sparse_rows(const DecodeArgs &a, cudaStream_t st) {
  const cudaError_t e = a.kv_dtype == KVO_BF16 ? dec::launch_kv<KVO_BF16, true>(a, st)
                                               : dec::launch_kv<KVO_F16, true>(a, st);
  return cuda_status(e, "sparse rows kernel launch");
}

}  // namespace kvo

using namespace kvo;

extern "C" int kvo_staging_worthwhile(int64_t rows, int64_t k_pad, int64_t num_pages_used, int64_t page_size) {
  if (rows < 0 || k_pad < 0 || num_pages_used < 0 || page_size < 0) return 0;
  return rows * k_pad > 2 * num_pages_used * page_size ? 1 : 0;
}

extern "C" size_t kvo_attn_sparse_rows_workspace_bytes(int64_t rows, int64_t n_q_heads, int64_t n_kv_heads,
                                                       int64_t head_dim, int64_t k_pad, int64_t rows_per_launch,
                                                       int64_t page_size, int64_t num_pages_used,
                                                       size_t arena_bytes) {
  if (rows <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || k_pad < 0 || rows_per_launch <= 0 ||
      page_size <= 0 || num_pages_used < 0)
    return 0;
  int slots = 0;
  const int64_t ap = arena_pages_of(arena_bytes, page_size * n_kv_heads * head_dim * 2, num_pages_used, &slots);
  const int64_t n_b = ap > 0 ? (num_pages_used + ap - 1) / ap : 0;
  return sparse_workspace(rows, n_q_heads, head_dim, k_pad, rows_per_launch, n_b).total;
}

extern "C" int kvo_attn_sparse_rows(const void *q, int q_dtype, int64_t rows, int64_t n_q_heads,
                                    int64_t n_kv_heads, int64_t head_dim, const void *k_pages,
                                    const void *v_pages, int dtype, int64_t page_size, int64_t n_pages,
                                    const int32_t *block_table, int64_t num_pages_used,
                                    const int32_t *indices, int64_t k_pad, float scale, void *arena,
                                    size_t arena_bytes, int64_t rows_per_launch, float *out,
                                    void *workspace, size_t workspace_bytes, void *stream) {
  clear_error();
  cudaStream_t st = (cudaStream_t)stream;
  const char *fn = "kvo_attn_sparse_rows";
  if (rows < 0 || k_pad < 0 || n_q_heads < 1 || n_kv_heads < 1 || page_size < 1 || n_pages < 0 ||
      num_pages_used < 0 || rows_per_launch < 1)
    return fail(KVO_ERR_ARG, "%s: bad size", fn);
  if (rows == 0) return KVO_OK;
  if (dtype != KVO_F16 && dtype != KVO_BF16)
    return fail(KVO_ERR_UNSUPPORTED, "%s: cache dtype must be f16 or bf16", fn);
  if (q_dtype != dtype) return fail(KVO_ERR_UNSUPPORTED, "%s: q dtype must equal the cache dtype", fn);
  if (n_q_heads % n_kv_heads) return fail(KVO_ERR_ARG, "%s: n_q_heads %% n_kv_heads", fn);
  const int64_t group = n_q_heads / n_kv_heads;
  if (group > 8 || n_kv_heads > 8 || (head_dim != 64 && head_dim != 128))
    return fail(KVO_ERR_UNSUPPORTED, "%s: group %lld, kv heads %lld, head_dim %lld", fn, (long long)group,
                (long long)n_kv_heads, (long long)head_dim);
  if (num_pages_used > n_pages) return fail(KVO_ERR_ARG, "%s: num_pages_used > n_pages", fn);
  const int64_t rb = n_kv_heads * head_dim * 2;
  const int64_t page_bytes = page_size * rb;
  if (!q || !out || !indices || (num_pages_used > 0 && !block_table))
    return fail(KVO_ERR_ARG, "%s: NULL q/out/indices/block_table", fn);
  if (!aligned16(q) || !aligned16(out) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(workspace))
    return fail(KVO_ERR_ALIGN, "%s: q/out/pages/workspace must be 16-byte aligned", fn);
  const size_t qbytes = (size_t)rows * n_q_heads * head_dim;
  if (classify(q, qbytes * 2) != kDeviceMem || classify(out, qbytes * 4) != kDeviceMem)
    return fail(KVO_ERR_NOT_MAPPED, "%s: q/out must be device memory", fn);
  if (k_pad > 0 && !classify(indices, (size_t)rows * k_pad * 4))
    return fail(KVO_ERR_NOT_MAPPED, "%s: indices not device-accessible", fn);
  if (num_pages_used > 0) {
    if (!classify(block_table, (size_t)num_pages_used * 4))
      return fail(KVO_ERR_NOT_MAPPED, "%s: block_table not device-accessible", fn);
    if (!classify(k_pages, (size_t)n_pages * page_bytes) || !classify(v_pages, (size_t)n_pages * page_bytes))
      return fail(KVO_ERR_NOT_MAPPED, "%s: k_pages/v_pages not device-accessible", fn);
  }
  const bool staged = arena != nullptr && arena_bytes > 0 && num_pages_used > 0;
  int64_t arena_pages = 0, n_b = 0;
  int slots = 0;
  if (staged) {
    arena_pages = arena_pages_of(arena_bytes, page_bytes, num_pages_used, &slots);
    if (arena_pages < 1) return fail(KVO_ERR_ARG, "%s: arena smaller than 2 pages", fn);
    if (!aligned16(arena)) return fail(KVO_ERR_ALIGN, "%s: arena alignment", fn);
    if (classify(arena, arena_bytes) != kDeviceMem)
      return fail(KVO_ERR_NOT_MAPPED, "%s: arena must be device memory", fn);
    n_b = (num_pages_used + arena_pages - 1) / arena_pages;
    if ((n_b + 1) * 4 > (int64_t)kPartitionSmem)
      return fail(KVO_ERR_UNSUPPORTED, "%s: %lld arena buckets (arena too small for the pages in use)", fn,
                  (long long)n_b);
  }
  const SparseWs lay = sparse_workspace(rows, n_q_heads, head_dim, k_pad, rows_per_launch, n_b);
  if (!workspace || workspace_bytes < lay.total || classify(workspace, lay.total) != kDeviceMem)
    return fail(KVO_ERR_WORKSPACE, "%s: workspace needs %zu bytes of device memory", fn, lay.total);
  uint32_t *err = device_error_word();
  if (!err) return fail(KVO_ERR_CUDA, "%s: device error word unavailable", fn);

  uint8_t *ws = (uint8_t *)workspace;
  float *run_acc = (float *)(ws + lay.run_acc);             // [rows][Hq][D]
  float *run_ml = (float *)(ws + lay.run_ml);               // [rows][Hq][2]
  float *part = (float *)(ws + lay.part);                   // one row block's chunk partials
  int32_t *grouped = (int32_t *)(ws + lay.grouped);         // staged: [rows][k_pad]
  int32_t *offs = (int32_t *)(ws + lay.offs);               // staged: [rows][n_b + 1]
  const int64_t rbk = row_block(rows, rows_per_launch);
  int chunk = 0, n_chunks = 0;

  DecodeArgs base;
  base.q_dtype = q_dtype;
  base.n_q_heads = (int)n_q_heads; base.n_kv_heads = (int)n_kv_heads;
  base.head_dim = (int)head_dim; base.group = (int)group;
  base.kv_dtype = dtype; base.row_bytes = rb;
  base.ctx_len = nullptr; base.max_ctx = k_pad; base.n_vram = 0; base.hi_device = 0;
  base.lo_seq_stride_rows = 0; base.hi_seq_stride_rows = 0;
  base.scale_log2 = scale * 1.4426950408889634f;
  base.k_hi = (const uint8_t *)k_pages; base.v_hi = (const uint8_t *)v_pages;
  base.block_table = block_table; base.page_size = page_size; base.n_pages_total = n_pages;
  base.err = err;
  base.k_lo = base.v_lo = nullptr;

  if (staged) {
    // group every row's picks by bucket once
    if (k_pad > 0) {
      int warps = (int)(kPartitionSmem / ((n_b + 1) * 4));
      if (warps > 8) warps = 8;
      const size_t smem = (size_t)warps * (n_b + 1) * 4;
      cudaError_t e = cudaFuncSetAttribute(partition_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return cuda_status(e, "partition smem attribute");
      partition_kernel<<<(unsigned)((rows + warps - 1) / warps), 32 * warps, smem, st>>>(
          indices, rows, k_pad, num_pages_used * page_size, arena_pages * page_size, (int)n_b, grouped, offs);
      e = cudaGetLastError();
      if (e != cudaSuccess) return cuda_status(e, "partition kernel launch");
    } else {
      const cudaError_t e = cudaMemsetAsync(offs, 0, (size_t)rows * (n_b + 1) * 4, st);
      if (e != cudaSuccess) return cuda_status(e, "cudaMemsetAsync");
    }
  }

  // Two slots: slot bk % 2 is gathered on the library's side stream once the
  // caller's stream has finished scoring the bucket that used it before.
  static std::mutex ring_mu;
  std::unique_lock<std::mutex> lock(ring_mu, std::defer_lock);
  Ring *rg = nullptr;
  if (staged && slots == 2) {
    lock.lock();
    rg = ring(1);
    if (!rg) return fail(KVO_ERR_CUDA, "%s: library streams unavailable", fn);
    int e = cuda_status(cudaEventRecord(rg->fork, st), "cudaEventRecord");
    if (!e) e = cuda_status(cudaStreamWaitEvent(rg->side, rg->fork, 0), "cudaStreamWaitEvent");
    if (e) return e;
  }
  const size_t slot_bytes = 2 * (size_t)arena_pages * page_bytes;
  const int64_t n_buckets = staged ? n_b : 1;
  for (int64_t bk = 0; bk < n_buckets; ++bk) {
    const int64_t p0 = bk * arena_pages;
    const int64_t np = staged ? (num_pages_used - p0 < arena_pages ? num_pages_used - p0 : arena_pages) : 0;
    const int slot = rg ? (int)(bk & 1) : 0;
    if (staged) {
      base.k_lo = (const uint8_t *)arena + slot * slot_bytes;
      base.v_lo = base.k_lo + (size_t)arena_pages * page_bytes;
      cudaStream_t gs = rg ? rg->side : st;
      if (rg && bk >= 2) {
        const int e = cuda_status(cudaStreamWaitEvent(gs, rg->freed[slot], 0), "cudaStreamWaitEvent");
        if (e) return e;
      }
      const cudaError_t e = launch_page_gather(k_pages, v_pages, page_bytes, block_table, p0, np, n_pages,
                                               (void *)base.k_lo, (void *)base.v_lo, err,
                                               rg != nullptr, gs);
      if (e != cudaSuccess) return cuda_status(e, "page gather launch");
      if (rg) {
        int e2 = cuda_status(cudaEventRecord(rg->ready[slot], gs), "cudaEventRecord");
        if (!e2) e2 = cuda_status(cudaStreamWaitEvent(st, rg->ready[slot], 0), "cudaStreamWaitEvent");
        if (e2) return e2;
      }
    }
    for (int64_t r0 = 0; r0 < rows; r0 += rbk) {
      const int64_t nr = rows - r0 < rbk ? rows - r0 : rbk;
      DecodeArgs a = base;
      a.q = (const uint16_t *)q + (size_t)r0 * n_q_heads * head_dim;
      a.batch = (int)nr;
      sparse_geometry(nr, k_pad, &chunk, &n_chunks);
      a.split_cells = chunk; a.n_splits = n_chunks;
      a.part_acc = part;
      a.part_ml = part + (size_t)nr * n_chunks * n_q_heads * head_dim;
      a.out = out + (size_t)r0 * n_q_heads * head_dim;
      if (staged) {
        a.sparse_staged = 1;
        a.all_ring = 1;
        if (rg && num_sms() > 2 * kGatherSms) a.grid_cap = num_sms() - kGatherSms;
        a.indices = grouped + (size_t)r0 * k_pad;
        a.offs = offs + (size_t)r0 * (n_b + 1);
        a.offs_stride = n_b + 1;
        a.bucket = bk;
        a.win_lo = p0 * page_size;
        a.win_hi = (p0 + np) * page_size;
        a.run_acc = run_acc + (size_t)r0 * n_q_heads * head_dim;
        a.run_ml = run_ml + (size_t)r0 * n_q_heads * 2;
        a.init = bk == 0;
        a.finalize = bk == n_buckets - 1;
        if (n_chunks == 1) {                 // one chunk per row: the split kernel folds it
          a.fold_in_split = 1;
          a.phase = 1;
        }
      } else {
        a.sparse_staged = 0;
        a.indices = indices + (size_t)r0 * k_pad;
        a.win_lo = 0;
        a.win_hi = num_pages_used * page_size;
      }
      const int e = launch_sparse_rows(a, st);
      if (e) return e;
    }
    if (rg) {
      const int e = cuda_status(cudaEventRecord(rg->freed[slot], st), "cudaEventRecord");
      if (e) return e;
    }
  }
  return KVO_OK;
}

// ExLlamaV3 qsa-kv-offload patch, copy_page: host-resident pages are copied
// by the CPU after the device stream is drained (a page may still be read or
// written by queued GPU work, and a host memcpy is outside the stream's
// ordering).
extern "C" int kvo_copy_pages_host(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                                   int64_t page_tokens, int64_t token_bytes, int64_t from_page,
                                   int64_t to_page, int64_t num_tokens, void *stream) {
  clear_error();
  const char *fn = "kvo_copy_pages_host";
  if (page_tokens < 1 || token_bytes < 1 || from_page < 0 || to_page < 0 || num_tokens < 0 ||
      num_tokens > page_tokens)
    return fail(KVO_ERR_ARG, "%s: bad size", fn);
  if (!src_k || !src_v || !dst_k || !dst_v) return fail(KVO_ERR_ARG, "%s: NULL plane", fn);
  const size_t off_src = (size_t)from_page * page_tokens * token_bytes;
  const size_t off_dst = (size_t)to_page * page_tokens * token_bytes;
  const size_t bytes = (size_t)num_tokens * token_bytes;
  const void *ptrs[4] = {src_k, src_v, dst_k, dst_v};
  for (const void *p : ptrs) {
    if (classify(p, 1) == kDeviceMem) return fail(KVO_ERR_NOT_MAPPED, "%s: planes must be host memory", fn);
    // a VMM tier's tail is host memory mapped for the device only: the CPU
    // has no mapping of it
    if (vmm_host_backed(p) >= 0)
      return fail(KVO_ERR_NOT_MAPPED, "%s: VMM tier memory is not host-addressable", fn);
  }
  const cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e, "cudaStreamSynchronize");
  if (bytes == 0) return KVO_OK;
  memmove((uint8_t *)dst_k + off_dst, (const uint8_t *)src_k + off_src, bytes);
  memmove((uint8_t *)dst_v + off_dst, (const uint8_t *)src_v + off_src, bytes);
  return KVO_OK;
}
