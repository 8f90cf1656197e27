// Tiered decode: split geometry, workspace size and dtype dispatch.  The
// kernels themselves live in decode_impl.cuh.
#include <mutex>

#include "kvo_internal.cuh"

namespace kvo {
namespace dec {
template <int KVT, bool SP> cudaError_t launch_kv(const DecodeArgs &a, cudaStream_t st);
constexpr int kMaxChunkTiles = 20;   // chunks of at most 640 cells
}  // namespace dec

void decode_geometry(int64_t batch, int64_t max_ctx, int64_t head_dim, int *split_cells,
                     int *n_splits) {
  (void)head_dim;
  // Chunk length C (32..640 cells, whole 32-cell tiles) minimising the work
  // of the busiest CTA when batch * ceil(max_ctx / C) chunks are dealt
  // round-robin to one persistent CTA per SM: its waves times (the chunk's
  // tiles plus a fixed cost of kChunkCostTiles per chunk -- the query load,
  // the pipeline fill, the partial and its share of the combine); ties go to
  // the longer chunk (fewer partials to combine).  Without the fixed cost a
  // context such as 110,592 cells came out as 3,456 chunks of 32 cells
  // (753 us against 212 us for 102,400 cells).
  constexpr int64_t kChunkCostTiles = 2;
  const int64_t sms = num_sms();
  const int64_t bt = batch > 0 ? batch : 1;
  int64_t best_c = 32, best_cost = -1;
  for (int64_t tiles = 1; tiles <= dec::kMaxChunkTiles; ++tiles) {
    const int64_t c = tiles * 32;
    const int64_t chunks = (max_ctx + c - 1) / c;
    const int64_t waves = (bt * chunks + sms - 1) / sms;
    const int64_t cost = (waves > 0 ? waves : 1) * (tiles + kChunkCostTiles);
    if (best_cost < 0 || cost <= best_cost) {
      best_cost = cost;
      best_c = c;
    }
    if (chunks <= 1) break;                 // longer chunks change nothing
  }
  *split_cells = (int)best_c;
  const int64_t ns = (max_ctx + best_c - 1) / best_c;
  *n_splits = (int)(ns > 0 ? ns : 1);
}

size_t decode_workspace_bytes(int64_t batch, int64_t n_q_heads, int64_t head_dim, int64_t max_ctx) {
  int sc, ns;
  decode_geometry(batch, max_ctx, head_dim, &sc, &ns);
  const size_t parts = (size_t)batch * ns * n_q_heads;
  return parts * head_dim * sizeof(float) + parts * 2 * sizeof(float);
}

int launch_decode(const DecodeArgs &a, cudaStream_t st) {
  cudaError_t e;
  if (a.kv_dtype == KVO_Q8_0) e = dec::launch_kv<KVO_Q8_0, false>(a, st);
  else if (a.kv_dtype == KVO_BF16) e = dec::launch_kv<KVO_BF16, false>(a, st);
  else e = dec::launch_kv<KVO_F16, false>(a, st);
  return cuda_status(e, "decode kernel launch");
}

StagedPlan staged_plan(int64_t batch, int split_cells, int n_splits, int64_t n_vram) {
  // The chunks wholly in VRAM are decoded first, then the chunks of each copy
  // part as soon as it has landed while the next part is in flight.  A launch
  // lasts about one chunk time per wave of its items over the SMs, so this
  // only pays when the items fill more than one wave: then there is one part
  // per wave of host chunks (at most four), else a single part and a single
  // launch after the whole copy.
  StagedPlan pl;
  const int64_t sms = num_sms();
  const bool multi_wave = batch * n_splits > sms;
  pl.c_v = multi_wave ? n_vram / split_cells : 0;
  const int64_t hc = n_splits - pl.c_v;          // >= 1: the last chunk holds host rows
  const int64_t waves = (batch * hc + sms - 1) / sms;
  pl.parts = multi_wave ? (waves < 4 ? (int)waves : 4) : 1;
  for (int p = 0; p < pl.parts; ++p) {           // even parts of the chunks [c_v, n_splits)
    pl.ch_lo[p] = pl.c_v + hc * p / pl.parts;
    pl.ch_hi[p] = pl.c_v + hc * (p + 1) / pl.parts;
  }
  return pl;
}

int launch_decode_staged(DecodeArgs a, const void *k_host, const void *v_host, int64_t host_stride,
                         void *staging_k, void *staging_v, cudaStream_t st) {
  // The copy runs on a library stream in the parts of staged_plan.  A chunk's
  // partial is the same whichever launch computes it, so the one combine at
  // the end gives the bits of a single launch over an all-VRAM cache.
  const int64_t C = a.split_cells, n_lo = a.n_vram, n_hi = a.max_ctx - a.n_vram;
  const size_t rb = (size_t)a.row_bytes;
  const StagedPlan pl = staged_plan(a.batch, a.split_cells, a.n_splits, n_lo);
  const int parts = pl.parts;
  const int64_t c_v = pl.c_v;
  if (parts == 1 && c_v == 0) {                  // one wave: copy, then one launch, on `st`
    for (int64_t b = 0; b < a.batch; ++b) {
      const size_t bytes = (size_t)n_hi * rb;
      const size_t src = (size_t)b * host_stride * rb, dst = (size_t)b * n_hi * rb;
      int e = cuda_status(cudaMemcpyAsync((uint8_t *)staging_k + dst, (const uint8_t *)k_host + src, bytes,
                                          cudaMemcpyDefault, st), "staging copy K");
      if (!e) e = cuda_status(cudaMemcpyAsync((uint8_t *)staging_v + dst, (const uint8_t *)v_host + src, bytes,
                                              cudaMemcpyDefault, st), "staging copy V");
      if (e) return e;
    }
    a.k_hi = (const uint8_t *)staging_k;
    a.v_hi = (const uint8_t *)staging_v;
    a.hi_seq_stride_rows = n_hi;
    a.hi_device = 1;
    return launch_decode(a, st);
  }
  static std::mutex mu;                          // one staged call at a time uses the events
  std::lock_guard<std::mutex> lock(mu);
  Ring *rg = ring(2);
  if (!rg) return fail(KVO_ERR_CUDA, "staged decode: library streams unavailable");
  int e = cuda_status(cudaEventRecord(rg->fork, st), "cudaEventRecord");
  if (!e) e = cuda_status(cudaStreamWaitEvent(rg->side, rg->fork, 0), "cudaStreamWaitEvent");
  if (e) return e;
  const int64_t *ch_lo = pl.ch_lo, *ch_hi = pl.ch_hi;
  for (int p = 0; p < parts; ++p) {
    const int64_t r0 = ch_lo[p] * C > n_lo ? ch_lo[p] * C : n_lo;
    const int64_t r1 = ch_hi[p] * C < a.max_ctx ? ch_hi[p] * C : a.max_ctx;
    for (int64_t b = 0; b < a.batch && r1 > r0; ++b) {
      const size_t bytes = (size_t)(r1 - r0) * rb;
      const size_t src = ((size_t)b * host_stride + (size_t)(r0 - n_lo)) * rb;
      const size_t dst = ((size_t)b * n_hi + (size_t)(r0 - n_lo)) * rb;
      e = cuda_status(cudaMemcpyAsync((uint8_t *)staging_k + dst, (const uint8_t *)k_host + src, bytes,
                                      cudaMemcpyDefault, rg->side), "staging copy K");
      if (!e) e = cuda_status(cudaMemcpyAsync((uint8_t *)staging_v + dst, (const uint8_t *)v_host + src, bytes,
                                              cudaMemcpyDefault, rg->side), "staging copy V");
      if (e) return e;
    }
    e = cuda_status(cudaEventRecord(rg->part[p], rg->side), "cudaEventRecord");
    if (e) return e;
  }
  a.k_hi = (const uint8_t *)staging_k;
  a.v_hi = (const uint8_t *)staging_v;
  a.hi_seq_stride_rows = n_hi;
  a.hi_device = 1;
  a.phase = 1;
  if (c_v > 0) {
    a.item_lo = 0;
    a.item_hi = c_v * a.batch;
    e = launch_decode(a, st);
    if (e) return e;
  }
  for (int p = 0; p < parts; ++p) {
    e = cuda_status(cudaStreamWaitEvent(st, rg->part[p], 0), "cudaStreamWaitEvent");
    if (e) return e;
    a.item_lo = ch_lo[p] * a.batch;
    a.item_hi = ch_hi[p] * a.batch;
    e = launch_decode(a, st);
    if (e) return e;
  }
  a.phase = 2;
  return launch_decode(a, st);
}

}  // namespace kvo

// Measured staged/direct rule of the dense calls (include/kvo.h).
extern "C" int kvo_dense_staging_worthwhile(int prefill, int64_t n_vram_cells, int64_t n_tail_cells) {
  if (n_tail_cells <= 0 || n_vram_cells < 0) return 0;
  if (prefill) return 1;
  return n_vram_cells >= 65536 && 5 * n_tail_cells <= n_vram_cells ? 1 : 0;
}
