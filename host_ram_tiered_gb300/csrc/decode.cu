// Tiered decode: split geometry, workspace size and dtype dispatch.  The
// kernels themselves live in decode_impl.cuh.
#include "kvo_internal.cuh"

namespace kvo {
namespace dec {
template <int KVT, bool SP> cudaError_t launch_kv(const DecodeArgs &a, cudaStream_t st);
constexpr int kMaxChunkTiles = 20;   // chunks of at most 640 cells
}  // namespace dec

void decode_geometry(int64_t batch, int64_t max_ctx, int64_t head_dim, int *split_cells,
                     int *n_splits) {
  (void)head_dim;
  // Chunk length C (32..640 cells, whole 32-cell tiles) minimising the tiles
  // of the busiest CTA when batch * ceil(max_ctx / C) chunks are dealt
  // round-robin to one persistent CTA per SM; ties go to the longer chunk
  // (fewer partials to combine).
  const int64_t sms = num_sms();
  const int64_t bt = batch > 0 ? batch : 1;
  int64_t best_c = 32, best_cost = -1;
  for (int64_t tiles = 1; tiles <= dec::kMaxChunkTiles; ++tiles) {
    const int64_t c = tiles * 32;
    const int64_t chunks = (max_ctx + c - 1) / c;
    const int64_t waves = (bt * chunks + sms - 1) / sms;
    const int64_t cost = (waves > 0 ? waves : 1) * tiles;
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

}  // namespace kvo
