// Tiered decode: split geometry, workspace size and dtype dispatch.  The
// kernels themselves live in decode_impl.cuh.
#include "kvo_internal.cuh"

namespace kvo {
namespace dec {
template <int KVT> cudaError_t launch_kv(const DecodeArgs &a, cudaStream_t st);
constexpr int kMinSplit = 64;
}  // namespace dec

void decode_geometry(int64_t batch, int64_t max_ctx, int64_t head_dim, int *split_cells,
                     int *n_splits) {
  (void)head_dim;
  // About four CTAs per SM over the whole batch; splits are multiples of 32
  // cells (every tile size divides them) and at least kMinSplit cells.
  const int64_t target = (int64_t)num_sms() * 4;
  int64_t per = (max_ctx * (batch > 0 ? batch : 1) + target - 1) / target;
  per = (per + 31) / 32 * 32;
  if (per < dec::kMinSplit) per = dec::kMinSplit;
  *split_cells = (int)per;
  const int64_t ns = (max_ctx + per - 1) / per;
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
  if (a.kv_dtype == KVO_Q8_0) e = dec::launch_kv<KVO_Q8_0>(a, st);
  else if (a.kv_dtype == KVO_BF16) e = dec::launch_kv<KVO_BF16>(a, st);
  else e = dec::launch_kv<KVO_F16>(a, st);
  return cuda_status(e, "decode kernel launch");
}

}  // namespace kvo
