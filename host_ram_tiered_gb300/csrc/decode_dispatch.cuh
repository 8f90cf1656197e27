// Dispatch of the tiered-decode kernels over the group shape: which
// heads-per-warp instantiation of launch_d serves a call.  launch_d itself
// (decode_impl.cuh) is instantiated in the decode_k_*.cu units, one per K/V
// dtype, head_dim and mode, so that they compile in parallel.
#pragma once
#include "kvo_internal.cuh"

namespace kvo {
namespace dec {

template <int KVT, int QT, int G, int D, bool SP>
cudaError_t launch_d(const DecodeArgs &a, cudaStream_t st);

template <int KVT, int QT, int G, bool SP>
cudaError_t launch_g(const DecodeArgs &a, cudaStream_t st) {
  if (a.head_dim == 128) return launch_d<KVT, QT, G, 128, SP>(a, st);
  return launch_d<KVT, QT, G, 64, SP>(a, st);
}

// Warps per kv head: the largest power of two w dividing the group with
// n_kv_heads * w <= 8 warps, or <= 16 warps when each warp is then left with
// at most two query heads; each warp takes group / w query heads.
inline int warps_per_kv_head(const DecodeArgs &a) {
  int w = 1;
  while (a.group % (w * 2) == 0) {
    const int warps = a.n_kv_heads * w * 2, heads = a.group / (w * 2);
    if (warps > (heads <= 2 ? 16 : 8)) break;
    w *= 2;
  }
  return w;
}

// The query type is the cache's 16-bit type (fp16 for a q8_0 cache); the
// entry points reject other pairs.
template <int KVT, bool SP = false>
cudaError_t launch_kv(const DecodeArgs &a, cudaStream_t st) {
  constexpr int QT = KVT == KVO_BF16 ? KVO_BF16 : KVO_F16;
  switch (a.group / warps_per_kv_head(a)) {
    case 1: return launch_g<KVT, QT, 1, SP>(a, st);
    case 2: return launch_g<KVT, QT, 2, SP>(a, st);
    case 3: return launch_g<KVT, QT, 3, SP>(a, st);
    case 4: return launch_g<KVT, QT, 4, SP>(a, st);
    case 5: return launch_g<KVT, QT, 5, SP>(a, st);
    case 6: return launch_g<KVT, QT, 6, SP>(a, st);
    case 7: return launch_g<KVT, QT, 7, SP>(a, st);
    default: return launch_g<KVT, QT, 8, SP>(a, st);
  }
}

}  // namespace dec
}  // namespace kvo
