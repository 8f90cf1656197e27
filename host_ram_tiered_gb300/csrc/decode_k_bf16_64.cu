// Split kernels of the tiered decode: bf16 K/V, head_dim 64 (see decode_impl.cuh).
#include "decode_impl.cuh"

namespace kvo {
namespace dec {
#define KVO_LAUNCH_D(G) \
  template cudaError_t launch_d<KVO_BF16, KVO_BF16, G, 64, false>(const DecodeArgs &, cudaStream_t);
KVO_LAUNCH_D(1) KVO_LAUNCH_D(2) KVO_LAUNCH_D(3) KVO_LAUNCH_D(4)
KVO_LAUNCH_D(5) KVO_LAUNCH_D(6) KVO_LAUNCH_D(7) KVO_LAUNCH_D(8)
#undef KVO_LAUNCH_D
}  // namespace dec
}  // namespace kvo
