// Tiered-decode dispatch for f16 K/V (kernels: decode_k_f16_*.cu).
#include "decode_dispatch.cuh"

namespace kvo {
namespace dec {
template cudaError_t launch_kv<KVO_F16, false>(const DecodeArgs &a, cudaStream_t st);
}  // namespace dec
}  // namespace kvo
