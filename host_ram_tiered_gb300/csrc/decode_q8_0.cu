// Tiered-decode dispatch for q8_0 K/V (kernels: decode_k_q8_0_*.cu).
#include "decode_dispatch.cuh"

namespace kvo {
namespace dec {
template cudaError_t launch_kv<KVO_Q8_0, false>(const DecodeArgs &a, cudaStream_t st);
}  // namespace dec
}  // namespace kvo
