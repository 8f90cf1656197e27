// Tiered-decode dispatch for bf16 K/V (kernels: decode_k_bf16_*.cu).
#include "decode_dispatch.cuh"

namespace kvo {
namespace dec {
template cudaError_t launch_kv<KVO_BF16, false>(const DecodeArgs &a, cudaStream_t st);
}  // namespace dec
}  // namespace kvo
