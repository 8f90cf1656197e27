// Decode kernels for bf16 K/V (see decode_impl.cuh).
#include "decode_impl.cuh"

namespace kvo {
namespace dec {
template cudaError_t launch_kv<KVO_BF16, false>(const DecodeArgs &a, cudaStream_t st);
}  // namespace dec
}  // namespace kvo
