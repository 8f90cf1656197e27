// Decode kernels for q8_0 K/V (see decode_impl.cuh).
#include "decode_impl.cuh"

namespace kvo {
namespace dec {
template cudaError_t launch_kv<KVO_Q8_0, false>(const DecodeArgs &a, cudaStream_t st);
}  // namespace dec
}  // namespace kvo
