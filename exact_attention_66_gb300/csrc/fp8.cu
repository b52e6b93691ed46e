// FP8 path (placeholder until the e4m3 kernels land).
#include "launch.h"
namespace attn {
cudaError_t launch_fwd_fp8(const Fp8Launch&, bool, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_hadamard_quant(const void*, const void*, const void*, void*, void*, void*, float*,
                                  const int8_t*, int, int, int, int, unsigned*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace attn
