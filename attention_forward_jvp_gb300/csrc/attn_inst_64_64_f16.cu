// Instantiations of the attention kernel for Dqk = 64, Dv = 64, f16
// storage (with and without tangents, each bias / mask mode); one file per
// head-dim pair and element type so the build compiles them in parallel.
#include "attn_kernel.cuh"

namespace attn {
template cudaError_t launch_attn<64, 64, true, kNoBias, true>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, true, kBiasRing, true>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, true, kBiasGlobal, true>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, false, kNoBias, true>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, false, kBiasRing, true>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, false, kBiasGlobal, true>(const KernelParams&, int, cudaStream_t);
// the lean ping-pong variants (dense, non-causal, whole key tiles)
template cudaError_t launch_attn<64, 64, true, kNoBias, true, false, true>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, false, kNoBias, true, false, true>(const KernelParams&, int, cudaStream_t);
}  // namespace attn
