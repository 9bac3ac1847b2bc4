// Instantiations of the attention kernel for Dqk = 64, Dv = 64, bf16
// storage (with and without tangents, each bias / mask mode); one file per
// head-dim pair and element type so the build compiles them in parallel.
#include "attn_kernel.cuh"

namespace attn {
template cudaError_t launch_attn<64, 64, true, kNoBias, false>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, true, kBiasRing, false>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, true, kBiasGlobal, false>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, false, kNoBias, false>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, false, kBiasRing, false>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, false, kBiasGlobal, false>(const KernelParams&, int, cudaStream_t);
// the lean ping-pong variants (dense, non-causal, whole key tiles)
template cudaError_t launch_attn<64, 64, true, kNoBias, false, false, true>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, false, kNoBias, false, false, true>(const KernelParams&, int, cudaStream_t);
}  // namespace attn
