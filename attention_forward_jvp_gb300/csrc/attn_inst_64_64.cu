// Instantiations of the attention kernel for Dqk = 64, Dv = 64
// (with and without tangents, each bias / mask mode); one file per head-dim pair so the build
// compiles them in parallel.
#include "attn_kernel.cuh"

namespace attn {
template cudaError_t launch_attn<64, 64, true, kNoBias>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, true, kBiasRing>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, true, kBiasGlobal>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, false, kNoBias>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, false, kBiasRing>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 64, false, kBiasGlobal>(const KernelParams&, int, cudaStream_t);
}  // namespace attn
