// Instantiations of the attention kernel for Dqk = 128, Dv = 128, bf16
// storage (with and without tangents, each bias / mask mode); one file per
// head-dim pair and element type so the build compiles them in parallel.
#include "attn_kernel.cuh"

namespace attn {
template cudaError_t launch_attn<128, 128, true, kNoBias, false>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<128, 128, true, kBiasRing, false>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<128, 128, true, kBiasGlobal, false>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<128, 128, false, kNoBias, false>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<128, 128, false, kBiasRing, false>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<128, 128, false, kBiasGlobal, false>(const KernelParams&, int, cudaStream_t);
}  // namespace attn
