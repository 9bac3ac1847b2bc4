// Instantiations of the attention kernel for Dqk = 256, Dv = 64, fp16
// storage.  With tangents: no bias / mask, or bias / mask read per thread
// (Q and tQ take 128 KB of shared memory, which leaves no room for a bias
// ring); without tangents every bias / mask mode.
#include "attn_kernel.cuh"

namespace attn {
template cudaError_t launch_attn<256, 64, true, kNoBias, true>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<256, 64, true, kBiasGlobal, true>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<256, 64, false, kNoBias, true>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<256, 64, false, kBiasRing, true>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<256, 64, false, kBiasGlobal, true>(const KernelParams&, int, cudaStream_t);
}  // namespace attn
