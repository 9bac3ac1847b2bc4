// Instantiations of the attention kernel for Dqk = Dv = 256, bf16 storage,
// forward only (each bias / mask mode).
#include "attn_kernel.cuh"

namespace attn {
template cudaError_t launch_attn<256, 256, false, kNoBias, false>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<256, 256, false, kBiasRing, false>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<256, 256, false, kBiasGlobal, false>(const KernelParams&, int, cudaStream_t);
}  // namespace attn
