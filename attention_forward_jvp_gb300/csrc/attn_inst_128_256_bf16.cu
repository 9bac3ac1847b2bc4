// Instantiations of the attention kernel for Dqk = 128, Dv = 256, bf16
// storage: forward only (each bias / mask mode).  With tangents, Dv = 256
// runs as two column slices of the Dqk = 128, Dv = 128 kernel.
#include "attn_kernel.cuh"

namespace attn {
template cudaError_t launch_attn<128, 256, false, kNoBias, false>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<128, 256, false, kBiasRing, false>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<128, 256, false, kBiasGlobal, false>(const KernelParams&, int, cudaStream_t);
}  // namespace attn
