// Instantiations of the attention kernel for Dqk = 64, Dv = 256, fp16
// storage: forward only (each bias / mask mode).  With tangents, Dv = 256
// runs as two column slices of the Dqk = 64, Dv = 128 kernel.
#include "attn_kernel.cuh"

namespace attn {
template cudaError_t launch_attn<64, 256, false, kNoBias, true>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 256, false, kBiasRing, true>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 256, false, kBiasGlobal, true>(const KernelParams&, int, cudaStream_t);
}  // namespace attn
