// Instantiations of the attention kernel for Dqk = 128, Dv = 64
// (with and without tangents, with and without bias / mask); one file per head-dim pair so the build
// compiles them in parallel.
#include "attn_kernel.cuh"

namespace attn {
template cudaError_t launch_attn<128, 64, true, false>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<128, 64, true, true>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<128, 64, false, false>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<128, 64, false, true>(const KernelParams&, int, cudaStream_t);
}  // namespace attn
