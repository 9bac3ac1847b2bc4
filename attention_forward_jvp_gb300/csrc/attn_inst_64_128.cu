// Instantiations of the attention kernel for Dqk = 64, Dv = 128
// (with and without tangents); one file per head-dim pair so the build
// compiles them in parallel.
#include "attn_kernel.cuh"

namespace attn {
template cudaError_t launch_attn<64, 128, true>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<64, 128, false>(const KernelParams&, int, cudaStream_t);
}  // namespace attn
