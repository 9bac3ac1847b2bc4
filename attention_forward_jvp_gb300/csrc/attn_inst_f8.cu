// Instantiations of the e5m2 (fp8) forward kernel: head dims 64 and 128,
// no tangents, no bias.
#include "attn_kernel.cuh"

namespace attn {
template cudaError_t launch_attn<64, 64, false, kNoBias, false, true>(const KernelParams&, int, cudaStream_t);
template cudaError_t launch_attn<128, 128, false, kNoBias, false, true>(const KernelParams&, int, cudaStream_t);
}  // namespace attn
