// Explicit instantiations of the attention backward kernels, Dqk = 128,
// Dv = 128, f16 storage: the dQ pass and the dK / dV pass, each without and with a bias / mask.
#include "attn_bwd_kernel.cuh"

namespace attn {
template cudaError_t launch_attn_bwd<128, 128, false, true, false>(const BwdParams&, int, cudaStream_t);
template cudaError_t launch_attn_bwd<128, 128, false, true, true>(const BwdParams&, int, cudaStream_t);
template cudaError_t launch_attn_bwd<128, 128, true, true, false>(const BwdParams&, int, cudaStream_t);
template cudaError_t launch_attn_bwd<128, 128, true, true, true>(const BwdParams&, int, cudaStream_t);
}  // namespace attn
