// Explicit instantiations of the attention backward kernels, Dqk = 128,
// Dv = 64, bf16 storage: the dQ pass and the dK / dV pass, each without and with a bias / mask.
#include "attn_bwd_kernel.cuh"

namespace attn {
template cudaError_t launch_attn_bwd<128, 64, false, false, false>(const BwdParams&, int, cudaStream_t);
template cudaError_t launch_attn_bwd<128, 64, false, false, true>(const BwdParams&, int, cudaStream_t);
template cudaError_t launch_attn_bwd<128, 64, true, false, false>(const BwdParams&, int, cudaStream_t);
template cudaError_t launch_attn_bwd<128, 64, true, false, true>(const BwdParams&, int, cudaStream_t);
}  // namespace attn
