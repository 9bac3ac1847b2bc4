// Work list for jagged launches: every (sequence, query tile) pair that has
// rows, ordered by decreasing cost (key tiles it visits), so that the
// attention kernel's snake walk over the list gives each SM a near-equal
// share (longest-processing-time-first).  One block, counting sort by cost.
#include <cuda_runtime.h>

#include "attn_plan.h"

namespace attn {

namespace {

constexpr int kPlanThreads = 512;

__device__ __forceinline__ int pair_cost(int len, int mt, int causal) {
  const int hi = causal ? min(len, (mt + 1) * kPlanBM) : len;
  return (hi + kPlanBN - 1) / kPlanBN;
}

__global__ void __launch_bounds__(kPlanThreads) plan_jagged_kernel(const int* offsets, int B,
                                                                   int max_seq_len, int causal,
                                                                   int2* list, int* count,
                                                                   int capacity) {
  extern __shared__ int bins[];  // one counter per cost 0 .. nbins-1
  const int nbins = (max_seq_len + kPlanBN - 1) / kPlanBN + 1;
  for (int i = threadIdx.x; i < nbins; i += blockDim.x) bins[i] = 0;
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int len = min(offsets[b + 1] - offsets[b], max_seq_len);
    for (int mt = 0; mt * kPlanBM < len; ++mt) atomicAdd(&bins[pair_cost(len, mt, causal)], 1);
  }
  __syncthreads();
  __shared__ int total;
  if (threadIdx.x == 0) {  // bin starts, costliest bin first
    int acc = 0;
    for (int c = nbins - 1; c >= 0; --c) {
      const int n = bins[c];
      bins[c] = acc;
      acc += n;
    }
    total = acc;
    count[0] = acc <= capacity ? acc : -1;  // -1: list not written, use the slot order
  }
  __syncthreads();
  if (total > capacity) return;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int len = min(offsets[b + 1] - offsets[b], max_seq_len);
    for (int mt = 0; mt * kPlanBM < len; ++mt) {
      const int pos = atomicAdd(&bins[pair_cost(len, mt, causal)], 1);
      list[pos] = make_int2(b, mt);
    }
  }
}

}  // namespace

bool plan_jagged_supported(int max_seq_len) { return max_seq_len >= 0 && max_seq_len <= kPlanMaxSeqLen; }

cudaError_t launch_plan_jagged(const int* offsets, int B, int max_seq_len, int causal, int2* list,
                               int* count, int capacity, cudaStream_t stream) {
  const int nbins = (max_seq_len + kPlanBN - 1) / kPlanBN + 1;
  const size_t smem = static_cast<size_t>(nbins) * sizeof(int);
  plan_jagged_kernel<<<1, kPlanThreads, smem, stream>>>(offsets, B, max_seq_len, causal, list,
                                                        count, capacity);
  return cudaGetLastError();
}

}  // namespace attn
