// Jagged work-list planning (see attn_plan.cu).
#pragma once
#include <cuda_runtime.h>

namespace attn {

constexpr int kPlanBM = 128;             // query rows per work unit
constexpr int kPlanBN = 64;              // keys per pipeline step
constexpr int kPlanMaxSeqLen = 65536;    // cost bins held in shared memory
constexpr int kPlanListBytes = 1 << 20;  // list capacity in the per-device scratch

bool plan_jagged_supported(int max_seq_len);

// Writes count[0] = number of (sequence, query tile) pairs with rows (or -1
// when more than `capacity`) and list[0 .. count) = those pairs as
// (sequence, tile), costliest first.  Asynchronous on `stream`.
cudaError_t launch_plan_jagged(const int* offsets, int B, int max_seq_len, int causal, int2* list,
                               int* count, int capacity, cudaStream_t stream);

}  // namespace attn
