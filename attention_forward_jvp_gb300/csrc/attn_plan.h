// Jagged work-list planning (see attn_plan.cu).
#pragma once
#include <cuda_runtime.h>

namespace attn {

constexpr int kPlanBM = 128;             // query rows per work unit
constexpr int kPlanBN = 64;              // keys per pipeline step
constexpr int kPlanMaxSeqLen = 65536;    // cost bins held in shared memory
constexpr int kPlanListBytes = 1 << 20;  // list capacity in the per-device scratch

bool plan_jagged_supported(int max_seq_len);

// Writes count[0] = number of (sequence, row tile) pairs with rows (or -1
// when more than `capacity`) and list[0 .. count) = those pairs as
// (sequence, tile), costliest first.  The cost of a pair is the number of
// 64-wide tiles its row tile streams: keys for a query tile (kv = 0, the
// forward and the backward's dQ pass), queries for a key tile (kv = 1, the
// backward's dK / dV pass: under the causal mask, those from the tile's
// first row to the sequence end).  Asynchronous on `stream`.
cudaError_t launch_plan_jagged(const int* offsets, int B, int max_seq_len, int causal, int2* list,
                               int* count, int capacity, cudaStream_t stream, int kv = 0);

// Writes keylen[b * H + h] = 1 + the last key j < N with mask[b, h, ., j]
// nonzero (0 when none), bit 31 set when every key below it is nonzero, for
// a [B, H, 1, N] view of a key mask that does not depend on the query row
// (element strides stride[0], stride[1], stride[3]).  One block per (b, h),
// asynchronous on `stream`.
cudaError_t launch_plan_keylen(const unsigned char* mask, const long long* stride, int B, int H, int N,
                               int* keylen, cudaStream_t stream);

}  // namespace attn
