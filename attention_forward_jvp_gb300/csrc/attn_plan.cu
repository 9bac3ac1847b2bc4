// Work list for jagged launches: every (sequence, row tile) pair that has
// rows, ordered by decreasing cost (the 64-wide tiles it streams), so that
// the attention kernels' snake walk over the list gives each SM a
// near-equal share (longest-processing-time-first).  One block, counting
// sort by cost.
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_plan.h"

namespace attn {

namespace {

constexpr int kPlanThreads = 512;

__device__ __forceinline__ int pair_cost(int len, int mt, int causal, int kv) {
  if (kv) {
    // the queries of a key tile: from its first row on under the causal mask
    const int all = (len + kPlanBN - 1) / kPlanBN;
    return causal ? all - mt * (kPlanBM / kPlanBN) : all;
  }
  const int hi = causal ? min(len, (mt + 1) * kPlanBM) : len;
  return (hi + kPlanBN - 1) / kPlanBN;
}

__global__ void __launch_bounds__(kPlanThreads) plan_jagged_kernel(const int* offsets, int B,
                                                                   int max_seq_len, int causal,
                                                                   int2* list, int* count,
                                                                   int capacity, int kv) {
  extern __shared__ int bins[];  // one counter per cost 0 .. nbins-1
  // the attention kernel after this one may start its prologue now (it
  // waits for this kernel to complete before it reads the list)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int nbins = (max_seq_len + kPlanBN - 1) / kPlanBN + 1;
  for (int i = threadIdx.x; i < nbins; i += blockDim.x) bins[i] = 0;
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int len = min(offsets[b + 1] - offsets[b], max_seq_len);
    for (int mt = 0; mt * kPlanBM < len; ++mt) atomicAdd(&bins[pair_cost(len, mt, causal, kv)], 1);
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
      const int pos = atomicAdd(&bins[pair_cost(len, mt, causal, kv)], 1);
      list[pos] = make_int2(b, mt);
    }
  }
}

// Key length of each (b, h) under a key mask that does not depend on the
// query row: one block per (b, h) finds the last key j < N whose mask byte
// is nonzero and the first key whose byte is zero, and writes j + 1 (0 when
// none), with bit 31 set when no key below j + 1 is masked (the mask is a
// key prefix).  Keys at or past j + 1 are masked for every row, so the
// attention kernel need not visit them; under a prefix it need not read
// the mask at all.
__global__ void __launch_bounds__(256) plan_keylen_kernel(const unsigned char* mask, long long s0,
                                                          long long s1, long long s3, int H, int N,
                                                          int* keylen) {
  // the attention kernel after this one may start its prologue now (it
  // waits for this kernel to complete before it reads the key lengths)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh % H;
  const unsigned char* row = mask + b * s0 + h * s1;
  int last = -1, first_zero = N;
  if (s3 == 1 && (reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
    // 16 keys per load: a key row of up to 4096 bytes in one pass
    for (int j0 = threadIdx.x * 16; j0 < N; j0 += blockDim.x * 16) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (j0 + 16 <= N) {
        v = __ldg(reinterpret_cast<const uint4*>(row + j0));
      } else {
        unsigned char t[16] = {};
        for (int c = 0; j0 + c < N; ++c) t[c] = row[j0 + c];
        v = make_uint4(t[0] | t[1] << 8 | t[2] << 16 | static_cast<uint32_t>(t[3]) << 24,
                       t[4] | t[5] << 8 | t[6] << 16 | static_cast<uint32_t>(t[7]) << 24,
                       t[8] | t[9] << 8 | t[10] << 16 | static_cast<uint32_t>(t[11]) << 24,
                       t[12] | t[13] << 8 | t[14] << 16 | static_cast<uint32_t>(t[15]) << 24);
      }
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        if (j0 + c >= N) break;
        if ((w[c >> 2] >> ((c & 3) * 8)) & 0xffu) last = j0 + c;
        else first_zero = min(first_zero, j0 + c);
      }
    }
  } else {
    for (int j = threadIdx.x; j < N; j += blockDim.x) {
      if (row[j * s3] != 0) last = j;
      else first_zero = min(first_zero, j);
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    first_zero = min(first_zero, __shfl_xor_sync(0xffffffffu, first_zero, o));
  }
  __shared__ int wmax[8], wmin[8];
  if ((threadIdx.x & 31) == 0) {
    wmax[threadIdx.x >> 5] = last;
    wmin[threadIdx.x >> 5] = first_zero;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int m = -1, z = N;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
      m = max(m, wmax[w]);
      z = min(z, wmin[w]);
    }
    const bool prefix = z > m;  // keys 0 .. m all attended
    keylen[bh] = (m + 1) | (prefix ? static_cast<int>(0x80000000u) : 0);
  }
}

}  // namespace

cudaError_t launch_plan_keylen(const unsigned char* mask, const long long* stride, int B, int H, int N,
                               int* keylen, cudaStream_t stream) {
  plan_keylen_kernel<<<B * H, 256, 0, stream>>>(mask, stride[0], stride[1], stride[3], H, N, keylen);
  return cudaGetLastError();
}

bool plan_jagged_supported(int max_seq_len) { return max_seq_len >= 0 && max_seq_len <= kPlanMaxSeqLen; }

cudaError_t launch_plan_jagged(const int* offsets, int B, int max_seq_len, int causal, int2* list,
                               int* count, int capacity, cudaStream_t stream, int kv) {
  const int nbins = (max_seq_len + kPlanBN - 1) / kPlanBN + 1;
  const size_t smem = static_cast<size_t>(nbins) * sizeof(int);
  plan_jagged_kernel<<<1, kPlanThreads, smem, stream>>>(offsets, B, max_seq_len, causal, list,
                                                        count, capacity, kv);
  return cudaGetLastError();
}

}  // namespace attn
