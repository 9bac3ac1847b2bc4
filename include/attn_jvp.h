/*
 * attn_jvp.h -- C ABI of the fused attention forward + JVP library for
 * NVIDIA GB300 (sm_103a).
 *
 * One pass over the keys computes, for every query row i:
 *
 *   S   = sm_scale * Q K^T + bias          (keys outside the valid set: -inf)
 *   P   = softmax(S)                       (row-wise)
 *   O   = P V
 *   LSE = log sum_j exp(S_ij)              (natural log, fp32)
 *   tS  = sm_scale * (tQ K^T + Q tK^T)     (0 outside the valid set)
 *   tO  = P tV + (P o tS) V - rowsum(P o tS) o O
 *
 * which is the forward pass of softmax attention together with its
 * Jacobian-vector product along the tangents (tQ, tK, tV).  Sources:
 *   - "Flash Attention v2 with JVP" (flm/utils/jvp.py): _attn_fwd_inner
 *     (score tangent, running max m, denominator l and tangent sum r) and
 *     the _attn_fwd epilogue (O = acc / l, tO = (acc_A + acc_B - r O) / l,
 *     LSE as a natural log, empty-row guard);
 *   - "_06_fused_attention_blockptr_jvp.py" (Triton fused attention with
 *     JVP): the same epilogue written as g_acc/l - (mu/l) O + p_tv_acc/l;
 *   - "flash_attention.py" (triton_flashattn): _attn_fwd_inner additive
 *     bias after the sm_scale product, boolean mask (nonzero = attend),
 *     unequal head dims Dqk != Dv;
 *   - "triton_multi_head_jagged_flash_attention.py" (FBGEMM): jagged
 *     [H, T, D] layout with offsets[B + 1], lengths capped at max_seq_len.
 *
 * Valid set of row i: key j < key length; j <= i when causal (in-sequence
 * indices for jagged); mask[b,h,i,j] != 0 when a mask is given.  A row
 * whose valid set is empty gets O = tO = 0 and LSE = -inf.
 *
 * Conventions for every entry point:
 *   - Pointers q..lse are DEVICE pointers owned by the caller; the library
 *     keeps none of them after the call returns.  Every one of them must be
 *     16-byte aligned (bulk tensor copies), else ATTN_ERR_MISALIGNED.
 *   - q, k, v, tq, tk, tv, o, to are bf16 (raw 16-bit storage), lse fp32;
 *     the *_f16 entry points take fp16 instead of bf16.
 *   - Dense layouts (offsets == NULL), all contiguous, row-major:
 *       q, tq [B, H, M, Dqk]   k, tk [B, H, N, Dqk]   v, tv [B, H, N, Dv]
 *       o, to [B, H, M, Dv]    lse   [B, H, M]
 *   - Jagged layouts (offsets != NULL), packed total-token layout:
 *       q, k, tq, tk [H, T, Dqk]   v, tv, o, to [H, T, Dv]   lse [H, T]
 *     offsets is a device int32 array [B + 1], offsets[0] = 0,
 *     non-decreasing, offsets[B] <= T.  Sequence b owns tokens
 *     [offsets[b], offsets[b+1]) and attends within its first
 *     L_b = min(offsets[b+1] - offsets[b], max_seq_len) tokens; its rows
 *     past L_b are written as empty rows; rows >= offsets[B] are not
 *     written.  The device offsets are not checked by the host; keys of
 *     neighbouring sequences may be read by a tile and are masked, so the
 *     whole of v and tv must hold finite values.
 *   - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *     default stream).  Argument errors are returned synchronously and
 *     launch nothing.  A device-side failure (a pipeline wait that ran out
 *     of time) is recorded in a per-device error word and reported by the
 *     next attn_sync_check on that device.
 *   - Supported head dims (forward, with and without tangents): Dqk, Dv
 *     each in {16, 32, 64, 128, 256}, independently (16 and 32 run
 *     zero-padded to 64 inside the kernel); otherwise ATTN_ERR_UNSUPPORTED.
 *     With tangents, Dv = 256 runs as two work units per query tile, one
 *     per 128-column half of O and tO (O and tO of 256 columns each would
 *     fill the tensor memory), each recomputing the scores; Dqk = 256 with
 *     tangents keeps one key stage in shared memory beside Q and tQ.  Rows
 *     of every tensor are D elements, contiguous.
 *   - The library allocates, on first use, one small per-device scratch
 *     buffer (error word) and, for jagged calls, one 1 MB work-list buffer
 *     per (device, stream); it keeps them until the process exits.  A
 *     jagged call launches a one-block planning kernel before the attention
 *     kernel, on the same stream.
 */
#ifndef ATTN_JVP_H
#define ATTN_JVP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, causal with M != N (dense) */
  ATTN_ERR_UNSUPPORTED = 2,   /* head dim outside the entry point's set, option not supported */
  ATTN_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned */
  ATTN_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed (no GPU, launch error) */
  ATTN_ERR_TIMEOUT = 5        /* a device pipeline wait ran out of time; outputs undefined */
} attn_status;

/* Problem shape.  Dense: B, H, M (query length), N (key length), Dqk, Dv;
 * T and max_seq_len ignored.  Jagged: B = number of sequences, H, Dqk, Dv,
 * T = total tokens, max_seq_len = cap on a sequence's length; M and N are
 * ignored. */
typedef struct {
  int32_t B, H, M, N, Dqk, Dv;
  int64_t T;
  int32_t max_seq_len;
} attn_shape;

/* Optional additive bias and boolean mask over [B, H, M, N] (dense only).
 * Strides are in elements; a stride of 0 broadcasts that dimension (a key
 * padding mask is {N, 0, 0, 1}).  A NULL pointer means "absent".  The
 * bias is fp32 and added after the sm_scale product (it is not scaled and
 * has no tangent); the mask is uint8, nonzero = attend.  Both may be given
 * together ("flash_attention.py", _attn_fwd_inner). */
typedef struct {
  const float* bias;
  int64_t bias_stride[4];
  const uint8_t* mask;
  int64_t mask_stride[4];
} attn_bias;

/* Forward + JVP in one pass ("Flash Attention v2 with JVP", _attn_fwd).
 * sm_scale: NaN selects the default Dqk^-1/2 (_attention.forward).
 * causal: nonzero = row i attends to keys j <= i; dense causal requires
 * M == N (ATTN_ERR_INVALID_ARG otherwise).  bias may be NULL.
 * Writes o, to (bf16) and lse (fp32). */
attn_status attn_fwd_jvp(const attn_shape* shape,
                         const void* q, const void* k, const void* v,
                         const void* tq, const void* tk, const void* tv,
                         const int32_t* offsets, const attn_bias* bias,
                         int causal, float sm_scale,
                         void* o, void* to, float* lse, void* stream);

/* Forward only: the same operation without tangents (the FA2 forward of
 * "flash_attention.py", _attn_fwd, and of the FBGEMM jagged forward with
 * sm_scale and without its 1/max_seq_len factor).  Writes o and lse. */
attn_status attn_fwd(const attn_shape* shape,
                     const void* q, const void* k, const void* v,
                     const int32_t* offsets, const attn_bias* bias,
                     int causal, float sm_scale,
                     void* o, float* lse, void* stream);

/* attn_fwd_jvp and attn_fwd with fp16 storage: q, k, v, tq, tk, tv, o and
 * to are IEEE half precision instead of bf16 (lse stays fp32); P and its
 * tangent product enter the output MMAs as fp16.  Everything else is as
 * above.  The Triton kernels of "Flash Attention v2 with JVP" and of the
 * fused-attention JVP tutorial accept fp16 and bf16 inputs alike.  P is at
 * most 2^8 here (the lazy rescale threshold) and P o tS at most 2^8 |tS|,
 * so fp16 holds them for |tS| below ~256. */
attn_status attn_fwd_jvp_f16(const attn_shape* shape,
                             const void* q, const void* k, const void* v,
                             const void* tq, const void* tk, const void* tv,
                             const int32_t* offsets, const attn_bias* bias,
                             int causal, float sm_scale,
                             void* o, void* to, float* lse, void* stream);
attn_status attn_fwd_f16(const attn_shape* shape,
                         const void* q, const void* k, const void* v,
                         const int32_t* offsets, const attn_bias* bias,
                         int causal, float sm_scale,
                         void* o, float* lse, void* stream);

/* FP8 forward (no tangents): the FP8 path of the Triton fused-attention
 * tutorial (q, k, v in float8 e5m2, V stored transposed, P cast to e5m2
 * before the P V product, O written in e5m2).  Dense only.
 *   q  [B, H, M, D] e5m2     k [B, H, N, D] e5m2
 *   vt [B, H, D, N] e5m2     (V transposed: vt[b,h,d,j] = V[b,h,j,d])
 *   o  [B, H, M, D] e5m2     lse [B, H, M] fp32 (natural log)
 * D = Dqk = Dv in {64, 128} (else ATTN_ERR_UNSUPPORTED); N a multiple of
 * 16 (the rows of vt are N bytes and bulk copies need 16-byte strides;
 * else ATTN_ERR_UNSUPPORTED); causal requires M == N.  S is accumulated in
 * fp32 from the e5m2 products, the row sum is taken from the fp32 weights,
 * P is then rounded to e5m2 for the P V product (the tutorial's order), and
 * O = (e5m2(P) V) / sum is rounded to e5m2 (nearest even, saturating).
 * Other conventions as attn_fwd.
 * Pointers, shape fields T / max_seq_len: as attn_fwd (T ignored). */
attn_status attn_fwd_f8(const attn_shape* shape,
                        const void* q, const void* k, const void* vt,
                        int causal, float sm_scale,
                        void* o, float* lse, void* stream);

/* attn_fwd_jvp for callers that may not allocate device memory: a framework
 * that owns every device allocation, a runtime that forbids cudaMalloc
 * while it records work, a real-time path with a frozen memory budget.
 * The pages have no counterpart of this entry point.
 *
 * Same arguments, layouts and results as attn_fwd_jvp.  The library's only
 * scratch (the kernel's error word, one 4-byte word whatever the problem
 * size) lives in a fixed 256-byte device array inside the library instead
 * of a buffer from cudaMalloc; every device that loads the library holds it
 * until the process exits.  A problem that would need more scratch than
 * the array holds is rejected with ATTN_ERR_UNSUPPORTED; no problem the
 * current kernels accept does.  Jagged calls here skip the cost-ordered
 * work list (it needs a buffer) and walk the units in the fixed slot order,
 * which balances less well.  Nothing here calls cudaMalloc, cudaFree or
 * any allocating library routine.
 *
 * The first call on a device (with that device current) looks up the
 * array's device address; make that first call before any stream capture.
 * Each call clears the error word on `stream` before its launch.  All calls
 * share the array, so calls that overlap on the GPU (other streams) race on
 * it.  A wait that runs out of time in this variant is reported by the next
 * attn_sync_check on the device, which reads (and clears) this array's
 * error word too and allocates nothing. */
attn_status attn_fwd_jvp_noalloc(const attn_shape* shape,
                                 const void* q, const void* k, const void* v,
                                 const void* tq, const void* tk, const void* tv,
                                 const int32_t* offsets, const attn_bias* bias,
                                 int causal, float sm_scale,
                                 void* o, void* to, float* lse, void* stream);

/* Backward of softmax attention: given the forward's inputs q, k, v (and
 * its bias / mask), its output o and log-sum-exp lse (as attn_fwd writes
 * them) and the gradient dout = dL/dO of a loss L, writes
 *
 *   Delta = rowsum(dout o O)             delta [B, H, M] fp32
 *   dV    = P^T dout                     dv    [B, H, N, Dv]
 *   dS    = P o (dout V^T - Delta)
 *   dQ    = sm_scale dS K                dq    [B, H, M, Dqk]
 *   dK    = sm_scale dS^T Q              dk    [B, H, N, Dqk]
 *
 * with P = exp(sm_scale Q K^T + bias - LSE) over the valid set (0 elsewhere
 * and on rows with LSE = -inf); the bias gets no gradient.  Sources: the Triton fused-attention tutorial's
 * backward (_attn_bwd_preprocess for Delta, _attn_bwd_dkdv and _attn_bwd_dq
 * recomputing P from the stored log-sum-exp); "flash_attention.py"
 * (triton_flashattn) _attn_bwd_dkdv_inner / _attn_bwd_dq_inner.
 *
 * bias: as in attn_fwd (the same pointers and strides the forward was
 * given; dense only, ATTN_ERR_UNSUPPORTED with offsets; ATTN_ERR_MISALIGNED
 * for a bias not 4-byte aligned).  Dqk, Dv in {16, 32, 64, 128} (16 and 32
 * zero-padded to 64 inside; unequal dims as in "flash_attention.py");
 * otherwise ATTN_ERR_UNSUPPORTED.  Dense (offsets NULL; causal requires M == N) or
 * jagged (offsets != NULL, the FBGEMM jagged backward's layout:
 * q, k, v, o, dout, dq, dk, dv [H, T, D], lse and delta [H, T]); a jagged
 * token past its sequence's min(length, max_seq_len) gets dq = dk = dv = 0,
 * tokens >= offsets[B] are not written.  Layouts, element types (bf16; fp16
 * for attn_bwd_f16), pointer ownership and alignment, sm_scale and stream
 * semantics are those of attn_fwd.  lse must be the forward's (natural log);
 * a row's lse decides its P, so a stale or mismatched lse gives wrong
 * gradients, not an error.  delta is a caller-owned output that the two
 * gradient kernels also read.  Launches on `stream`: Delta, (jagged) a
 * one-block-per-sequence zero fill of the capped tokens, the dQ pass, the
 * dK / dV pass; no atomics, each output element is written once.  Dense
 * M == 0 writes zero dK and dV; N == 0 writes zero dQ (and delta). */
attn_status attn_bwd(const attn_shape* shape,
                     const void* q, const void* k, const void* v,
                     const void* o, const void* dout, const float* lse,
                     const int32_t* offsets, const attn_bias* bias,
                     int causal, float sm_scale,
                     void* dq, void* dk, void* dv, float* delta, void* stream);
attn_status attn_bwd_f16(const attn_shape* shape,
                         const void* q, const void* k, const void* v,
                         const void* o, const void* dout, const float* lse,
                         const int32_t* offsets, const attn_bias* bias,
                         int causal, float sm_scale,
                         void* dq, void* dk, void* dv, float* delta, void* stream);

/* The launches of attn_bwd / attn_bwd_f16, selected by `stages` (a nonzero
 * OR of the flags below; other bits: ATTN_ERR_INVALID_ARG): Delta; the dQ
 * pass (reads delta); the dK / dV pass (reads delta).  Given delta the two
 * gradient passes are independent, so a caller may run them on different
 * streams, or time them one by one.  f16 nonzero selects fp16 storage.
 * Arguments, validation (every pointer of attn_bwd is still required),
 * layouts and results are those of attn_bwd; a stage writes only its own
 * outputs. */
enum {
  ATTN_BWD_DELTA = 1,
  ATTN_BWD_DQ = 2,
  ATTN_BWD_DKDV = 4,
  ATTN_BWD_ALL = 7
};
attn_status attn_bwd_stages(const attn_shape* shape,
                            const void* q, const void* k, const void* v,
                            const void* o, const void* dout, const float* lse,
                            const int32_t* offsets, const attn_bias* bias,
                            int causal, float sm_scale,
                            void* dq, void* dk, void* dv, float* delta,
                            int f16, unsigned stages, void* stream);

/* Synchronises `stream`, then reads and clears the error words of the
 * current device: the scratch of the allocating entry points and the fixed
 * array of attn_fwd_jvp_noalloc, each once a call on the device has set it
 * up (nothing is allocated here).  Returns ATTN_ERR_TIMEOUT if a launch
 * since the last check reported a timed-out wait, ATTN_ERR_CUDA on a CUDA
 * error, else ATTN_OK. */
attn_status attn_sync_check(void* stream);

/* Static description of a status code; never NULL. */
const char* attn_status_string(attn_status s);

/* Number of kernels this library has launched in this process. */
uint64_t attn_launch_count(void);

/* Upper bound, in nanoseconds, on any single pipeline wait inside the
 * kernels (default 2e9).  Values below 1e6 are raised to 1e6. */
void attn_set_wait_timeout_ns(uint64_t ns);

/* Test hook for failure detection: when nonzero, the next launches skip
 * the first query-tile load, so the consumer's bounded wait runs out and
 * the call reports ATTN_ERR_TIMEOUT through attn_sync_check.  0 restores
 * normal operation. */
void attn_debug_skip_first_load(int enable);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_JVP_H */
