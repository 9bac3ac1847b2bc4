// Fused attention forward (+ JVP) for sm_103a: one persistent kernel
// family, templated on the head dims and on whether tangents are carried.
//
// Method ("Flash Attention v2 with JVP", _attn_fwd_inner / _attn_fwd):
// for a tile of 128 query rows, stream the keys in tiles of 64 and keep
// per row a running max m, denominator l and tangent sum r, plus the
// accumulators O_acc = sum p V and tO_acc = sum p tV + sum (p tS) V, where
// p = exp2(x - m) and x = S * sm_scale * log2(e) (+ bias * log2(e)).
// The epilogue writes O = O_acc / l, tO = (tO_acc - r O) / l and
// LSE = (m + log2 l) ln 2.
//
// GB300 mapping (one CTA per SM, 12 warps):
//   warp 0      bulk-tensor (TMA) producer: Q, tQ once per work unit; K, tK
//               into a ring of NK stages.
//   warp 2      bulk-tensor producer of V, tV into a ring of NV stages.
//   warp 1      tcgen05 issuer, per key tile:
//                 [S | Q tK^T] = Q [K ; tK]^T      one N = 128 MMA chain
//                 tS += tQ K^T                     N = 64
//                 [O | tO] += P [V | tV]           one N = 2 Dv MMA chain
//                 tO += H V                        N = Dv
//               so P tV + H V is the K = 2*BN contraction [P | H] [tV ; V]
//               accumulated into one tO.  S / tS are double buffered in
//               TMEM; P and H (bf16) are written back over the S / tS
//               columns they came from and read by the MMA from TMEM.
//   warp 3      release warp: frees each K stage (and Q at the end of a
//               unit) as soon as the score MMAs that read it are done.
//   warps 4..11 softmax / rescale / epilogue: two warps per TMEM lane
//               quadrant (row = TMEM lane).  Column halves: each warp
//               writes P / H for 32 of the 64 key columns of a tile and
//               reads all 64 scores for the row maximum (only the
//               per-thread global bias mode exchanges partial maxima
//               through shared memory).  Ping-pong (head dims 64, no bias
//               or mask): the two warps take alternate key tiles, all 64
//               columns, each into its own O / tO buffer, and merge their
//               row states and buffers once per unit.  Rescaling is lazy:
//               the reference max m moves (and O, tO, l, r are multiplied
//               by exp2(m_old - m_new)) only when the row maximum grows by
//               more than kRescaleThreshold; the result is exact because
//               l, r and the accumulators share the same stale reference.
//   Work units (query tile, head, batch or sequence) are walked by every
//   CTA in a snake over a longest-first order.
//
// Every mbarrier wait is bounded: on expiry the thread records
// ERR_TIMEOUT in the device error word, raises a CTA-wide abort flag and
// all roles leave their loops; in-flight copies and MMAs are drained with
// bounded waits before tensor memory is released.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"

namespace attn {

constexpr int kBM = 128;       // query rows per work unit (= TMEM lanes)
constexpr int kBN = 64;        // keys per pipeline step
constexpr int kHalf = kBN / 2; // key columns per softmax thread
constexpr int kThreads = 384;  // 12 warps = 3 warpgroups
// Register split (setmaxnreg): the kernel is launched with kLaunchRegs per
// thread; warpgroup 0 (producers, MMA issuer, release warp) gives registers
// back and the two softmax warpgroups take them:
//   4 warps x 32 x kLowRegs + 8 warps x 32 x kHighRegs = 384 x kLaunchRegs.
constexpr int kLaunchRegs = 168;
constexpr int kLowRegs = 56;
constexpr int kHighRegs = 224;
static_assert(4 * 32 * kLowRegs + 8 * 32 * kHighRegs == kThreads * kLaunchRegs,
              "register split must use exactly the launch allocation");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p <= 2^8 between rescales
constexpr int ERR_TIMEOUT = 1;
constexpr int ERR_SMEM_ALIGN = 2;

struct KernelParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_tq, tm_tk, tm_tv;
  // fp32 bias as a 4-D view {key, query row, head, batch}, box 32 x 128
  // (used when bias_tma is set); a broadcast head / batch dimension has
  // size 1 and is addressed at coordinate 0.
  CUtensorMap tm_bias;
  int bias_tma, bias_bcast_h, bias_bcast_b;
  int B, H, M, N;  // jagged: B = sequences, M = N = max_seq_len
  int jagged, causal;
  int n_mt;        // query tiles per (b, h) or per (sequence, h)
  // output column slices per query tile: 1, or 2 when the kernel's DV is
  // half of the output head dim (tangents at Dv = 256: O and tO of 256
  // columns each do not fit tensor memory beside the scores, so each slice
  // of 128 columns is its own work unit, which recomputes the scores)
  int n_vh;
  int num_units;   // units in the fixed slot order (B * H * n_mt * n_vh)
  // Jagged work list (optional): unit_count[0] (sequence, query tile) pairs,
  // costliest first, at unit_list (x = sequence, y = tile); unit u is pair
  // u / H, head u % H.  A count of -1 means the list was not written.
  const int2* unit_list;
  const int* unit_count;
  // Dense, with a key mask that does not depend on the query row (optional):
  // bits 0-30 of keylen[b * H + h] = 1 + the last key any row of (b, h)
  // attends, bit 31 set when every key below it is attended (the mask is
  // then a key prefix, and the key length alone masks the rest); the units
  // visit only the key tiles below it (a planning kernel earlier on the
  // stream writes it).
  const int* keylen;
  float scale_log2;  // sm_scale * log2(e)
  float sm_scale;
  const int* offsets;
  const float* bias;
  long long bias_stride[4];
  const unsigned char* mask;
  long long mask_stride[4];
  uint16_t* o;   // bf16 or fp16 storage (the kernel's element type)
  uint16_t* to;
  float* lse;
  long long T;
  int max_seq_len;
  // output head dim (row stride of o / to): DV, or 16 / 32 when the kernel
  // runs a smaller head dim zero-padded to DV = 64 (columns past dv_out are
  // computed as zeros and not stored)
  int dv_out;
  int* err;
  unsigned long long timeout_ns;
  int skip_first_load;
};

// Bias / mask handling of a kernel instantiation.
//   kNoBias:     neither; every tile's row maximum is local.
//   kBiasRing:   bias tiles copied by tensor copies into a shared-memory
//                ring (and / or a boolean mask read per thread); both halves
//                of a row see every column, so the row maximum is local.
//   kBiasGlobal: bias read per thread from global memory (layouts a tensor
//                map cannot describe); the two warps of a row exchange their
//                partial maxima.
constexpr int kNoBias = 0, kBiasRing = 1, kBiasGlobal = 2;

// Shared-memory and tensor-memory plan for one instantiation.
// F8: e5m2 operands (forward only): a row of Q or K (D <= 128 bytes) is
// one 128-byte swizzled chunk, and V arrives transposed, a tile being Dv
// rows of 64 keys (64-byte rows, 64-byte swizzle).
template <int DQK, int DV, bool JVP, int BMODE, bool F8 = false>
struct Plan {
  static_assert(!F8 || (!JVP && BMODE == 0 && DQK <= 128 && DV <= 128), "e5m2: forward only, no bias");
  static constexpr int NQ = JVP ? 2 : 1;   // primal (+ tangent) operands
  static constexpr int CH = F8 ? 1 : DQK / 64;  // 128-byte chunks per Q / K row
  // Bias stage: the fp32 bias of one key tile, two 128-row x 32-key boxes
  // (one per softmax half), 128-byte swizzled rows.
  static constexpr int BIAS_BOX = kBM * 32 * 4;
  static constexpr int BIAS_STAGE = 2 * BIAS_BOX;
  static constexpr int Q_SUB = kBM * 128;  // one 64-column swizzled sub-tile
  static constexpr int K_SUB = kBN * 128;
  static constexpr int V_SUB = kBN * 128;
  static constexpr int Q_TILE = CH * Q_SUB;
  static constexpr int V_TILE = F8 ? DV * 64 : (DV / 64) * V_SUB;
  // K stage: for each 64-column chunk c, [K rows | tK rows] side by side so
  // that Q [K ; tK]^T is one N = 128 operand.
  static constexpr int K_GROUP = NQ * K_SUB;
  static constexpr int K_STAGE = CH * K_GROUP;
  // V stage: [V chunks | tV chunks], uniform 64-column stride, so that
  // [V | tV] is one N = 2 Dv operand.
  static constexpr int V_STAGE = NQ * V_TILE;
  static constexpr int QSET = NQ * Q_TILE;  // one Q (+ tQ) buffer
  // Ping-pong softmax (head dims 64, no bias / mask, 16-bit operands): the
  // two softmax warps of a TMEM lane quadrant take alternate key tiles of a
  // unit (all 64 columns each) instead of the two column halves of every
  // tile, each with its own running max, sums and O / tO accumulator (the
  // two O buffers); the epilogue merges the two.  The two warps of a
  // sub-partition then work on different tiles, so their latencies overlap.
  static constexpr bool PP = !F8 && BMODE == kNoBias && DQK == 64 && DV == 64;
  // exchange slots between the two softmax warps of a row:
  // [parity][half][row] plus one [row] array (the epilogue's third value);
  // ping-pong: [unit parity][value][tile parity][row], four values
  static constexpr int XCHG_FLOATS = PP ? 2 * 4 * 2 * kBM : 2 * 2 * kBM + kBM;
  static constexpr int BUDGET = 227 * 1024 - 512 - XCHG_FLOATS * 4;
  // Q buffers: two (the next unit's Q loads while the current unit runs and
  // score MMAs flow across unit boundaries) when they fit beside three K and
  // two V stages, else one.  Kernels with a bias ring keep one.
  static constexpr int NQB =
      (BMODE != kBiasRing && 2 * QSET + 3 * K_STAGE + 2 * V_STAGE <= BUDGET) ? 2 : 1;
  static constexpr int FIXED = NQB * QSET;
  // bias stages (kernels with bias / mask only): two when two K and two V
  // stages still fit beside them, else one
  static constexpr int NB = BMODE != kBiasRing ? 0 : (FIXED + 2 * BIAS_STAGE + 2 * K_STAGE + 2 * V_STAGE <= BUDGET) ? 2 : 1;
  static constexpr int RING = BUDGET - NB * BIAS_STAGE;
  // (one K stage only when two do not fit: Dqk = 256 with tangents, whose
  // Q and tQ take 128 KB)
  // With one Q buffer and K / V stages of the same size (Dqk = Dv = 128
  // with tangents, no bias), three K stages and two V stages fit, and so do
  // two and three: the second measured faster (causal B2 H16 N4096:
  // 257.7 -> 250.7 us), so there the V ring gets the third stage.
  static constexpr bool V3 = !F8 && BMODE == kNoBias && NQB == 1 && K_STAGE == V_STAGE &&
                             FIXED + 2 * K_STAGE + 3 * V_STAGE <= RING &&
                             FIXED + 3 * K_STAGE + 3 * V_STAGE > RING;
  static constexpr int NK = V3 ? 2
                            : (FIXED + 4 * K_STAGE + 4 * V_STAGE <= RING) ? 4
                            : (FIXED + 3 * K_STAGE + 2 * V_STAGE <= RING) ? 3
                            : (FIXED + 2 * K_STAGE + V_STAGE <= RING)     ? 2
                                                                          : 1;
  static constexpr int NV = (FIXED + NK * K_STAGE + 4 * V_STAGE <= RING)   ? 4
                            : (FIXED + NK * K_STAGE + 3 * V_STAGE <= RING) ? 3
                            : (FIXED + NK * K_STAGE + 2 * V_STAGE <= RING) ? 2
                                                                           : 1;
  // One K stage only (Dqk = 256 with tangents): it is kept as CH chunk
  // stages of 64 columns ([K | tK] of one chunk each), released one by one
  // as the score MMAs that read them finish, so that the next tile's chunks
  // load while the rest of this tile's score chain runs.
  static constexpr bool KCH = JVP && NK == 1 && CH > 1;
  static constexpr int NKB = KCH ? CH : NK;  // K full / empty barrier pairs
  static constexpr int OFF_Q = 0;       // buffer b at OFF_Q + b * QSET
  static constexpr int OFF_TQ = Q_TILE;  // buffer b at OFF_TQ + b * QSET
  static constexpr int OFF_K = FIXED;
  static constexpr int OFF_V = OFF_K + NK * K_STAGE;
  static constexpr int OFF_BIAS = OFF_V + NV * V_STAGE;  // 1024-byte aligned (stages are)
  static constexpr int OFF_BAR = OFF_BIAS + NB * BIAS_STAGE;
  // barriers: q_full, q_empty, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV],
  //           s_full[2], p_full[2], mma_drain, pair[4] (the two softmax warps
  //           of a quadrant).  v_empty of tile t's stage completes when the
  //           output MMAs of tile t (and every MMA before them) are done; the
  //           softmax warps wait on it too (lazy rescale, epilogue).
  //           k_empty and q_empty are arrived on by the release warp once the
  //           score MMAs that read the stage (Q: of the unit's last tile) are
  //           done.
  //           With two O buffers, o_empty[b] completes when the softmax
  //           warps have read buffer b in a unit's epilogue.
  static constexpr int SBUF = 2 * kBN;
  static constexpr int COL_O = 2 * SBUF;
  static constexpr int OBUF = (JVP ? 2 : 1) * DV;  // columns of one [O | tO] buffer
  // O buffers: two (a unit's epilogue runs after the next unit's first tile,
  // whose output MMAs write the other buffer) with two Q buffers, when the
  // tensor memory holds them.
  static constexpr int NOB = (NQB == 2 && COL_O + 2 * OBUF <= 512) ? 2 : 1;
  static_assert(!PP || (NQB == 2 && NOB == 2), "ping-pong softmax: two Q and two O buffers");
  static constexpr int B_QF = 0, B_QE = B_QF + NQB, B_KF = B_QE + NQB, B_KE = B_KF + NKB,
                       B_VF = B_KE + NKB, B_VE = B_VF + NV, B_SF = B_VE + NV, B_PF = B_SF + 2,
                       B_DRAIN = B_PF + 2, B_PAIR = B_DRAIN + 1, B_BF = B_PAIR + 4,
                       B_BE = B_BF + NB, B_OE = B_BE + NB, NBAR = B_OE + NOB;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem address, abort flag
  static constexpr int OFF_XCHG = OFF_MISC + 16;
  static constexpr int SMEM_BYTES = OFF_XCHG + XCHG_FLOATS * 4;
  // TMEM columns: buffer b holds S at [b*SBUF, b*SBUF + BN) and tS (or, in
  // the forward-only kernel, scratch) in the next BN columns; then NOB
  // buffers of O_acc and tO_acc side by side (buffer b at COL_O + b * OBUF).  Softmax half h writes its bf16 P (16 columns) and
  // H (16 columns) over its own 32 tS columns, which no other thread reads,
  // so the S columns stay intact for both halves' row maxima.
  static constexpr int COLS_USED = COL_O + NOB * OBUF;
  static constexpr int TMEM_COLS = COLS_USED <= 256 ? 256 : 512;
  // Requested dynamic shared memory: never less than half an SM's, so one
  // CTA (and its TMEM allocation) owns an SM.
  static constexpr int SMEM_LAUNCH = SMEM_BYTES > 120 * 1024 ? SMEM_BYTES : 120 * 1024;
  // whether the plan fits one CTA's shared memory (the host does not launch
  // an instantiation that does not: a bias ring at Dqk = 256 with tangents
  // falls back to per-thread bias loads)
  static constexpr bool FITS = SMEM_BYTES <= 227 * 1024;
  static_assert(COLS_USED <= 512, "tensor memory plan exceeds 512 columns");
  static_assert(DQK % 64 == 0 && DV % 64 == 0, "head dims are multiples of 64");
  static_assert(V_TILE % 1024 == 0, "V tiles keep 1024-byte alignment");
  static_assert(NQ * DV <= 256, "[O | tO] MMA needs N <= 256");
};

struct Unit {
  int z;            // third tensor-map coordinate: b*H + h (dense) or h (jagged)
  int row0;         // first row of this (b, h) / sequence in the tensor map
  int mt;           // query tile index
  int q_len;        // query rows of this (b, h) / sequence
  int kv_len;       // keys of this (b, h) / sequence
  int nt;           // key tiles visited
  int b, h;
  long long out0;   // row index of query 0 in the [.., rows] output view
  int vh;           // output column slice: columns [vh * DV, vh * DV + DV)
  bool mask_on;     // the key mask has to be read (false: a key prefix, in kv_len)
  bool active;
};

// Work unit u.  Causal dense units and (without a work list) jagged units
// are ordered by descending query tile, so the costliest units start first;
// a jagged work list is already ordered by cost.  SLICES: the kernel may
// run output column slices (tangents with a 128-wide kernel DV); other
// kernels carry no slice arithmetic.  NG > 1: causal dense units take the
// heads in NG groups, one group after the other.  LEAN: dense, non-causal,
// no key mask, every key tile whole (N a positive multiple of the key
// tile): unit u is query tile u % n_mt of (b, h) = u / n_mt.
template <bool SLICES, int NG, bool LEAN = false>
__device__ __forceinline__ Unit decode_unit(const KernelParams& p, int u, const int2* list) {
  Unit w;
  if constexpr (LEAN) {
    const int bh = u / p.n_mt;
    w.vh = 0;
    w.mask_on = false;
    w.b = bh / p.H;
    w.h = bh % p.H;
    w.z = bh;
    w.row0 = 0;
    w.mt = u % p.n_mt;
    w.q_len = p.M;
    w.kv_len = p.N;
    w.out0 = static_cast<long long>(bh) * p.M;
    w.active = true;
    w.nt = p.N / kBN;
    return w;
  }
  // the column slices of one query tile are adjacent units (they share Q, K
  // and V tiles through L2)
  w.vh = 0;
  w.mask_on = true;
  if constexpr (SLICES) {
    if (p.n_vh > 1) {
      w.vh = u % p.n_vh;
      u /= p.n_vh;
    }
  }
  const int BH = p.B * p.H;
  if (!p.jagged) {
    int bh, mt;
    if (p.causal) {
      if constexpr (NG > 1) {
        // heads in NG groups walked one after the other, costliest query
        // tile first within a group: a group's K / V stay in L2 (one group
        // when NG does not divide B H)
        const int ng = (BH % NG == 0) ? NG : 1;
        const int BHg = BH / ng;
        const int per = p.n_mt * BHg;
        const int grp = u / per, r = u % per;
        mt = p.n_mt - 1 - r / BHg;
        bh = grp * BHg + r % BHg;
      } else {
        mt = p.n_mt - 1 - u / BH;
        bh = u % BH;
      }
    } else {
      bh = u / p.n_mt;
      mt = u % p.n_mt;
    }
    w.b = bh / p.H;
    w.h = bh % p.H;
    w.z = bh;
    w.row0 = 0;
    w.mt = mt;
    w.q_len = p.M;
    w.kv_len = p.N;
    if (p.keylen != nullptr) {
      const int kl = __ldg(p.keylen + bh);
      w.kv_len = min(p.N, kl & 0x7fffffff);
      w.mask_on = kl >= 0;
    }
    w.out0 = static_cast<long long>(bh) * p.M;
  } else {
    int mt, b, h;
    if (list != nullptr) {
      const int2 e = list[u / p.H];
      b = e.x;
      mt = e.y;
      h = u % p.H;
    } else {
      mt = p.n_mt - 1 - u / BH;
      const int r = u % BH;
      b = r / p.H;
      h = r % p.H;
    }
    const int begin = __ldg(p.offsets + b), end = __ldg(p.offsets + b + 1);
    const int len = min(end - begin, p.max_seq_len);
    w.b = b;
    w.h = h;
    w.z = h;
    w.row0 = begin;
    w.mt = mt;
    w.q_len = len;
    w.kv_len = len;
    w.out0 = static_cast<long long>(h) * p.T + begin;
  }
  w.active = w.mt * kBM < w.q_len;
  int hi = w.kv_len;
  if (p.causal) hi = min(hi, (w.mt + 1) * kBM);
  w.nt = w.active ? (hi + kBN - 1) / kBN : 0;
  return w;
}

// The unit a CTA processes in its round `rnd`: rounds walk the longest-first
// unit order in a snake (even rounds CTA 0 -> G-1, odd rounds G-1 -> 0), so
// the CTA that took the costliest unit of one round takes the cheapest of
// the next.  Every role of a CTA walks the same sequence.
__device__ __forceinline__ int unit_of_round(int rnd) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return rnd * G + ((rnd & 1) ? (G - 1 - c) : c);
}

// Key tiles ahead of its use at which a bias box is pulled into L2.
constexpr int kBiasLead = 4;

struct Waiter {
  volatile int* abort_flag;
  int* err;
  unsigned long long timeout_ns;
};

// Bounded wait for the phase of `bar` with parity `parity`.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Waiter& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*w.abort_flag) return false;
      if (globaltimer_ns() - t0 > w.timeout_ns) {
        *w.abort_flag = 1;
        atomicCAS(w.err, 0, ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// wait_bar for a warp with nothing else to do: it sleeps inside the poll.
__device__ __forceinline__ bool wait_bar_sleep(uint32_t bar, uint32_t parity, const Waiter& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*w.abort_flag) return false;
    if (globaltimer_ns() - t0 > w.timeout_ns) {
      *w.abort_flag = 1;
      atomicCAS(w.err, 0, ERR_TIMEOUT);
      return false;
    }
  }
}

// Bounded wait that ignores the abort flag (teardown drains).
__device__ __forceinline__ bool drain_bar(uint32_t bar, uint32_t parity, unsigned long long ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > ns) return false;
  }
  return true;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// n32 packed bf16x2 words (a multiple of 4) to global memory with 16-byte
// stores.
__device__ __forceinline__ void store_row_bf16(uint16_t* dst, const uint32_t* packed, int n32) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < n32 / 4; ++i)
    d[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
}


// Transpose 4 x 4 blocks across each quad of lanes: lane q of a quad holds
// chunks 0..3 (C words each) of its own row; afterwards it holds chunk q of
// the quad's four rows, slot k taken from lane k.  Two rounds of paired
// shuffles (lanes q, q^2 then q, q^1), indices fixed at compile time.
template <int C>
__device__ __forceinline__ void quad_transpose(uint32_t (&a)[4 * C], int q) {
  const bool hi2 = (q & 2) != 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
#pragma unroll
    for (int w = 0; w < C; ++w) {
      const uint32_t send = hi2 ? a[j * C + w] : a[(j + 2) * C + w];
      const uint32_t got = __shfl_xor_sync(0xffffffffu, send, 2);
      if (hi2) a[j * C + w] = got;
      else a[(j + 2) * C + w] = got;
    }
  }
  const bool hi1 = (q & 1) != 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
#pragma unroll
    for (int w = 0; w < C; ++w) {
      const uint32_t send = hi1 ? a[2 * j * C + w] : a[(2 * j + 1) * C + w];
      const uint32_t got = __shfl_xor_sync(0xffffffffu, send, 1);
      if (hi1) a[2 * j * C + w] = got;
      else a[(2 * j + 1) * C + w] = got;
    }
  }
}

// C packed words to global memory: one 32-byte store when C == 8 and the
// address is 32-byte aligned, one 8-byte store when C == 2, else 16-byte
// stores.
template <int C>
__device__ __forceinline__ void store_chunk(uint16_t* dst, const uint32_t* w, bool aligned32) {
  if constexpr (C == 2) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    return;
  }
  if (C == 8 && aligned32) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
  } else {
#pragma unroll
    for (int i = 0; i < C / 4; ++i)
      reinterpret_cast<uint4*>(dst)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  }
}

// Mask bytes of 32 keys from key0 (nonzero = attend), four per word; keys
// at or past kv_len read as 0.
__device__ __forceinline__ void load_mask32(const unsigned char* mrow, int key0, int kv_len,
                                            long long stride, bool row_ok, uint32_t (&mv)[8]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) mv[c] = 0u;
  if (!row_ok) return;
  const unsigned char* mp = mrow + static_cast<long long>(key0) * stride;
  if (stride == 1 && (reinterpret_cast<uintptr_t>(mp) & 15u) == 0 && key0 + 32 <= kv_len) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint4 t4 = __ldg(reinterpret_cast<const uint4*>(mp) + c);
      mv[4 * c] = t4.x;
      mv[4 * c + 1] = t4.y;
      mv[4 * c + 2] = t4.z;
      mv[4 * c + 3] = t4.w;
    }
  } else {
    for (int c = 0; c < 32; ++c)
      if (key0 + c < kv_len && __ldg(mp + c * stride) != 0) mv[c >> 2] |= 1u << ((c & 3) * 8);
  }
}

// Bit c set when key key_start + c (c < 32) is below kv_len and, for
// causal attention, at most qi.
__device__ __forceinline__ uint32_t keep_bits(int key_start, int kv_len, int qi, bool causal) {
  int n = kv_len - key_start;
  if (causal) n = min(n, qi - key_start + 1);
  return n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
}

// Bit c set when mask byte c (byte c % 4 of word c / 4) is nonzero: a
// per-byte compare, then the four 0/1 bytes of a word gathered into four
// adjacent bits by one multiply (0x01020408 moves byte i's bit 8i to bit
// 24 + i; no other partial product lands on bits 24..27).
__device__ __forceinline__ uint32_t mask_bits32(const uint32_t (&mv)[8]) {
  uint32_t bits = 0;
#pragma unroll
  for (int wd = 0; wd < 8; ++wd) {
    const uint32_t nz = __vcmpne4(mv[wd], 0u) & 0x01010101u;
    bits |= ((nz * 0x01020408u) >> 24) << (4 * wd);
  }
  return bits;
}

// Row maximum of 32 values, 3-input max tree.
__device__ __forceinline__ float rowmax32(const float* x) {
  float a[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) a[i] = max3f(x[3 * i], x[3 * i + 1], x[3 * i + 2]);
  a[10] = fmaxf(x[30], x[31]);
  const float b0 = max3f(a[0], a[1], a[2]), b1 = max3f(a[3], a[4], a[5]);
  const float b2 = max3f(a[6], a[7], a[8]), b3 = fmaxf(a[9], a[10]);
  return fmaxf(max3f(b0, b1, b2), b3);
}

// BMODE: kNoBias, kBiasRing or kBiasGlobal (see Plan).  Each mode compiles
// only its own bias / mask code, which keeps the per-tile loop small.
// F16: fp16 inputs, MMA operands and outputs instead of bf16.
template <int DQK, int DV, bool JVP, int BMODE, bool F16, bool F8 = false, bool LEAN = false>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ KernelParams p) {
  using P = Plan<DQK, DV, JVP, BMODE, F8>;
  // LEAN: the ping-pong kernel compiled for dense non-causal problems whose
  // key tiles are all whole (no masking, no jagged or causal unit decode,
  // no empty rows): the kernel's speed depends on its code size
  static_assert(!LEAN || P::PP, "the lean variant is a ping-pong kernel");
  // output column slices (tangents at Dv = 256 run the 128-wide kernels)
  constexpr bool kSlices = JVP && DV == 128;
  // causal units at Dqk = 256 walk the heads in four groups: each query
  // tile's score work re-reads K / V (two column slices with tangents), and
  // keeping a quarter of the heads' K / V in L2 outweighs the coarser
  // balance (measured: 930 -> 857 us on B2 H16 N4096; at Dqk = 128, where
  // the reads are far from the HBM roof, grouping was slower)
  constexpr int kHeadGroups = DQK >= 256 ? 4 : 1;
  constexpr bool BM = BMODE != kNoBias;
  constexpr bool RING = BMODE == kBiasRing;
  constexpr bool GLOB = BMODE == kBiasGlobal;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Launched as a programmatic dependent, this kernel may start while the
  // kernel before it on the stream (a planning kernel, or the previous
  // call) is still running: the prologue below touches only shared and
  // tensor memory and the kernel parameters, and every thread waits for
  // the kernels before it to complete before the first global access.
  griddep_launch_dependents();
  // 128-byte swizzled operands need 1024-byte aligned tiles; the dynamic
  // shared window starts aligned, and a launch where it does not reports
  // an error instead of computing.
  if ((smem_u32(smem) & 1023u) != 0) {
    griddep_wait();
    if (threadIdx.x == 0) atomicCAS(p.err, 0, ERR_SMEM_ALIGN);
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + P::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + P::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P::OFF_MISC + 4);
  float* xchg = reinterpret_cast<float*>(smem + P::OFF_XCHG);

  if (threadIdx.x == 0) {
    for (int i = 0; i < P::NQB; ++i) {
      mbar_init(bar(P::B_QF + i), 1);
      mbar_init(bar(P::B_QE + i), 1);
    }
    for (int i = 0; i < P::NOB; ++i) mbar_init(bar(P::B_OE + i), 8);  // one arrival per softmax warp
    for (int i = 0; i < P::NKB; ++i) {
      mbar_init(bar(P::B_KF + i), 1);
      mbar_init(bar(P::B_KE + i), 1);
    }
    for (int i = 0; i < P::NV; ++i) {
      mbar_init(bar(P::B_VF + i), 1);
      mbar_init(bar(P::B_VE + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(P::B_SF + i), 1);
      // one arrival per softmax warp of the tile (all eight, or the four of
      // its parity in the ping-pong softmax) + the release warp
      mbar_init(bar(P::B_PF + i), P::PP ? 5 : 9);
    }
    mbar_init(bar(P::B_DRAIN), 1);
    for (int i = 0; i < 4; ++i) mbar_init(bar(P::B_PAIR + i), 64);
    for (int i = 0; i < P::NB; ++i) {
      mbar_init(bar(P::B_BF + i), 1);
      mbar_init(bar(P::B_BE + i), 8);  // one arrival per softmax warp
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
    if (JVP) {
      prefetch_tmap(&p.tm_tq);
      prefetch_tmap(&p.tm_tk);
      prefetch_tmap(&p.tm_tv);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), P::TMEM_COLS);
    tmem_relinquish();
  }
  griddep_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Waiter W{abort_flag, p.err, p.timeout_ns};
  // The units this launch walks: a jagged work list when one was written
  // (by the planning kernel earlier on the stream), else the slot order.
  const int2* list = nullptr;
  int num_units = p.num_units;
  if (!LEAN && p.unit_list != nullptr) {
    const int c = __ldg(p.unit_count);
    if (c >= 0) {
      list = p.unit_list;
      num_units = c * p.H * (kSlices && p.n_vh > 1 ? p.n_vh : 1);
    }
  }

  if (warp < 4) {
  setmaxnreg_dec<kLowRegs>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t qfill = 0, kfill = 0;
      int kpart = 0;  // chunk stages issued for tile kfill (chunked K only)
      const bool first_q_loaded = p.skip_first_load == 0;
      bool skip = !first_q_loaded;
      bool ok = true;
      for (int rnd = 0; ok; ++rnd) {
        const int u = unit_of_round(rnd);
        if (u >= num_units) break;
        const Unit w = decode_unit<kSlices, kHeadGroups, LEAN>(p, u, list);
        if (w.nt == 0) continue;
        const uint32_t qb = qfill % P::NQB;
        ok = wait_bar(bar(P::B_QE + qb), ((qfill / P::NQB) & 1u) ^ 1u, W);
        if (!ok) break;
        if (!skip) {
          mbar_arrive_expect_tx(bar(P::B_QF + qb), P::QSET);
          const int r = w.row0 + w.mt * kBM;
          const uint32_t qdst = sbase + qb * P::QSET;
#pragma unroll
          for (int c = 0; c < P::CH; ++c) {
            tma_load_3d(qdst + P::OFF_Q + c * P::Q_SUB, &p.tm_q, bar(P::B_QF + qb), c * 64, r, w.z);
            if (JVP)
              tma_load_3d(qdst + P::OFF_TQ + c * P::Q_SUB, &p.tm_tq, bar(P::B_QF + qb), c * 64, r,
                          w.z);
          }
        }
        skip = false;
        ++qfill;
        for (int j = 0; j < w.nt; ++j) {
          const int r = w.row0 + j * kBN;
          if constexpr (P::KCH) {
            // chunk stages: chunk c of this tile once the score MMAs of the
            // previous tile that read chunk c are done
            kpart = 0;
#pragma unroll 1
            for (int c = 0; c < P::CH && ok; ++c) {
              ok = wait_bar(bar(P::B_KE + c), (kfill & 1u) ^ 1u, W);
              if (!ok) break;
              mbar_arrive_expect_tx(bar(P::B_KF + c), P::K_GROUP);
              const uint32_t kdst = sbase + P::OFF_K + c * P::K_GROUP;
              tma_load_3d(kdst, &p.tm_k, bar(P::B_KF + c), c * 64, r, w.z);
              if constexpr (JVP) tma_load_3d(kdst + P::K_SUB, &p.tm_tk, bar(P::B_KF + c), c * 64, r, w.z);
              kpart = c + 1;
            }
            if (!ok) break;
            kpart = 0;
          } else {
          const uint32_t ks = kfill % P::NK;
          ok = wait_bar(bar(P::B_KE + ks), ((kfill / P::NK) & 1u) ^ 1u, W);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(P::B_KF + ks), P::K_STAGE);
          const uint32_t kdst = sbase + P::OFF_K + ks * P::K_STAGE;
#pragma unroll
          for (int c = 0; c < P::CH; ++c) {
            tma_load_3d(kdst + c * P::K_GROUP, &p.tm_k, bar(P::B_KF + ks), c * 64, r, w.z);
            if (JVP)
              tma_load_3d(kdst + c * P::K_GROUP + P::K_SUB, &p.tm_tk, bar(P::B_KF + ks), c * 64, r,
                          w.z);
          }
          }
          ++kfill;
        }
      }
      // Teardown: every issued copy must have landed before the CTA exits.
      if constexpr (P::KCH) {
        // chunks of an interrupted tile (the first kpart) were filled for
        // tile kfill; the others last for tile kfill - 1
        for (int c = 0; c < P::CH; ++c) {
          if (c < kpart) drain_bar(bar(P::B_KF + c), kfill & 1u, p.timeout_ns);
          else if (kfill > 0) drain_bar(bar(P::B_KF + c), (kfill - 1) & 1u, p.timeout_ns);
        }
      } else {
        for (uint32_t s = 0; s < P::NK && s < kfill; ++s) {
          const uint32_t nf = (kfill - s + P::NK - 1) / P::NK;
          drain_bar(bar(P::B_KF + s), (nf - 1) & 1u, p.timeout_ns);
        }
      }
      // (a skipped first load leaves its buffer's barrier incomplete)
      for (uint32_t s = 0; s < static_cast<uint32_t>(P::NQB) && s < qfill; ++s) {
        const uint32_t f = qfill - 1 - s;  // the last fill of buffer f % NQB
        if (f == 0 && !first_q_loaded) continue;
        drain_bar(bar(P::B_QF + f % P::NQB), (f / P::NQB) & 1u, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ---------------------------------------------------- V / tV producer
    // Separate from the K ring so that a K load never waits for a V slot.
    // With a bias that has a tensor map it also loads each key tile's bias
    // (two 128 x 32 fp32 boxes) into the bias ring.
    if (lane == 0) {
      uint32_t vfill = 0, bfill = 0;
      const bool bias_ring = P::NB > 0 && p.bias_tma != 0;
      bool ok = true;
      for (int rnd = 0; ok; ++rnd) {
        const int u = unit_of_round(rnd);
        if (u >= num_units) break;
        const Unit w = decode_unit<kSlices, kHeadGroups, LEAN>(p, u, list);
        for (int j = 0; j < w.nt; ++j) {
          const int r = w.row0 + j * kBN;
          if constexpr (P::NB > 0) {
            // The bias goes first: its stage frees as soon as the softmax
            // warps have read tile j - NB's bias, well before the output
            // MMAs of that tile release its V stage, so its copy is not
            // held back behind the V wait.
            if (bias_ring) {
              // the bias streams from HBM once: its boxes are pulled into L2
              // kBiasLead tiles ahead of their copy into the ring
              const int hb = p.bias_bcast_h ? 0 : w.h, bb = p.bias_bcast_b ? 0 : w.b;
              for (int jj = (j == 0 ? 0 : j + kBiasLead); jj <= j + kBiasLead && jj < w.nt; ++jj) {
                tma_prefetch_l2_4d(&p.tm_bias, jj * kBN, w.mt * kBM, hb, bb);
                tma_prefetch_l2_4d(&p.tm_bias, jj * kBN + 32, w.mt * kBM, hb, bb);
              }
              const uint32_t bs = bfill % P::NB;
              ok = wait_bar(bar(P::B_BE + bs), ((bfill / P::NB) & 1u) ^ 1u, W);
              if (!ok) break;
              mbar_arrive_expect_tx(bar(P::B_BF + bs), P::BIAS_STAGE);
              const uint32_t bdst = sbase + P::OFF_BIAS + bs * P::BIAS_STAGE;
              tma_load_4d(bdst, &p.tm_bias, bar(P::B_BF + bs), j * kBN, w.mt * kBM, hb, bb);
              tma_load_4d(bdst + P::BIAS_BOX, &p.tm_bias, bar(P::B_BF + bs), j * kBN + 32,
                          w.mt * kBM, hb, bb);
              ++bfill;
            }
          }
          const uint32_t vs = vfill % P::NV;
          ok = wait_bar(bar(P::B_VE + vs), ((vfill / P::NV) & 1u) ^ 1u, W);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(P::B_VF + vs), P::V_STAGE);
          const uint32_t vdst = sbase + P::OFF_V + vs * P::V_STAGE;
          if constexpr (F8) {
            // V^T: Dv rows of this tile's 64 keys (x = key, y = row of V^T)
            tma_load_3d(vdst, &p.tm_v, bar(P::B_VF + vs), r, 0, w.z);
          } else {
#pragma unroll
          for (int c = 0; c < DV / 64; ++c) {
            const int x = w.vh * DV + c * 64;  // this unit's column slice
            tma_load_3d(vdst + c * P::V_SUB, &p.tm_v, bar(P::B_VF + vs), x, r, w.z);
            if (JVP) tma_load_3d(vdst + P::V_TILE + c * P::V_SUB, &p.tm_tv, bar(P::B_VF + vs), x, r, w.z);
          }
          }
          ++vfill;
        }
      }
      for (uint32_t s = 0; s < P::NV && s < vfill; ++s) {
        const uint32_t nf = (vfill - s + P::NV - 1) / P::NV;
        drain_bar(bar(P::B_VF + s), (nf - 1) & 1u, p.timeout_ns);
      }
      if constexpr (P::NB > 0) {
        if (bias_ring) {
          for (uint32_t s = 0; s < static_cast<uint32_t>(P::NB) && s < bfill; ++s) {
            const uint32_t nf = (bfill - s + P::NB - 1) / P::NB;
            drain_bar(bar(P::B_BF + s), (nf - 1) & 1u, p.timeout_ns);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------- release warp
    // Frees the K stage of tile g (and Q after a unit's last tile) as soon
    // as the score MMAs of tile g are done, without costing the MMA issuer
    // a commit.  It also arrives on p_full of tile g, so the output MMAs of
    // tile g -- and hence the score MMAs of tile g+2, the next phase of the
    // same s_full barrier -- cannot be issued before it has seen s_full of
    // tile g: its parity waits are unambiguous.
    uint32_t g = 0, qu = 0;  // tiles, units with keys
    bool ok = true;
    for (int rnd = 0; ok; ++rnd) {
      const int u = unit_of_round(rnd);
      if (u >= num_units) break;
      const Unit w = decode_unit<kSlices, kHeadGroups, LEAN>(p, u, list);
      if (w.nt == 0) continue;
      for (int j = 0; j < w.nt; ++j, ++g) {
        ok = __all_sync(0xffffffffu, wait_bar_sleep(bar(P::B_SF + (g & 1u)), (g >> 1) & 1u, W));
        if (!ok) break;
        if (lane == 0) {
          if constexpr (!P::KCH) mbar_arrive(bar(P::B_KE + g % P::NK));
          if (j == w.nt - 1) mbar_arrive(bar(P::B_QE + qu % P::NQB));
          mbar_arrive(bar(P::B_PF + (g & 1u)));
        }
        __syncwarp();
      }
      ++qu;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp walks the issue loop, so descriptors and addresses are
    // warp-uniform values; one lane, elected once, issues every tcgen05
    // instruction.  (An issuer running alone in a diverged warp competes
    // for issue slots with the softmax warps of its sub-partition and lets
    // the tensor pipe run dry between MMAs.)  Each mbarrier poll stalls
    // issue for a round trip even when the barrier is already complete, so
    // the waits for the K / V tiles of the next batches are placed in the
    // middle of a batch, while the tensor pipe still holds queued MMAs.
    const bool leader = elect_one();
    constexpr uint32_t idesc_s = F8 ? idesc_e5m2(kBM, kBN)
                                    : idesc_16(kBM, JVP ? 2 * kBN : kBN, false, F16);  // [S | Q tK^T]
    constexpr uint32_t idesc_t = idesc_16(kBM, kBN, false, F16);                   // tQ K^T
    constexpr uint32_t idesc_o = F8 ? idesc_e5m2(kBM, DV)                         // O (V^T K-major)
                                    : idesc_16(kBM, P::NQ * DV, true, F16);       // [O | tO]
    constexpr uint32_t idesc_h = idesc_16(kBM, DV, true, F16);                     // H V
    auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, wait_bar(b, parity, W));
    };
    // K tile t sits in stage t % NK (fill round t / NK), V tile t in stage
    // t % NV.  Q / K / V arrive by bulk copy: the mbarrier wait alone orders
    // them before the MMAs that read them (no tcgen05 fence needed).
    // In the middle of a batch the tiles of the next batch are only polled
    // once (k_seen / v_seen record a tile found resident); a tile not yet
    // resident is waited for just before the batch that reads it, so a slow
    // copy never holds back the rest of the current batch.
    uint32_t k_seen = 0xffffffffu, v_seen = 0xffffffffu;
    auto poll_k = [&](uint32_t t) {
      if constexpr (!P::KCH)
        if (__all_sync(0xffffffffu, mbar_try_wait(bar(P::B_KF + t % P::NK), (t / P::NK) & 1u))) k_seen = t;
    };
    auto poll_v = [&](uint32_t t) {
      if (__all_sync(0xffffffffu, mbar_try_wait(bar(P::B_VF + t % P::NV), (t / P::NV) & 1u))) v_seen = t;
    };
    auto wait_k = [&](uint32_t t) {
      return k_seen == t || wait_all(bar(P::B_KF + t % P::NK), (t / P::NK) & 1u);
    };
    auto wait_v = [&](uint32_t t) {
      return v_seen == t || wait_all(bar(P::B_VF + t % P::NV), (t / P::NV) & 1u);
    };

    // Descriptor low words of Q buffer 0, K stage 0 (K-major) and V stage 0
    // (MN-major, 64-column chunks V_SUB apart); a buffer / stage / K step is
    // a constant added to the low word (see sdesc_lo), which keeps the issue
    // loop to one add per operand per MMA.
    constexpr uint32_t kHi = sdesc_hi_sw128(1024);
    const uint32_t lo_q = sdesc_lo(sbase + P::OFF_Q, 16);
    const uint32_t lo_k = sdesc_lo(sbase + P::OFF_K, 16);
    const uint32_t lo_v = sdesc_lo(sbase + P::OFF_V, F8 ? 16 : P::V_SUB);
    constexpr uint32_t kHi64 = sdesc_hi_sw64(512);  // e5m2 V^T tiles: 64-byte rows
    // K steps of one score chain: 16 elements (32 bytes) for 16-bit types,
    // 32 elements (32 bytes) for e5m2
    constexpr int KS = F8 ? DQK / 32 : DQK / 16;

    // [S | Q tK^T] = Q [K ; tK]^T, tS += tQ K^T for tile t; `mid` runs after
    // the first half of the first chain.
    auto issue_s = [&](uint32_t t, uint32_t qb, auto&& mid) -> bool {
      const uint32_t lq = lo_q + qb * (P::QSET >> 4);
      const uint32_t dS = tmem + (t & 1u) * P::SBUF;
      if constexpr (P::KCH) {
        // per 64-column chunk c: its four [S | Q tK^T] K steps, then its
        // four tQ K^T steps (accumulating onto the Q tK^T columns the first
        // step initialised), then a commit that frees chunk stage c
#pragma unroll 1
        for (int c = 0; c < P::CH; ++c) {
          if (!wait_all(bar(P::B_KF + c), t & 1u)) return false;
          const uint32_t lk = lo_k + ((c * P::K_GROUP) >> 4);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const uint32_t oq = (c * P::Q_SUB + k4 * 32) >> 4;
            if (leader)
              mma_ss(dS, sdesc_join(lq + oq, kHi), sdesc_join(lk + ((k4 * 32) >> 4), kHi), idesc_s,
                     (c > 0 || k4 > 0) ? 1u : 0u);
            __syncwarp();
          }
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const uint32_t oq = (P::OFF_TQ - P::OFF_Q + c * P::Q_SUB + k4 * 32) >> 4;
            if (leader) mma_ss(dS + kBN, sdesc_join(lq + oq, kHi), sdesc_join(lk + ((k4 * 32) >> 4), kHi), idesc_t, 1u);
            __syncwarp();
          }
          if (leader) tc_commit(bar(P::B_KE + c));
          __syncwarp();
          if (c == P::CH / 2 - 1) mid();
        }
        if (leader) tc_commit(bar(P::B_SF + (t & 1u)));
        __syncwarp();
        return true;
      }
      if (!wait_k(t)) return false;
      const uint32_t lk = lo_k + (t % P::NK) * (P::K_STAGE >> 4);
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        const uint32_t oq = ((kk >> 2) * P::Q_SUB + (kk & 3) * 32) >> 4;
        const uint32_t ok_ = ((kk >> 2) * P::K_GROUP + (kk & 3) * 32) >> 4;
        if (leader) {
          if constexpr (F8)
            mma_ss_f8(dS, sdesc_join(lq + oq, kHi), sdesc_join(lk + ok_, kHi), idesc_s, kk > 0 ? 1u : 0u);
          else
            mma_ss(dS, sdesc_join(lq + oq, kHi), sdesc_join(lk + ok_, kHi), idesc_s, kk > 0 ? 1u : 0u);
        }
        __syncwarp();
        if (kk == KS / 2 - 1) mid();
      }
      if (JVP) {
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint32_t oq = (P::OFF_TQ - P::OFF_Q + (kk >> 2) * P::Q_SUB + (kk & 3) * 32) >> 4;
          const uint32_t ok_ = ((kk >> 2) * P::K_GROUP + (kk & 3) * 32) >> 4;
          if (leader) mma_ss(dS + kBN, sdesc_join(lq + oq, kHi), sdesc_join(lk + ok_, kHi), idesc_t, 1u);
          __syncwarp();
        }
      }
      if (leader) tc_commit(bar(P::B_SF + (t & 1u)));
      __syncwarp();
      return true;
    };

    // [O | tO] += P [V | tV] ; tO += H V for tile t of unit un (O buffer
    // un % NOB), once its P and H are written; `mid` runs after the first
    // half of the first chain.  The first output MMAs of a unit overwrite
    // the O buffer: with two buffers they wait until the epilogue of unit
    // un - 2 has read it.
    // jt: the tile's index within its unit.  Ping-pong softmax: tile t
    // accumulates into O buffer t % 2 (the buffer of the softmax warps that
    // take the tiles of its global parity); the first write of a unit into
    // each buffer (tiles jt = 0 and 1) overwrites it, once the previous
    // unit's merge has read both buffers: the unit's first tile waits for
    // that on both o_empty barriers, so every unit waits each barrier's
    // phases in order.
    auto issue_pv = [&](uint32_t t, int jt, uint32_t un, auto&& mid) -> bool {
      const uint32_t sb = t & 1u;
      const bool first = P::PP ? jt < 2 : jt == 0;
      if (!wait_v(t) || !wait_all(bar(P::B_PF + sb), (t >> 1) & 1u)) return false;
      if constexpr (P::PP) {
        if (jt == 0 && !(wait_all(bar(P::B_OE + 0), (un & 1u) ^ 1u) &&
                         wait_all(bar(P::B_OE + 1), (un & 1u) ^ 1u)))
          return false;
      } else {
        if (P::NOB == 2 && first && !wait_all(bar(P::B_OE + un % P::NOB), ((un / P::NOB) & 1u) ^ 1u))
          return false;
      }
      tc_fence_after();
      const uint32_t colo = P::COL_O + (P::PP ? sb : un % P::NOB) * P::OBUF;
      const uint32_t lv = lo_v + (t % P::NV) * (P::V_STAGE >> 4);
      // keys [16 kk, 16 kk + 16): P at column base + 32 (kk / 2) + 8 (kk % 2),
      // H 16 columns further (the layout the softmax halves write)
      const uint32_t aP = tmem + sb * P::SBUF + kBN;
      if constexpr (F8) {
        // keys [32 kk, 32 kk + 32): e5m2 P in the 8 columns of softmax half
        // kk; V^T rows of 64 keys, the K step 32 bytes along the row
#pragma unroll
        for (int kk = 0; kk < kBN / 32; ++kk) {
          const uint64_t dv = sdesc_join(lv + ((kk * 32) >> 4), kHi64);
          if (leader) mma_ts_f8(tmem + colo, aP + 8 * kk, dv, idesc_o, (first && kk == 0) ? 0u : 1u);
          __syncwarp();
          if (kk == 0) mid();
        }
      } else {
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk) {
        const uint64_t dv = sdesc_join(lv + ((kk * 2048) >> 4), kHi);
        if (leader)
          mma_ts(tmem + colo, aP + 32 * (kk >> 1) + 8 * (kk & 1), dv, idesc_o,
                 (first && kk == 0) ? 0u : 1u);
        __syncwarp();
        if (kk == kBN / 32 - 1) mid();
      }
      }
      if (JVP) {
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t dv = sdesc_join(lv + ((kk * 2048) >> 4), kHi);
          if (leader) mma_ts(tmem + colo + DV, aP + 32 * (kk >> 1) + 16 + 8 * (kk & 1), dv, idesc_h, 1u);
          __syncwarp();
        }
      }
      if (leader) tc_commit(bar(P::B_VE + t % P::NV));
      __syncwarp();
      return true;
    };

    uint32_t quse = 0, g = 0;  // units with keys; g: global tile counter (same in every role)
    bool ok = true;
    if constexpr (P::NQB == 1) {
      // Issue order per unit: S(t0), S(t0+1), PV(t0), S(t0+2), PV(t0+1), ...,
      // PV(last).  The K tile of S(t+1) is polled inside the batch before it
      // (S(t0) for t0+1, else PV(t-1)); the V tile of PV(t) inside S(t+1)
      // (S(last) for the unit's last tile).
      for (int rnd = 0; ok; ++rnd) {
        const int u = unit_of_round(rnd);
        if (u >= num_units) break;
        const Unit w = decode_unit<kSlices, kHeadGroups, LEAN>(p, u, list);
        if (w.nt == 0) continue;
        ok = wait_all(bar(P::B_QF), quse & 1u);
        if (!ok) break;
        // step j: S(t0 + j) (j < nt), then PV(t0 + j - 1) (j > 0): one call
        // site per batch kind keeps the issue loop's code small
        for (int j = 0; j <= w.nt; ++j) {
          if (j < w.nt) {
            ok = issue_s(g, 0, [&]() {
              if (j > 0) poll_v(g - 1);
              if (j == w.nt - 1) poll_v(g);
              else if (j == 0) poll_k(g + 1);
            });
            if (!ok) break;
            ++g;
          }
          if (j > 0) {
            ok = issue_pv(g - 1 - (j < w.nt ? 1u : 0u), j - 1, quse, [&]() {
              if (j + 1 < w.nt) poll_k(g);
            });
            if (!ok) break;
          }
        }
        if (!ok) break;
        ++quse;
      }
    } else {
      // Two Q buffers: the tiles of consecutive units form one stream,
      // S(t+1) issued before PV(t) also when t ends a unit.  The pending
      // output batch (tile pt of unit pu, its index in the unit: pj)
      // is issued after the next score batch; polls as above.
      bool pend = false;
      int pj = 0;
      uint32_t pt = 0, pu = 0;
      for (int rnd = 0; ok; ++rnd) {
        const int u = unit_of_round(rnd);
        if (u >= num_units) break;
        const Unit w = decode_unit<kSlices, kHeadGroups, LEAN>(p, u, list);
        if (w.nt == 0) continue;
        const uint32_t qb = quse % P::NQB;
        ok = wait_all(bar(P::B_QF + qb), (quse / P::NQB) & 1u);
        if (!ok) break;
        for (int j = 0; j < w.nt; ++j, ++g) {
          ok = issue_s(g, qb, [&]() {
            if (pend) poll_v(pt);
          });
          if (!ok) break;
          if (pend) {
            ok = issue_pv(pt, pj, pu, [&]() { poll_k(g + 1); });
            if (!ok) break;
          }
          pend = true;
          pt = g;
          pj = j;
          pu = quse;
        }
        if (!ok) break;
        ++quse;
      }
      if (ok && pend) ok = issue_pv(pt, pj, pu, []() {});
    }
    // Teardown: all MMAs issued by the leader complete before TMEM is freed.
    if (leader) {
      tc_commit(bar(P::B_DRAIN));
      drain_bar(bar(P::B_DRAIN), 0, p.timeout_ns);
    }
    __syncwarp();
  }
  } else {
    setmaxnreg_inc<kHighRegs>();
    // -------------------------------------------- softmax / rescale / epilogue
    const int quad = warp & 3;         // TMEM lane quadrant this warp may access
    const int half = (warp - 4) >> 2;  // which 32 of the 64 key columns
    const int row = quad * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    // Bounded rendezvous of the two warps of this quadrant (64 arrivals per
    // phase); shared-memory writes before it are visible after it.
    uint32_t pair_phase = 0;
    auto pair_sync = [&]() -> bool {
      tc_fence_before();
      mbar_arrive(bar(P::B_PAIR + quad));
      const bool r = __all_sync(0xffffffffu, wait_bar(bar(P::B_PAIR + quad), pair_phase & 1u, W));
      ++pair_phase;
      tc_fence_after();
      return r;
    };
    const bool has_bias = BM && p.bias != nullptr;
    const bool has_mask = BM && p.mask != nullptr;
    float* my_x0 = xchg + (0 * 2 + half) * kBM + row;
    float* my_x1 = xchg + (1 * 2 + half) * kBM + row;
    const float* other_x0 = xchg + (0 * 2 + (half ^ 1)) * kBM + row;
    const float* other_x1 = xchg + (1 * 2 + (half ^ 1)) * kBM + row;
    constexpr int DVH = DV / 2;  // output columns per softmax thread
    const uint64_t scale2 = f2_make(p.sm_scale, p.sm_scale);
    const bool out32 = ((reinterpret_cast<uintptr_t>(p.o) | (JVP ? reinterpret_cast<uintptr_t>(p.to) : 0)) & 31u) == 0;
    // One unit's row state, kept until its epilogue runs.
    struct Epi {
      int mt, q_len;
      long long out0;
      float m_run;
      uint64_t l2, lt2, r2;
      uint32_t g_end;  // one past the unit's last tile
      uint32_t un;     // unit index among units with keys (O buffer un % NOB)
      int vh;          // output column slice
    };
    float* my_xl = xchg + 4 * kBM + row;  // the epilogue's third value (l of half 1)
    // Normalise and store one unit's O, tO and LSE rows.
    auto epilogue = [&](const Epi& e) -> bool {
      const int qi = e.mt * kBM + row;
      const bool row_ok = qi < e.q_len;
      // combine the two halves' partial sums through shared memory (this
      // overlaps the output MMAs of the unit's last tile): both write lt and
      // r, the second half also its l, which only the first half needs
      float l_a, l_b, lt_a, lt_b, r_a, r_b;
      f2_split(e.l2, l_a, l_b);
      f2_split(e.lt2, lt_a, lt_b);
      f2_split(e.r2, r_a, r_b);
      float l_sum = l_a + l_b, lt_sum = lt_a + lt_b, r_sum = r_a + r_b;
      if constexpr (GLOB) {
        if (!pair_sync()) return false;  // both halves are done with the max slots
      }
      *my_x0 = lt_sum;
      *my_x1 = r_sum;
      if (half == 1) *my_xl = l_sum;
      if (!pair_sync()) return false;
      lt_sum += *other_x0;
      r_sum += *other_x1;
      if (half == 0) l_sum += *my_xl;
      if (!pair_sync()) return false;  // slots free for the next use
      // every MMA of the unit is done once the output MMAs of its last tile
      // are; the phase after that one needs a P that this thread has not
      // written yet (at most the next unit's first tile is done), so the
      // parity wait is unambiguous
      const uint32_t gl = e.g_end - 1;
      if (!__all_sync(0xffffffffu, wait_bar(bar(P::B_VE + gl % P::NV), (gl / P::NV) & 1u, W))) return false;
      tc_fence_after();

      // O = O_acc / lt, tO = (tO_acc - r O) / lt as packed bf16 pairs, this
      // thread's DVH columns of its row
      const uint32_t colo = P::COL_O + (e.un % P::NOB) * P::OBUF;
      // (both halves hold the full lt; only the first half has the full l.
      // lt > 0 exactly when the row has a valid key: its largest weight is
      // at least 1 because the reference max trails the row max by < 8)
      const bool empty = !(lt_sum > 0.f);
      const float inv_l = empty ? 0.f : 1.f / lt_sum;
      constexpr int EPW = F8 ? 4 : 2;  // output elements per packed word
      constexpr int NW = DVH / EPW;    // packed words per half row
      constexpr int CW = NW / 4;       // words per chunk (four chunks per half row)
      uint32_t po[NW], pt[NW];
#pragma unroll
      for (int c0 = 0; c0 < DVH; c0 += 32) {
        uint32_t ov[32];
        uint32_t tv[32];
        tmem_ld_32x32b_x32(tl + colo + half * DVH + c0, ov);
        if constexpr (JVP) tmem_ld_32x32b_x32(tl + colo + DV + half * DVH + c0, tv);
        tmem_wait_ld_regs(ov);
        if constexpr (JVP) tmem_regs_ready(tv);
        if constexpr (F8) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            po[c0 / 4 + i / 4] = pack_e5m2x4(__uint_as_float(ov[i]) * inv_l, __uint_as_float(ov[i + 1]) * inv_l,
                                             __uint_as_float(ov[i + 2]) * inv_l, __uint_as_float(ov[i + 3]) * inv_l);
          continue;
        }
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float o0 = __uint_as_float(ov[i]) * inv_l;
          const float o1 = __uint_as_float(ov[i + 1]) * inv_l;
          po[c0 / 2 + i / 2] = pack2<F16>(o0, o1);
          if constexpr (JVP) {
            const float t0 = (__uint_as_float(tv[i]) - r_sum * o0) * inv_l;
            const float t1 = (__uint_as_float(tv[i + 1]) - r_sum * o1) * inv_l;
            pt[c0 / 2 + i / 2] = pack2<F16>(t0, t1);
          }
        }
      }
      if constexpr (P::NOB == 2) {
        // this warp has read the O buffer: the unit after next may reuse it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(P::B_OE + e.un % P::NOB));
      }
      if (row_ok && half == 0 && e.vh == 0)
        p.lse[e.out0 + qi] = empty ? -INFINITY : (e.m_run + __log2f(l_sum)) * kLn2;
      // Rows are stored a quad of lanes at a time: after the transpose lane q
      // of a quad holds chunk q of the quad's four rows, so each store
      // instruction writes eight whole row segments (contiguous per quad).
      const int q = lane & 3;
      quad_transpose<CW>(po, q);
      if constexpr (JVP) quad_transpose<CW>(pt, q);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int qk = e.mt * kBM + quad * 32 + (lane & ~3) + k;       // row of slot k
        const int col = e.vh * DV + half * DVH + q * EPW * CW;          // first column of the chunk
        if (qk < e.q_len && col < p.dv_out) {
          const long long off = (e.out0 + qk) * p.dv_out + col;
          if constexpr (F8)
            store_chunk<CW>(reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(p.o) + off), po + k * CW, false);
          else
            store_chunk<CW>(p.o + off, po + k * CW, out32);
          if constexpr (JVP) store_chunk<CW>(p.to + off, pt + k * CW, out32);
        }
      }
      return true;
    };
    bool ok = true;
    if constexpr (P::PP) {
      // ------------------------------------------------ ping-pong softmax
      // This warp takes the key tiles whose global index (the counter every
      // role keeps) is par mod 2 -- the tiles of score buffer par -- all 64
      // key columns, accumulating through O buffer par; the two parities of
      // a row merge their (m, l, lt, r) and O / tO once per unit (after each
      // one's first tile of the next unit, see pp_merge).  Binding the warp
      // to the buffer, not to the tile's index within its unit, makes it
      // wait every phase of its s_full and p_full barriers in order: after
      // a unit with an odd tile count the in-unit parity would hand it a
      // tile whose barrier's previous phase belonged to the other warp and
      // could still be pending, and a parity wait two phases behind returns
      // at once.
      const int par = half;
      const uint32_t colo_par = P::COL_O + static_cast<uint32_t>(par) * P::OBUF;
      const uint64_t sc2 = f2_make(p.scale_log2, p.scale_log2);
      uint32_t un = 0;  // units with keys seen so far
      uint32_t g = 0;   // global key-tile counter of the unit's first tile (same in every role)
      // Merge the two parities' state of unit e and store its rows.  It
      // runs after this warp's first tile of the next unit (or at once
      // when there is none): that tile's softmax needs neither O buffer,
      // and the next unit's output MMAs wait for o_empty of the merge.
      auto pp_merge = [&](const Epi& e) -> bool {
        const int qi = e.mt * kBM + row;
        const bool row_ok = qi < e.q_len;
        float l_a, l_b, lt_a, lt_b, r_a, r_b;
        f2_split(e.l2, l_a, l_b);
        f2_split(e.lt2, lt_a, lt_b);
        f2_split(e.r2, r_a, r_b);
        // slots [unit parity][value][tile parity][row]: a warp can reuse a
        // unit parity's slots only after the next unit's rendezvous, which
        // its partner reaches after reading them
        float* slot = xchg + (e.un & 1u) * (8 * kBM);
        slot[(0 * 2 + par) * kBM + row] = e.m_run;
        slot[(1 * 2 + par) * kBM + row] = l_a + l_b;
        slot[(2 * 2 + par) * kBM + row] = lt_a + lt_b;
        slot[(3 * 2 + par) * kBM + row] = r_a + r_b;
        if (!pair_sync()) return false;
        // weights of buffer 0 / 1 relative to the merged reference max (an
        // empty parity weighs 0; both warps compute identical sums)
        const float m0 = slot[(0 * 2 + 0) * kBM + row], m1 = slot[(0 * 2 + 1) * kBM + row];
        const float m = fmaxf(m0, m1);
        const float a0 = (m0 == -INFINITY) ? 0.f : ex2(m0 - m);
        const float a1 = (m1 == -INFINITY) ? 0.f : ex2(m1 - m);
        const float l_sum = a0 * slot[(1 * 2 + 0) * kBM + row] + a1 * slot[(1 * 2 + 1) * kBM + row];
        const float lt_sum = a0 * slot[(2 * 2 + 0) * kBM + row] + a1 * slot[(2 * 2 + 1) * kBM + row];
        const float r_sum = a0 * slot[(3 * 2 + 0) * kBM + row] + a1 * slot[(3 * 2 + 1) * kBM + row];
        // every MMA of the unit is done once the output MMAs of its last
        // tile are; the phase after that one is tile gl + NV (NV >= 3), a
        // tile of the next unit past the first one of each parity, whose P
        // neither warp of this quadrant has written
        const uint32_t gl = e.g_end - 1u;
        if (!__all_sync(0xffffffffu, wait_bar(bar(P::B_VE + gl % P::NV), (gl / P::NV) & 1u, W))) return false;
        tc_fence_after();
        const bool empty = !(lt_sum > 0.f);
        const float inv_l = empty ? 0.f : 1.f / lt_sum;
        // a buffer holds no tile of this unit when its parity had none (its
        // weight is then 0 and its stale contents are not read into the sum)
        const bool use0 = a0 != 0.f, use1 = a1 != 0.f;
        constexpr int NW = DVH / 2;  // packed words of this warp's columns
        constexpr int CW = NW / 4;
        uint32_t po[NW], pt[NW];
#pragma unroll
        for (int c0 = 0; c0 < DVH; c0 += 32) {
          uint32_t ov0[32], ov1[32], tv0[32], tv1[32];
          tmem_ld_32x32b_x32(tl + P::COL_O + par * DVH + c0, ov0);
          tmem_ld_32x32b_x32(tl + P::COL_O + P::OBUF + par * DVH + c0, ov1);
          if constexpr (JVP) {
            tmem_ld_32x32b_x32(tl + P::COL_O + DV + par * DVH + c0, tv0);
            tmem_ld_32x32b_x32(tl + P::COL_O + P::OBUF + DV + par * DVH + c0, tv1);
          }
          tmem_wait_ld_regs(ov0);
          tmem_regs_ready(ov1);
          if constexpr (JVP) {
            tmem_regs_ready(tv0);
            tmem_regs_ready(tv1);
          }
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float o[2], t[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float oa = use0 ? a0 * __uint_as_float(ov0[i + e]) : 0.f;
              if (use1) oa = fmaf(a1, __uint_as_float(ov1[i + e]), oa);
              o[e] = oa * inv_l;
              if constexpr (JVP) {
                float ta = use0 ? a0 * __uint_as_float(tv0[i + e]) : 0.f;
                if (use1) ta = fmaf(a1, __uint_as_float(tv1[i + e]), ta);
                t[e] = (ta - r_sum * o[e]) * inv_l;
              }
            }
            po[c0 / 2 + i / 2] = pack2<F16>(o[0], o[1]);
            if constexpr (JVP) pt[c0 / 2 + i / 2] = pack2<F16>(t[0], t[1]);
          }
        }
        // this warp has read both O buffers: the next unit's output MMAs
        // may write them
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(P::B_OE + 0));
          mbar_arrive(bar(P::B_OE + 1));
        }
        if (row_ok && par == 0) p.lse[e.out0 + qi] = empty ? -INFINITY : (m + __log2f(l_sum)) * kLn2;
        // quad-of-lanes transpose, then whole row segments per store
        const int q = lane & 3;
        quad_transpose<CW>(po, q);
        if constexpr (JVP) quad_transpose<CW>(pt, q);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int qk = e.mt * kBM + quad * 32 + (lane & ~3) + k;  // row of slot k
          const int col = par * DVH + q * 2 * CW;                     // first column of the chunk
          if (qk < e.q_len && col < p.dv_out) {
            const long long off = (e.out0 + qk) * p.dv_out + col;
            store_chunk<CW>(p.o + off, po + k * CW, out32);
            if constexpr (JVP) store_chunk<CW>(p.to + off, pt + k * CW, out32);
          }
        }
        return true;
      };
      // One walk over units and this warp's tiles, flattened so that the
      // merge has a single call site (its code is large; one inlined copy
      // keeps the loop's instruction footprint small): each step takes the
      // next unit when the last one is done, then this warp's next tile of
      // it, then the previous unit's merge if one is pending (after the
      // first tile of the next unit, or at once when this parity has no
      // tile in it or no unit is left).
      Epi ppend{};
      bool has_ppend = false;
      Unit w{};
      int rnd = 0, j = 0, qi = 0;
      bool have = false, fresh = true;
      float m_run = -INFINITY;
      uint64_t l2 = 0, lt2 = 0, r2 = 0;
      for (;;) {
        if (fresh) {
          // the next unit with keys; units without keys get empty rows
          fresh = false;
          have = false;
          for (;;) {
            const int u = unit_of_round(rnd);
            if (u >= num_units) break;
            ++rnd;
            w = decode_unit<kSlices, kHeadGroups, LEAN>(p, u, list);
            if (!w.active) continue;
            qi = w.mt * kBM + row;
            const bool row_ok = qi < w.q_len;
            if (!LEAN && w.nt == 0) {  // no keys at all: empty rows (this warp: columns [par DVH, ...))
              const int ncol = min(DVH, p.dv_out - par * DVH);
              if (row_ok && ncol > 0) {
                uint32_t z[DVH / 2];
#pragma unroll
                for (int i = 0; i < DVH / 2; ++i) z[i] = 0u;
                store_row_bf16(p.o + (w.out0 + qi) * p.dv_out + par * DVH, z, ncol / 2);
                if (JVP) store_row_bf16(p.to + (w.out0 + qi) * p.dv_out + par * DVH, z, ncol / 2);
              }
              if (row_ok && par == 0) p.lse[w.out0 + qi] = -INFINITY;
              continue;
            }
            have = true;
            j = (par ^ static_cast<int>(g)) & 1;
            m_run = -INFINITY;
            l2 = lt2 = r2 = 0;
            break;
          }
        }
        if (have && j < w.nt) {
          const uint32_t gt = g + static_cast<uint32_t>(j);
          const uint32_t sb = gt & 1u;
          ok = __all_sync(0xffffffffu, wait_bar(bar(P::B_SF + sb), (gt >> 1) & 1u, W));
          if (!ok) break;
          tc_fence_after();
          const bool diag = !LEAN && p.causal && (j * kBN + kBN - 1 > w.mt * kBM);
          const bool fast = LEAN || (!diag && (j * kBN + kBN <= w.kv_len));
          uint32_t s0[kHalf], s1[kHalf];
          tmem_ld_32x32b_x32(tl + sb * P::SBUF, s0);
          tmem_ld_32x32b_x32(tl + sb * P::SBUF + kHalf, s1);
          tmem_wait_ld_regs(s0);
          tmem_regs_ready(s1);
          float x0[kHalf], x1[kHalf];
#pragma unroll
          for (int c = 0; c < kHalf; ++c) {
            x0[c] = __uint_as_float(s0[c]);
            x1[c] = __uint_as_float(s1[c]);
          }
          uint32_t km0 = 0xffffffffu, km1 = 0xffffffffu;
          if (!fast) {
            // causal diagonal / ragged tail: masked keys at -inf (raw scores;
            // the exponent scales them by s log2 e > 0)
            km0 = keep_bits(j * kBN, w.kv_len, qi, p.causal);
            km1 = keep_bits(j * kBN + kHalf, w.kv_len, qi, p.causal);
#pragma unroll
            for (int c = 0; c < kHalf; ++c) {
              x0[c] = ((km0 >> c) & 1u) ? x0[c] : -INFINITY;
              x1[c] = ((km1 >> c) & 1u) ? x1[c] : -INFINITY;
            }
          }
          const float mx = fmaxf(rowmax32(x0), rowmax32(x1)) * p.scale_log2;
          // lazy online-softmax update of this parity's reference max
          const float m_new = fmaxf(m_run, mx);
          float alpha = 1.f;
          bool resc = false;
          if (m_new > m_run + kRescaleThreshold) {
            if (m_run != -INFINITY) {
              alpha = ex2(m_run - m_new);
              resc = true;
            }
            m_run = m_new;
          }
          const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
          const uint64_t nm2 = f2_make(neg_m, neg_m);
          uint64_t ls = 0;
          float lt0 = 0.f, lt1 = 0.f, rt0 = 0.f, rt1 = 0.f;
          // one 32-column half: P (16 columns) then H (16 columns) over the
          // half's own tS columns, whose load is issued before P is stored
          auto half_step = [&](const float (&x)[kHalf], uint32_t km, int hh) {
            const uint32_t colh = tl + sb * P::SBUF + kBN + hh * kHalf;
            uint32_t tr[kHalf];
            if constexpr (JVP) tmem_ld_32x32b_x32(colh, tr);
            uint64_t pv[kHalf / 2];
            uint32_t pk[kHalf / 2];
#pragma unroll
            for (int c = 0; c < kHalf; c += 2) {
              float a0, a1;
              f2_split(f2_fma(f2_make(x[c], x[c + 1]), sc2, nm2), a0, a1);
              const float p0 = ex2(a0), p1 = ex2(a1);
              const uint64_t pp = f2_make(p0, p1);
              pv[c / 2] = pp;
              ls = f2_add(ls, pp);
              const uint32_t pw = pack2<F16>(p0, p1);
              pk[c / 2] = pw;
              add2_f32<F16>(pw, lt0, lt1);
            }
            tmem_st_32x32b_x16(colh, pk);
            if constexpr (JVP) {
              tmem_wait_ld_regs(tr);
              if (!fast) {
#pragma unroll
                for (int c = 0; c < kHalf; ++c) tr[c] = ((km >> c) & 1u) ? tr[c] : 0u;
              }
              uint32_t hk[kHalf / 2];
#pragma unroll
              for (int c = 0; c < kHalf; c += 2) {
                const uint64_t ts = f2_mul(f2_make(__uint_as_float(tr[c]), __uint_as_float(tr[c + 1])), scale2);
                float h0, h1;
                f2_split(f2_mul(pv[c / 2], ts), h0, h1);
                const uint32_t hw = pack2<F16>(h0, h1);
                hk[c / 2] = hw;
                add2_f32<F16>(hw, rt0, rt1);
              }
              tmem_st_32x32b_x16(colh + kHalf / 2, hk);
            }
          };
          half_step(x0, km0, 0);
          half_step(x1, km1, 1);
          const uint64_t a2 = f2_make(alpha, alpha);
          l2 = f2_fma(l2, a2, ls);
          lt2 = f2_fma(lt2, a2, f2_make(lt0, lt1));
          if constexpr (JVP) r2 = f2_fma(r2, a2, f2_make(rt0, rt1));
          if (__any_sync(0xffffffffu, resc)) {
            // O buffer par is rescaled in place once the previous output MMAs
            // into it (tile gt - 2 of this unit: a parity's first tile never
            // rescales) are done; the phase after that one needs this tile's
            // P, so the parity wait is unambiguous
            const uint32_t gp = gt - 2u;
            ok = __all_sync(0xffffffffu, wait_bar(bar(P::B_VE + gp % P::NV), (gp / P::NV) & 1u, W));
            if (!ok) break;
            tc_fence_after();
            const float a = resc ? alpha : 1.f;
#pragma unroll 1
            for (int c0 = 0; c0 < P::OBUF; c0 += 32) {
              uint32_t v[32];
              tmem_ld_32x32b_x32(tl + colo_par + c0, v);
              tmem_wait_ld_regs(v);
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * a);
              tmem_st_32x32b_x32(tl + colo_par + c0, v);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(P::B_PF + sb));
          j += 2;
        }
        if (has_ppend) {
          has_ppend = false;
          ok = pp_merge(ppend);
          if (!ok) break;
        }
        if (!have) break;
        if (j >= w.nt) {
          ppend = Epi{w.mt, w.q_len, w.out0, m_run, l2, lt2, r2, g + static_cast<uint32_t>(w.nt), un, 0};
          has_ppend = true;
          g += static_cast<uint32_t>(w.nt);
          ++un;
          fresh = true;
        }
      }
    } else {
      uint32_t un = 0;         // units with keys seen so far
      Epi pend{};              // with two O buffers: the unit whose epilogue is due
      bool has_pend = false;
      uint32_t g = 0;           // global key-tile counter (same in every role)
      uint32_t gen = 0;         // masked tiles seen (slot parity of the max exchange)
      for (int rnd = 0; ok; ++rnd) {
        const int u = unit_of_round(rnd);
        if (u >= num_units) break;
        const Unit w = decode_unit<kSlices, kHeadGroups, LEAN>(p, u, list);
        if (!w.active) continue;
        const int qi = w.mt * kBM + row;
        const bool row_ok = qi < w.q_len;
        if (w.nt == 0) {  // no keys at all: empty rows
          // this half's output columns: [c0, min(c0 + DVH, dv_out))
          const int c0 = w.vh * DV + half * DVH;
          const int ncol = min(DVH, p.dv_out - c0);
          if (row_ok && ncol > 0) {
            uint32_t z[DVH / 2];
#pragma unroll
            for (int i = 0; i < DVH / 2; ++i) z[i] = 0u;
            if constexpr (F8) {
              // e5m2 output: one byte per element
              uint8_t* orow8 = reinterpret_cast<uint8_t*>(p.o) + (w.out0 + qi) * p.dv_out + c0;
              store_row_bf16(reinterpret_cast<uint16_t*>(orow8), z, ncol / 4);
            } else {
              uint16_t* orow = p.o + (w.out0 + qi) * p.dv_out + c0;
              uint16_t* torow = JVP ? p.to + (w.out0 + qi) * p.dv_out + c0 : nullptr;
              store_row_bf16(orow, z, ncol / 2);
              if (JVP) store_row_bf16(torow, z, ncol / 2);
            }
          }
          if (row_ok && half == 0 && w.vh == 0) p.lse[w.out0 + qi] = -INFINITY;
          continue;
        }
        const float* brow = nullptr;
        const unsigned char* mrow = nullptr;
        if (has_bias)
          brow = p.bias + w.b * p.bias_stride[0] + w.h * p.bias_stride[1] +
                 static_cast<long long>(qi) * p.bias_stride[2];
        // a mask that is a key prefix of this (b, h) is already in kv_len
        const bool umask = has_mask && w.mask_on;
        if (umask)
          mrow = p.mask + w.b * p.mask_stride[0] + w.h * p.mask_stride[1] +
                 static_cast<long long>(qi) * p.mask_stride[2];

        // m_run: reference max (log2 units), shared by both halves of a row.
        // l2: exact partial sum of p (for LSE); lt2 / r2: partial sums of the
        // bf16 values of p and p*tS that the MMAs consume, so O and tO are
        // normalised by the weights actually used.  Pairs of fp32 lanes.
        float m_run = -INFINITY;
        uint64_t l2 = 0, lt2 = 0, r2 = 0;
        const uint32_t colo_cur = P::COL_O + (un % P::NOB) * P::OBUF;  // this unit's O buffer
        for (int j = 0; j < w.nt; ++j, ++g) {
          const uint32_t sb = g & 1u;
          const int key0 = j * kBN + half * kHalf;  // first key of this thread's columns
          // Bias rows stream from HBM once: pull this thread's segment of the
          // tile two steps ahead into L2 (the first two tiles at unit start),
          // then load this tile's entries before waiting on S.
          if (GLOB && has_bias && row_ok && p.bias_stride[3] == 1) {
            const float* bp = brow + half * kHalf;
            if (j == 0) {
              prefetch_l2(bp);
              if (w.nt > 1) prefetch_l2(bp + kBN);
            }
            if (j + 2 < w.nt) prefetch_l2(bp + (j + 2) * kBN);
          }
          float bv[kHalf];
          uint32_t mv[kHalf / 4];
          uint32_t mvo[kHalf / 4];  // the partner's columns (local row maximum)
          if (GLOB && has_bias) {
#pragma unroll
            for (int c = 0; c < kHalf; ++c) bv[c] = 0.f;
            if (row_ok) {
              const float* bp = brow + static_cast<long long>(key0) * p.bias_stride[3];
              if (p.bias_stride[3] == 1 && (reinterpret_cast<uintptr_t>(bp) & 15u) == 0 &&
                  key0 + kHalf <= w.kv_len) {
#pragma unroll
                for (int c = 0; c < kHalf / 4; ++c) {
                  const float4 t4 = __ldg(reinterpret_cast<const float4*>(bp) + c);
                  bv[4 * c] = t4.x;
                  bv[4 * c + 1] = t4.y;
                  bv[4 * c + 2] = t4.z;
                  bv[4 * c + 3] = t4.w;
                }
              } else {
                for (int c = 0; c < kHalf; ++c)
                  if (key0 + c < w.kv_len) bv[c] = __ldg(bp + c * p.bias_stride[3]);
              }
            }
          }
          if (umask) {
            load_mask32(mrow, key0, w.kv_len, p.mask_stride[3], row_ok, mv);
            if (RING) load_mask32(mrow, j * kBN + (half ^ 1) * kHalf, w.kv_len, p.mask_stride[3], row_ok, mvo);
          }

          ok = __all_sync(0xffffffffu, wait_bar(bar(P::B_SF + sb), (g >> 1) & 1u, W));
          if (!ok) break;
          tc_fence_after();
          if constexpr (RING) {
            if (has_bias) {
              // this tile's bias stage, waited for before the score loads so
              // that the wait overlaps them (the stage is waited on even when
              // unused, so that its next fill cannot start before this one
              // has landed)
              constexpr int NBR = P::NB > 0 ? P::NB : 1;
              ok = __all_sync(0xffffffffu, wait_bar(bar(P::B_BF + g % NBR), (g / NBR) & 1u, W));
              if (!ok) break;
            }
          }
          // Each warp also reads the partner half's 32 score columns and takes
          // the row maximum over all 64 itself, so the two warps of a quadrant
          // never wait for each other: unmasked tiles (`fast`) and masked tiles
          // (`local`: causal diagonal, ragged tail, mask, and bias read from
          // the shared-memory ring), the mask applied to both halves.  Only a
          // bias read per thread from global memory makes the two warps
          // exchange partial maxima through shared memory instead.
          const bool diag = p.causal && (j * kBN + kBN - 1 > w.mt * kBM);
          const bool fast = !BM && !diag && (j * kBN + kBN <= w.kv_len);
          const bool local = !GLOB && !fast;
          uint32_t sr[kHalf];
          uint32_t so[kHalf];
          uint32_t tr[kHalf];
          tmem_ld_32x32b_x32(tl + sb * P::SBUF + half * kHalf, sr);
          if (fast) {
            tmem_ld_32x32b_x32(tl + sb * P::SBUF + (half ^ 1) * kHalf, so);
            tmem_wait_ld_regs(sr);
            tmem_regs_ready(so);
            // the tangent scores are needed only after the exponentials, so
            // their load overlaps the row maximum and exp2 below
            if constexpr (JVP) tmem_ld_32x32b_x32(tl + sb * P::SBUF + kBN + half * kHalf, tr);
          } else {
            if (local) tmem_ld_32x32b_x32(tl + sb * P::SBUF + (half ^ 1) * kHalf, so);
            if constexpr (JVP) tmem_ld_32x32b_x32(tl + sb * P::SBUF + kBN + half * kHalf, tr);
            tmem_wait_ld_regs(sr);
            tmem_regs_ready(so);
            if constexpr (JVP) tmem_regs_ready(tr);
          }
          float x[kHalf];
#pragma unroll
          for (int c = 0; c < kHalf; ++c) x[c] = __uint_as_float(sr[c]);

          float sc;  // factor taking x to log2 units inside the exponent
          float mx;
          bool dead = false;  // no key of the tile kept for any row of this warp
          if (fast) {
            sc = p.scale_log2;
            float xo[kHalf];
#pragma unroll
            for (int c = 0; c < kHalf; ++c) xo[c] = __uint_as_float(so[c]);
            mx = fmaxf(rowmax32(x), rowmax32(xo)) * p.scale_log2;
          } else if (RING) {
            // bias from the shared-memory ring (rows 128-byte swizzled: 16-byte
            // chunk k of row r at chunk k ^ (r mod 8)) for both halves'
            // columns, so the row maximum needs no exchange
            sc = 1.f;
            constexpr int NBR = P::NB > 0 ? P::NB : 1;
            const int keyo = j * kBN + (half ^ 1) * kHalf;
            uint32_t km = keep_bits(key0, w.kv_len, qi, p.causal);
            uint32_t kmo = keep_bits(keyo, w.kv_len, qi, p.causal);
            if (umask) {
              // Most tiles of a key-padding or block mask are wholly kept or
              // wholly masked: only mixed mask bytes need the bit gather.
              uint32_t any_set = 0u, any_zero = 0u;
#pragma unroll
              for (int wd = 0; wd < kHalf / 4; ++wd) {
                any_set |= mv[wd] | mvo[wd];
                any_zero |= __vcmpeq4(mv[wd], 0u) | __vcmpeq4(mvo[wd], 0u);
              }
              if (any_set == 0u) {
                km = 0u;
                kmo = 0u;
              } else if (any_zero != 0u) {
                km &= mask_bits32(mv);
                kmo &= mask_bits32(mvo);
              }
            }
            // warp-uniform tile classes: every key kept (no per-element
            // selects) or none kept (no arithmetic; P = H = 0)
            const bool all_keep = __all_sync(0xffffffffu, (km & kmo) == 0xffffffffu);
            dead = __all_sync(0xffffffffu, (km | kmo) == 0u);
            const uint8_t* bbase = smem + P::OFF_BIAS + (g % NBR) * P::BIAS_STAGE + row * 128;
            float xo[kHalf];
            if (dead) {
              mx = -INFINITY;
            } else if (all_keep && !has_bias) {
              // as without a mask: the row maximum of the raw scores, scaled once
              sc = p.scale_log2;
#pragma unroll
              for (int c = 0; c < kHalf; ++c) xo[c] = __uint_as_float(so[c]);
              mx = fmaxf(rowmax32(x), rowmax32(xo)) * p.scale_log2;
            } else if (all_keep) {
              // x = s S + bias in natural units (one packed FMA per pair); the
              // exponent's factor becomes log2 e
              sc = kLog2e;
              const uint64_t s2 = f2_make(p.sm_scale, p.sm_scale);
#pragma unroll
              for (int k4 = 0; k4 < kHalf / 4; ++k4) {
                const int phys = (k4 ^ (row & 7)) * 16;
                const float4 b4 = *reinterpret_cast<const float4*>(bbase + half * P::BIAS_BOX + phys);
                const float4 bo4 = *reinterpret_cast<const float4*>(bbase + (half ^ 1) * P::BIAS_BOX + phys);
                const int c = 4 * k4;
                f2_split(f2_fma(f2_make(x[c], x[c + 1]), s2, f2_make(b4.x, b4.y)), x[c], x[c + 1]);
                f2_split(f2_fma(f2_make(x[c + 2], x[c + 3]), s2, f2_make(b4.z, b4.w)), x[c + 2], x[c + 3]);
                f2_split(f2_fma(f2_make(__uint_as_float(so[c]), __uint_as_float(so[c + 1])), s2,
                                f2_make(bo4.x, bo4.y)),
                         xo[c], xo[c + 1]);
                f2_split(f2_fma(f2_make(__uint_as_float(so[c + 2]), __uint_as_float(so[c + 3])), s2,
                                f2_make(bo4.z, bo4.w)),
                         xo[c + 2], xo[c + 3]);
              }
              mx = fmaxf(rowmax32(x), rowmax32(xo)) * kLog2e;
            } else {
#pragma unroll
              for (int k4 = 0; k4 < kHalf / 4; ++k4) {
                float4 b4 = make_float4(0.f, 0.f, 0.f, 0.f), bo4 = b4;
                if (has_bias) {
                  const int phys = (k4 ^ (row & 7)) * 16;
                  b4 = *reinterpret_cast<const float4*>(bbase + half * P::BIAS_BOX + phys);
                  bo4 = *reinterpret_cast<const float4*>(bbase + (half ^ 1) * P::BIAS_BOX + phys);
                }
                const float bo[4] = {bo4.x, bo4.y, bo4.z, bo4.w};
                const float bw[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int c = 4 * k4 + e;
                  const float v = fmaf(bw[e], kLog2e, x[c] * p.scale_log2);
                  const float vo = fmaf(bo[e], kLog2e, __uint_as_float(so[c]) * p.scale_log2);
                  x[c] = ((km >> c) & 1u) ? v : -INFINITY;
                  xo[c] = ((kmo >> c) & 1u) ? vo : -INFINITY;
                  if constexpr (JVP) tr[c] = ((km >> c) & 1u) ? tr[c] : 0u;
                }
              }
              mx = fmaxf(rowmax32(x), rowmax32(xo));
            }
            if (has_bias) {
              // this warp is done with the tile's bias
              __syncwarp();
              if (lane == 0) mbar_arrive(bar(P::B_BE + g % NBR));
            }
          } else {
            sc = 1.f;
            if constexpr (!BM) {
              // causal diagonal / ragged tail: both halves under the same mask
              const int keyo = j * kBN + (half ^ 1) * kHalf;
              const uint32_t km = keep_bits(key0, w.kv_len, qi, p.causal);
              const uint32_t kmo = keep_bits(keyo, w.kv_len, qi, p.causal);
              float xo[kHalf];
#pragma unroll
              for (int c = 0; c < kHalf; ++c) {
                x[c] = ((km >> c) & 1u) ? x[c] * p.scale_log2 : -INFINITY;
                xo[c] = ((kmo >> c) & 1u) ? __uint_as_float(so[c]) * p.scale_log2 : -INFINITY;
                if constexpr (JVP) tr[c] = ((km >> c) & 1u) ? tr[c] : 0u;
              }
              mx = fmaxf(rowmax32(x), rowmax32(xo));
            } else {
              uint32_t km = keep_bits(key0, w.kv_len, qi, p.causal);
              if (umask) km &= mask_bits32(mv);
#pragma unroll
              for (int c = 0; c < kHalf; ++c) {
                float v = x[c] * p.scale_log2;
                if (has_bias) v = fmaf(bv[c], kLog2e, v);
                x[c] = ((km >> c) & 1u) ? v : -INFINITY;
                if constexpr (JVP) tr[c] = ((km >> c) & 1u) ? tr[c] : 0u;
              }
              mx = rowmax32(x);
              // the pair's row maximum over all 64 columns of the tile; the
              // slot alternates per tile, and a writer can only come back to a
              // slot after the rendezvous of the tile in between
              float* mine = (gen & 1u) ? my_x1 : my_x0;
              const float* theirs = (gen & 1u) ? other_x1 : other_x0;
              ++gen;
              *mine = mx;
              ok = pair_sync();
              if (!ok) break;
              mx = fmaxf(mx, *theirs);
            }
          }

          // lazy online-softmax update (identical in both halves)
          const float m_new = fmaxf(m_run, mx);
          float alpha = 1.f;
          bool resc = false;
          if (m_new > m_run + kRescaleThreshold) {
            if (m_run != -INFINITY) {
              alpha = ex2(m_run - m_new);
              resc = true;
            }
            m_run = m_new;
          }
          const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
          const uint64_t sc2 = f2_make(sc, sc), nm2 = f2_make(neg_m, neg_m);
          uint64_t ls = 0;
          float lt0 = 0.f, lt1 = 0.f, rt0 = 0.f, rt1 = 0.f;
          uint64_t pv[kHalf / 2];
          if (!F8 && dead) {
            // P = H = 0 for the output MMAs; m, l and r stay as they are
            uint32_t zk[kHalf / 2];
#pragma unroll
            for (int c = 0; c < kHalf / 2; ++c) zk[c] = 0u;
            tmem_st_32x32b_x16(tl + sb * P::SBUF + kBN + half * kHalf, zk);
            if constexpr (JVP) tmem_st_32x32b_x16(tl + sb * P::SBUF + kBN + half * kHalf + kHalf / 2, zk);
          } else if constexpr (F8) {
            // four e5m2 weights per column, half h in the 8 columns at 8 h
            uint32_t pk8[kHalf / 4];
#pragma unroll
            for (int c = 0; c < kHalf; c += 4) {
              float a0, a1, a2, a3;
              f2_split(f2_fma(f2_make(x[c], x[c + 1]), sc2, nm2), a0, a1);
              f2_split(f2_fma(f2_make(x[c + 2], x[c + 3]), sc2, nm2), a2, a3);
              const float p0 = ex2(a0), p1 = ex2(a1), p2 = ex2(a2), p3 = ex2(a3);
              ls = f2_add(ls, f2_add(f2_make(p0, p1), f2_make(p2, p3)));
              pk8[c / 4] = pack_e5m2x4(p0, p1, p2, p3);
            }
            // the normaliser is the row sum of the unrounded weights: the
            // tutorial takes it before the cast to e5m2
            f2_split(ls, lt0, lt1);
            tmem_st_32x32b_x8(tl + sb * P::SBUF + kBN + half * (kHalf / 4), pk8);
          } else {
          uint32_t pk[kHalf / 2];
#pragma unroll
          for (int c = 0; c < kHalf; c += 2) {
            float a0, a1;
            f2_split(f2_fma(f2_make(x[c], x[c + 1]), sc2, nm2), a0, a1);
            const float p0 = ex2(a0), p1 = ex2(a1);
            const uint64_t pp = f2_make(p0, p1);
            pv[c / 2] = pp;
            ls = f2_add(ls, pp);
            const uint32_t pw = pack2<F16>(p0, p1);
            pk[c / 2] = pw;
            add2_f32<F16>(pw, lt0, lt1);
          }
          tmem_st_32x32b_x16(tl + sb * P::SBUF + kBN + half * kHalf, pk);
          }
          if (JVP && !dead) {
            uint32_t hk[kHalf / 2];
            tmem_wait_ld_regs(tr);
#pragma unroll
            for (int c = 0; c < kHalf; c += 2) {
              const uint64_t ts =
                  f2_mul(f2_make(__uint_as_float(tr[c]), __uint_as_float(tr[c + 1])), scale2);
              float h0, h1;
              f2_split(f2_mul(pv[c / 2], ts), h0, h1);
              const uint32_t hw = pack2<F16>(h0, h1);
              hk[c / 2] = hw;
              add2_f32<F16>(hw, rt0, rt1);
            }
            tmem_st_32x32b_x16(tl + sb * P::SBUF + kBN + half * kHalf + kHalf / 2, hk);
          }
          const uint64_t a2 = f2_make(alpha, alpha);
          l2 = f2_fma(l2, a2, ls);
          lt2 = f2_fma(lt2, a2, f2_make(lt0, lt1));
          if constexpr (JVP) r2 = f2_fma(r2, a2, f2_make(rt0, rt1));

          if (__any_sync(0xffffffffu, resc)) {
            // O and tO are rescaled in place, so the previous tile's output
            // MMAs must have completed: phase (g-1) / NV of v_empty of its
            // stage.  The phase after it needs the output MMAs of tile
            // g-1+NV > g, whose P this thread has not written yet, so the
            // parity wait is unambiguous.  (resc is never set on a unit's
            // first tile, where m_run starts at -inf.)
            ok = __all_sync(0xffffffffu, wait_bar(bar(P::B_VE + (g - 1) % P::NV), ((g - 1) / P::NV) & 1u, W));
            if (!ok) break;
            tc_fence_after();
            {
              // (rare: kept as a rolled loop so the tile loop's code stays small)
              const float a = resc ? alpha : 1.f;
#pragma unroll 1
              for (int c0 = 0; c0 < DVH; c0 += 32) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tl + colo_cur + half * DVH + c0, v);
                tmem_wait_ld_regs(v);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * a);
                tmem_st_32x32b_x32(tl + colo_cur + half * DVH + c0, v);
                if constexpr (JVP) {
                  tmem_ld_32x32b_x32(tl + colo_cur + DV + half * DVH + c0, v);
                  tmem_wait_ld_regs(v);
#pragma unroll
                  for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * a);
                  tmem_st_32x32b_x32(tl + colo_cur + DV + half * DVH + c0, v);
                }
              }
            }
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(P::B_PF + sb));
          if (P::NOB == 2 && j == 0 && has_pend) {
            // the previous unit's epilogue, now that this unit's first output
            // MMAs can run
            has_pend = false;
            ok = epilogue(pend);
            if (!ok) break;
          }
        }
        if (!ok) break;

        // ------------------------------------------------------------ epilogue
        const Epi cur{w.mt, w.q_len, w.out0, m_run, l2, lt2, r2, g, un, w.vh};
        ++un;
        if constexpr (P::NOB == 2) {
          // runs after the next unit's first tile
          pend = cur;
          has_pend = true;
        } else {
          ok = epilogue(cur);
          if (!ok) break;
        }
      }
      if (ok && has_pend) ok = epilogue(pend);
    }

    // Jagged rows past max_seq_len inside their sequence: empty rows.  (The
    // e5m2 kernel is dense only.)
    if (!F8 && ok && p.jagged) {
      const int t256 = threadIdx.x - 128;
      for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
        const int begin = __ldg(p.offsets + b), end = __ldg(p.offsets + b + 1);
        const int kept = min(end - begin, p.max_seq_len);
        for (int h = 0; h < p.H; ++h) {
          for (int rr = begin + kept + t256; rr < end; rr += 256) {
            const long long o_row = static_cast<long long>(h) * p.T + rr;
            uint32_t z[DV / 2];
#pragma unroll
            for (int i = 0; i < DV / 2; ++i) z[i] = 0u;
            // the whole row (every column slice), DV columns at a time
            for (int c0 = 0; c0 < p.dv_out; c0 += DV) {
              const int n = min(DV, p.dv_out - c0);
              store_row_bf16(p.o + o_row * p.dv_out + c0, z, n / 2);
              if (JVP) store_row_bf16(p.to + o_row * p.dv_out + c0, z, n / 2);
            }
            p.lse[o_row] = -INFINITY;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, P::TMEM_COLS);
}

template <int DQK, int DV, bool JVP, int BMODE, bool F16, bool F8 = false, bool LEAN = false>
cudaError_t launch_attn(const KernelParams& kp, int grid, cudaStream_t stream) {
  using P = Plan<DQK, DV, JVP, BMODE, F8>;
  static_assert(P::FITS, "shared memory plan exceeds 227 KB");
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_done[dev]) {
    // The register split is only valid for the launch allocation it was
    // computed for; a build that compiled to another count is refused
    // (setmaxnreg.inc would otherwise wait for registers that never free).
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, attn_fwd_kernel<DQK, DV, JVP, BMODE, F16, F8, LEAN>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kLaunchRegs || fa.maxThreadsPerBlock < kThreads)
      return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(attn_fwd_kernel<DQK, DV, JVP, BMODE, F16, F8, LEAN>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, P::SMEM_LAUNCH);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  // a programmatic dependent of the kernel before it on the stream (the
  // kernel waits for it before its first global access)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = P::SMEM_LAUNCH;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_fwd_kernel<DQK, DV, JVP, BMODE, F16, F8, LEAN>, kp);
}

}  // namespace attn
