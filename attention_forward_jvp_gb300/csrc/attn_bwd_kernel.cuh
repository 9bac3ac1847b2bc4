// Attention backward for sm_103a: gradients dQ, dK, dV of a loss through
// O = softmax(s Q K^T + bias) V (keys outside the valid set -- causal, key
// mask -- at -inf), given dO and the forward's log-sum-exp.  The bias gets
// no gradient.
//
// Method (the Triton fused-attention tutorial's backward, "_attn_bwd_dkdv"
// and "_attn_bwd_dq"; "flash_attention.py" "_attn_bwd_dkdv_inner" /
// "_attn_bwd_dq_inner"): P is recomputed from the stored LSE, no running
// maximum, and
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - Delta),  dQ = s dS K,  dK = s dS^T Q
// with Delta = rowsum(dO o O) from a preprocessing pass.  Two passes, each
// a persistent kernel of this template:
//   dQ pass (KV = false): a unit is 128 query rows; key tiles of 64 stream
//     by.  Row operands Q, dO; streamed K, V.  Scores S = Q K^T, dP = dO V^T;
//     dQ += dS K.
//   dK / dV pass (KV = true): a unit is 128 key rows; query tiles of 64
//     stream by.  Row operands K, V; streamed Q, dO.  S^T = K Q^T,
//     dP^T = V dO^T; dV += P^T dO, dK += dS^T Q.
// Neither pass needs atomics: each owns its output rows.
//
// GB300 mapping (one CTA per SM, 12 warps, as the forward kernel):
//   warp 0  bulk-tensor producer: the unit's two row operands, then the
//           two streamed operands of each tile into a ring of NS stages.
//   warp 1  tcgen05 issuer (whole warp, one elected lane): per tile the two
//           score chains (N = 64 each) into a double-buffered TMEM pair,
//           then the previous tile's output chain(s) from TMEM operands.
//           A commit after a unit's last score chain frees the row operands
//           (a commit completes its barrier exactly once, when the MMAs
//           before it are done, so no waiter can mistake one phase for
//           another).
//   warps 4..11  elementwise warps, two per TMEM lane quadrant, 32 of the 64
//           columns each: P = exp2(S s log2e - LSE log2e), dS = P (dP - Delta),
//           written as 16-bit operands over the thread's own dP columns;
//           the epilogue scales and stores the accumulators.
#pragma once
#include <type_traits>

#include "attn_kernel.cuh"

namespace attn {

struct BwdParams {
  CUtensorMap tm_r1, tm_r2;  // row operands, box 64 x 128 (dQ: Q, dO; KV: K, V)
  CUtensorMap tm_t1, tm_t2;  // streamed operands, box 64 x 64 (dQ: K, V; KV: Q, dO)
  int B, H, M, N;
  int causal;
  int jagged;          // [H, T, D] layout with offsets[B + 1]
  const int* offsets;  // jagged: device offsets
  long long T;         // jagged: total tokens
  int max_seq_len;     // jagged: cap on a sequence's length
  int n_rt;       // row tiles of 128 per (b, h) (jagged: per max_seq_len)
  int num_units;  // B * H * n_rt
  // Jagged work list (optional): unit_count[0] (sequence, row tile) pairs,
  // costliest first, at unit_list (x = sequence, y = tile); unit u is pair
  // u / H, head u % H.  A count of -1 means the list was not written.
  const int2* unit_list;
  const int* unit_count;
  float scale_log2;  // sm_scale * log2(e)
  float sm_scale;
  const float* lse;    // [B, H, M] (jagged [H, T]), natural log
  const float* delta;  // same layout as lse
  uint16_t* out1;      // dQ pass: dQ; KV pass: dK
  uint16_t* out2;      // KV pass: dV
  int d_qk;            // row width of q, k, dq, dk (Dqk; 16 / 32 run padded to 64)
  int d_v;             // row width of v, o, do, dv
  // dense only, both optional: fp32 additive bias and uint8 mask (nonzero =
  // attend) over [B, H, M, N], element strides, 0 = broadcast
  const float* bias;
  long long bias_stride[4];
  const unsigned char* mask;
  long long mask_stride[4];
  int* err;
  unsigned long long timeout_ns;
};

template <int DQK, int DV, bool KV>
struct BwdPlan {
  static constexpr int TN = 64;                      // streamed rows per tile
  static constexpr int R_SUB = kBM * 128;            // 64-column chunk of a row operand
  static constexpr int T_SUB = TN * 128;             // 64-column chunk of a streamed tile
  // row operands R1 (Q / K, Dqk wide) then R2 (dO / V, Dv wide); streamed
  // T1 (K / Q, Dqk) then T2 (V / dO, Dv)
  static constexpr int R1_TILE = (DQK / 64) * R_SUB;
  static constexpr int R2_TILE = (DV / 64) * R_SUB;
  static constexpr int T1_TILE = (DQK / 64) * T_SUB;
  static constexpr int T2_TILE = (DV / 64) * T_SUB;
  static constexpr int RSET = R1_TILE + R2_TILE;
  static constexpr int T_STAGE = T1_TILE + T2_TILE;
  static constexpr int BUDGET = 227 * 1024 - 4096;
  static constexpr int NS = (RSET + 4 * T_STAGE <= BUDGET) ? 4 : (RSET + 3 * T_STAGE <= BUDGET) ? 3 : 2;
  // TMEM: score buffer b = [X (64 fp32: S or S^T) | Y (64 fp32: dP or dP^T)]
  // at b * 128, three buffers where the accumulators leave room, else two;
  // accumulators after them: dQ pass dQ (Dqk); KV pass dV (Dv), dK (Dqk)
  static constexpr int SBUF = 2 * TN;
  static constexpr int NACC = KV ? DV + DQK : DQK;
  static constexpr int NSB = (3 * SBUF + NACC <= 512) ? 3 : 2;
  static constexpr int COL_A = NSB * SBUF;
  static constexpr int COLS_USED = COL_A + NACC;
  static constexpr int TMEM_COLS = COLS_USED <= 256 ? 256 : 512;
  static constexpr int OFF_R = 0;
  static constexpr int OFF_T = RSET;
  static constexpr int OFF_BAR = OFF_T + NS * T_STAGE;
  // barriers: r_full, r_empty, t_full[NS], t_empty[NS], s_full[NSB],
  // p_full[NSB], drain (score issuer), o_done[NSB] (the output chain that
  // read score buffer b is done), drain (output issuer)
  static constexpr int B_RF = 0, B_RE = 1, B_TF = 2, B_TE = B_TF + NS, B_SF = B_TE + NS,
                       B_PF = B_SF + NSB, B_DRAIN = B_PF + NSB, B_OD = B_DRAIN + 1,
                       B_DRAIN2 = B_OD + NSB, NBAR = B_DRAIN2 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // KV pass: per elementwise warp, the current query tile's 32 column
  // values of -LSE log2(e) then -Delta
  static constexpr int OFF_COLV = (OFF_MISC + 16 + 15) / 16 * 16;
  static constexpr int SMEM_BYTES = OFF_COLV + (KV ? 8 * 64 * 4 : 0);
  static constexpr int SMEM_LAUNCH = SMEM_BYTES > 120 * 1024 ? SMEM_BYTES : 120 * 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory plan exceeds 227 KB");
  static_assert(COLS_USED <= 512, "tensor memory plan exceeds 512 columns");
  static_assert((DQK == 64 || DQK == 128) && (DV == 64 || DV == 128), "head dims 64 or 128");
};

struct BwdUnit {
  int z;            // tensor-map z: b * H + h (dense) or h (jagged)
  int rt;           // row tile
  int t0;           // first streamed tile (KV causal: the diagonal)
  int nt;           // streamed tiles (rows with none get zero gradients)
  int rows;         // valid positions of this pass's rows (queries for dQ, keys for KV)
  int cols;         // valid positions of the streamed dimension (keys for dQ, queries for KV)
  int row0;         // tensor-map row of position 0 (jagged: the sequence's first token)
  long long orow0;  // output row of position 0 of this pass's rows
  long long qrow0;  // LSE / Delta index of query 0
  int b, h;         // batch entry and head (dense)
};

// Unit u, costliest first: dense causal dQ units by descending query tile,
// causal KV units by ascending key tile (more query tiles above the
// diagonal); jagged units from the work list when one was written (ordered
// by cost), else by descending row tile (a high tile only exists in a long
// sequence) except causal KV, ascending.  A jagged unit past its
// sequence's length has no rows and nt = 0.
template <bool KV>
__device__ __forceinline__ BwdUnit bwd_unit(const BwdParams& p, int u) {
  const int BH = p.B * p.H;
  BwdUnit w;
  int q_len, k_len;
  if (!p.jagged) {
    if (p.causal) {
      w.rt = KV ? u / BH : p.n_rt - 1 - u / BH;
      w.z = u % BH;
    } else {
      w.z = u / p.n_rt;
      w.rt = u % p.n_rt;
    }
    q_len = p.M;
    k_len = p.N;
    w.row0 = 0;
    w.qrow0 = static_cast<long long>(w.z) * p.M;
    w.orow0 = static_cast<long long>(w.z) * (KV ? p.N : p.M);
  } else {
    int b, h;
    if (p.unit_list != nullptr && __ldg(p.unit_count) >= 0) {
      const int2 e = p.unit_list[u / p.H];
      b = e.x;
      w.rt = e.y;
      h = u % p.H;
    } else {
      const int tile = u / BH, r = u % BH;
      w.rt = (KV && p.causal) ? tile : p.n_rt - 1 - tile;
      b = r / p.H;
      h = r % p.H;
    }
    const int begin = __ldg(p.offsets + b), end = __ldg(p.offsets + b + 1);
    const int len = max(0, min(end - begin, p.max_seq_len));
    q_len = k_len = len;
    w.z = h;
    w.row0 = begin;
    w.qrow0 = static_cast<long long>(h) * p.T + begin;
    w.orow0 = w.qrow0;
  }
  w.rows = KV ? k_len : q_len;
  w.cols = KV ? q_len : k_len;
  w.b = p.jagged ? 0 : w.z / p.H;
  w.h = p.jagged ? w.z : w.z % p.H;
  const bool active = w.rt * kBM < w.rows;
  if (!KV) {
    int hi = k_len;
    if (p.causal) hi = min(hi, (w.rt + 1) * kBM);
    w.t0 = 0;
    w.nt = active ? (hi + 63) / 64 : 0;
  } else {
    const int nq = (q_len + 63) / 64;
    w.t0 = p.causal ? (w.rt * kBM) / 64 : 0;
    w.nt = active ? max(0, nq - w.t0) : 0;
  }
  return w;
}

// BM: the launch has a bias and / or a mask (their loads and terms are
// compiled only into those instantiations).
template <int DQK, int DV, bool KV, bool F16, bool BM>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_kernel(const __grid_constant__ BwdParams p) {
  using P = BwdPlan<DQK, DV, KV>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicCAS(p.err, 0, ERR_SMEM_ALIGN);
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + P::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + P::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    mbar_init(bar(P::B_RF), 1);
    mbar_init(bar(P::B_RE), 1);
    for (int i = 0; i < P::NS; ++i) {
      mbar_init(bar(P::B_TF + i), 1);
      mbar_init(bar(P::B_TE + i), 1);
    }
    for (int i = 0; i < P::NSB; ++i) {
      mbar_init(bar(P::B_SF + i), 1);
      mbar_init(bar(P::B_PF + i), 8);  // one arrival per elementwise warp
      mbar_init(bar(P::B_OD + i), 1);
    }
    mbar_init(bar(P::B_DRAIN), 1);
    mbar_init(bar(P::B_DRAIN2), 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.tm_r1);
    prefetch_tmap(&p.tm_r2);
    prefetch_tmap(&p.tm_t1);
    prefetch_tmap(&p.tm_t2);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), P::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Waiter W{abort_flag, p.err, p.timeout_ns};
  auto unit_at = [&](int rnd) { return unit_of_round(rnd); };
  // The units this launch walks: a jagged work list when one was written
  // (by the planning kernel earlier on the stream), else the slot order;
  // read from the parameters at each unit, so the dense kernels' loops
  // carry nothing for it.
  auto units_end = [&]() -> int {
    if (p.unit_list != nullptr) {
      const int c = __ldg(p.unit_count);
      if (c >= 0) return c * p.H;
    }
    return p.num_units;
  };

  if (warp < 4) {
    setmaxnreg_dec<kLowRegs>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        uint32_t rfill = 0, tfill = 0;
        bool ok = true;
        for (int rnd = 0; ok; ++rnd) {
          const int u = unit_at(rnd);
          if (u >= units_end()) break;
          const BwdUnit w = bwd_unit<KV>(p, u);
          if (w.nt == 0) continue;
          ok = wait_bar(bar(P::B_RE), (rfill & 1u) ^ 1u, W);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(P::B_RF), P::RSET);
          const int r = w.row0 + w.rt * kBM;
#pragma unroll
          for (int c = 0; c < DQK / 64; ++c)
            tma_load_3d(sbase + P::OFF_R + c * P::R_SUB, &p.tm_r1, bar(P::B_RF), c * 64, r, w.z);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c)
            tma_load_3d(sbase + P::OFF_R + P::R1_TILE + c * P::R_SUB, &p.tm_r2, bar(P::B_RF), c * 64, r,
                        w.z);
          ++rfill;
          for (int j = 0; j < w.nt; ++j) {
            const int tr = w.row0 + (w.t0 + j) * P::TN;
            const uint32_t ts = tfill % P::NS;
            ok = wait_bar(bar(P::B_TE + ts), ((tfill / P::NS) & 1u) ^ 1u, W);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(P::B_TF + ts), P::T_STAGE);
            const uint32_t dst = sbase + P::OFF_T + ts * P::T_STAGE;
#pragma unroll
            for (int c = 0; c < DQK / 64; ++c)
              tma_load_3d(dst + c * P::T_SUB, &p.tm_t1, bar(P::B_TF + ts), c * 64, tr, w.z);
#pragma unroll
            for (int c = 0; c < DV / 64; ++c)
              tma_load_3d(dst + P::T1_TILE + c * P::T_SUB, &p.tm_t2, bar(P::B_TF + ts), c * 64, tr, w.z);
            ++tfill;
          }
        }
        for (uint32_t s = 0; s < P::NS && s < tfill; ++s) {
          const uint32_t nf = (tfill - s + P::NS - 1) / P::NS;
          drain_bar(bar(P::B_TF + s), (nf - 1) & 1u, p.timeout_ns);
        }
        if (rfill > 0) drain_bar(bar(P::B_RF), (rfill - 1) & 1u, p.timeout_ns);
      }
      __syncwarp();
    } else if (warp == 1 || warp == 3) {
      // ------------------------------------------------------- MMA issuers
      // Two issuing warps on different sub-partitions: warp 1 the score
      // chains, warp 3 the output chains.  An issuing warp's waits, commits
      // and fences queue behind its own MMAs, so a single issuer stalls at
      // every wait while the tensor pipe drains; with two, each one's waits
      // overlap the other's MMAs.  Ordering between them runs through
      // barriers completed by tcgen05.commit of the warp whose MMAs must
      // finish first: s_full (scores of tile g ready) -> elementwise ->
      // p_full -> output chain of g -> o_done (its score buffer may be
      // overwritten) -> score chains of tile g + NSB.  Each wait is gated by
      // a phase the waiter itself enables, so no parity wait can alias.
      const bool leader = elect_one();
      constexpr uint32_t idesc_s = idesc_16(kBM, P::TN, false, F16);  // score chains, N = 64
      constexpr uint32_t idesc_k = idesc_16(kBM, DQK, true, F16);     // dQ / dK chains, N = Dqk
      constexpr uint32_t idesc_v = idesc_16(kBM, DV, true, F16);      // dV chain, N = Dv
      auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, wait_bar(b, parity, W));
      };
      // Descriptor low words (the issue loop is instruction-bound: a score
      // MMA lasts ~48 cycles, so each MMA gets one 32-bit add per operand):
      // row operands and ring stage 0, K-major; ring stage 0 MN-major (the
      // output chains' B, 64-column chunks T_SUB apart).
      constexpr uint32_t kHi = sdesc_hi_sw128(1024);
      const uint32_t lo_r1 = sdesc_lo(sbase + P::OFF_R, 16);
      const uint32_t lo_r2 = lo_r1 + (P::R1_TILE >> 4);
      const uint32_t lo_t = sdesc_lo(sbase + P::OFF_T, 16);
      const uint32_t lo_tmn = sdesc_lo(sbase + P::OFF_T, P::T_SUB);
      bool ok = true;
      uint32_t g = 0;  // tile counter over units with tiles (same in every role)
      if (warp == 1) {
        uint32_t ruse = 0;
        for (int rnd = 0; ok; ++rnd) {
          const int u = unit_at(rnd);
          if (u >= units_end()) break;
          const BwdUnit w = bwd_unit<KV>(p, u);
          if (w.nt == 0) continue;
          ok = wait_all(bar(P::B_RF), ruse & 1u);
          if (!ok) break;
          for (int j = 0; j < w.nt; ++j, ++g) {
            const uint32_t ts = g % P::NS, sb = g % P::NSB;
            // the tile's operands, and the output chain that last read this
            // score buffer (tile g - NSB; a fresh barrier passes)
            ok = wait_all(bar(P::B_TF + ts), (g / P::NS) & 1u) &&
                 wait_all(bar(P::B_OD + sb), ((g / P::NSB) & 1u) ^ 1u);
            if (!ok) break;
            tc_fence_after();
            const uint32_t lt = lo_t + ts * (P::T_STAGE >> 4);
            const uint32_t dX = tmem + sb * P::SBUF;
            // both chains from the elected lane in one pass (the rest of the
            // warp waits at the commit's warp sync)
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < DQK / 16; ++kk) {
                const uint32_t oa = ((kk >> 2) * P::R_SUB + (kk & 3) * 32) >> 4;
                const uint32_t ob = ((kk >> 2) * P::T_SUB + (kk & 3) * 32) >> 4;
                mma_ss(dX, sdesc_join(lo_r1 + oa, kHi), sdesc_join(lt + ob, kHi), idesc_s, kk > 0 ? 1u : 0u);
              }
#pragma unroll
              for (int kk = 0; kk < DV / 16; ++kk) {
                const uint32_t oa = ((kk >> 2) * P::R_SUB + (kk & 3) * 32) >> 4;
                const uint32_t ob = (P::T1_TILE + (kk >> 2) * P::T_SUB + (kk & 3) * 32) >> 4;
                mma_ss(dX + P::TN, sdesc_join(lo_r2 + oa, kHi), sdesc_join(lt + ob, kHi), idesc_s, kk > 0 ? 1u : 0u);
              }
              tc_commit(bar(P::B_SF + sb));
              // the unit's last score chain: the row operands are free once
              // it is done (the output chains never read them)
              if (j == w.nt - 1) tc_commit(bar(P::B_RE));
            }
            __syncwarp();
          }
          ++ruse;
        }
        if (leader) {
          tc_commit(bar(P::B_DRAIN));
          drain_bar(bar(P::B_DRAIN), 0, p.timeout_ns);
        }
      } else {
        for (int rnd = 0; ok; ++rnd) {
          const int u = unit_at(rnd);
          if (u >= units_end()) break;
          const BwdUnit w = bwd_unit<KV>(p, u);
          if (w.nt == 0) continue;
          for (int j = 0; j < w.nt; ++j, ++g) {
            const uint32_t sb = g % P::NSB, ts = g % P::NS;
            ok = wait_all(bar(P::B_PF + sb), (g / P::NSB) & 1u);
            if (!ok) break;
            tc_fence_after();
            const bool first = j == 0;  // zero-initialises the accumulators
            const uint32_t lm = lo_tmn + ts * (P::T_STAGE >> 4);
            // 16-bit operands over the Y columns: half h at Y + 32 h holds
            // P^T (KV pass) at +0 and dS at +16 (KV) / +0 (dQ pass), 8
            // packed columns per 16 streamed rows
            const uint32_t aY = tmem + sb * P::SBUF + P::TN;
            // dQ += dS K   /   dK += dS^T Q
            const uint32_t acc = tmem + P::COL_A + (KV ? DV : 0);
            const uint32_t ds_off = KV ? 16u : 0u;
            if (leader) {
              if (KV) {
                // dV += P^T dO
#pragma unroll
                for (int kk = 0; kk < P::TN / 16; ++kk) {
                  const uint64_t db = sdesc_join(lm + ((P::T1_TILE + kk * 2048) >> 4), kHi);
                  mma_ts(tmem + P::COL_A, aY + 32 * (kk >> 1) + 8 * (kk & 1), db, idesc_v,
                         (first && kk == 0) ? 0u : 1u);
                }
              }
#pragma unroll
              for (int kk = 0; kk < P::TN / 16; ++kk) {
                const uint64_t db = sdesc_join(lm + ((kk * 2048) >> 4), kHi);
                mma_ts(acc, aY + 32 * (kk >> 1) + ds_off + 8 * (kk & 1), db, idesc_k,
                       (first && kk == 0) ? 0u : 1u);
              }
              tc_commit(bar(P::B_TE + ts));  // stage free (the tile's score chains finished first)
              tc_commit(bar(P::B_OD + sb));  // score buffer free
            }
            __syncwarp();
          }
        }
        if (leader) {
          tc_commit(bar(P::B_DRAIN2));
          drain_bar(bar(P::B_DRAIN2), 0, p.timeout_ns);
        }
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<kHighRegs>();
    // ---------------------------------------------- elementwise / epilogue
    const int quad = warp & 3;
    const int half = (warp - 4) >> 2;
    const int row = quad * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    constexpr float kLog2eF = 1.4426950408889634f;
    // KV pass: this warp's 64-float slot of column terms
    float* colv = reinterpret_cast<float*>(smem + P::OFF_COLV) + (KV ? (warp - 4) * 64 : 0);
    uint32_t g = 0, tuse = 0;
    bool ok = true;
    for (int rnd = 0; ok; ++rnd) {
      const int u = unit_at(rnd);
      if (u >= units_end()) break;
      const BwdUnit w = bwd_unit<KV>(p, u);
      const int ri = w.rt * kBM + row;  // this thread's row (query for dQ, key for KV)
      const bool row_ok = ri < w.rows;
      if (w.nt == 0) {
        // no streamed tile touches these rows: zero gradients
        if (row_ok) {
          // this half's columns of each output row (a multiple of 8 each)
          auto zero_row = [&](uint16_t* out, int width, int d_real) {
            const int ncol = min(width / 2, d_real - half * (width / 2));
            const long long off = (w.orow0 + ri) * d_real + half * (width / 2);
            for (int c = 0; c < ncol; c += 8)
              *reinterpret_cast<uint4*>(out + off + c) = make_uint4(0u, 0u, 0u, 0u);
          };
          zero_row(p.out1, DQK, p.d_qk);
          if (KV) zero_row(p.out2, DV, p.d_v);
        }
        continue;
      }
      // Per-row (dQ pass) or per-column (KV pass) terms of the exponent and
      // of dS, pre-negated: nl = -LSE log2(e) and nd = -Delta, with
      // nl = -inf for empty rows and padding rows / columns so that their P
      // is exactly 0 without a test.
      const int q_len = KV ? w.cols : w.rows;
      auto neg_terms = [&](int i, float& nl, float& nd) {
        nl = -INFINITY;
        nd = 0.f;
        if (i < q_len) {
          const float l = __ldg(p.lse + w.qrow0 + i);
          nl = l == -INFINITY ? -INFINITY : -l * kLog2eF;
          nd = -__ldg(p.delta + w.qrow0 + i);
        }
      };
      float nl_r = -INFINITY, nd_r = 0.f;   // dQ pass: this row's terms
      float nl_c = -INFINITY, nd_c = 0.f;   // KV pass: this lane's column of the next tile
      if (!KV) neg_terms(ri, nl_r, nd_r);
      else neg_terms((w.t0) * 64 + half * 32 + lane, nl_c, nd_c);
      const uint64_t sc2 = f2_make(p.scale_log2, p.scale_log2);
      const bool has_bias = BM && p.bias != nullptr, has_mask = BM && p.mask != nullptr;
      // this thread's row of the bias / mask: a query row (dQ pass, keys
      // along it) or a key column (KV pass, queries along it)
      const float* bbase = nullptr;
      const unsigned char* mbase = nullptr;
      long long bstep = 0, mstep = 0;  // element step along the streamed dimension
      if (has_bias) {
        bbase = p.bias + w.b * p.bias_stride[0] + w.h * p.bias_stride[1] +
                static_cast<long long>(ri) * p.bias_stride[KV ? 3 : 2];
        bstep = p.bias_stride[KV ? 2 : 3];
      }
      if (has_mask) {
        mbase = p.mask + w.b * p.mask_stride[0] + w.h * p.mask_stride[1] +
                static_cast<long long>(ri) * p.mask_stride[KV ? 3 : 2];
        mstep = p.mask_stride[KV ? 2 : 3];
      }
      for (int j = 0; j < w.nt; ++j, ++g, ++tuse) {
        const uint32_t sb = g % P::NSB;
        const int col0 = (w.t0 + j) * 64 + half * 32;  // first column (key or query) of this thread
        if (KV) {
          // publish this tile's column terms to the warp's slot, then fetch
          // the next tile's (their latency hides behind this tile)
          __syncwarp();
          colv[lane] = nl_c;
          colv[32 + lane] = nd_c;
          __syncwarp();
          if (j + 1 < w.nt) neg_terms(col0 + 64 + lane, nl_c, nd_c);
        }
        // valid columns [lo, hi) of this thread's 32 (the others get P = 0):
        // dQ pass keys < N and, causal, <= the query; KV pass, causal,
        // queries >= the key (queries >= M already have nl = -inf)
        int lo = 0, hi = 32;
        if (!KV) hi = (p.causal ? min(w.cols, ri + 1) : w.cols) - col0;
        else if (p.causal) lo = ri - col0;
        // keep bit c: column col0 + c in [lo, hi) and, with a mask, attended
        uint32_t keep = 0xffffffffu;
        if (lo > 0) keep = lo >= 32 ? 0u : keep << lo;
        if (hi < 32) keep &= hi <= 0 ? 0u : (1u << hi) - 1u;
        // bias values of this thread's 32 columns (log2 units; 0 past the
        // valid columns), loaded before the scores are waited for
        float bl[BM ? 32 : 1];
        if constexpr (BM) {
        if (has_bias) {
#pragma unroll
          for (int c = 0; c < 32; ++c) bl[c] = 0.f;
          if (row_ok) {
            const float* bp = bbase + static_cast<long long>(col0) * bstep;
            if (bstep == 1 && (reinterpret_cast<uintptr_t>(bp) & 15u) == 0 && col0 + 32 <= w.cols) {
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const float4 t4 = __ldg(reinterpret_cast<const float4*>(bp) + c);
                bl[4 * c] = t4.x * kLog2eF;
                bl[4 * c + 1] = t4.y * kLog2eF;
                bl[4 * c + 2] = t4.z * kLog2eF;
                bl[4 * c + 3] = t4.w * kLog2eF;
              }
            } else {
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (col0 + c < w.cols) bl[c] = __ldg(bp + c * bstep) * kLog2eF;
            }
          }
        }
        }
        if (has_mask && row_ok) {
          const unsigned char* mp = mbase + static_cast<long long>(col0) * mstep;
          uint32_t mb = 0u;
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (col0 + c < w.cols && __ldg(mp + c * mstep) != 0) mb |= 1u << c;
          keep &= mb;
        }
        const bool full = keep == 0xffffffffu;
        // a sleeping wait: a spinning one would take issue slots from the
        // MMA issuer on the same sub-partition
        ok = __all_sync(0xffffffffu, wait_bar_sleep(bar(P::B_SF + sb), (g / P::NSB) & 1u, W));
        if (!ok) break;
        tc_fence_after();
        uint32_t xr[32], yr[32];
        tmem_ld_32x32b_x32(tl + sb * P::SBUF + half * 32, xr);
        tmem_ld_32x32b_x32(tl + sb * P::SBUF + P::TN + half * 32, yr);
        tmem_wait_ld_regs(xr);
        tmem_regs_ready(yr);
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          float4 nl4, nd4;
          if (KV) {
            nl4 = *reinterpret_cast<const float4*>(colv + c);
            nd4 = *reinterpret_cast<const float4*>(colv + 32 + c);
          } else {
            nl4 = make_float4(nl_r, nl_r, nl_r, nl_r);
            nd4 = make_float4(nd_r, nd_r, nd_r, nd_r);
          }
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int cc = c + e;
            const float nla = e == 0 ? nl4.x : nl4.z, nlb = e == 0 ? nl4.y : nl4.w;
            const float nda = e == 0 ? nd4.x : nd4.z, ndb = e == 0 ? nd4.y : nd4.w;
            // x = S s log2(e) - LSE log2(e);  P = 2^x;  dS = P (dP - Delta)
            uint64_t x = f2_fma(f2_make(__uint_as_float(xr[cc]), __uint_as_float(xr[cc + 1])), sc2,
                                f2_make(nla, nlb));
            if constexpr (BM) {
              if (has_bias) x = f2_add(x, f2_make(bl[cc], bl[cc + 1]));
            }
            float x0, x1;
            f2_split(x, x0, x1);
            float p0 = ex2(x0), p1 = ex2(x1);
            if (!full) {
              p0 = ((keep >> cc) & 1u) ? p0 : 0.f;
              p1 = ((keep >> (cc + 1)) & 1u) ? p1 : 0.f;
            }
            const uint64_t d = f2_add(f2_make(__uint_as_float(yr[cc]), __uint_as_float(yr[cc + 1])),
                                      f2_make(nda, ndb));
            float d0, d1;
            f2_split(f2_mul(f2_make(p0, p1), d), d0, d1);
            pk[cc / 2] = pack2<F16>(p0, p1);
            dk[cc / 2] = pack2<F16>(d0, d1);
          }
        }
        const uint32_t yb = tl + sb * P::SBUF + P::TN + half * 32;
        if (KV) {
          tmem_st_32x32b_x16(yb, pk);
          tmem_st_32x32b_x16(yb + 16, dk);
        } else {
          tmem_st_32x32b_x16(yb, dk);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(P::B_PF + sb));
      }
      if (!ok) break;
      // ------------------------------------------------------------ epilogue
      // every MMA of the unit is done once the last tile's output MMAs are
      // (their commit is the last tile's ring-stage release; the phase after
      // it needs a tile this thread has not processed yet)
      const uint32_t tl_last = tuse - 1;
      ok = __all_sync(0xffffffffu, wait_bar_sleep(bar(P::B_TE + tl_last % P::NS), (tl_last / P::NS) & 1u, W));
      if (!ok) break;
      tc_fence_after();
      const int q = lane & 3;
      // one accumulator of W columns: scale, round, transpose across lane
      // quads, store whole row segments
      auto store_acc = [&](auto width, uint32_t colA, float f, uint16_t* out, int d_real) {
        constexpr int W = decltype(width)::value;
        constexpr int DH = W / 2;   // columns per thread
        constexpr int NW = DH / 2;  // packed words
        constexpr int CW = NW / 4;
        uint32_t pw[NW];
#pragma unroll
        for (int c0 = 0; c0 < DH; c0 += 32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tl + colA + half * DH + c0, v);
          tmem_wait_ld_regs(v);
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            pw[c0 / 2 + i / 2] = pack2<F16>(__uint_as_float(v[i]) * f, __uint_as_float(v[i + 1]) * f);
        }
        quad_transpose<CW>(pw, q);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int rk = w.rt * kBM + quad * 32 + (lane & ~3) + k;
          const int col = half * DH + q * 2 * CW;
          if (rk < w.rows && col < d_real) {
            const long long off = (w.orow0 + rk) * d_real + col;
            store_chunk<CW>(out + off, pw + k * CW, false);
          }
        }
      };
      if (KV) {
        // dV (unscaled) then dK (scaled by s)
        store_acc(std::integral_constant<int, DV>{}, P::COL_A, 1.f, p.out2, p.d_v);
        store_acc(std::integral_constant<int, DQK>{}, P::COL_A + DV, p.sm_scale, p.out1, p.d_qk);
      } else {
        store_acc(std::integral_constant<int, DQK>{}, P::COL_A, p.sm_scale, p.out1, p.d_qk);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, P::TMEM_COLS);
}

template <int DQK, int DV, bool KV, bool F16, bool BM>
cudaError_t launch_attn_bwd(const BwdParams& bp, int grid, cudaStream_t stream) {
  using P = BwdPlan<DQK, DV, KV>;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_done[dev]) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, attn_bwd_kernel<DQK, DV, KV, F16, BM>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kLaunchRegs || fa.maxThreadsPerBlock < kThreads) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(attn_bwd_kernel<DQK, DV, KV, F16, BM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             P::SMEM_LAUNCH);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  attn_bwd_kernel<DQK, DV, KV, F16, BM><<<grid, kThreads, P::SMEM_LAUNCH, stream>>>(bp);
  return cudaGetLastError();
}

// Delta = rowsum(dO o O) over [rows, d], fp32 sums.  A warp takes four rows
// at a time, each lane d / 32 consecutive elements of each (one 8-, 4- or
// 2-byte load per row and operand), so eight loads are in flight per lane
// before the first reduction; d = 16 leaves half the lanes idle.
template <bool F16>
__device__ __forceinline__ float dot2(uint32_t a, uint32_t b) {
  float a0, a1, b0, b1;
  if constexpr (F16) {
    a0 = __half2float(__ushort_as_half(static_cast<uint16_t>(a & 0xffffu)));
    a1 = __half2float(__ushort_as_half(static_cast<uint16_t>(a >> 16)));
    b0 = __half2float(__ushort_as_half(static_cast<uint16_t>(b & 0xffffu)));
    b1 = __half2float(__ushort_as_half(static_cast<uint16_t>(b >> 16)));
  } else {
    a0 = __uint_as_float(a << 16);
    a1 = __uint_as_float(a & 0xffff0000u);
    b0 = __uint_as_float(b << 16);
    b1 = __uint_as_float(b & 0xffff0000u);
  }
  return fmaf(a1, b1, a0 * b0);
}

template <bool F16>
__global__ void attn_bwd_delta_kernel(const uint16_t* o, const uint16_t* dout, float* delta,
                                      long long rows, int d) {
  const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int per = d >> 5;  // elements per lane: 4, 2, 1 (d = 128, 64, 32); 0 for d = 16
  for (long long r0 = wid * 4; r0 < rows; r0 += nw * 4) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const long long r = r0 + k;
      if (r >= rows) break;
      const long long base = r * d;
      if (per == 4) {
        const uint2 a = *reinterpret_cast<const uint2*>(o + base + lane * 4);
        const uint2 b = *reinterpret_cast<const uint2*>(dout + base + lane * 4);
        acc[k] = dot2<F16>(a.x, b.x) + dot2<F16>(a.y, b.y);
      } else if (per == 2) {
        acc[k] = dot2<F16>(*reinterpret_cast<const uint32_t*>(o + base + lane * 2),
                           *reinterpret_cast<const uint32_t*>(dout + base + lane * 2));
      } else {
        for (int c = lane; c < d; c += 32) {
          const uint32_t a = o[base + c], b = dout[base + c];
          acc[k] = fmaf(F16 ? __half2float(__ushort_as_half(static_cast<uint16_t>(a))) : __uint_as_float(a << 16),
                        F16 ? __half2float(__ushort_as_half(static_cast<uint16_t>(b))) : __uint_as_float(b << 16),
                        acc[k]);
        }
      }
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], s);
    if (lane < 4 && r0 + lane < rows) {
      float v = acc[0];
#pragma unroll
      for (int k = 1; k < 4; ++k)
        if (lane == k) v = acc[k];
      delta[r0 + lane] = v;
    }
  }
}

}  // namespace attn
