// fa_bwd_main.cuh -- the backward main pass of head dims 64 and 128 (sm_103a): its
// shared-memory and TMEM layout, the kernel, and its launchers. Included by fa_bwd.cu (default
// layout) and fa_bwd_strided.cu (bshd layouts), so that the two sets of instantiations compile
// in parallel. The method is described at the top of fa_bwd.cu.
#pragma once
#include <float.h>

#include "fa_bwd_common.cuh"
#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {

// HD: head dim of Q, K (and dQ, dK); DV: head dim of V, O, dO (and dV).
template <int HD, int DV>
struct BwdLayout {
  using T = BwdTraits<HD>;
  static constexpr int BM = T::BM;
  static constexpr int DH = HD / T::DSPLIT;   // head-dim slice of dK this CTA produces
  static constexpr int DVH = DV / T::DSPLIT;  // ... of dV
  static constexpr int KCH = HD / 64;
  static constexpr int VCH = DV / 64;
  static constexpr int K_BYTES = kBN * HD * 2;
  static constexpr int V_BYTES = kBN * DV * 2;
  static constexpr int QT_BYTES = BM * HD * 2;
  static constexpr int DOT_BYTES = BM * DV * 2;
  static constexpr int DS_BYTES = kBN * BM * 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + K_BYTES;
  static constexpr int OFF_Q = OFF_V + V_BYTES;                 // ST x Q tile
  static constexpr int OFF_DO = OFF_Q + T::ST * QT_BYTES;       // ST x dO tile
  static constexpr int OFF_DS = OFF_DO + T::ST * DOT_BYTES;     // 2 x dS^T [kv][q] swizzled
  static constexpr int OFF_L = OFF_DS + 2 * DS_BYTES;           // ST x BM f32
  static constexpr int OFF_D = OFF_L + T::ST * BM * 4;          // ST x BM f32
  static constexpr int OFF_STG = OFF_D + T::ST * BM * 4;            // dQ staging [BM][HD] f32
  static constexpr int STG_BYTES = T::DQ_BULK ? BM * HD * 4 : 0;
  static constexpr int OFF_END = OFF_STG + STG_BYTES;
  static constexpr int SMEM_BYTES = OFF_END + 1024;
  // TMEM columns: S^T buffers, dP^T buffers (also holding dQ), dV, dK
  static constexpr int COL_S0 = 0;
  static constexpr int COL_DP0 = T::NSB * BM;
  static constexpr int COL_DV = (T::NSB + 2) * BM;
  static constexpr int COL_DK = COL_DV + DVH;
  static constexpr int TMEM_USED = COL_DK + DH;
  static constexpr int TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
  static constexpr int DQ_COLS = T::DQT ? BM : HD;
  // WG0 (warps 0-3): P^T; WG1 (warps 4-7): dS^T and the dK/dV epilogue; WG2 (warps 8-11):
  // the dQ drain; warp 12: TMA; warp 13: MMA (with SPLIT_MMA: S^T and dP^T only); warp 14:
  // issues the bulk dQ reductions; warp 15 (SPLIT_MMA): the dV, dK and dQ MMAs.
  static constexpr int THREADS = 512;
  static constexpr int TMA_WARP = 12, MMA_WARP = 13, BULK_WARP = 14, MMA2_WARP = 15;
  static_assert(TMEM_USED <= 512, "TMEM budget");
  static_assert(DQ_COLS <= BM, "dQ tile must fit in a dP^T buffer");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(T::DQT ? DH == 128 : BM == 128, "every MMA has M = 128");
  static_assert(T::LOOKAHEAD ? T::ST >= (T::NSB == 2 ? 3 : 2) : true, "ring too shallow");
  static_assert(!T::SPLIT_MMA || (T::NSB == 2 && T::LOOKAHEAD), "split issue order");
  static_assert(T::DQ_BULK && T::DSPLIT == 1, "the dQ drain stages whole head-dim rows");
  static_assert(!T::DQ_BULK || (T::DQT ? BM : HD) / 4 == kDqChunks, "staged dQ tile layout");
  static_assert(T::DSPLIT == 1 || DV == HD, "a split head dim needs DV == HD");
  static_assert(DVH % 16 == 0 && DVH >= 16 && DVH <= 256, "dV MMA N");
};

// ------------------------------------------------------------------------ main kernel
// STRIDED: instantiated for calls with a bshd layout only, so that the default-layout kernels
// carry no code for it (with the layout tested at run time instead, the head_dim-128 main pass
// measured 651 -> 669 us on the 4k GQA shape).
template <int HD, int DV, int BAND, int MASKT, bool VARLEN, bool STRIDED>
__global__ void __launch_bounds__(BwdLayout<HD, DV>::THREADS, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                    const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mDO,
                    const BwdKParams p) {
  using T = BwdTraits<HD>;
  const bool q_bshd = STRIDED && p.q_bshd != 0, kv_bshd = STRIDED && p.kv_bshd != 0;
  using LY = BwdLayout<HD, DV>;
  constexpr int BM = T::BM, DH = LY::DH, KCH = LY::KCH, ST = T::ST, NSB = T::NSB;
  constexpr int DVH = LY::DVH, VCH = LY::VCH;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ uint64_t kv_full, qdo_full[ST], qdo_empty[ST];
  __shared__ uint64_t s_full[NSB], p_ready[NSB], p_consumed[NSB];
  __shared__ uint64_t dp_full[2], ds_ready[2], dq_full[2], dq_free[2];
  __shared__ uint64_t acc_full, mma_drain, mma_drain2;
  __shared__ uint64_t dv_done[NSB];  // SPLIT_MMA: dV(it) has read P^T(it) from its S^T buffer
  __shared__ uint64_t stg_full, stg_free;  // dQ staging handshake of the bulk drain
  __shared__ uint32_t tmem_base_s;
  __shared__ WaitCtl wctl;

  const int warp = warp_id(), lane = lane_id();
  // Launch order, heaviest (causal) kv tile first either way. Fixed length: tile-major, so
  // that every group's heaviest tile starts in the first wave and the light ones fill the
  // tail. Variable-length batch: the kv tiles of one (sequence, kv head) next to each other,
  // so that the Q / dO tiles they all walk stay in L2 (measured: 7.6 -> 5.0 ms on a mix of
  // 16 sequences, where tile-major order read ~48 GB from HBM per launch).
  const int gidx = p.tiles_fast ? (int)blockIdx.y : (int)blockIdx.x;
  const int dh = gidx % T::DSPLIT;
  const int bkh = gidx / T::DSPLIT;  // b * Hk + kh
  const int b = bkh / p.Hk, kh = bkh % p.Hk;
  const int G = p.H / p.Hk;
  const int n0 = (int)(p.tiles_fast ? blockIdx.x : blockIdx.y) * kBN;
  // the rows of this problem: one (batch, kv head) of fixed length, or in a variable-length
  // batch sequence b's own rows of the packed heads (tensor-map z = head, rows offset)
  int ql = p.ql, kl = p.kl;
  int krow0 = 0, qrow0 = 0;
  int kb = b, krows = p.kl;  // dK / dV: batch and rows of this problem (row of key 0: krow0)
  // (kb is also the batch coordinate of the tile loads: 0 in a packed batch)
  if constexpr (VARLEN) {
    int qs, ks;
    const bool bad = varlen_seq(p.cu_q, b, p.total_q, p.ql, qs, ql) |
                     varlen_seq(p.cu_k, b, p.total_k, p.kl, ks, kl);
    if (bad && threadIdx.x == 0 && p.status) atomicCAS(p.status, kStatusOk, kStatusBadInput);
    krow0 = ks;
    qrow0 = qs;
    kb = 0;
    krows = p.total_k;
  }
  if (n0 >= kl) return;  // a kv tile past this sequence's keys (the whole CTA leaves)
  int m_first, m_last;
  constexpr bool WIN = BAND == kBandWindow;
  bwd_mtile_range<HD, BAND>(n0, p, ql, kl, m_first, m_last);
  const int nm = m_last - m_first + 1;  // query tiles per head (0 if none)
  const int n_iter = G * nm;          // (head, query tile) pairs this CTA visits
  const bool split_mma = T::SPLIT_MMA && p.skip_dq;  // two MMA issuers (see BwdTraits)

  if (threadIdx.x == 0) {
    wait_ctl_init(&wctl, p.wait_limit_ns);
    mbar_init(&kv_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&qdo_full[s], 1);
      mbar_init(&qdo_empty[s], 1);
    }
    for (int s = 0; s < NSB; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_ready[s], 128);
      mbar_init(&p_consumed[s], 128);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&dp_full[s], 1);
      mbar_init(&ds_ready[s], 128);
      mbar_init(&dq_full[s], 1);
      mbar_init(&dq_free[s], 128);
    }
    mbar_init(&acc_full, 1);
    mbar_init(&mma_drain, 1);
    mbar_init(&mma_drain2, 1);
    for (int s = 0; s < NSB; ++s) mbar_init(&dv_done[s], 1);
    mbar_init(&stg_full, 128);
    mbar_init(&stg_free, 1);
    fence_barrier_init();
  }
  if (warp == LY::MMA_WARP) {
    tmem_alloc(&tmem_base_s, LY::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_s;
  // the prologue above overlaps the pre-pass's tail; L, D and the zeroed accumulator are its
  // output
  grid_dep_wait();
  grid_dep_trigger();

  if (warp == LY::TMA_WARP) {
    // ------------------------------------------------------------------ TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mV);
      tma_prefetch_desc(&mDO);
      int last_use[ST];
      for (int s = 0; s < ST; ++s) last_use[s] = -1;
      mbar_arrive_expect_tx(&kv_full, LY::K_BYTES + LY::V_BYTES);
      for (int c = 0; c < KCH; ++c)
        tma_load_bh(smem + LY::OFF_K + c * kBN * 128, &mK, &kv_full, c * 64, krow0 + n0, kh, kb,
                    p.Hk, kv_bshd);
      for (int c = 0; c < VCH; ++c)
        tma_load_bh(smem + LY::OFF_V + c * kBN * 128, &mV, &kv_full, c * 64, krow0 + n0, kh, kb,
                    p.Hk, kv_bshd);
      for (int it = 0; it < n_iter; ++it) {
        const int st = it % ST;
        const uint32_t use = it / ST;
        if (it >= ST && !mbar_wait(&qdo_empty[st], (use - 1) & 1, &wctl)) break;
        const int h = kh * G + it / nm;
        const int q0 = (m_first + it % nm) * BM;
        const int bh = b * p.H + h;
        mbar_arrive_expect_tx(&qdo_full[st], LY::QT_BYTES + LY::DOT_BYTES + 2 * BM * 4);
        for (int c = 0; c < KCH; ++c)
          tma_load_bh(smem + LY::OFF_Q + st * LY::QT_BYTES + c * BM * 128, &mQ, &qdo_full[st],
                      c * 64, qrow0 + q0, h, kb, p.H, q_bshd);
        for (int c = 0; c < VCH; ++c)
          tma_load_bh(smem + LY::OFF_DO + st * LY::DOT_BYTES + c * BM * 128, &mDO,
                      &qdo_full[st], c * 64, qrow0 + q0, h, kb, p.H, q_bshd);
        bulk_load(smem + LY::OFF_L + st * BM * 4, p.lse2 + (size_t)bh * p.ql_pad + q0, BM * 4,
                  &qdo_full[st]);
        bulk_load(smem + LY::OFF_D + st * BM * 4, p.dvec + (size_t)bh * p.ql_pad + q0, BM * 4,
                  &qdo_full[st]);
        last_use[st] = it;
      }
      mbar_wait_drain(&kv_full, 0);
      for (int s = 0; s < ST; ++s)
        if (last_use[s] >= 0) mbar_wait_drain(&qdo_full[s], (last_use[s] / ST) & 1);
    }
  } else if (split_mma && (warp == LY::MMA_WARP || warp == LY::MMA2_WARP)) {
    // ------------------------------------------------------------------ MMA issuers (split)
    // Warp 13 issues S^T(it) and dP^T(it); warp 15 issues dV(it), dK(it) and dQ(it). Each
    // stream keeps the order the single issuer had, and the one hazard between them that the
    // issue order used to cover (S^T(it) overwriting the score buffer that dV(it - NSB) reads
    // P^T from) is covered by the dv_done barrier.
    if constexpr (T::SPLIT_MMA) {
      if (elect_one()) {
        const uint32_t sK = smem_u32(smem + LY::OFF_K), sV = smem_u32(smem + LY::OFF_V);
        const Desc kd = make_desc(sK, 16, 1024);          // K as a K-major operand
        const Desc vd = make_desc(sV, 16, 1024);          // V as a K-major operand
        const Desc kmn = make_desc(sK, kBN * 128, 1024);  // K as an MN-major operand
        const uint32_t id_s = idesc_bf16(128, BM, 0, 0);      // S^T, dP^T: [kv x q]
        const uint32_t id_dv = idesc_bf16(128, DVH, 0, 1);    // dV: A tmem, B MN-major
        const uint32_t id_dk = idesc_bf16(128, DH, 0, 1);     // dK: A tmem, B MN-major
        const uint32_t id_dq = idesc_bf16(DH, BM, 1, 1);      // dQ^T: [d x q]
        const uint32_t tDV = tbase + LY::COL_DV, tDK = tbase + LY::COL_DK;
        const uint32_t slice = (dh * DH / 64) * (BM * 128);
        const uint32_t vslice = (dh * DVH / 64) * (BM * 128);
        bool ok = mbar_wait(&kv_full, 0, &wctl);
        if (warp == LY::MMA_WARP) {
          for (int it = 0; it < n_iter && ok; ++it) {
            const int st = it % ST;
            ok = mbar_wait(&qdo_full[st], (it / ST) & 1, &wctl);
            // S^T(it) = K Q^T, into the score buffer of it - NSB once WG1 and dV(it - NSB) have
            // read P^T(it - NSB) from it
            if (ok && it >= NSB) {
              ok = mbar_wait(&p_consumed[it % NSB], ((it - NSB) / NSB) & 1, &wctl);
              if (ok) ok = mbar_wait(&dv_done[it % NSB], ((it - NSB) / NSB) & 1, &wctl);
            }
            if (!ok) break;
            tc_fence_after();
            const Desc qd = make_desc(smem_u32(smem + LY::OFF_Q + st * LY::QT_BYTES), 16, 1024);
            const uint32_t tS = tbase + LY::COL_S0 + (it % NSB) * BM;
#pragma unroll
            for (int ks = 0; ks < HD / 16; ++ks) {
              const uint32_t ko = (ks / 4) * (kBN * 128) + (ks % 4) * 32;
              const uint32_t qo = (ks / 4) * (BM * 128) + (ks % 4) * 32;
              mma_ss2(tS, kd.at(ko), kd.hi, qd.at(qo), qd.hi, id_s, ks > 0 ? 1u : 0u);
            }
            mma_commit(&s_full[it % NSB]);
            // dP^T(it) = V dO^T, into the buffer that dQ(it - 2) used, once WG2 has drained it
            if (it >= 2) {
              ok = mbar_wait(&dq_free[it % 2], ((it - 2) / 2) & 1, &wctl);
              if (!ok) break;
              tc_fence_after();
            }
            const Desc dod = make_desc(smem_u32(smem + LY::OFF_DO + st * LY::DOT_BYTES), 16, 1024);
            const uint32_t tDP = tbase + LY::COL_DP0 + (it % 2) * BM;
#pragma unroll
            for (int ks = 0; ks < DV / 16; ++ks) {
              const uint32_t ko = (ks / 4) * (kBN * 128) + (ks % 4) * 32;
              const uint32_t qo = (ks / 4) * (BM * 128) + (ks % 4) * 32;
              mma_ss2(tDP, vd.at(ko), vd.hi, dod.at(qo), dod.hi, id_s, ks > 0 ? 1u : 0u);
            }
            mma_commit(&dp_full[it % 2]);
          }
          mma_commit(&mma_drain2);
          mbar_wait_drain(&mma_drain2, 0);
        } else {
          for (int it = 0; it < n_iter && ok; ++it) {
            const int st = it % ST;
            // (the stage barrier is observed for the tensor core's reads of Q and dO; its next
            // phase needs dK(it) below, so it cannot have moved on)
            ok = mbar_wait(&qdo_full[st], (it / ST) & 1, &wctl);
            if (ok) ok = mbar_wait(&p_ready[it % NSB], (it / NSB) & 1, &wctl);
            if (!ok) break;
            tc_fence_after();
            const Desc qmn = make_desc(smem_u32(smem + LY::OFF_Q + st * LY::QT_BYTES), BM * 128, 1024);
            const Desc domn = make_desc(smem_u32(smem + LY::OFF_DO + st * LY::DOT_BYTES), BM * 128, 1024);
            const uint32_t tS = tbase + LY::COL_S0 + (it % NSB) * BM;
            const uint32_t tDP = tbase + LY::COL_DP0 + (it % 2) * BM;
            const Desc dsd = make_desc(smem_u32(smem + LY::OFF_DS + (it % 2) * LY::DS_BYTES), kBN * 128, 1024);
            // dV += P^T dO
#pragma unroll
            for (int ks = 0; ks < BM / 16; ++ks)
              mma_ts2(tDV, tS + ks * 8, domn.at(vslice + ks * 2048), domn.hi, id_dv,
                      (it > 0 || ks > 0) ? 1u : 0u);
            mma_commit(&dv_done[it % NSB]);
            // dK += dS^T Q
            ok = mbar_wait(&ds_ready[it % 2], (it / 2) & 1, &wctl);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < BM / 16; ++ks)
              mma_ts2(tDK, tDP + ks * 8, qmn.at(slice + ks * 2048), qmn.hi, id_dk,
                      (it > 0 || ks > 0) ? 1u : 0u);
            mma_commit(&qdo_empty[st]);
            // dQ^T[d, q] = sum_kv K[kv, d] dS^T[kv, q], into the dP^T buffer (its dS^T has just
            // been read by dK); with skip_dq the commit still hands the buffers on
            if (!p.skip_dq) {
              const uint32_t kslice = (dh * DH / 64) * (kBN * 128);
#pragma unroll
              for (int ks = 0; ks < kBN / 16; ++ks)
                mma_ss2(tDP, kmn.at(kslice + ks * 2048), kmn.hi, dsd.at(ks * 2048), dsd.hi, id_dq,
                        ks > 0 ? 1u : 0u);
            }
            mma_commit(&dq_full[it % 2]);
          }
          mma_commit(&acc_full);
          mma_commit(&mma_drain);
          mbar_wait_drain(&mma_drain, 0);
        }
      }
    }
  } else if (warp == LY::MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    {
    if (elect_one()) {
      const uint32_t sK = smem_u32(smem + LY::OFF_K), sV = smem_u32(smem + LY::OFF_V);
      const Desc kd = make_desc(sK, 16, 1024);          // K as a K-major operand
      const Desc vd = make_desc(sV, 16, 1024);          // V as a K-major operand
      const Desc kmn = make_desc(sK, kBN * 128, 1024);  // K as an MN-major operand
      const uint32_t id_s = idesc_bf16(128, BM, 0, 0);      // S^T, dP^T: [kv x q]
      const uint32_t id_dv = idesc_bf16(128, DVH, 0, 1);    // dV: A tmem, B MN-major
      const uint32_t id_dk = idesc_bf16(128, DH, 0, 1);     // dK: A tmem, B MN-major
      const uint32_t id_dq = T::DQT ? idesc_bf16(DH, BM, 1, 1) : idesc_bf16(BM, HD, 1, 1);
      const uint32_t tDV = tbase + LY::COL_DV, tDK = tbase + LY::COL_DK;
      // head-dim slices of Q (for dK, N = DH) and dO (for dV, N = DVH): MN-major B operands
      const uint32_t slice = (dh * DH / 64) * (BM * 128);
      const uint32_t vslice = (dh * DVH / 64) * (BM * 128);
      bool ok = mbar_wait(&kv_full, 0, &wctl);
      int q_ready = -1;  // highest iteration whose Q/dO stage wait is done

      auto stage_ready = [&](int it) {
        if (it > q_ready) {
          ok = ok && mbar_wait(&qdo_full[it % ST], (it / ST) & 1, &wctl);
          q_ready = it;
          tc_fence_after();
        }
      };
      auto issue_s = [&](int it) {  // S^T(it) = K Q^T
        stage_ready(it);
        if (!ok) return;
        const Desc qd = make_desc(smem_u32(smem + LY::OFF_Q + (it % ST) * LY::QT_BYTES), 16, 1024);
        const uint32_t tS = tbase + LY::COL_S0 + (it % NSB) * BM;
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t ko = (ks / 4) * (kBN * 128) + (ks % 4) * 32;
          const uint32_t qo = (ks / 4) * (BM * 128) + (ks % 4) * 32;
          mma_ss2(tS, kd.at(ko), kd.hi, qd.at(qo), qd.hi, id_s, ks > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[it % NSB]);
      };
      auto issue_dp = [&](int it) {  // dP^T(it) = V dO^T, into the buffer dQ(it-2) used
        stage_ready(it);
        if (ok && it >= 2) {
          ok = mbar_wait(&dq_free[it % 2], ((it - 2) / 2) & 1, &wctl);
          tc_fence_after();
        }
        if (!ok) return;
        const Desc dod = make_desc(smem_u32(smem + LY::OFF_DO + (it % ST) * LY::DOT_BYTES), 16, 1024);
        const uint32_t tDP = tbase + LY::COL_DP0 + (it % 2) * BM;
#pragma unroll
        for (int ks = 0; ks < DV / 16; ++ks) {  // contraction over the value head dim
          const uint32_t ko = (ks / 4) * (kBN * 128) + (ks % 4) * 32;
          const uint32_t qo = (ks / 4) * (BM * 128) + (ks % 4) * 32;
          mma_ss2(tDP, vd.at(ko), vd.hi, dod.at(qo), dod.hi, id_s, ks > 0 ? 1u : 0u);
        }
        mma_commit(&dp_full[it % 2]);
      };

      if (n_iter > 0 && ok) {
        issue_s(0);
        issue_dp(0);
      }
      for (int it = 0; it < n_iter && ok; ++it) {
        const int st = it % ST;
        const Desc qmn = make_desc(smem_u32(smem + LY::OFF_Q + st * LY::QT_BYTES), BM * 128, 1024);
        const Desc domn = make_desc(smem_u32(smem + LY::OFF_DO + st * LY::DOT_BYTES), BM * 128, 1024);
        const uint32_t tS = tbase + LY::COL_S0 + (it % NSB) * BM;
        const uint32_t tDP = tbase + LY::COL_DP0 + (it % 2) * BM;
        const Desc dsd = make_desc(smem_u32(smem + LY::OFF_DS + (it % 2) * LY::DS_BYTES), kBN * 128, 1024);
        // dV += P^T dO
        ok = mbar_wait(&p_ready[it % NSB], (it / NSB) & 1, &wctl);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < BM / 16; ++ks)
          mma_ts2(tDV, tS + ks * 8, domn.at(vslice + ks * 2048), domn.hi, id_dv,
                  (it > 0 || ks > 0) ? 1u : 0u);
        if constexpr (T::LOOKAHEAD && NSB == 2) {
          // S^T(it + 1), then dP^T(it + 1). S^T(it + 1) goes into the buffer that held P^T(it - 1),
          // free once the dS warpgroup has read it (dV(it - 1) was issued before). Forming S^T
          // one tile ahead, not two, keeps a Q/dO stage in use for two tiles instead of three,
          // so the three-stage ring has a stage to prefetch into (a stage takes ~1 us to refill);
          // S^T before dP^T lets the P^T warpgroup start sooner. Measured on the 4k GQA shape:
          // main pass 666 -> 648 us; window workload 2346 -> 2281 us.
          if (it + 1 < n_iter) {
            if (it >= 1) {
              ok = mbar_wait(&p_consumed[(it - 1) % NSB], ((it - 1) / NSB) & 1, &wctl);
              if (!ok) break;
              tc_fence_after();
            }
            issue_s(it + 1);
            if (!ok) break;
            issue_dp(it + 1);
            if (!ok) break;
          }
        } else if constexpr (T::LOOKAHEAD) {
          if (it + 1 < n_iter) {
            issue_dp(it + 1);
            if (!ok) break;
          }
          // the next S^T into this tile's score buffer, as soon as the dS warpgroup has read
          // P^T(it) from it (dV(it), issued above, reads it first: same-thread MMAs run in order)
          if (it + NSB < n_iter) {
            ok = mbar_wait(&p_consumed[it % NSB], (it / NSB) & 1, &wctl);
            if (!ok) break;
            tc_fence_after();
            issue_s(it + NSB);
            if (!ok) break;
          }
        }
        // dK += dS^T Q
        ok = mbar_wait(&ds_ready[it % 2], (it / 2) & 1, &wctl);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < BM / 16; ++ks)
          mma_ts2(tDK, tDP + ks * 8, qmn.at(slice + ks * 2048), qmn.hi, id_dk,
                  (it > 0 || ks > 0) ? 1u : 0u);
        mma_commit(&qdo_empty[st]);
        if constexpr (!T::LOOKAHEAD) {
          if (it + 1 < n_iter) {
            issue_s(it + 1);
            issue_dp(it + 1);
            if (!ok) break;
          }
        }
        // dQ of this tile, into the dP^T buffer (its dS^T has just been read by dK). With
        // skip_dq the commit below still tells WG1 and WG2 that dK has read the buffers.
        if (p.skip_dq) {
        } else if constexpr (T::DQT) {
          // dQ^T[d, q] = sum_kv K[kv, d] dS^T[kv, q]: A = K slice (MN-major), B = dS^T
          const uint32_t kslice = (dh * DH / 64) * (kBN * 128);
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks)
            mma_ss2(tDP, kmn.at(kslice + ks * 2048), kmn.hi, dsd.at(ks * 2048), dsd.hi, id_dq,
                    ks > 0 ? 1u : 0u);
        } else {
          // dQ[q, d] = sum_kv dS^T[kv, q] K[kv, d]: A = dS^T (MN-major), B = K (MN-major)
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks)
            mma_ss2(tDP, dsd.at(ks * 2048), dsd.hi, kmn.at(ks * 2048), kmn.hi, id_dq,
                    ks > 0 ? 1u : 0u);
        }
        mma_commit(&dq_full[it % 2]);
      }
      mma_commit(&acc_full);
      mma_commit(&mma_drain);
      mbar_wait_drain(&mma_drain, 0);
    }
    }
  } else if (warp == LY::BULK_WARP) {
    // ------------------------------------------------------------------ bulk dQ reductions
    if constexpr (T::DQ_BULK) {
      if (!p.skip_dq && elect_one()) {
        const float* stg = reinterpret_cast<const float*>(smem + LY::OFF_STG);
        for (int it = 0; it < n_iter; ++it) {
          if (!mbar_wait(&stg_full, it & 1, &wctl)) break;
          const int h = kh * G + it / nm;
          const int q0 = (m_first + it % nm) * BM;
          const int bh = b * p.H + h;
          bulk_reduce_add_f32(p.dqacc + ((size_t)bh * p.ql_pad + q0) * HD, stg, BM * HD * 4);
          bulk_commit();
          bulk_wait_read<0>();  // the staging buffer has been read
          mbar_arrive(&stg_free);
        }
        bulk_wait<0>();  // every reduction has landed before the CTA exits
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------------ WG0: P^T, dQ drain
    const int j = warp * 32 + lane;  // kv row within the tile == TMEM lane
    const int kv = n0 + j;
    const bool kv_live = kv < kl;
    const uint32_t lane_base = tbase + ((uint32_t)(warp * 32) << 16);
    const float c2 = p.scale_log2;
    const uint64_t c2v = f2_pack(c2, c2);
    bool ok = true;

    for (int it = 0; it < n_iter && ok; ++it) {
      const int st = it % ST;
      const int h = kh * G + it / nm;
      const int q0 = (m_first + it % nm) * BM;
      const float* sL = reinterpret_cast<const float*>(smem + LY::OFF_L + st * BM * 4);
      const uint32_t colS = LY::COL_S0 + (it % NSB) * BM;
      // column q (row q0 + q) sees this key iff qlo <= q <= qhi (no upper limit without a
      // window)
      const int off = kl - ql;
      const int hi_off = WIN ? p.hi_off : 0;
      const int qlo = kv - off - hi_off - q0;
      const int qhi = WIN ? kv - off - p.lo_off - q0 : BM;
      // interior pair: the first query row sees the tile's last key and the last query row its
      // first key; otherwise some element is hidden (uniform over the warpgroup)
      const bool edge = BAND != kBandNone && !(q0 >= n0 + kBN - 1 - off - hi_off &&
                                               (!WIN || q0 + BM - 1 <= n0 - off - p.lo_off));
      // columns outside [qcut_lo, qcut_hi] get P = 0: the band on edge tiles, every column for
      // kv rows past the end (qcut_lo = BM)
      const bool need_mask = edge || !kv_live;
      const int qcut_lo = !kv_live ? BM : (edge ? qlo : 0);
      const int qcut_hi = edge ? qhi : BM;
      const void* mcol = nullptr;
      if (MASKT != 0 && kv_live) {
        const size_t es = MASKT == 1 ? 4 : MASKT == 2 ? 2 : 1;
        mcol = reinterpret_cast<const uint8_t*>(p.mask) +
               (b * p.msb + (long long)h * p.msh + (long long)q0 * p.msq + kv) * es;
      }

      // the stage's L rows came with the Q/dO copies; observe that barrier here too (its
      // next phase needs this tile's dK MMA, so it cannot have moved on)
      ok = __all_sync(0xffffffffu, mbar_wait(&qdo_full[st], (it / ST) & 1, &wctl));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&s_full[it % NSB], (it / NSB) & 1, &wctl));
      if (!ok) break;
      tc_fence_after();
      const float4* sL4 = reinterpret_cast<const float4*>(sL);  // -L*log2(e) per query
      constexpr int GRP = BM / 32 < 2 ? BM / 32 : 2;  // 32-column chunks loaded per wait
#pragma unroll
      for (int g0 = 0; g0 < BM / 32; g0 += GRP) {
        uint32_t rs[GRP][32];
#pragma unroll
        for (int g = 0; g < GRP; ++g) tmem_ld32(lane_base + colS + (g0 + g) * 32, rs[g]);
        tmem_wait_ld();
#pragma unroll
        for (int g = 0; g < GRP; ++g) {
          const int c32 = g0 + g;
          uint32_t pk[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 nl = sL4[c32 * 8 + e4];
            const int q = c32 * 32 + e4 * 4;
            uint64_t b01 = f2_pack(nl.x, nl.y), b23 = f2_pack(nl.z, nl.w);
            if (MASKT != 0) {
              float m4[4];
#pragma unroll
              for (int k = 0; k < 4; ++k)
                m4[k] = (mcol != nullptr && q0 + q + k < ql)
                            ? mask_log2_b<MASKT>(mcol, (long long)(q + k) * p.msq)
                            : 0.0f;
              b01 = f2_add(b01, f2_pack(m4[0], m4[1]));
              b23 = f2_add(b23, f2_pack(m4[2], m4[3]));
            }
            const uint32_t* r = rs[g];
            const uint64_t s01 = f2_fma(f2_pack(__uint_as_float(r[4 * e4]), __uint_as_float(r[4 * e4 + 1])), c2v, b01);
            const uint64_t s23 = f2_fma(f2_pack(__uint_as_float(r[4 * e4 + 2]), __uint_as_float(r[4 * e4 + 3])), c2v, b23);
            float a0, a1, a2, a3;
            f2_unpack(s01, a0, a1);
            f2_unpack(s23, a2, a3);
            float p0 = ex2(a0), p1 = ex2(a1), p2 = ex2(a2), p3 = ex2(a3);
            if (need_mask) {  // hidden columns (band) and kv rows past the end
              p0 = (q >= qcut_lo && (!WIN || q <= qcut_hi)) ? p0 : 0.0f;
              p1 = (q + 1 >= qcut_lo && (!WIN || q + 1 <= qcut_hi)) ? p1 : 0.0f;
              p2 = (q + 2 >= qcut_lo && (!WIN || q + 2 <= qcut_hi)) ? p2 : 0.0f;
              p3 = (q + 3 >= qcut_lo && (!WIN || q + 3 <= qcut_hi)) ? p3 : 0.0f;
            }
            pk[2 * e4] = pack_bf16(p0, p1);
            pk[2 * e4 + 1] = pack_bf16(p2, p3);
          }
          // P^T as bf16 into the S columns (A operand of dV += P^T dO; read again by WG1)
          tmem_st16(lane_base + colS + c32 * 16, pk);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_ready[it % NSB]);
    }
  } else if (warp >= 8 && warp < 12) {
    // ------------------------------------------------------------------ WG2: dQ drain
    const int j = (warp - 8) * 32 + lane;  // TMEM lane (head-dim row of dQ^T, or query row)
    const uint32_t lane_base = tbase + ((uint32_t)((warp - 8) * 32) << 16);
    bool ok = true;
    // dQ of iteration `it` into the f32 accumulator (its MMA followed that tile's dK)
    auto drain = [&](int it) {
      const int h = kh * G + it / nm;
      const int q0 = (m_first + it % nm) * BM;
      const int bh = b * p.H + h;
      const uint32_t colDQ = LY::COL_DP0 + (it % 2) * BM;
      ok = __all_sync(0xffffffffu, mbar_wait(&dq_full[it % 2], (it / 2) & 1, &wctl));
      if (!ok) return;
      tc_fence_after();
      if (p.skip_dq) {  // nothing to drain: hand the buffer straight back
        tc_fence_before();
        mbar_arrive(&dq_free[it % 2]);
        return;
      }
      if constexpr (T::DQ_BULK && T::DQT) {
        // lane = head-dim index d, column = query row: stage the tile transposed and
        // chunk-major (chunk c = query rows 4c .. 4c+3 of row d at float4 position c * HD + d;
        // the accumulator keeps this tile layout and the dQ convert kernel turns it back), so
        // that the 16-byte stores of a warp cover 512 contiguous bytes. The bulk warp adds the
        // tile with one reduction; the buffer is handed over with mbarriers (stg_full once
        // written, stg_free once read).
        float* stg = reinterpret_cast<float*>(smem + LY::OFF_STG);
        uint32_t rq[BM / 32][32];
#pragma unroll
        for (int c32 = 0; c32 < BM / 32; ++c32) tmem_ld32(lane_base + colDQ + c32 * 32, rq[c32]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&dq_free[it % 2]);
        if (it > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(&stg_free, (it - 1) & 1, &wctl));
          if (!ok) return;
        }
        static_assert(BM / 4 == kDqChunks, "chunk-major dQ tile");
        float4* st4 = reinterpret_cast<float4*>(stg) + j;
#pragma unroll
        for (int c = 0; c < BM / 4; ++c) {  // chunk c: query rows 4c .. 4c+3
          const uint32_t* r = &rq[c / 8][(c % 8) * 4];
          st4[c * HD] = make_float4(__uint_as_float(r[0]), __uint_as_float(r[1]),
                                    __uint_as_float(r[2]), __uint_as_float(r[3]));
        }
        fence_proxy_async();  // staging writes -> visible to the bulk copy
        mbar_arrive(&stg_full);
      } else {
        // lane = query row j, column = head-dim index: stage the row (HD f32) with its 16-byte
        // chunks XOR-rotated by (j & 15); the bulk warp adds the tile with one reduction
        float* stg = reinterpret_cast<float*>(smem + LY::OFF_STG);
        uint32_t rq[HD / 32][32];
#pragma unroll
        for (int c32 = 0; c32 < HD / 32; ++c32) tmem_ld32(lane_base + colDQ + c32 * 32, rq[c32]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&dq_free[it % 2]);
        if (it > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(&stg_free, (it - 1) & 1, &wctl));
          if (!ok) return;
        }
        float4* row = reinterpret_cast<float4*>(stg + j * HD);
#pragma unroll
        for (int c = 0; c < HD / 4; ++c) {  // chunk c: head-dim 4c .. 4c+3
          const uint32_t* r = &rq[c / 8][(c % 8) * 4];
          row[c ^ (j & (kDqChunks - 1))] = make_float4(__uint_as_float(r[0]), __uint_as_float(r[1]),
                                                       __uint_as_float(r[2]), __uint_as_float(r[3]));
        }
        fence_proxy_async();  // staging writes -> visible to the bulk copy
        mbar_arrive(&stg_full);
      }
    };

    for (int it = 0; it < n_iter && ok; ++it) drain(it);
  } else if (warp < 8) {
    // ------------------------------------------------------------------ WG1: dS^T, epilogue
    const int wl = warp - 4;
    const int j = wl * 32 + lane;
    const int kv = n0 + j;
    const uint32_t lane_base = tbase + ((uint32_t)(wl * 32) << 16);
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      const int st = it % ST;
      const float* sD = reinterpret_cast<const float*>(smem + LY::OFF_D + st * BM * 4);
      const uint32_t colS = LY::COL_S0 + (it % NSB) * BM;
      const uint32_t colDP = LY::COL_DP0 + (it % 2) * BM;
      ok = __all_sync(0xffffffffu, mbar_wait(&dp_full[it % 2], (it / 2) & 1, &wctl));
      // (p_ready also makes the stage's D rows visible: the P warpgroup observed the Q/dO stage
      // barrier before it arrived on p_ready)
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&p_ready[it % NSB], (it / NSB) & 1, &wctl));
      // the dQ MMA of tile it-2 must be done reading this dS^T buffer
      if (ok && it >= 2)
        ok = __all_sync(0xffffffffu, mbar_wait(&dq_full[it % 2], ((it - 2) / 2) & 1, &wctl));
      if (!ok) break;
      tc_fence_after();
      uint8_t* sds = smem + LY::OFF_DS + (it % 2) * LY::DS_BYTES;
      const float4* sD4 = reinterpret_cast<const float4*>(sD);
      constexpr int GRP = BM / 32 < 2 ? BM / 32 : 2;  // 32-column chunks loaded per wait
#pragma unroll
      for (int g0 = 0; g0 < BM / 32; g0 += GRP) {
        uint32_t rd[GRP][32];
        uint32_t rp[32];  // P^T bf16 pairs of these 2 x 32 columns (first 16 or 32 used)
#pragma unroll
        for (int g = 0; g < GRP; ++g) tmem_ld32(lane_base + colDP + (g0 + g) * 32, rd[g]);
        if (GRP == 2) {
          tmem_ld32(lane_base + colS + g0 * 16, rp);
        } else {
          tmem_ld16(lane_base + colS + g0 * 16, *reinterpret_cast<uint32_t(*)[16]>(rp));
        }
        tmem_wait_ld();
        if (g0 + GRP >= BM / 32) {  // every column of P^T(it) is in registers: free its buffer
          tc_fence_before();
          mbar_arrive(&p_consumed[it % NSB]);
        }
#pragma unroll
        for (int g = 0; g < GRP; ++g) {
          const int c32 = g0 + g;
          const uint32_t* r = rd[g];
          uint32_t pk[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 dd = sD4[c32 * 8 + e4];
            // P of columns q .. q+3 from the packed pairs (bf16 -> f32 is a shift)
            const uint32_t pp0 = rp[g * 16 + 2 * e4];
            const uint32_t pp1 = rp[g * 16 + 2 * e4 + 1];
            const uint64_t pv01 = f2_pack(__uint_as_float(pp0 << 16), __uint_as_float(pp0 & 0xffff0000u));
            const uint64_t pv23 = f2_pack(__uint_as_float(pp1 << 16), __uint_as_float(pp1 & 0xffff0000u));
            const uint64_t t01 = f2_add(f2_pack(__uint_as_float(r[4 * e4]), __uint_as_float(r[4 * e4 + 1])),
                                        f2_pack(-dd.x, -dd.y));
            const uint64_t t23 = f2_add(f2_pack(__uint_as_float(r[4 * e4 + 2]), __uint_as_float(r[4 * e4 + 3])),
                                        f2_pack(-dd.z, -dd.w));
            const uint64_t u01 = f2_mul(t01, pv01);
            const uint64_t u23 = f2_mul(t23, pv23);
            float d0, d1, d2, d3;
            f2_unpack(u01, d0, d1);
            f2_unpack(u23, d2, d3);
            pk[2 * e4] = pack_bf16(d0, d1);
            pk[2 * e4 + 1] = pack_bf16(d2, d3);
          }
          tmem_st16(lane_base + colDP + c32 * 16, pk);
          // dS^T row j, columns c32*32 .. +31: 4 granules of the 64-column chunk c32/2 (also
          // written with skip_dq: a branch here costs the default path more than the stores)
          uint8_t* chunk = sds + (c32 / 2) * (kBN * 128);
#pragma unroll
          for (int gg = 0; gg < 4; ++gg)
            st_swizzled(chunk, j, (c32 % 2) * 4 + gg,
                        make_uint4(pk[4 * gg], pk[4 * gg + 1], pk[4 * gg + 2], pk[4 * gg + 3]));
        }
      }
      fence_proxy_async();  // generic-proxy writes of dS^T -> visible to the tensor core
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&ds_ready[it % 2]);
    }

    // ---------------------------------------------------------------- dK, dV epilogue
    bool have = false;
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(&acc_full, 0, &wctl));
      tc_fence_after();
      have = ok && n_iter > 0;
    }
    const long long kvr = krow0 + (kv < kl ? kv : 0);  // row of this key in dK / dV
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {
      const uint32_t col = which == 0 ? LY::COL_DV : LY::COL_DK;
      const float mul = which == 0 ? 1.0f : p.scale;
      const int width = which == 0 ? DVH : DH;  // columns of the slice this CTA owns
      __nv_bfloat16* out =
          which == 0 ? p.dv + bhsd_offset(kb, kh, kvr, p.Hk, krows, DV, kv_bshd) + dh * DVH
                     : p.dk + bhsd_offset(kb, kh, kvr, p.Hk, krows, HD, kv_bshd) + dh * DH;
#pragma unroll 1
      for (int c = 0; c < width; c += 32) {
        uint32_t r[32];
        if (have) {
          tmem_ld32(lane_base + col + c, r);
          tmem_wait_ld();
        }
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = have ? pack_bf16(__uint_as_float(r[2 * e]) * mul, __uint_as_float(r[2 * e + 1]) * mul)
                       : 0u;
        if (kv < kl) {
          uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == LY::MMA_WARP) tmem_dealloc(tbase, LY::TMEM_COLS);
  if (threadIdx.x == 0) report_abort(&wctl, p.status);
}

template <int HD, int DV, int BAND, bool STRIDED, int MASKT, bool VARLEN = false>
static cudaError_t launch_main_t(const BwdArgs& a, const BwdMaps& m, cudaStream_t s) {
  using LY = BwdLayout<HD, DV>;
  auto kern = bwd_main_kernel<HD, DV, BAND, MASKT, VARLEN, STRIDED>;
  static OncePerKey<> smem_attr;  // per instantiation and device
  {
    const cudaError_t e = set_smem_once(smem_attr, kern, LY::SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  BwdKParams kp = make_bwd_kparams(a);
  const int groups = a.B * a.Hk * BwdTraits<HD>::DSPLIT, ktiles = (a.kl + kBN - 1) / kBN;
  kp.tiles_fast = a.cu_q != nullptr && groups <= 65535;  // (grid y limit)
  dim3 grid(kp.tiles_fast ? ktiles : groups, kp.tiles_fast ? groups : ktiles);
  profile_mark(kKernBwdMain, 0, s);
  const cudaError_t e = launch_pdl(kern, grid, dim3(LY::THREADS), LY::SMEM_BYTES, s, m.q, m.k,
                                   m.v, m.dO, kp);
  profile_mark(kKernBwdMain, 1, s);
  return e;
}

template <int HD, int DV, int BAND, bool STRIDED>
static cudaError_t launch_main_m(const BwdArgs& a, const BwdMaps& m, cudaStream_t s) {
  if (a.cu_q) return launch_main_t<HD, DV, BAND, STRIDED, 0, true>(a, m, s);  // (no mask)
  if (!a.mask) return launch_main_t<HD, DV, BAND, STRIDED, 0>(a, m, s);
  switch (a.mask_type) {
    case 0: return launch_main_t<HD, DV, BAND, STRIDED, 1>(a, m, s);
    case 1: return launch_main_t<HD, DV, BAND, STRIDED, 2>(a, m, s);
    default: return launch_main_t<HD, DV, BAND, STRIDED, 3>(a, m, s);
  }
}

// The main pass of head dims 64 and 128 in either layout class (the bshd instantiations live in
// fa_bwd_strided.cu, compiled in parallel with fa_bwd.cu).
template <int HD, int DV, bool STRIDED>
static cudaError_t launch_main_layout(const BwdArgs& a, const BwdMaps& m, cudaStream_t s) {
  return a.band == kBandNone     ? launch_main_m<HD, DV, kBandNone, STRIDED>(a, m, s)
         : a.band == kBandCausal ? launch_main_m<HD, DV, kBandCausal, STRIDED>(a, m, s)
                                 : launch_main_m<HD, DV, kBandWindow, STRIDED>(a, m, s);
}

// Defined in fa_bwd_strided.cu: the main pass of a call with a bshd layout (head dims 64, 128).
cudaError_t launch_main_strided(const BwdArgs& a, const BwdMaps& m, cudaStream_t s);

}  // namespace fa
