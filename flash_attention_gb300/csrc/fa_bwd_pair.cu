// fa_bwd_pair.cu -- the backward main pass at head_dim 256, on a pair of CTAs (a 2-CTA
// cluster) that share one kv tile (sm_103a).
//
// Method: as in fa_bwd.cu (page "mlx-native tests/test_flash_attn_train.rs",
// `sdpa_backward_reference_f32`, with the kv-tile-major decomposition of page "tang
// src/compute/cuda.rs", `causal_attention_backward`): per kv tile of 128 keys and per query tile
// of 64 rows of every query head sharing the kv head,
//   S^T = K Q^T,  P^T = exp2(S^T * scale * log2(e) + mask * log2(e) - L * log2(e)),
//   dP^T = V dO^T,  dS^T = P^T o (dP^T - D),
//   dV += P^T dO,  dK += dS^T Q,  dQ^T += K^T dS^T  (f32, across CTAs).
//
// Why a pair: at head_dim 256 the f32 dK and dV of a 128-key tile fill all 512 TMEM columns of
// one CTA, so each CTA can own only one 128-wide half of them. Two CTAs that each computed S^T
// and dP^T for their half would repeat 2 of the 5 contractions, and K, V, Q and dO would fill
// their shared memory. Here the two CTAs of a cluster split the work instead:
//   rank 0 holds K, computes S^T and P^T, dV and dK for head-dim columns 0-127, and all of dQ;
//   rank 1 holds V, computes dP^T and dS^T, dV and dK for columns 128-255.
// Each CTA stages the bf16 tile it produced (P^T from rank 0, dS^T from rank 1) in its own shared
// memory and sends it to the other CTA with one bulk copy (cp.async.bulk shared::cta to
// shared::cluster) that completes a transaction on the other CTA's barrier; its own copy also
// goes to TMEM as the A operand of its own dV (rank 0) or dK (rank 1) MMA. (128 threads storing
// their rows into the other CTA directly measured 1.3-2 us per tile, most of an iteration.) Every contraction is done once, and each CTA holds only what it multiplies: a two-stage
// Q/dO ring fits next to K or V, the exchange buffers and (rank 0) a dQ staging tile for bulk
// reductions.
//
// Roles (384 threads): warps 0-3 compute P^T (rank 0) or dS^T (rank 1), one kv row per thread
// (= TMEM lane), and write that CTA's dK/dV half at the end; warps 4-7 (rank 0) drain dQ^T from
// TMEM into a staging tile; warp 8 issues the TMA loads; warp 9 issues the MMAs, polling the
// barriers of the three MMA groups of its rank so that whichever is ready goes first; warp 10
// (rank 0) adds the staged dQ^T tiles into the f32 accumulator with bulk reductions; warp 11
// sends the staged tile to the other CTA; on rank 1, warp 10 tells rank 0 when rank 1's exchange
// buffer may be rewritten. Every wait is bounded.
#include "fa_bwd_common.cuh"

namespace fa {

namespace {
constexpr int kPM = 64;   // query rows per tile (N of S^T and dP^T; K of dV and dK)
constexpr int kPD = 256;  // head dim of q, k, v and dO
constexpr int kPST = 2;   // depth of the Q / dO ring
}  // namespace

// One shared-memory layout for both ranks; what a region holds depends on the rank.
struct PairLayout {
  static constexpr int KV_BYTES = kBN * kPD * 2;          // K (rank 0) or V (rank 1), 64 KB
  static constexpr int FULL_BYTES = kPM * kPD * 2;        // Q (rank 0) or dO (rank 1), 32 KB
  static constexpr int HALF_BYTES = kPM * (kPD / 2) * 2;  // dO[:, 0:128] (0) / Q[:, 128:256] (1)
  static constexpr int STAGE_BYTES = FULL_BYTES + HALF_BYTES;
  static constexpr int X_BYTES = kBN * kPM * 2;           // a [kv][q] bf16 tile, 16 KB
  static constexpr int STG_BYTES = 128 * kPM * 4;         // rank 0: 128 head-dim rows x 64 f32
  static constexpr int OFF_KV = 0;
  static constexpr int OFF_ST = OFF_KV + KV_BYTES;            // kPST stages
  static constexpr int OFF_X = OFF_ST + kPST * STAGE_BYTES;   // 2 exchange buffers
  static constexpr int OFF_STG = OFF_X + 2 * X_BYTES;  // rank 0: dQ^T staging; 1: dS^T out
  static constexpr int OFF_L = OFF_STG + STG_BYTES;           // kPST x kPM f32: -L log2(e)
  static constexpr int OFF_D = OFF_L + kPST * kPM * 4;        // kPST x kPM f32: D
  static constexpr int OFF_END = OFF_D + kPST * kPM * 4;
  static constexpr int SMEM_BYTES = OFF_END + 1024;
  // TMEM columns: two 64-column buffers (rank 0: S^T then P^T as bf16; rank 1: dP^T then dS^T),
  // rank 0's dQ^T (two 128-row halves of 64 columns), and the dV and dK halves.
  static constexpr int COL_X0 = 0;
  static constexpr int COL_DQ = 128;
  static constexpr int COL_DV = 256;
  static constexpr int COL_DK = 384;
  static constexpr int TMEM_COLS = 512;
  static constexpr int THREADS = 384;
  static constexpr int TMA_WARP = 8, MMA_WARP = 9, BULK_WARP = 10, LINK_WARP = 11;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(kPM / 4 == kDqChunks, "staged dQ^T tile layout");
};

template <int BAND, int MASKT, bool VARLEN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairLayout::THREADS, 1)
    bwd_pair_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                    const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mDO,
                    const BwdKParams p) {
  using LY = PairLayout;
  constexpr int BM = kPM, ST = kPST, HD = kPD;
  constexpr bool WIN = BAND == kBandWindow;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ uint64_t kv_full, qdo_full[ST], qdo_empty[ST];
  __shared__ uint64_t mine_full[2];  // rank 0: S^T(it) in TMEM; rank 1: dP^T(it)
  __shared__ uint64_t own_ready[2];  // 128 arrivals: P^T (0) / dS^T (1) written to TMEM as bf16
  __shared__ uint64_t x_ready[2];    // the peer's tile has landed in x buffer (bulk-copy bytes)
  __shared__ uint64_t x_free[2];     // rank 0: rank 1's x buffer may be rewritten (remote)
  __shared__ uint64_t x_done[2];     // MMA commit: this CTA's MMAs have read its x buffer
  __shared__ uint64_t out_staged[2]; // 128 arrivals: this CTA's outgoing tile is staged
  __shared__ uint32_t n_sent;        // tiles sent to the peer (read by the peer at the end)
  __shared__ uint64_t dq_full, dq_free, stg_full, stg_free, acc_full, mma_drain;
  __shared__ uint32_t tmem_base_s;
  __shared__ WaitCtl wctl;

  const int warp = warp_id(), lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  // The pair is along x. Fixed length: x = (batch, kv head) pair, y = kv tile (tile-major: the
  // heaviest causal tiles launch first). Variable length: x = kv tile pair, y = (sequence, kv
  // head), so that one sequence's tiles run together and share its Q / dO through L2.
  const int bkh = p.tiles_fast ? (int)blockIdx.y : (int)(blockIdx.x >> 1);
  const int b = bkh / p.Hk, kh = bkh % p.Hk;
  const int G = p.H / p.Hk;
  const int n0 = (int)(p.tiles_fast ? (blockIdx.x >> 1) : blockIdx.y) * kBN;
  int ql = p.ql, kl = p.kl;
  int kz = bkh, qzb = b * p.H, krow0 = 0, qrow0 = 0;
  size_t kvrow0 = (size_t)bkh * p.kl;  // dK / dV row of key 0
  if constexpr (VARLEN) {
    int qs, ks;
    const bool bad = varlen_seq(p.cu_q, b, p.total_q, p.ql, qs, ql) |
                     varlen_seq(p.cu_k, b, p.total_k, p.kl, ks, kl);
    if (bad && threadIdx.x == 0 && rank == 0 && p.status)
      atomicCAS(p.status, kStatusOk, kStatusBadInput);
    kz = kh;
    qzb = 0;
    krow0 = ks;
    qrow0 = qs;
    kvrow0 = (size_t)kh * p.total_k + ks;
  }
  if (n0 >= kl) return;  // a kv tile past this sequence's keys: both CTAs of the pair leave
  int m_first, m_last;
  bwd_mtile_range<HD, BAND>(n0, p, ql, kl, m_first, m_last);
  const int nm = m_last - m_first + 1;  // query tiles per head (0 if none)
  const int n_iter = G * nm;            // (head, query tile) pairs this pair of CTAs visits
  const bool do_dq = rank == 0 && !p.skip_dq;

  if (threadIdx.x == 0) {
    wait_ctl_init(&wctl, p.wait_limit_ns);
    mbar_init(&kv_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&qdo_full[s], 1);
      mbar_init(&qdo_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&mine_full[s], 1);
      mbar_init(&own_ready[s], 128);
      mbar_init(&x_ready[s], 1);
      mbar_init(&x_free[s], 1);
      mbar_init(&x_done[s], 1);
      mbar_init(&out_staged[s], 128);
    }
    n_sent = 0;
    mbar_init(&dq_full, 1);
    mbar_init(&dq_free, 128);
    mbar_init(&stg_full, 128);
    mbar_init(&stg_free, 1);
    mbar_init(&acc_full, 1);
    mbar_init(&mma_drain, 1);
    // rank 1 receives P^T(0) and P^T(1) into armed phases (later phases are armed as buffers
    // free up; rank 0 arms each phase before it sends the P^T the peer answers with dS^T)
    if (rank == 1)
      for (int s = 0; s < 2 && s < n_iter; ++s) mbar_arrive_expect_tx(&x_ready[s], LY::X_BYTES);
    fence_barrier_init();
  }
  if (warp == LY::MMA_WARP) {
    tmem_alloc(&tmem_base_s, LY::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();  // the peer's barriers are initialised before any remote arrive
  const uint32_t tbase = tmem_base_s;
  const uint32_t x_local = smem_u32(smem + LY::OFF_X);

  if (warp == LY::TMA_WARP) {
    // ------------------------------------------------------------------ TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mV);
      tma_prefetch_desc(&mDO);
      int last_use[ST];
      for (int s = 0; s < ST; ++s) last_use[s] = -1;
      const CUtensorMap* mkv = rank == 0 ? &mK : &mV;
      const CUtensorMap* mfull = rank == 0 ? &mQ : &mDO;  // the tile this rank needs whole
      const CUtensorMap* mhalf = rank == 0 ? &mDO : &mQ;  // ... and the half it needs
      const int half_c0 = rank == 0 ? 0 : 2;              // first 64-column chunk of that half
      mbar_arrive_expect_tx(&kv_full, LY::KV_BYTES);
      for (int c = 0; c < HD / 64; ++c)
        tma_load_3d(smem + LY::OFF_KV + c * kBN * 128, mkv, &kv_full, c * 64, krow0 + n0, kz);
      for (int it = 0; it < n_iter; ++it) {
        const int st = it % ST;
        const uint32_t use = it / ST;
        if (it >= ST && !mbar_wait(&qdo_empty[st], (use - 1) & 1, &wctl)) break;
        const int h = kh * G + it / nm;
        const int q0 = (m_first + it % nm) * BM;
        const int bh = b * p.H + h;
        uint8_t* sbase = smem + LY::OFF_ST + st * LY::STAGE_BYTES;
        mbar_arrive_expect_tx(&qdo_full[st], LY::STAGE_BYTES + 2 * BM * 4);
        for (int c = 0; c < HD / 64; ++c)
          tma_load_3d(sbase + c * BM * 128, mfull, &qdo_full[st], c * 64, qrow0 + q0, qzb + h);
        for (int c = 0; c < 2; ++c)
          tma_load_3d(sbase + LY::FULL_BYTES + c * BM * 128, mhalf, &qdo_full[st],
                      (half_c0 + c) * 64, qrow0 + q0, qzb + h);
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
  } else if (warp == LY::MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    // Three groups per iteration it, issued in dependence order but interleaved across
    // iterations by polling: X(it) = S^T (rank 0) or dP^T (rank 1) into TMEM buffer it % 2;
    // V(it) = dV half (rank 0: A = P^T in TMEM; rank 1: A = P^T in the exchange buffer);
    // K(it) = dK half (rank 0: A = dS^T in the exchange buffer; rank 1: A = dS^T in TMEM) and,
    // on rank 0, dQ^T. Conditions: X(i) needs its Q/dO stage and its TMEM buffer free (rank 0:
    // V(i-2) issued; rank 1: K(i-2) issued: MMAs of one thread run in issue order); V(i) needs
    // X(i) issued and P^T(i); K(i) needs V(i) issued (so that the stage-release commit after it
    // covers every reader of the stage) and dS^T(i), and dQ(i) the drain of dQ(i-1).
    if (elect_one()) {
      const uint32_t sKV = smem_u32(smem + LY::OFF_KV);
      const Desc akv = make_desc(sKV, 16, 1024);          // K or V as a K-major operand
      const Desc kmn = make_desc(sKV, kBN * 128, 1024);   // K as an MN-major operand (dQ^T)
      const uint32_t id_x = idesc_bf16(128, BM, 0, 0);    // S^T, dP^T: [kv x q]
      const uint32_t id_acc = idesc_bf16(128, 128, 0, 1); // dV, dK halves: B MN-major
      const uint32_t id_dq = idesc_bf16(128, BM, 1, 1);   // dQ^T half: [d x q]
      const uint32_t tDV = tbase + LY::COL_DV, tDK = tbase + LY::COL_DK;
      bool ok = mbar_wait(&kv_full, 0, &wctl);
      int nx = 0, nv = 0, nk = 0;
      const bool every_poll = wctl.limit_ns < 100000ull;
      uint64_t t_idle = 0;
      uint32_t spins = 0;
      while (ok && nk < n_iter) {
        bool progressed = false;
        // ---- K(nk): dK half (+ dQ^T on rank 0)
        if (nk < nv) {
          const int bb = nk & 1;
          const uint32_t ph = (nk >> 1) & 1;
          bool ready = rank == 0 ? mbar_test_wait_cluster(&x_ready[bb], ph)
                                 : mbar_test_wait(&own_ready[bb], ph);
          if (ready && do_dq && nk > 0) ready = mbar_test_wait(&dq_free, (nk - 1) & 1);
          if (ready) {
            tc_fence_after();
            fence_proxy_async();
            const int st = nk % ST;
            const uint32_t sst = smem_u32(smem + LY::OFF_ST + st * LY::STAGE_BYTES);
            if (rank == 0) {
              // dK[:, 0:128] += dS^T Q[:, 0:128]: A = dS^T (exchange buffer, K-major), B = Q
              // half (MN-major: the first two chunks of the stage's Q tile)
              const Desc dsk = make_desc(x_local + bb * LY::X_BYTES, 16, 1024);
              const Desc qmn = make_desc(sst, BM * 128, 1024);
#pragma unroll
              for (int ks = 0; ks < BM / 16; ++ks)
                mma_ss2(tDK, dsk.at(ks * 32), dsk.hi, qmn.at(ks * 2048), qmn.hi, id_acc,
                        (nk > 0 || ks > 0) ? 1u : 0u);
            } else {
              // dK[:, 128:256] += dS^T Q[:, 128:256]: A = dS^T (TMEM), B = the stage's Q half
              const Desc qmn = make_desc(sst + LY::FULL_BYTES, BM * 128, 1024);
              const uint32_t tX = tbase + LY::COL_X0 + bb * BM;
#pragma unroll
              for (int ks = 0; ks < BM / 16; ++ks)
                mma_ts2(tDK, tX + ks * 8, qmn.at(ks * 2048), qmn.hi, id_acc,
                        (nk > 0 || ks > 0) ? 1u : 0u);
            }
            mma_commit(&qdo_empty[st]);
            if (do_dq) {
              // dQ^T[d, q] = sum_kv K[kv, d] dS^T[kv, q], two 128-row halves of d
              const Desc dsn = make_desc(x_local + bb * LY::X_BYTES, kBN * 128, 1024);
#pragma unroll
              for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int ks = 0; ks < kBN / 16; ++ks)
                  mma_ss2(tbase + LY::COL_DQ + hh * BM, kmn.at(2 * hh * (kBN * 128) + ks * 2048),
                          kmn.hi, dsn.at(ks * 2048), dsn.hi, id_dq, ks > 0 ? 1u : 0u);
              mma_commit(&dq_full);
            }
            mma_commit(&x_done[bb]);
            ++nk;
            progressed = true;
          }
        }
        // ---- X(nx): S^T (rank 0) or dP^T (rank 1)
        if (nx < n_iter && nx <= (rank == 0 ? nv : nk) + 1 &&
            mbar_test_wait(&qdo_full[nx % ST], (nx / ST) & 1)) {
          tc_fence_after();
          const Desc bd = make_desc(smem_u32(smem + LY::OFF_ST + (nx % ST) * LY::STAGE_BYTES), 16,
                                    1024);  // Q (rank 0) or dO (rank 1), K-major
          const uint32_t tX = tbase + LY::COL_X0 + (nx & 1) * BM;
#pragma unroll
          for (int ks = 0; ks < HD / 16; ++ks) {
            const uint32_t ko = (ks / 4) * (kBN * 128) + (ks % 4) * 32;
            const uint32_t qo = (ks / 4) * (BM * 128) + (ks % 4) * 32;
            mma_ss2(tX, akv.at(ko), akv.hi, bd.at(qo), bd.hi, id_x, ks > 0 ? 1u : 0u);
          }
          mma_commit(&mine_full[nx & 1]);
          ++nx;
          progressed = true;
        }
        // ---- V(nv): dV half
        if (nv < nx) {
          const int bb = nv & 1;
          const uint32_t ph = (nv >> 1) & 1;
          const bool ready = rank == 0 ? mbar_test_wait(&own_ready[bb], ph)
                                       : mbar_test_wait_cluster(&x_ready[bb], ph);
          if (ready) {
            tc_fence_after();
            fence_proxy_async();
            const int st = nv % ST;
            const uint32_t sst = smem_u32(smem + LY::OFF_ST + st * LY::STAGE_BYTES);
            if (rank == 0) {
              // dV[:, 0:128] += P^T dO[:, 0:128]: A = P^T (TMEM), B = the stage's dO half
              const Desc dmn = make_desc(sst + LY::FULL_BYTES, BM * 128, 1024);
              const uint32_t tX = tbase + LY::COL_X0 + bb * BM;
#pragma unroll
              for (int ks = 0; ks < BM / 16; ++ks)
                mma_ts2(tDV, tX + ks * 8, dmn.at(ks * 2048), dmn.hi, id_acc,
                        (nv > 0 || ks > 0) ? 1u : 0u);
            } else {
              // dV[:, 128:256] += P^T dO[:, 128:256]: A = P^T (exchange buffer, K-major),
              // B = chunks 2, 3 of the stage's dO tile (MN-major)
              const Desc pk = make_desc(x_local + bb * LY::X_BYTES, 16, 1024);
              const Desc dmn = make_desc(sst + 2 * (BM * 128), BM * 128, 1024);
#pragma unroll
              for (int ks = 0; ks < BM / 16; ++ks)
                mma_ss2(tDV, pk.at(ks * 32), pk.hi, dmn.at(ks * 2048), dmn.hi, id_acc,
                        (nv > 0 || ks > 0) ? 1u : 0u);
            }
            ++nv;
            progressed = true;
          }
        }
        if (progressed) {
          spins = 0;
          t_idle = 0;
          continue;
        }
        __nanosleep(32);  // (leave issue slots to the warps that share this scheduler)
        if ((++spins & 63u) == 0 || every_poll) {
          if (*reinterpret_cast<volatile int*>(&wctl.abort)) break;
          const uint64_t now = globaltimer();
          if (t_idle == 0) {
            t_idle = now;
          } else if (now - t_idle > wctl.limit_ns) {
            *reinterpret_cast<volatile int*>(&wctl.abort) = 1;
            break;
          }
        }
      }
      mma_commit(&acc_full);
      mma_commit(&mma_drain);
      mbar_wait_drain(&mma_drain, 0);
    }
  } else if (warp == LY::BULK_WARP && rank == 1) {
    // ------------------------------------------------------------------ rank 1: releases
    // Once rank 1's MMAs of iteration it have read its exchange buffer it % 2 (P^T(it), for dV),
    // the buffer may receive P^T(it + 2): arm that phase, then tell rank 0.
    if (elect_one()) {
      const uint32_t free_peer = mapa_shared(smem_u32(&x_free[0]), peer);
      for (int it = 0; it + 2 < n_iter; ++it) {
        if (!mbar_wait(&x_done[it & 1], (it >> 1) & 1, &wctl)) break;
        mbar_arrive_expect_tx(&x_ready[it & 1], LY::X_BYTES);
        mbar_arrive_remote(free_peer + (it & 1) * 8);
      }
    }
  } else if (warp == LY::BULK_WARP) {
    // ------------------------------------------------------------------ bulk dQ reductions
    if (do_dq && elect_one()) {
      const float* stg = reinterpret_cast<const float*>(smem + LY::OFF_STG);
      for (int it = 0; it < n_iter; ++it) {
        const int h = kh * G + it / nm;
        const int q0 = (m_first + it % nm) * BM;
        const int bh = b * p.H + h;
        bool ok = true;
        for (int hh = 0; hh < 2 && ok; ++hh) {
          const int k = 2 * it + hh;
          ok = mbar_wait(&stg_full, k & 1, &wctl);
          if (!ok) break;
          bulk_reduce_add_f32(p.dqacc + ((size_t)bh * p.ql_pad + q0) * HD + hh * 128 * BM, stg,
                              128 * BM * 4);
          bulk_commit();
          bulk_wait_read<0>();  // the staging tile has been read
          mbar_arrive(&stg_free);
        }
        if (!ok) break;
      }
      bulk_wait<0>();  // every reduction has landed before the CTA exits
    }
  } else if (warp == LY::LINK_WARP) {
    // ------------------------------------------------------------------ sending staged tiles
    // Rank 0 sends P^T(it) from its exchange buffer it % 2 (dS^T(it) from rank 1 lands there
    // afterwards: rank 1 answers only once P^T(it) has arrived) into rank 1's buffer, once rank 1
    // has freed it, after arming its own phase for the answer. Rank 1 sends dS^T(it) from its
    // staging tile; rank 0 has armed the phase before it sent P^T(it), and the staging tile is
    // not rewritten before rank 0 has consumed this one (rank 1 rewrites it only after P^T(it+2)
    // arrives, which rank 0 sends only after its MMAs have read dS^T(it)).
    if (elect_one()) {
      const uint32_t x_peer = mapa_shared(x_local, peer);
      const uint32_t ready_peer = mapa_shared(smem_u32(&x_ready[0]), peer);
      const uint8_t* src0 = smem + (rank == 0 ? LY::OFF_X : LY::OFF_STG);
      for (int it = 0; it < n_iter; ++it) {
        const int bb = it & 1;
        if (!mbar_wait(&out_staged[bb], (it >> 1) & 1, &wctl)) break;
        if (rank == 0) {
          if (it >= 2 && !mbar_wait_cluster(&x_free[bb], ((it - 2) >> 1) & 1, &wctl)) break;
          mbar_arrive_expect_tx(&x_ready[bb], LY::X_BYTES);  // for dS^T(it)
        }
        bulk_copy_to_peer(x_peer + bb * LY::X_BYTES, src0 + bb * LY::X_BYTES, LY::X_BYTES,
                          ready_peer + bb * 8);
        *reinterpret_cast<volatile uint32_t*>(&n_sent) = it + 1;
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------------ P^T or dS^T, epilogue
    const int j = warp * 32 + lane;  // kv row within the tile == TMEM lane
    const int kv = n0 + j;
    const bool kv_live = kv < kl;
    const uint32_t lane_base = tbase + ((uint32_t)(warp * 32) << 16);
    bool ok = true;
    for (int it = 0; it < n_iter && ok; ++it) {
      const int st = it % ST;
      const int bb = it & 1;
      const uint32_t colX = LY::COL_X0 + bb * BM;
      uint32_t pk[BM / 2];  // this row's 64 bf16 results as packed pairs
      ok = __all_sync(0xffffffffu, mbar_wait(&qdo_full[st], (it / ST) & 1, &wctl));
      if (ok)
        ok = __all_sync(0xffffffffu, mbar_wait(&mine_full[bb], (it >> 1) & 1, &wctl));
      if (rank == 0) {
        // P^T(it) from S^T(it): as the single-CTA kernel's P^T warpgroup
        const int h = kh * G + it / nm;
        const int q0 = (m_first + it % nm) * BM;
        const int off = kl - ql;
        const int hi_off = WIN ? p.hi_off : 0;
        const int qlo = kv - off - hi_off - q0;
        const int qhi = WIN ? kv - off - p.lo_off - q0 : BM;
        const bool edge = BAND != kBandNone && !(q0 >= n0 + kBN - 1 - off - hi_off &&
                                                 (!WIN || q0 + BM - 1 <= n0 - off - p.lo_off));
        const bool need_mask = edge || !kv_live;
        const int qcut_lo = !kv_live ? BM : (edge ? qlo : 0);
        const int qcut_hi = edge ? qhi : BM;
        const void* mcol = nullptr;
        if (MASKT != 0 && kv_live) {
          const size_t es = MASKT == 1 ? 4 : MASKT == 2 ? 2 : 1;
          mcol = reinterpret_cast<const uint8_t*>(p.mask) +
                 (b * p.msb + (long long)h * p.msh + (long long)q0 * p.msq + kv) * es;
        }
        if (!ok) break;
        tc_fence_after();
        const float4* sL4 = reinterpret_cast<const float4*>(smem + LY::OFF_L + st * BM * 4);
        const float c2 = p.scale_log2;
        const uint64_t c2v = f2_pack(c2, c2);
        uint32_t rs[2][32];
        tmem_ld32(lane_base + colX, rs[0]);
        tmem_ld32(lane_base + colX + 32, rs[1]);
        tmem_wait_ld();
#pragma unroll
        for (int c32 = 0; c32 < 2; ++c32) {
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
            const uint32_t* r = rs[c32];
            const uint64_t s01 = f2_fma(
                f2_pack(__uint_as_float(r[4 * e4]), __uint_as_float(r[4 * e4 + 1])), c2v, b01);
            const uint64_t s23 = f2_fma(
                f2_pack(__uint_as_float(r[4 * e4 + 2]), __uint_as_float(r[4 * e4 + 3])), c2v, b23);
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
            pk[c32 * 16 + 2 * e4] = pack_bf16(p0, p1);
            pk[c32 * 16 + 2 * e4 + 1] = pack_bf16(p2, p3);
          }
        }
      } else {
        // dS^T(it) = P^T(it) o (dP^T(it) - D): P^T from the exchange buffer (written by rank 0)
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_cluster(&x_ready[bb], (it >> 1) & 1, &wctl));
        if (!ok) break;
        tc_fence_after();
        const float4* sD4 = reinterpret_cast<const float4*>(smem + LY::OFF_D + st * BM * 4);
        uint32_t rd[2][32];
        tmem_ld32(lane_base + colX, rd[0]);
        tmem_ld32(lane_base + colX + 32, rd[1]);
        uint32_t rp[BM / 2];  // P^T bf16 pairs of this row
        const uint8_t* xrow = smem + LY::OFF_X + bb * LY::X_BYTES + j * 128;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint4 v = *reinterpret_cast<const uint4*>(xrow + ((g ^ (j & 7)) << 4));
          rp[4 * g] = v.x;
          rp[4 * g + 1] = v.y;
          rp[4 * g + 2] = v.z;
          rp[4 * g + 3] = v.w;
        }
        tmem_wait_ld();
#pragma unroll
        for (int c32 = 0; c32 < 2; ++c32) {
          const uint32_t* r = rd[c32];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 dd = sD4[c32 * 8 + e4];
            const uint32_t pp0 = rp[c32 * 16 + 2 * e4];
            const uint32_t pp1 = rp[c32 * 16 + 2 * e4 + 1];
            const uint64_t pv01 =
                f2_pack(__uint_as_float(pp0 << 16), __uint_as_float(pp0 & 0xffff0000u));
            const uint64_t pv23 =
                f2_pack(__uint_as_float(pp1 << 16), __uint_as_float(pp1 & 0xffff0000u));
            const uint64_t t01 = f2_add(
                f2_pack(__uint_as_float(r[4 * e4]), __uint_as_float(r[4 * e4 + 1])),
                f2_pack(-dd.x, -dd.y));
            const uint64_t t23 = f2_add(
                f2_pack(__uint_as_float(r[4 * e4 + 2]), __uint_as_float(r[4 * e4 + 3])),
                f2_pack(-dd.z, -dd.w));
            const uint64_t u01 = f2_mul(t01, pv01);
            const uint64_t u23 = f2_mul(t23, pv23);
            float d0, d1, d2, d3;
            f2_unpack(u01, d0, d1);
            f2_unpack(u23, d2, d3);
            pk[c32 * 16 + 2 * e4] = pack_bf16(d0, d1);
            pk[c32 * 16 + 2 * e4 + 1] = pack_bf16(d2, d3);
          }
        }
      }
      // stage row j of the outgoing tile (rank 0: into its exchange buffer bb, once its MMAs
      // have read dS^T(it - 2) there; rank 1: into its staging tile bb) for the link warp
      if (rank == 0 && it >= 2) {
        ok = __all_sync(0xffffffffu, mbar_wait(&x_done[bb], ((it - 2) >> 1) & 1, &wctl));
        if (!ok) break;
      }
      uint8_t* orow = smem + (rank == 0 ? LY::OFF_X : LY::OFF_STG) + bb * LY::X_BYTES + j * 128;
#pragma unroll
      for (int g = 0; g < 8; ++g)
        *reinterpret_cast<uint4*>(orow + ((g ^ (j & 7)) << 4)) =
            make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
      fence_proxy_async();  // generic writes -> visible to the bulk copy
      mbar_arrive(&out_staged[bb]);
      // this CTA's own copy as bf16 over the fp32 tile in TMEM: A operand of its dV (rank 0)
      // or dK (rank 1) MMA
      tmem_st16(lane_base + colX, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
      tmem_st16(lane_base + colX + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&own_ready[bb]);
    }

    // ---------------------------------------------------------------- dK, dV epilogue
    bool have = false;
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(&acc_full, 0, &wctl));
      tc_fence_after();
      have = ok && n_iter > 0;
    }
    const size_t kvrow = kvrow0 + (kv < kl ? kv : 0);
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {
      const uint32_t col = which == 0 ? LY::COL_DV : LY::COL_DK;
      const float mul = which == 0 ? 1.0f : p.scale;
      __nv_bfloat16* out =
          (which == 0 ? p.dv : p.dk) + kvrow * HD + rank * (HD / 2);  // this rank's half
#pragma unroll 1
      for (int c = 0; c < HD / 2; c += 32) {
        uint32_t r[32];
        if (have) {
          tmem_ld32(lane_base + col + c, r);
          tmem_wait_ld();
        }
        uint32_t pkk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pkk[e] = have ? pack_bf16(__uint_as_float(r[2 * e]) * mul,
                                    __uint_as_float(r[2 * e + 1]) * mul)
                        : 0u;
        if (kv < kl) {
          uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[v4] = make_uint4(pkk[4 * v4], pkk[4 * v4 + 1], pkk[4 * v4 + 2], pkk[4 * v4 + 3]);
        }
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------------ rank 0: dQ^T drain
    // lane = head-dim row within a 128-row half, column = query row. Each half is staged as
    // 128 rows of 64 f32 with the 16-byte chunks of row d XOR-rotated by (d & 15), the
    // accumulator's tile layout; the bulk warp adds it with one reduction.
    if (do_dq) {
      const int j = (warp - 4) * 32 + lane;
      const uint32_t lane_base = tbase + ((uint32_t)((warp - 4) * 32) << 16);
      float* stg = reinterpret_cast<float*>(smem + LY::OFF_STG);
      bool ok = true;
      for (int it = 0; it < n_iter && ok; ++it) {
        ok = __all_sync(0xffffffffu, mbar_wait(&dq_full, it & 1, &wctl));
        if (!ok) break;
        tc_fence_after();
        for (int hh = 0; hh < 2; ++hh) {
          const int k = 2 * it + hh;  // use of the staging tile
          uint32_t rq[2][32];
          tmem_ld32(lane_base + LY::COL_DQ + hh * BM, rq[0]);
          tmem_ld32(lane_base + LY::COL_DQ + hh * BM + 32, rq[1]);
          tmem_wait_ld();
          if (hh == 1) {  // both halves are in registers: the TMEM tile is free
            tc_fence_before();
            mbar_arrive(&dq_free);
          }
          if (k > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&stg_free, (k - 1) & 1, &wctl));
            if (!ok) break;
          }
          float4* row = reinterpret_cast<float4*>(stg + j * BM);
#pragma unroll
          for (int c = 0; c < BM / 4; ++c) {  // chunk c: query rows 4c .. 4c+3
            const uint32_t* r = &rq[c / 8][(c % 8) * 4];
            row[c ^ (j & (kDqChunks - 1))] =
                make_float4(__uint_as_float(r[0]), __uint_as_float(r[1]), __uint_as_float(r[2]),
                            __uint_as_float(r[3]));
          }
          fence_proxy_async();  // staging writes -> visible to the bulk copy
          mbar_arrive(&stg_full);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == LY::MMA_WARP) tmem_dealloc(tbase, LY::TMEM_COLS);
  // Neither CTA leaves while the other may still write into its shared memory or arrive on
  // its barriers: after both have left their loops, each lets the tiles the other sent land
  // (normally already consumed; after a bounded wait ran out perhaps not), then both leave.
  cluster_sync_all();
  if (threadIdx.x == 0) {
    const int sent = (int)ld_cluster_u32(mapa_shared(smem_u32(&n_sent), peer));
    for (int it = sent - 2 < 0 ? 0 : sent - 2; it < sent; ++it)
      mbar_wait_drain(&x_ready[it & 1], (it >> 1) & 1);
  }
  cluster_sync_all();
  if (threadIdx.x == 0) report_abort(&wctl, p.status);
}

// ------------------------------------------------------------------------ host side
template <int BAND, int MASKT, bool VARLEN>
static cudaError_t launch_pair_t(const BwdArgs& a, const BwdMaps& m, cudaStream_t s) {
  using LY = PairLayout;
  auto kern = bwd_pair_kernel<BAND, MASKT, VARLEN>;
  static OncePerKey<> smem_attr;  // per instantiation and device
  {
    const cudaError_t e = set_smem_once(smem_attr, kern, LY::SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  BwdKParams kp = make_bwd_kparams(a);
  const int groups = a.B * a.Hk, ktiles = (a.kl + kBN - 1) / kBN;
  kp.tiles_fast = a.cu_q != nullptr && groups <= 65535;  // (grid y limit)
  dim3 grid(kp.tiles_fast ? 2 * ktiles : 2 * groups, kp.tiles_fast ? groups : ktiles);
  profile_mark(kKernBwdMain, 0, s);
  kern<<<grid, LY::THREADS, LY::SMEM_BYTES, s>>>(m.q, m.k, m.v, m.dO, kp);
  cudaError_t e = cudaGetLastError();
  profile_mark(kKernBwdMain, 1, s);
  return e;
}

template <int BAND>
static cudaError_t launch_pair_m(const BwdArgs& a, const BwdMaps& m, cudaStream_t s) {
  if (a.cu_q) return launch_pair_t<BAND, 0, true>(a, m, s);  // (no mask with varlen)
  if (!a.mask) return launch_pair_t<BAND, 0, false>(a, m, s);
  switch (a.mask_type) {
    case 0: return launch_pair_t<BAND, 1, false>(a, m, s);
    case 1: return launch_pair_t<BAND, 2, false>(a, m, s);
    default: return launch_pair_t<BAND, 3, false>(a, m, s);
  }
}

cudaError_t launch_bwd_pair(const BwdArgs& a, const BwdMaps& m, cudaStream_t s) {
  if (a.d != kPD || a.dval != kPD) return cudaErrorInvalidValue;
  switch (a.band) {
    case kBandNone: return launch_pair_m<kBandNone>(a, m, s);
    case kBandCausal: return launch_pair_m<kBandCausal>(a, m, s);
    default: return launch_pair_m<kBandWindow>(a, m, s);
  }
}

}  // namespace fa
