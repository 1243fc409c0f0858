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
// one CTA. Two CTAs that each owned one half of the head dimension would both have to form S^T
// and dP^T (2 of the 5 contractions twice), with K, V, Q and dO filling their shared memory.
// Here the two CTAs of a cluster split the work by what they multiply:
//   rank 0 holds K: S^T, P^T, all of dV (A = its own P^T in TMEM) and head-dim rows 0-127
//   of dQ^T;
//   rank 1 holds V and the upper half of K: dP^T, dS^T, all of dK (A = its own dS^T in TMEM)
//   and head-dim rows 128-255 of dQ^T.
// The dQ^T split matters because one SM pushes only ~30-50 GB/s of f32 reductions towards L2
// (measured on a GB300 with 38, 76 and 152 SMs pushing at once: the rate per SM is the same).
// With all 64 KB of a step's dQ^T on rank 0, that push, not the tensor core, set the step
// time.
// The two tiles each rank needs from the other travel through shared memory: rank 0 stages
// P^T in its exchange buffer and sends it with one bulk copy (cp.async.bulk shared::cta to
// shared::cluster) that completes a transaction on rank 1's barrier; rank 1 computes dS^T,
// writes it over P^T in the same buffer and sends it back the same way. (128 threads storing
// their rows into the other CTA directly measured 1.3-2 us per tile.) Each rank's Q/dO stage is
// read only by its own MMAs, so rank 0 frees it once dV is issued, without waiting for rank 1.
// Buffer reuse: rank 0 stages P^T(it + 2) in its buffer only after its dQ MMAs have read
// dS^T(it) there. Rank 0 sends P^T(it + 2) into rank 1's buffer only after rank 1's dQ MMAs
// have read dS^T(it) from it: rank 1 tells it with a remote arrive once they complete. Rank 1
// read P^T(it) there before writing dS^T(it) over it, so the buffer is free.
//
// Roles (384 threads): warps 0-3 compute P^T (rank 0) or dS^T (rank 1), one kv row per thread
// (= TMEM lane), and write that rank's dV or dK at the end. Warps 4-7 drain this rank's half of
// dQ^T from TMEM. On rank 0 they stage it for warp 11, which adds it to the f32 accumulator
// with a bulk reduction. On rank 1, whose shared memory holds the K half instead of a staging
// tile, they add it with 16-byte vector reductions. Warp 8 issues the TMA loads (one lane per
// ring). Warp 9 issues the MMAs, polling the barriers of its rank's MMA groups so that
// whichever is ready goes first. Warp 10 sends the staged tiles. Every wait is bounded.
#include "fa_bwd_common.cuh"

namespace fa {

namespace {
constexpr int kPM = 64;   // query rows per tile (N of S^T and dP^T; K of dV and dK)
constexpr int kPD = 256;  // head dim of q, k, v and dO
constexpr int kPST = 2;   // depth of the Q / dO ring
}  // namespace

// One shared-memory layout for both ranks; what a region holds depends on the rank.
struct PairLayout {
  static constexpr int KV_BYTES = kBN * kPD * 2;    // K (rank 0) or V (rank 1), 64 KB
  static constexpr int TILE_BYTES = kPM * kPD * 2;  // one 64 x 256 bf16 tile, 32 KB
  static constexpr int X_BYTES = kBN * kPM * 2;     // a [kv][q] bf16 exchange tile, 16 KB
  static constexpr int STG_BYTES = 128 * kPM * 4;   // rank 0: half a dQ^T tile in f32, 32 KB
  static constexpr int KH_BYTES = kBN * 128 * 2;     // rank 1: K columns 128-255, 32 KB
  // Two rings with the lifetimes of their operands: F holds the tile that only S^T / dP^T read
  // (rank 0: Q; rank 1: dO), freed as soon as that MMA completes, so one stage suffices; R
  // holds the tile that dV / dK read (rank 0: dO; rank 1: Q) and the row vector the P^T / dS^T
  // warps read (-L log2(e) or D), freed after dV / dK, two stages.
  static constexpr int OFF_KV = 0;
  static constexpr int OFF_F = OFF_KV + KV_BYTES;           // 1 stage
  static constexpr int OFF_R = OFF_F + TILE_BYTES;          // kPST stages
  static constexpr int OFF_X = OFF_R + kPST * TILE_BYTES;   // 2 exchange buffers
  static constexpr int OFF_STG = OFF_X + 2 * X_BYTES;       // rank 0: dQ^T staging; rank 1: K half
  static constexpr int OFF_LD = OFF_STG + STG_BYTES;        // kPST x kPM f32 (ring R)
  static constexpr int OFF_END = OFF_LD + kPST * kPM * 4;
  static constexpr int SMEM_BYTES = OFF_END + 1024;
  // TMEM columns: two 64-column buffers (rank 0: S^T then P^T as bf16; rank 1: dP^T then dS^T),
  // two 64-column buffers for this rank's 128-row half of dQ^T (one per step parity), and the
  // 256-column accumulator (rank 0: dV; rank 1: dK).
  static constexpr int COL_X0 = 0;
  static constexpr int COL_DQ = 128;
  static constexpr int COL_ACC = 256;
  static constexpr int TMEM_COLS = 512;
  static constexpr int THREADS = 384;
  static constexpr int TMA_WARP = 8, MMA_WARP = 9, LINK_WARP = 10, BULK_WARP = 11;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(KH_BYTES == STG_BYTES, "rank 1 keeps its K half where rank 0 stages dQ^T");
  static_assert(kPM / 4 == kDqChunks, "dQ^T tile layout of the accumulator");
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
  __shared__ uint64_t kv_full, f_full, f_empty, r_full[ST], r_empty[ST];
  __shared__ uint64_t mine_full[2];   // rank 0: S^T(it) in TMEM; rank 1: dP^T(it)
  __shared__ uint64_t own_ready[2];   // 128 arrivals: P^T (0) / dS^T (1) written to TMEM as bf16
  __shared__ uint64_t x_ready[2];     // the peer's tile has landed in x buffer (bulk-copy bytes)
  __shared__ uint64_t x_done[2];      // rank 0: its dQ MMAs have read dS^T in x buffer
  __shared__ uint64_t out_staged[2];  // 128 arrivals: this rank's outgoing tile is in x buffer
  __shared__ uint64_t dq_full[2], dq_free[2];  // this rank's dQ^T half in TMEM buffer it % 2
  __shared__ uint64_t peer_read[2];  // rank 0: rank 1's dQ MMAs have read dS^T in its x buffer
  __shared__ uint64_t stg_full, stg_free, acc_full, mma_drain;
  __shared__ uint32_t n_sent;         // tiles sent to the peer (read by the peer at the end)
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
  int krow0 = 0, qrow0 = 0;
  int kb = b, krows = p.kl;  // dK / dV: batch and rows of this problem (row of key 0: krow0)
  if constexpr (VARLEN) {
    int qs, ks;
    const bool bad = varlen_seq(p.cu_q, b, p.total_q, p.ql, qs, ql) |
                     varlen_seq(p.cu_k, b, p.total_k, p.kl, ks, kl);
    if (bad && threadIdx.x == 0 && rank == 0 && p.status)
      atomicCAS(p.status, kStatusOk, kStatusBadInput);
    krow0 = ks;
    qrow0 = qs;
    kb = 0;
    krows = p.total_k;
  }
  if (n0 >= kl) return;  // a kv tile past this sequence's keys: both CTAs of the pair leave
  int m_first, m_last;
  bwd_mtile_range<HD, BAND>(n0, p, ql, kl, m_first, m_last);
  const int nm = m_last - m_first + 1;  // query tiles per head (0 if none)
  const int n_iter = G * nm;            // (head, query tile) pairs this pair of CTAs visits
  const bool do_dq = !p.skip_dq;  // both ranks form and add a half of dQ^T

  if (threadIdx.x == 0) {
    wait_ctl_init(&wctl, p.wait_limit_ns);
    mbar_init(&kv_full, 1);
    mbar_init(&f_full, 1);
    mbar_init(&f_empty, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&r_full[s], 1);
      mbar_init(&r_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&mine_full[s], 1);
      mbar_init(&own_ready[s], 128);
      mbar_init(&x_ready[s], 1);
      mbar_init(&x_done[s], 1);
      mbar_init(&out_staged[s], 128);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&dq_full[s], 1);
      mbar_init(&dq_free[s], 128);
      mbar_init(&peer_read[s], 1);
    }
    mbar_init(&stg_full, 128);
    mbar_init(&stg_free, 1);
    mbar_init(&acc_full, 1);
    mbar_init(&mma_drain, 1);
    n_sent = 0;
    // every phase of x_ready expects one tile; it is armed before that tile can be sent: rank 1
    // arms P^T(0), P^T(1) here and P^T(it + 2) before it sends dS^T(it); rank 0 arms dS^T(it)
    // before it sends P^T(it)
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
  cluster_sync_all();  // the peer's barriers are initialised before any copy reaches them
  const uint32_t tbase = tmem_base_s;
  const uint32_t x_local = smem_u32(smem + LY::OFF_X);

  if (warp == LY::TMA_WARP) {
    // ------------------------------------------------------------------ TMA producers
    // lane 0: K or V, then ring F; lane 1: ring R (each waits only on its own ring)
    const CUtensorMap* mkv = rank == 0 ? &mK : &mV;
    const CUtensorMap* mfirst = rank == 0 ? &mQ : &mDO;   // read by S^T / dP^T (ring F)
    const CUtensorMap* msecond = rank == 0 ? &mDO : &mQ;  // read by dV / dK (ring R)
    const float* ld_src = rank == 0 ? p.lse2 : p.dvec;    // -L log2(e) (P^T) or D (dS^T)
    if (lane == 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mV);
      tma_prefetch_desc(&mDO);
      const bool k_half = rank == 1 && do_dq;  // rank 1's dQ^T rows need K columns 128-255
      mbar_arrive_expect_tx(&kv_full, LY::KV_BYTES + (k_half ? LY::KH_BYTES : 0));
      for (int c = 0; c < HD / 64; ++c)
        tma_load_bh(smem + LY::OFF_KV + c * kBN * 128, mkv, &kv_full, c * 64, krow0 + n0, kh, kb,
                    p.Hk, p.kv_bshd != 0);
      if (k_half)
        for (int c = 2; c < HD / 64; ++c)
          tma_load_bh(smem + LY::OFF_STG + (c - 2) * kBN * 128, &mK, &kv_full, c * 64,
                      krow0 + n0, kh, kb, p.Hk, p.kv_bshd != 0);
      int loaded = 0;
      for (int it = 0; it < n_iter; ++it) {
        if (it >= 1 && !mbar_wait(&f_empty, (it - 1) & 1, &wctl)) break;
        const int h = kh * G + it / nm;
        const int q0 = (m_first + it % nm) * BM;
        mbar_arrive_expect_tx(&f_full, LY::TILE_BYTES);
        for (int c = 0; c < HD / 64; ++c)
          tma_load_bh(smem + LY::OFF_F + c * BM * 128, mfirst, &f_full, c * 64, qrow0 + q0, h,
                      kb, p.H, p.q_bshd != 0);
        loaded = it + 1;
      }
      mbar_wait_drain(&kv_full, 0);
      if (loaded > 0) mbar_wait_drain(&f_full, (loaded - 1) & 1);
    } else if (lane == 1) {
      int last_use[ST];
      for (int s = 0; s < ST; ++s) last_use[s] = -1;
      for (int it = 0; it < n_iter; ++it) {
        const int st = it % ST;
        const uint32_t use = it / ST;
        if (it >= ST && !mbar_wait(&r_empty[st], (use - 1) & 1, &wctl)) break;
        const int h = kh * G + it / nm;
        const int q0 = (m_first + it % nm) * BM;
        const int bh = b * p.H + h;
        mbar_arrive_expect_tx(&r_full[st], LY::TILE_BYTES + BM * 4);
        for (int c = 0; c < HD / 64; ++c)
          tma_load_bh(smem + LY::OFF_R + st * LY::TILE_BYTES + c * BM * 128, msecond, &r_full[st],
                      c * 64, qrow0 + q0, h, kb, p.H, p.q_bshd != 0);
        bulk_load(smem + LY::OFF_LD + st * BM * 4, ld_src + (size_t)bh * p.ql_pad + q0, BM * 4,
                  &r_full[st]);
        last_use[st] = it;
      }
      for (int s = 0; s < ST; ++s)
        if (last_use[s] >= 0) mbar_wait_drain(&r_full[s], (last_use[s] / ST) & 1);
    }
  } else if (warp == LY::MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    // Groups of iteration it: X(it) = S^T (rank 0) or dP^T (rank 1) into TMEM buffer it % 2;
    // A(it) = dV += P^T dO (rank 0) or dK += dS^T Q (rank 1), A from this rank's TMEM;
    // Q(it) = this rank's 128-row half of dQ^T from dS^T in exchange buffer it % 2 (rank 0: as
    // received from rank 1; rank 1: its own, once staged). X(i) needs its stage and its TMEM
    // buffer (A(i - 2) issued: MMAs of one thread run in issue order); A(i) needs X(i) issued
    // and this rank's P^T / dS^T(i), and releases the stage; Q(i) needs dS^T(i) and the drain
    // of Q(i - 2), which used the same TMEM buffer.
    if (elect_one()) {
      const uint32_t sKV = smem_u32(smem + LY::OFF_KV);
      const Desc akv = make_desc(sKV, 16, 1024);          // K or V as a K-major operand
      // K columns 0-127 (rank 0) or 128-255 (rank 1) as the MN-major A operand of dQ^T
      const Desc kq = make_desc(rank == 0 ? sKV : smem_u32(smem + LY::OFF_STG), kBN * 128, 1024);
      const uint32_t id_x = idesc_bf16(128, BM, 0, 0);    // S^T, dP^T: [kv x q]
      const uint32_t id_acc = idesc_bf16(128, HD, 0, 1);  // dV, dK: A tmem, B MN-major, N = 256
      const uint32_t id_dq = idesc_bf16(128, BM, 1, 1);   // dQ^T half: [d x q], K = kv
      const uint32_t tACC = tbase + LY::COL_ACC;
      bool ok = mbar_wait(&kv_full, 0, &wctl);
      // (rank 0 runs the Q group in the deterministic mode too, without dQ MMAs: its commit
      // still tells the P^T warps that the exchange buffer has been read back)
      int nx = 0, na = 0, nq = (rank == 0 || do_dq) ? 0 : n_iter;
      const bool every_poll = wctl.limit_ns < 100000ull;
      uint64_t t_idle = 0;
      uint32_t spins = 0;
      while (ok && (na < n_iter || nq < n_iter)) {
        bool progressed = false;
        // ---- Q(nq): dQ^T rows of this rank's half = K^T dS^T
        if (nq < n_iter && (rank == 1 || nq < na)) {
          const int bb = nq & 1;
          bool ready = rank == 0 ? mbar_test_wait_cluster(&x_ready[bb], (nq >> 1) & 1)
                                 : mbar_test_wait(&out_staged[bb], (nq >> 1) & 1);
          if (ready && do_dq && nq >= 2)
            ready = mbar_test_wait(&dq_free[bb], ((nq - 2) >> 1) & 1);
          if (ready) {
            tc_fence_after();
            fence_proxy_async();
            if (do_dq) {
              const Desc dsn = make_desc(x_local + bb * LY::X_BYTES, kBN * 128, 1024);
#pragma unroll
              for (int ks = 0; ks < kBN / 16; ++ks)
                mma_ss2(tbase + LY::COL_DQ + bb * BM, kq.at(ks * 2048), kq.hi, dsn.at(ks * 2048),
                        dsn.hi, id_dq, ks > 0 ? 1u : 0u);
              mma_commit(&dq_full[bb]);
            }
            // rank 0: the P^T warps may stage P^T(nq + 2) in this buffer (rank 1 learns that
            // its buffer has been read from its drain warps, which wait for dq_full)
            if (rank == 0) mma_commit(&x_done[bb]);
            ++nq;
            progressed = true;
          }
        }
        // ---- X(nx): S^T (rank 0) or dP^T (rank 1)
        if (nx < n_iter && nx <= na + 1 && mbar_test_wait(&f_full, nx & 1)) {
          tc_fence_after();
          const Desc bd = make_desc(smem_u32(smem + LY::OFF_F), 16, 1024);  // Q or dO, K-major
          const uint32_t tX = tbase + LY::COL_X0 + (nx & 1) * BM;
#pragma unroll
          for (int ks = 0; ks < HD / 16; ++ks) {
            const uint32_t ko = (ks / 4) * (kBN * 128) + (ks % 4) * 32;
            const uint32_t qo = (ks / 4) * (BM * 128) + (ks % 4) * 32;
            mma_ss2(tX, akv.at(ko), akv.hi, bd.at(qo), bd.hi, id_x, ks > 0 ? 1u : 0u);
          }
          mma_commit(&mine_full[nx & 1]);
          mma_commit(&f_empty);  // ring F is free once this MMA has read it
          ++nx;
          progressed = true;
        }
        // ---- A(na): dV (rank 0) or dK (rank 1), accumulated over every iteration
        if (na < nx && mbar_test_wait(&own_ready[na & 1], (na >> 1) & 1) &&
            mbar_test_wait(&r_full[na % ST], (na / ST) & 1)) {
          tc_fence_after();
          const int st = na % ST;
          // B = dO (rank 0) or Q (rank 1) from ring R, MN-major, N = 256
          const Desc bmn = make_desc(smem_u32(smem + LY::OFF_R + st * LY::TILE_BYTES), BM * 128,
                                     1024);
          const uint32_t tX = tbase + LY::COL_X0 + (na & 1) * BM;
#pragma unroll
          for (int ks = 0; ks < BM / 16; ++ks)
            mma_ts2(tACC, tX + ks * 8, bmn.at(ks * 2048), bmn.hi, id_acc,
                    (na > 0 || ks > 0) ? 1u : 0u);
          mma_commit(&r_empty[st]);  // ring R's last reader on this rank
          ++na;
          progressed = true;
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
  } else if (warp == LY::LINK_WARP) {
    // ------------------------------------------------------------------ sending staged tiles
    if (elect_one()) {
      const uint32_t x_peer = mapa_shared(x_local, peer);
      const uint32_t ready_peer = mapa_shared(smem_u32(&x_ready[0]), peer);
      for (int it = 0; it < n_iter; ++it) {
        const int bb = it & 1;
        if (!mbar_wait(&out_staged[bb], (it >> 1) & 1, &wctl)) break;
        // rank 1 reads dS^T(it - 2) from the buffer P^T(it) lands in, for its own dQ MMAs
        if (rank == 0 && do_dq && it >= 2 &&
            !mbar_wait_cluster(&peer_read[bb], ((it - 2) >> 1) & 1, &wctl))
          break;
        if (rank == 0)
          mbar_arrive_expect_tx(&x_ready[bb], LY::X_BYTES);  // dS^T(it) will come back
        else if (it + 2 < n_iter)
          mbar_arrive_expect_tx(&x_ready[bb], LY::X_BYTES);  // P^T(it + 2) may follow
        bulk_copy_to_peer(x_peer + bb * LY::X_BYTES, smem + LY::OFF_X + bb * LY::X_BYTES,
                          LY::X_BYTES, ready_peer + bb * 8);
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
      uint8_t* xrow = smem + LY::OFF_X + bb * LY::X_BYTES + j * 128;
      uint32_t pk[BM / 2];  // this row's 64 bf16 results as packed pairs
      ok = __all_sync(0xffffffffu, mbar_wait(&r_full[st], (it / ST) & 1, &wctl));
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
        const float4* sL4 = reinterpret_cast<const float4*>(smem + LY::OFF_LD + st * BM * 4);
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
        // P^T to TMEM first (this rank's dV and the release of its stage need only that),
        // then to the exchange buffer, which holds dS^T(it - 2) until the dQ MMAs have read it
        tmem_st16(lane_base + colX, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
        tmem_st16(lane_base + colX + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&own_ready[bb]);
        if (it >= 2) {
          ok = __all_sync(0xffffffffu, mbar_wait(&x_done[bb], ((it - 2) >> 1) & 1, &wctl));
          if (!ok) break;
        }
      } else {
        // dS^T(it) = P^T(it) o (dP^T(it) - D): P^T from the exchange buffer (written by rank 0)
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_cluster(&x_ready[bb], (it >> 1) & 1, &wctl));
        if (!ok) break;
        tc_fence_after();
        const float4* sD4 = reinterpret_cast<const float4*>(smem + LY::OFF_LD + st * BM * 4);
        uint32_t rd[2][32];
        tmem_ld32(lane_base + colX, rd[0]);
        tmem_ld32(lane_base + colX + 32, rd[1]);
        uint32_t rp[BM / 2];  // P^T bf16 pairs of this row
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
      // the outgoing tile: row j of the exchange buffer (rank 1: over its own P^T(it) row,
      // already read), sent by the link warp
#pragma unroll
      for (int g = 0; g < 8; ++g)
        *reinterpret_cast<uint4*>(xrow + ((g ^ (j & 7)) << 4)) =
            make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
      fence_proxy_async();  // generic writes -> visible to the bulk copy
      mbar_arrive(&out_staged[bb]);
      if (rank == 1) {
        // dS^T as bf16 over dP^T in TMEM: A operand of this rank's dK MMA
        tmem_st16(lane_base + colX, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
        tmem_st16(lane_base + colX + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&own_ready[bb]);
      }
    }

    // ---------------------------------------------------------------- dV (0) / dK (1) epilogue
    bool have = false;
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(&acc_full, 0, &wctl));
      tc_fence_after();
      have = ok && n_iter > 0;
    }
    const long long kvr = krow0 + (kv < kl ? kv : 0);  // row of this key in dK / dV
    const float mul = rank == 0 ? 1.0f : p.scale;
    __nv_bfloat16* out =
        (rank == 0 ? p.dv : p.dk) + bhsd_offset(kb, kh, kvr, p.Hk, krows, HD, p.kv_bshd != 0);
#pragma unroll 1
    for (int c = 0; c < HD; c += 32) {
      uint32_t r[32];
      if (have) {
        tmem_ld32(lane_base + LY::COL_ACC + c, r);
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
  } else if (warp < 8) {
    // ------------------------------------------------------------------ dQ^T drain
    // lane = head-dim row d within this rank's 128-row half, column = query row. The
    // accumulator keeps each (head, query tile) as two chunk-major halves: the 16-byte chunk c
    // (query rows 4c .. 4c+3) of row d at position (d / 128) * 2048 + c * 128 + d % 128, which
    // the dQ convert kernel reads. Rank 0 stages its half in that layout (32 consecutive lanes
    // store 512 contiguous bytes) and the bulk warp adds it with one reduction. Rank 1 has no
    // staging tile (its shared memory holds the K half) and adds each chunk with a 16-byte
    // vector reduction, a warp covering 512 contiguous bytes per instruction.
    if (do_dq) {
      const int j = (warp - 4) * 32 + lane;
      const uint32_t lane_base = tbase + ((uint32_t)((warp - 4) * 32) << 16);
      float* stg = reinterpret_cast<float*>(smem + LY::OFF_STG);
      bool ok = true;
      for (int it = 0; it < n_iter && ok; ++it) {
        const int bb = it & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(&dq_full[bb], (it >> 1) & 1, &wctl));
        if (!ok) break;
        // rank 1: its dQ MMAs have read dS^T(it) from its exchange buffer; rank 0 may send
        // P^T(it + 2) into it
        if (rank == 1 && threadIdx.x == 128)
          mbar_arrive_remote(mapa_shared(smem_u32(&peer_read[bb]), 0));
        tc_fence_after();
        uint32_t rq[2][32];
        tmem_ld32(lane_base + LY::COL_DQ + bb * BM, rq[0]);
        tmem_ld32(lane_base + LY::COL_DQ + bb * BM + 32, rq[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&dq_free[bb]);  // the TMEM buffer may take dQ^T(it + 2)
        if (rank == 0) {
          if (it > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&stg_free, (it - 1) & 1, &wctl));
            if (!ok) break;
          }
          float4* s4 = reinterpret_cast<float4*>(stg);
#pragma unroll
          for (int c = 0; c < BM / 4; ++c) {
            const uint32_t* r = &rq[c / 8][(c % 8) * 4];
            s4[c * 128 + j] = make_float4(__uint_as_float(r[0]), __uint_as_float(r[1]),
                                          __uint_as_float(r[2]), __uint_as_float(r[3]));
          }
          fence_proxy_async();  // staging writes -> visible to the bulk copy
          mbar_arrive(&stg_full);
        } else {
          const int h = kh * G + it / nm;
          const int q0 = (m_first + it % nm) * BM;
          const int bh = b * p.H + h;
          float4* half1 = reinterpret_cast<float4*>(p.dqacc + ((size_t)bh * p.ql_pad + q0) * HD) +
                          128 * kDqChunks;
#pragma unroll
          for (int c = 0; c < BM / 4; ++c) {
            const uint32_t* r = &rq[c / 8][(c % 8) * 4];
            atomicAdd(half1 + c * 128 + j,
                      make_float4(__uint_as_float(r[0]), __uint_as_float(r[1]),
                                  __uint_as_float(r[2]), __uint_as_float(r[3])));
          }
        }
      }
    }
  } else if (warp == LY::BULK_WARP) {
    // ------------------------------------------------------------------ rank 0: dQ reductions
    if (rank == 0 && do_dq && elect_one()) {
      const float* stg = reinterpret_cast<const float*>(smem + LY::OFF_STG);
      for (int it = 0; it < n_iter; ++it) {
        const int h = kh * G + it / nm;
        const int q0 = (m_first + it % nm) * BM;
        const int bh = b * p.H + h;
        if (!mbar_wait(&stg_full, it & 1, &wctl)) break;
        bulk_reduce_add_f32(p.dqacc + ((size_t)bh * p.ql_pad + q0) * HD, stg, 128 * BM * 4);
        bulk_commit();
        bulk_wait_read<0>();  // the staging tile has been read
        mbar_arrive(&stg_free);
      }
      bulk_wait<0>();  // every reduction has landed before the CTA exits
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
