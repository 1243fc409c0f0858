// fa_fwd.cu -- forward kernel: O = softmax(scale * Q K^T + mask) V and the natural-log
// logsumexp L, one launch, sm_103a.
//
// Method: the online softmax of the mlx-native training forward (page "mlx-native
// tests/test_flash_attn_train.rs", `sdpa_reference_with_logsumexp`): scores taken to base 2 by
// multiplying the f32 dot product with scale*log2(e) and the mask with log2(e), a running row
// maximum that starts at the finite sentinel -FLT_MAX/2, p = exp2(s - max), and at the end
// L = max * ln(2) + ln(sum p), O = (sum p v) / sum p, with O = 0 and L = -inf for a row that
// sees no key. Causal masking is bottom-right: key j is visible to query row i iff
// j <= kl - ql + i.
//
// GB300 design:
//  * a CTA owns NQ query tiles of 128 rows of one (batch, head); each tile has its own
//    softmax warpgroup, in which thread r owns query row r: tcgen05.ld hands every thread one
//    full TMEM lane, so row maxima and sums need no shuffles;
//  * one warp streams K and V tiles with TMA (128-byte swizzle) through a STAGES-deep ring;
//  * one warp issues the tcgen05 MMAs: S = Q K^T into TMEM (both operands K-major in shared
//    memory) and O += P V with P read straight from TMEM (the softmax warps overwrite S with
//    P as packed bf16) and V MN-major in shared memory; O accumulates in TMEM in f32;
//  * the two query tiles ping-pong: while one warpgroup runs its softmax, the tensor core
//    works on the other tile's MMAs;
//  * O is rescaled lazily: the running maximum used for the exponentials is only moved when
//    the true maximum exceeds it by more than 8 (a factor 256), so most tiles skip the O
//    round trip through TMEM. The result is the same sum: O and the row sum are scaled by the
//    same 2^-m_used, which cancels in O / sum and is added back in L;
//  * with causal masking, key tiles that lie wholly above a query tile's diagonal are never
//    loaded or multiplied, and the CTAs with the most work are launched first.
#include <float.h>
#include "fa_band.cuh"
#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {

constexpr int kBM = 128;  // query rows per tile (the MMA M)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 of the largest p before O is rescaled

template <int HD>
struct FwdTraits;
// NQ query tiles per CTA, BN keys per kv tile, NS score buffers per query tile, STAGES-deep
// K/V ring. POLY: pair e of each 16-pair group of exponentials goes to the FMA-pipe
// polynomial when e % POLY == 0 (0 = all on MUFU, 16 or more = one pair in 16). A small share
// relieves the MUFU queue (16 exp2 per clock per SM); a larger one costs the softmax warps
// issue slots (measured best: 16 at head_dim 64 and 128). SPLIT: S = Q K^T and O += P V are
// issued by two warps (a busy scheduler starves a lone issuing thread less often when the
// two streams do not wait behind each other's barriers). S into a score buffer then waits for
// the completion of the P V that read it, not just for its issue: with one score buffer per
// tile (NS = 1) that wait is on the critical path (measured at head_dim 128: 230 -> 272 us on
// the 4k causal GQA shape), with two it is hidden (head_dim 256: 125 -> 121 us).
template <>
struct FwdTraits<64> {
  static constexpr int NQ = 2, BN = 128, NS = 1, STAGES = 3, POLY = 16;
  static constexpr bool SPLIT = false;
};
template <>
struct FwdTraits<128> {
  static constexpr int NQ = 2, BN = 128, NS = 1, STAGES = 2, POLY = 16;
  static constexpr bool SPLIT = false;
};
template <>
struct FwdTraits<256> {
  static constexpr int NQ = 1, BN = 64, NS = 2, STAGES = 2, POLY = 0;
  static constexpr bool SPLIT = true;
};

// HD: head dim of Q and K; DV: head dim of V and O (the value head dim).
template <int HD, int DV>
struct FwdLayout {
  using T = FwdTraits<HD>;
  static constexpr int KCH = HD / 64;                         // 128-byte column chunks of Q, K
  static constexpr int VCH = DV / 64;                         // ... of V
  static constexpr int Q_TILE_BYTES = kBM * HD * 2;
  static constexpr int K_TILE_BYTES = T::BN * HD * 2;
  static constexpr int V_TILE_BYTES = T::BN * DV * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + T::NQ * Q_TILE_BYTES;
  static constexpr int OFF_V = OFF_K + T::STAGES * K_TILE_BYTES;
  static constexpr int OFF_END = OFF_V + T::STAGES * V_TILE_BYTES;
  static constexpr int SMEM_BYTES = OFF_END + 1024;  // + alignment slack
  // TMEM columns of tile t: O at t*TILE_COLS, S buffer s at t*TILE_COLS + DV + s*BN.
  static constexpr int TILE_COLS = DV + T::NS * T::BN;
  static constexpr int TMEM_COLS_USED = T::NQ * TILE_COLS;
  static constexpr int TMEM_COLS = TMEM_COLS_USED <= 256 ? 256 : 512;
  // softmax warpgroups + TMA + MMA warps (with SPLIT: MMA_WARP issues S, MMA2_WARP P V)
  static constexpr int THREADS = T::NQ * 128 + (T::SPLIT ? 96 : 64);
  static constexpr int TMA_WARP = T::NQ * 4;
  static constexpr int MMA_WARP = T::NQ * 4 + 1;
  static constexpr int MMA2_WARP = T::NQ * 4 + 2;
  // two CTAs per SM when both fit (TMEM and shared memory), else one
  static constexpr int MIN_BLOCKS = (TMEM_COLS <= 256 && SMEM_BYTES <= 113 * 1024) ? 2 : 1;
  static_assert(TMEM_COLS_USED <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

struct FwdKParams {
  const void* mask;  // additive f32 / bf16, or bool (uint8), addressed with the strides below
  long long msb, msh, msq;  // mask strides (elements) of batch, head, query row; keys contiguous
  __nv_bfloat16* o;
  float* lse;
  const float* sinks;  // [H] natural-log sink logits, or nullptr
  const int32_t* cu_q;  // variable-length batch: sequence offsets, or nullptr
  const int32_t* cu_k;
  int total_q, total_k;
  int q_bshd, kv_bshd;  // 1: q, o / k, v are [batch, rows, heads, d] (else [b, heads, rows, d])
  int* status;
  int H, Hk, ql, kl, n_mblk;  // ql, kl: the longest sequence in a variable-length batch
  int tiles_fast;  // 1: blockIdx.x = query tile, y = (batch, head); 0: the other way round
  int lo_off, hi_off;  // key j is visible to row i iff q_abs + lo_off <= j <= q_abs + hi_off
  float scale_log2;    // scale * log2(e)
  unsigned long long wait_limit_ns;  // limit of one barrier wait
};

// Mask value of key column `j` for the row whose mask row starts at `mrow`, as a base-2
// additive term (0 or -inf for bool masks).
template <int MASKT>
__device__ __forceinline__ float mask_log2(const void* mrow, long long j) {
  if constexpr (MASKT == 1) return reinterpret_cast<const float*>(mrow)[j] * kLog2e;
  if constexpr (MASKT == 2)
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(mrow)[j]) * kLog2e;
  if constexpr (MASKT == 3) return reinterpret_cast<const uint8_t*>(mrow)[j] ? 0.0f : -INFINITY;
  return 0.0f;
}

// Kv tiles [first, last) that query tile t of the CTA at row m0 must visit: the tiles holding a
// key inside the row band [q_abs + lo_off, q_abs + hi_off] of any of its rows (q_abs = kl - ql +
// row). Without a window every range starts at tile 0 (an empty range is [0, 0), as for a tile
// wholly past the last query row). With one, a tile wholly past the last query row, or whose
// band misses every key, gets first = last = -1 and the caller places it at the end of the
// previous tile's range, so that the ranges of a CTA's tiles stay ordered.
template <int HD, int BAND>
__device__ __forceinline__ void fwd_tile_range(int m0, int t, const FwdKParams& p, int ql,
                                               int kl, int& first, int& last) {
  const int r0 = m0 + t * kBM;
  if (r0 >= ql) {  // a tile wholly past the last query row: nothing to visit
    first = last = BAND == kBandWindow ? -1 : 0;
    return;
  }
  const int r1 = min(m0 + (t + 1) * kBM, ql) - 1;  // last row of the tile (clamped)
  band_kv_tiles<FwdTraits<HD>::BN, BAND>(r0, r1, ql, kl, p.lo_off, p.hi_off, first, last);
}

template <int HD, int DV, int BAND, int MASKT, bool VARLEN>
__global__ void __launch_bounds__(FwdLayout<HD, DV>::THREADS, FwdLayout<HD, DV>::MIN_BLOCKS)
    fwd_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
               const __grid_constant__ CUtensorMap mV, const FwdKParams p) {
  using T = FwdTraits<HD>;
  using LY = FwdLayout<HD, DV>;
  constexpr int NQ = T::NQ, BN = T::BN, NS = T::NS, STAGES = T::STAGES, KCH = LY::KCH;
  constexpr int VCH = LY::VCH;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ uint64_t q_full;
  __shared__ uint64_t k_full[STAGES], k_empty[STAGES], v_full[STAGES], v_empty[STAGES];
  __shared__ uint64_t s_full[NQ][NS], p_full[NQ][NS], o_done[NQ], o_final[NQ];
  __shared__ uint64_t pv_done[NQ][NS];  // SPLIT: P V of a score buffer has read its P
  __shared__ uint64_t mma_drain, mma_drain2;
  __shared__ uint32_t tmem_base_s;
  __shared__ WaitCtl wctl;

  const int warp = warp_id();
  const int lane = lane_id();
  // Launch order, heaviest (causal) query tile first either way. Fixed length: tile-major, so
  // that every head's heaviest tile starts in the first wave and the light ones fill the tail.
  // Variable-length batch: the tiles of one (sequence, head) next to each other, so that they
  // share its K and V through L2 (tile-major, concurrent CTAs of every sequence thrash L2).
  const int bh = p.tiles_fast ? (int)blockIdx.y : (int)blockIdx.x;  // b * H + h
  const int mblk = p.n_mblk - 1 - (int)(p.tiles_fast ? blockIdx.x : blockIdx.y);
  const int m0 = mblk * NQ * kBM;
  const int b = bh / p.H, h = bh % p.H;
  // the rows of this problem: one (batch, head) of fixed length, or in a variable-length
  // batch sequence b's own rows of the packed head h (tensor-map z = head, rows offset)
  int ql = p.ql, kl = p.kl;
  int qrow0 = 0, krow0 = 0;
  size_t orow0 = (size_t)bh * p.ql;  // L row of query 0
  int ob = b, or0 = 0, orows = p.ql;  // O: batch, first row and rows of this problem
  const int kh = h / (p.H / p.Hk);
  int tb = b;  // batch coordinate of the tile loads (0 in a packed batch)
  if constexpr (VARLEN) {
    int qs, ks;
    const bool bad = varlen_seq(p.cu_q, b, p.total_q, p.ql, qs, ql) |
                     varlen_seq(p.cu_k, b, p.total_k, p.kl, ks, kl);
    if (bad && threadIdx.x == 0 && p.status) atomicCAS(p.status, kStatusOk, kStatusBadInput);
    qrow0 = qs;
    krow0 = ks;
    orow0 = (size_t)h * p.total_q + qs;
    ob = 0;
    tb = 0;
    or0 = qs;
    orows = p.total_q;
  }
  if (m0 >= ql) return;  // a query tile past this sequence's rows (the whole CTA leaves)

  // kv tile ranges of the query tiles, and their union [J0, J1)
  constexpr bool WIN = BAND == kBandWindow;
  int jt0[NQ], jt1[NQ];
#pragma unroll
  for (int t = 0; t < NQ; ++t) fwd_tile_range<HD, BAND>(m0, t, p, ql, kl, jt0[t], jt1[t]);
  int J0 = 0, J1 = 0;
  if (!WIN) {
#pragma unroll
    for (int t = 0; t < NQ; ++t) {
      jt0[t] = 0;
      J1 = max(J1, jt1[t]);
    }
  } else {
    bool any = false;
#pragma unroll
    for (int t = 0; t < NQ; ++t) {
      if (jt0[t] < 0) continue;
      J0 = any ? min(J0, jt0[t]) : jt0[t];
      J1 = any ? max(J1, jt1[t]) : jt1[t];
      any = true;
    }
#pragma unroll
    for (int t = 0; t < NQ; ++t)
      if (jt0[t] < 0) jt0[t] = jt1[t] = (t > 0 ? jt1[t - 1] : J0);  // empty, in order
  }

  if (threadIdx.x == 0) {
    wait_ctl_init(&wctl, p.wait_limit_ns);
    mbar_init(&q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < NQ; ++t) {
      for (int s = 0; s < NS; ++s) {
        mbar_init(&s_full[t][s], 1);
        mbar_init(&p_full[t][s], 128);
        mbar_init(&pv_done[t][s], 1);
      }
      mbar_init(&o_done[t], 1);
      mbar_init(&o_final[t], 1);
    }
    mbar_init(&mma_drain, 1);
    mbar_init(&mma_drain2, 1);
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
  // a following kernel launched with programmatic serialisation (the backward's pre-pass) may
  // be scheduled once every CTA of this grid is resident; it waits for this grid's completion
  grid_dep_trigger();

  if (warp == LY::TMA_WARP) {
    // ------------------------------------------------------------------ TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mV);
      const uint64_t pol_kv = policy_evict_last();
      int last_k[STAGES], last_v[STAGES];  // last kv tile loaded into each stage (-1: none)
      for (int s = 0; s < STAGES; ++s) last_k[s] = last_v[s] = -1;
      mbar_arrive_expect_tx(&q_full, NQ * LY::Q_TILE_BYTES);
      for (int t = 0; t < NQ; ++t)
        for (int c = 0; c < KCH; ++c)
          tma_load_bh(smem + LY::OFF_Q + t * LY::Q_TILE_BYTES + c * kBM * 128, &mQ, &q_full,
                      c * 64, qrow0 + m0 + t * kBM, h, tb, p.H, p.q_bshd != 0);
      for (int j = J0; j < J1; ++j) {
        const int st = (j - J0) % STAGES;
        const uint32_t use = (j - J0) / STAGES;
        if (use > 0 && !mbar_wait(&k_empty[st], (use - 1) & 1, &wctl)) break;
        mbar_arrive_expect_tx(&k_full[st], LY::K_TILE_BYTES);
        for (int c = 0; c < KCH; ++c)
          tma_load_bh_hint(smem + LY::OFF_K + st * LY::K_TILE_BYTES + c * BN * 128, &mK,
                           &k_full[st], c * 64, krow0 + j * BN, kh, tb, p.Hk, p.kv_bshd != 0,
                           pol_kv);
        last_k[st] = j - J0;
        if (use > 0 && !mbar_wait(&v_empty[st], (use - 1) & 1, &wctl)) break;
        mbar_arrive_expect_tx(&v_full[st], LY::V_TILE_BYTES);
        for (int c = 0; c < VCH; ++c)
          tma_load_bh_hint(smem + LY::OFF_V + st * LY::V_TILE_BYTES + c * BN * 128, &mV,
                           &v_full[st], c * 64, krow0 + j * BN, kh, tb, p.Hk, p.kv_bshd != 0,
                           pol_kv);
        last_v[st] = j - J0;
      }
      // Let every copy this thread started land before the CTA can exit.
      mbar_wait_drain(&q_full, 0);
      for (int s = 0; s < STAGES; ++s) {
        if (last_k[s] >= 0) mbar_wait_drain(&k_full[s], (last_k[s] / STAGES) & 1);
        if (last_v[s] >= 0) mbar_wait_drain(&v_full[s], (last_v[s] / STAGES) & 1);
      }
    }
  } else if (warp == LY::MMA_WARP || (T::SPLIT && warp == LY::MMA2_WARP)) {
    // ------------------------------------------------------------------ MMA issuer(s)
    if (elect_one()) {
      const uint32_t idesc_s = idesc_bf16(kBM, BN, 0, 0);
      const uint32_t idesc_o = idesc_bf16(kBM, DV, 0, 1);
      const uint32_t sq = smem_u32(smem + LY::OFF_Q);
      const uint32_t sk = smem_u32(smem + LY::OFF_K);
      const uint32_t sv = smem_u32(smem + LY::OFF_V);
      // K / V of kv tile j sit in stage (j - J0) % STAGES. A stage is released once every query
      // tile that uses the kv tile has issued its MMA on it. Without a window the last query
      // tile with rows uses every kv tile of the CTA (its range is the widest and all start at
      // 0), so it releases; with one, kleft / vleft count the users still to come (set when the
      // tile's full barrier is waited, in kv order).
      int k_ready = J0 - 1, v_ready = J0 - 1;  // highest kv tile whose K / V wait is done
      // without a window the last query tile that has rows uses every kv tile of the CTA
      const int t_rel = min(NQ - 1, (ql - 1 - m0) / kBM);
      int kleft[STAGES], vleft[STAGES];
      auto users = [&](int j) {
        int n = 0;
#pragma unroll
        for (int t = 0; t < NQ; ++t) n += (j >= jt0[t] && j < jt1[t]) ? 1 : 0;
        return n;
      };
      bool ok = mbar_wait(&q_full, 0, &wctl);
      tc_fence_after();

      auto issue_s = [&](int t, int j) {
        const int st = (j - J0) % STAGES;
        // wait the K tiles in order (without a window the next one is always j itself)
        while (ok && j > k_ready) {
          const int jw = WIN ? k_ready + 1 : j;
          ok = mbar_wait(&k_full[(jw - J0) % STAGES], ((jw - J0) / STAGES) & 1, &wctl);
          if (WIN) kleft[(jw - J0) % STAGES] = users(jw);
          k_ready = jw;
          tc_fence_after();
        }
        if (!ok) return;
        const int jj = j - jt0[t];  // == j without a window
        const uint32_t d_tmem = tbase + t * LY::TILE_COLS + DV + (jj % NS) * BN;
        const Desc qa = make_desc(sq + t * LY::Q_TILE_BYTES, 16, 1024);
        const Desc kb = make_desc(sk + st * LY::K_TILE_BYTES, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks)
          mma_ss2(d_tmem, qa.at((ks / 4) * (kBM * 128) + (ks % 4) * 32), qa.hi,
                  kb.at((ks / 4) * (BN * 128) + (ks % 4) * 32), kb.hi, idesc_s, ks > 0 ? 1u : 0u);
        mma_commit(&s_full[t][jj % NS]);
        if (WIN ? --kleft[st] == 0 : t == t_rel) mma_commit(&k_empty[st]);
      };

      if constexpr (T::SPLIT) {
        if (warp == LY::MMA_WARP) {
          // S of every (kv tile, query tile) in kv order; S(t, j) reuses the score buffer of
          // iteration j - NS of tile t once P V there has read P
          for (int j = J0; j < J1 && ok; ++j) {
#pragma unroll
            for (int t = 0; t < NQ; ++t) {
              if (!ok) break;
              if (j < jt0[t] || j >= jt1[t]) continue;
              const int jj = j - jt0[t];
              if (jj >= NS) {
                ok = mbar_wait(&pv_done[t][jj % NS], ((jj - NS) / NS) & 1, &wctl);
                if (!ok) break;
                tc_fence_after();
              }
              issue_s(t, j);
            }
          }
          mma_commit(&mma_drain2);
          mbar_wait_drain(&mma_drain2, 0);
        } else {
          for (int j = J0; j < J1 && ok; ++j) {
            const int st = (j - J0) % STAGES;
#pragma unroll
            for (int t = 0; t < NQ; ++t) {
              if (!ok) break;
              if (j < jt0[t] || j >= jt1[t]) continue;
              const int jj = j - jt0[t];
              const int sb = jj % NS;
              ok = mbar_wait(&p_full[t][sb], (jj / NS) & 1, &wctl);
              if (!ok) break;
              if (j > v_ready) {
                ok = mbar_wait(&v_full[st], ((j - J0) / STAGES) & 1, &wctl);
                if (!ok) break;
                if (WIN) vleft[st] = users(j);
                v_ready = j;
              }
              tc_fence_after();
              const uint32_t o_tmem = tbase + t * LY::TILE_COLS;
              const uint32_t p_tmem = o_tmem + DV + sb * BN;
              const Desc vb = make_desc(sv + st * LY::V_TILE_BYTES, BN * 128, 1024);
#pragma unroll
              for (int ks = 0; ks < BN / 16; ++ks)
                mma_ts2(o_tmem, p_tmem + ks * 8, vb.at(ks * 2048), vb.hi, idesc_o,
                        (jj > 0 || ks > 0) ? 1u : 0u);
              mma_commit(&o_done[t]);
              mma_commit(&pv_done[t][sb]);
              if (j == jt1[t] - 1) mma_commit(&o_final[t]);  // every PV of tile t issued
              if (WIN ? --vleft[st] == 0 : t == t_rel) mma_commit(&v_empty[st]);
            }
          }
          mma_commit(&mma_drain);
          mbar_wait_drain(&mma_drain, 0);
        }
      } else {
      // prologue: the first NS score tiles of every query tile
      for (int s0 = 0; s0 < NS && ok; ++s0)
#pragma unroll
        for (int t = 0; t < NQ; ++t)
          if (jt0[t] + s0 < jt1[t]) issue_s(t, jt0[t] + s0);

      for (int j = J0; j < J1 && ok; ++j) {
        const int st = (j - J0) % STAGES;
#pragma unroll
        for (int t = 0; t < NQ; ++t) {
          if (!ok) break;
          if (j < jt0[t] || j >= jt1[t]) continue;
          const int jj = j - jt0[t];  // iteration of this query tile
          const int sb = jj % NS;
          ok = mbar_wait(&p_full[t][sb], (jj / NS) & 1, &wctl);
          if (!ok) break;
          if (j > v_ready) {
            ok = mbar_wait(&v_full[st], ((j - J0) / STAGES) & 1, &wctl);
            if (!ok) break;
            if (WIN) vleft[st] = users(j);
            v_ready = j;
          }
          tc_fence_after();
          const uint32_t o_tmem = tbase + t * LY::TILE_COLS;
          const uint32_t p_tmem = o_tmem + DV + sb * BN;
          const Desc vb = make_desc(sv + st * LY::V_TILE_BYTES, BN * 128, 1024);
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks)
            mma_ts2(o_tmem, p_tmem + ks * 8, vb.at(ks * 2048), vb.hi, idesc_o,
                    (jj > 0 || ks > 0) ? 1u : 0u);
          mma_commit(&o_done[t]);
          if (j == jt1[t] - 1) mma_commit(&o_final[t]);  // every PV of tile t issued
          if (WIN ? --vleft[st] == 0 : t == t_rel) mma_commit(&v_empty[st]);
          if (j + NS < jt1[t]) issue_s(t, j + NS);
        }
      }
      // all MMAs complete before TMEM can be released
      mma_commit(&mma_drain);
      mbar_wait_drain(&mma_drain, 0);
      }
    }
  } else if (warp < 4 * NQ) {
    // ------------------------------------------------------------------ softmax warpgroups
    const int t = warp / 4;
    const int wl = warp % 4;
    const int r = wl * 32 + lane;  // row within the tile == TMEM lane
    const int i = m0 + t * kBM + r;
    // kv tiles [kt0, kt0 + ntt) of this query tile (an empty window range gives ntt = 0)
    int kt0, kt1;
    fwd_tile_range<HD, BAND>(m0, t, p, ql, kl, kt0, kt1);
    const int ntt = kt1 - kt0;
    const int off = kl - ql;
    // visible keys of this row: [klo_row, khi_row] (the row band, clipped to the keys)
    const int hi_off = WIN ? p.hi_off : 0;
    const int klo_row = WIN ? off + i + p.lo_off : 0;
    const int khi_row = BAND != kBandNone ? min(kl - 1, off + i + hi_off) : kl - 1;
    // the same bounds at the tile's first and last rows decide whether a kv tile is interior
    const int tile_row0 = m0 + t * kBM;
    const int tile_row1 = min(tile_row0 + kBM, ql) - 1;
    const int klo_tile = WIN ? off + tile_row1 + p.lo_off : 0;  // largest lo
    const int khi_tile =
        BAND != kBandNone ? min(kl - 1, off + tile_row0 + hi_off) : kl - 1;  // smallest hi
    const float c2 = p.scale_log2;
    const uint32_t lane_base = tbase + ((uint32_t)(wl * 32) << 16);
    const uint32_t o_col = t * LY::TILE_COLS;
    const void* mrow = nullptr;
    if (MASKT != 0 && i < ql) {
      const int b_ = bh / p.H, h_ = bh % p.H;
      const size_t es = MASKT == 1 ? 4 : MASKT == 2 ? 2 : 1;
      mrow = reinterpret_cast<const uint8_t*>(p.mask) +
             (b_ * p.msb + h_ * p.msh + (long long)i * p.msq) * es;
    }

    // running max (base 2, from the finite sentinel) and row sum over the keys; a sink joins
    // only in the epilogue
    float m_used = -FLT_MAX / 2.0f;
    float l = 0.0f;
    bool ok = true;

    for (int j = 0; j < ntt; ++j) {  // j: iteration of this query tile (kv tile kt0 + j)
      const int sb = j % NS;
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t][sb], (j / NS) & 1, &wctl));
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_addr = lane_base + o_col + DV + sb * BN;
      uint32_t sr[BN / 32][32];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(s_addr + c * 32, sr[c]);
      tmem_wait_ld();

      const int n0 = (kt0 + j) * BN;
      // does any element of this tile need masking (uniform over the warpgroup)?
      const bool edge = (n0 + BN - 1 > khi_tile) || (WIN && n0 < klo_tile);
      const int lim_lo = klo_row - n0, lim_hi = khi_row - n0;  // c visible iff lo <= c <= hi
      // scores in place of the loaded row: raw S, or (with a mask) the base-2 score; -inf
      // where the key is hidden. Tiles inside every row's band skip this.
      if (MASKT != 0 || edge) {
#pragma unroll
        for (int c32 = 0; c32 < BN / 32; ++c32) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int c = c32 * 32 + e;
            float v = __uint_as_float(sr[c32][e]);
            if (MASKT != 0) {
              const float mv = (mrow != nullptr && n0 + c < kl) ? mask_log2<MASKT>(mrow, n0 + c) : 0.0f;
              v = fmaf(v, c2, mv);
            }
            if ((WIN && c < lim_lo) || c > lim_hi) v = -INFINITY;
            sr[c32][e] = __float_as_uint(v);
          }
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c32 = 0; c32 < BN / 32; ++c32)
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          mx = fmax3(mx, __uint_as_float(sr[c32][e]), __uint_as_float(sr[c32][e + 1]));
      // row maximum in base-2 units
      const float m_tile = MASKT != 0 ? mx : mx * c2;
      const float m_new = fmaxf(m_used, m_tile);
      const bool need = m_new > m_used + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float factor = ex2(m_used - m_new);
        l *= factor;
        if (j > 0) {
          // O holds PV of tiles < j: wait for the last of them, then scale the row in place.
          // (S of tile j was committed after PV of tile j-NS, so at most NS-1 <= 1 phase of
          // o_done is outstanding here and the parity wait is exact.)
          ok = __all_sync(0xffffffffu, mbar_wait(&o_done[t], (j - 1) & 1, &wctl));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < DV; c += 32) {
            uint32_t orr[32];
            tmem_ld32(lane_base + o_col + c, orr);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e)
              orr[e] = __float_as_uint(__uint_as_float(orr[e]) * factor);
            tmem_st32(lane_base + o_col + c, orr);
          }
          tmem_wait_st();
        }
        m_used = m_new;
      }
      // p = exp2(x - m_used) on pairs, packed to bf16 in place of S, 32 columns at a time
      const uint64_t negm = f2_pack(-m_used, -m_used);
      const uint64_t c2v = f2_pack(c2, c2);
      float rs0 = 0.0f, rs1 = 0.0f;
#pragma unroll
      for (int c32 = 0; c32 < BN / 32; ++c32) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint64_t xv = f2_pack(__uint_as_float(sr[c32][2 * e]),
                                      __uint_as_float(sr[c32][2 * e + 1]));
          const uint64_t sv = MASKT != 0 ? f2_add(xv, negm) : f2_fma(xv, c2v, negm);
          float s0, s1;
          f2_unpack(sv, s0, s1);
          float p0, p1;
          if (T::POLY > 0 && (e % (T::POLY > 0 ? T::POLY : 1)) == 0) {
            p0 = ex2_poly(s0);
            p1 = ex2_poly(s1);
          } else {
            p0 = ex2(s0);
            p1 = ex2(s1);
          }
          rs0 += p0;
          rs1 += p1;
          pk[e] = pack_bf16(p0, p1);
        }
        tmem_st16(s_addr + c32 * 16, pk);
      }
      const float rs = rs0 + rs1;
      l += rs;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[t][sb]);
    }

    // ---------------------------------------------------------------- epilogue
    // o_final completes once, after the last PV of this tile (a single-phase barrier: o_done
    // may be anywhere between NS phases behind and done here, which a parity wait cannot
    // tell apart).
    if (ok && ntt > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&o_final[t], 0, &wctl));
      tc_fence_after();
    }
    // O = O_acc * inv and L from the keys' normaliser l * 2^m_used. A sink adds 2^s2 to the
    // normaliser here, in log2 form so that nothing overflows: keeping it out of the running
    // max leaves the largest key's weight at exactly 1, so the bf16 rounding of P costs a row
    // dominated by one key no more than without a sink. O exists in TMEM only when some kv
    // tile was visited.
    const bool have_o = ok && ntt > 0 && l > 0.0f;
    float inv = have_o ? 1.0f / l : 0.0f;
    float L = (ok && l > 0.0f) ? m_used * kLn2 + logf(l) : -INFINITY;
    if (p.sinks != nullptr && ok) {
      const float s2 = __ldg(p.sinks + bh % p.H) * kLog2e;  // -inf: no sink
      if (l > 0.0f) {
        const float lm = m_used + log2f(l);
        const float mx = fmaxf(lm, s2);
        const float L2 = mx + log2f(exp2f(lm - mx) + exp2f(s2 - mx));
        inv = exp2f(m_used - L2);
        L = L2 * kLn2;
      } else {
        L = s2 * kLn2;  // a row that sees no key: O = 0, L = sink
      }
    }
    __nv_bfloat16* orow =
        p.o + bhsd_offset(ob, h, or0 + (i < ql ? i : 0), p.H, orows, DV, p.q_bshd != 0);
#pragma unroll 1
    for (int c = 0; c < DV; c += 32) {
      uint32_t orr[32];
      if (ok && ntt > 0) {
        tmem_ld32(lane_base + o_col + c, orr);
        tmem_wait_ld();
      }
      uint32_t packed[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float a0 = have_o ? __uint_as_float(orr[2 * e]) * inv : 0.0f;
        float a1 = have_o ? __uint_as_float(orr[2 * e + 1]) * inv : 0.0f;
        packed[e] = pack_bf16(a0, a1);
      }
      if (i < ql) {
        uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)
          dst[v4] = make_uint4(packed[4 * v4], packed[4 * v4 + 1], packed[4 * v4 + 2],
                               packed[4 * v4 + 3]);
      }
    }
    if (i < ql) p.lse[orow0 + i] = L;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == LY::MMA_WARP) tmem_dealloc(tbase, LY::TMEM_COLS);
  if (threadIdx.x == 0) report_abort(&wctl, p.status);
}

int fwd_q_box_rows(int) { return kBM; }
int fwd_kv_box_rows(int d) {
  return d == 64 ? FwdTraits<64>::BN : d == 128 ? FwdTraits<128>::BN : FwdTraits<256>::BN;
}

template <int HD, int DV, int BAND, int MASKT, bool VARLEN = false>
static cudaError_t launch_fwd_t(const FwdArgs& a, const FwdMaps& m, cudaStream_t stream) {
  using LY = FwdLayout<HD, DV>;
  auto kern = fwd_kernel<HD, DV, BAND, MASKT, VARLEN>;
  static OncePerKey<> smem_attr;  // per instantiation and device
  {
    const cudaError_t e = set_smem_once(smem_attr, kern, LY::SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  FwdKParams kp;
  kp.mask = a.mask;
  kp.msb = a.mask_stride_b;
  kp.msh = a.mask_stride_h;
  kp.msq = a.mask_stride_q;
  kp.o = reinterpret_cast<__nv_bfloat16*>(a.o);
  kp.lse = a.lse;
  kp.sinks = a.sinks;
  kp.cu_q = a.cu_q;
  kp.cu_k = a.cu_k;
  kp.total_q = a.total_q;
  kp.q_bshd = a.q_bshd;
  kp.kv_bshd = a.kv_bshd;
  kp.total_k = a.total_k;
  kp.status = a.status;
  kp.wait_limit_ns = a.wait_limit_ns;
  kp.H = a.H;
  kp.Hk = a.Hk;
  kp.ql = a.ql;
  kp.kl = a.kl;
  kp.lo_off = a.lo_off;
  kp.hi_off = a.hi_off;
  kp.n_mblk = (a.ql + FwdTraits<HD>::NQ * kBM - 1) / (FwdTraits<HD>::NQ * kBM);
  kp.scale_log2 = a.scale * kLog2e;
  kp.tiles_fast = a.cu_q != nullptr && a.B * a.H <= 65535;  // (grid y limit)
  dim3 grid(kp.tiles_fast ? kp.n_mblk : a.B * a.H, kp.tiles_fast ? a.B * a.H : kp.n_mblk);
  profile_mark(kKernFwd, 0, stream);
  kern<<<grid, LY::THREADS, LY::SMEM_BYTES, stream>>>(m.q, m.k, m.v, kp);
  cudaError_t e = cudaGetLastError();
  profile_mark(kKernFwd, 1, stream);
  return e;
}

template <int HD, int DV, int BAND>
static cudaError_t launch_fwd_m(const FwdArgs& a, const FwdMaps& m, cudaStream_t s) {
  if (a.cu_q) return launch_fwd_t<HD, DV, BAND, 0, true>(a, m, s);  // (no mask with varlen)
  if (!a.mask) return launch_fwd_t<HD, DV, BAND, 0>(a, m, s);
  switch (a.mask_type) {
    case 0: return launch_fwd_t<HD, DV, BAND, 1>(a, m, s);
    case 1: return launch_fwd_t<HD, DV, BAND, 2>(a, m, s);
    default: return launch_fwd_t<HD, DV, BAND, 3>(a, m, s);
  }
}

template <int HD, int DV>
static cudaError_t launch_fwd_d(const FwdArgs& a, const FwdMaps& m, cudaStream_t s) {
  switch (a.band) {
    case kBandNone: return launch_fwd_m<HD, DV, kBandNone>(a, m, s);
    case kBandCausal: return launch_fwd_m<HD, DV, kBandCausal>(a, m, s);
    default: return launch_fwd_m<HD, DV, kBandWindow>(a, m, s);
  }
}

cudaError_t launch_fwd(const FwdArgs& a, const FwdMaps& m, cudaStream_t stream) {
  if (a.d == 64 && a.dval == 64) return launch_fwd_d<64, 64>(a, m, stream);
  if (a.d == 128 && a.dval == 128) return launch_fwd_d<128, 128>(a, m, stream);
  if (a.d == 256 && a.dval == 256) return launch_fwd_d<256, 256>(a, m, stream);
  if (a.d == 128 && a.dval == 64) return launch_fwd_d<128, 64>(a, m, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
