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
// K/V ring. POLY: one pair of exponentials in every POLY goes to the FMA-pipe polynomial
// (0 = all on MUFU); the MUFU unit (16 exp2 per clock per SM) would otherwise be as slow as
// the tensor core at head_dim 128 and the bottleneck at 64.
template <>
struct FwdTraits<64> {
  static constexpr int NQ = 2, BN = 128, NS = 1, STAGES = 3, POLY = 4;
};
template <>
struct FwdTraits<128> {
  static constexpr int NQ = 2, BN = 128, NS = 1, STAGES = 2, POLY = 8;
};
template <>
struct FwdTraits<256> {
  static constexpr int NQ = 1, BN = 64, NS = 2, STAGES = 2, POLY = 0;
};

template <int HD>
struct FwdLayout {
  using T = FwdTraits<HD>;
  static constexpr int KCH = HD / 64;                         // 128-byte column chunks
  static constexpr int Q_TILE_BYTES = kBM * HD * 2;
  static constexpr int KV_TILE_BYTES = T::BN * HD * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + T::NQ * Q_TILE_BYTES;
  static constexpr int OFF_V = OFF_K + T::STAGES * KV_TILE_BYTES;
  static constexpr int OFF_END = OFF_V + T::STAGES * KV_TILE_BYTES;
  static constexpr int SMEM_BYTES = OFF_END + 1024;  // + alignment slack
  // TMEM columns of tile t: O at t*TILE_COLS, S buffer s at t*TILE_COLS + HD + s*BN.
  static constexpr int TILE_COLS = HD + T::NS * T::BN;
  static constexpr int TMEM_COLS_USED = T::NQ * TILE_COLS;
  static constexpr int TMEM_COLS = TMEM_COLS_USED <= 256 ? 256 : 512;
  static constexpr int THREADS = T::NQ * 128 + 64;  // softmax warpgroups + TMA + MMA warps
  static constexpr int TMA_WARP = T::NQ * 4;
  static constexpr int MMA_WARP = T::NQ * 4 + 1;
  static_assert(TMEM_COLS_USED <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

struct FwdKParams {
  const float* mask;
  __nv_bfloat16* o;
  float* lse;
  int* status;
  int H, Hk, ql, kl, n_mblk;
  float scale_log2;  // scale * log2(e)
};

// Number of kv tiles query tile t of the CTA at row m0 must visit.
template <int HD, bool CAUSAL>
__device__ __forceinline__ int fwd_tiles_for(int m0, int t, int ql, int kl) {
  constexpr int BN = FwdTraits<HD>::BN;
  int kend = kl;
  if (CAUSAL) {
    // last row of the tile is m0 + (t+1)*BM - 1 (clamped to ql-1); it sees keys <= off + row
    int last_row = min(m0 + (t + 1) * kBM, ql) - 1;
    int lim = kl - ql + last_row + 1;  // exclusive key bound
    kend = min(kend, lim);
  }
  if (kend <= 0) return 0;
  return (kend + BN - 1) / BN;
}

template <int HD, bool CAUSAL, bool HAS_MASK>
__global__ void __launch_bounds__(FwdLayout<HD>::THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
               const __grid_constant__ CUtensorMap mV, const FwdKParams p) {
  using T = FwdTraits<HD>;
  using LY = FwdLayout<HD>;
  constexpr int NQ = T::NQ, BN = T::BN, NS = T::NS, STAGES = T::STAGES, KCH = LY::KCH;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ uint64_t q_full;
  __shared__ uint64_t k_full[STAGES], k_empty[STAGES], v_full[STAGES], v_empty[STAGES];
  __shared__ uint64_t s_full[NQ][NS], p_full[NQ][NS], o_done[NQ], o_final[NQ];
  __shared__ uint64_t mma_drain;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;

  const int warp = warp_id();
  const int lane = lane_id();
  const int bh = blockIdx.x;                     // b * H + h
  const int mblk = p.n_mblk - 1 - (int)blockIdx.y;  // heaviest (causal) first
  const int m0 = mblk * NQ * kBM;
  const int b = bh / p.H, h = bh % p.H;
  const int bkh = b * p.Hk + h / (p.H / p.Hk);

  int nt[NQ];
  int nt_max = 0;
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    nt[t] = fwd_tiles_for<HD, CAUSAL>(m0, t, p.ql, p.kl);
    nt_max = max(nt_max, nt[t]);
  }

  if (threadIdx.x == 0) {
    abort_flag = 0;
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
      }
      mbar_init(&o_done[t], 1);
      mbar_init(&o_final[t], 1);
    }
    mbar_init(&mma_drain, 1);
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
          tma_load_3d(smem + LY::OFF_Q + t * LY::Q_TILE_BYTES + c * kBM * 128, &mQ, &q_full,
                      c * 64, m0 + t * kBM, bh);
      for (int j = 0; j < nt_max; ++j) {
        const int st = j % STAGES;
        const uint32_t use = j / STAGES;
        if (j >= STAGES && !mbar_wait(&k_empty[st], (use - 1) & 1, &abort_flag)) break;
        mbar_arrive_expect_tx(&k_full[st], LY::KV_TILE_BYTES);
        for (int c = 0; c < KCH; ++c)
          tma_load_3d_hint(smem + LY::OFF_K + st * LY::KV_TILE_BYTES + c * BN * 128, &mK,
                           &k_full[st], c * 64, j * BN, bkh, pol_kv);
        last_k[st] = j;
        if (j >= STAGES && !mbar_wait(&v_empty[st], (use - 1) & 1, &abort_flag)) break;
        mbar_arrive_expect_tx(&v_full[st], LY::KV_TILE_BYTES);
        for (int c = 0; c < KCH; ++c)
          tma_load_3d_hint(smem + LY::OFF_V + st * LY::KV_TILE_BYTES + c * BN * 128, &mV,
                           &v_full[st], c * 64, j * BN, bkh, pol_kv);
        last_v[st] = j;
      }
      // Let every copy this thread started land before the CTA can exit.
      mbar_wait_drain(&q_full, 0);
      for (int s = 0; s < STAGES; ++s) {
        if (last_k[s] >= 0) mbar_wait_drain(&k_full[s], (last_k[s] / STAGES) & 1);
        if (last_v[s] >= 0) mbar_wait_drain(&v_full[s], (last_v[s] / STAGES) & 1);
      }
    }
  } else if (warp == LY::MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      const uint32_t idesc_s = idesc_bf16(kBM, BN, 0, 0);
      const uint32_t idesc_o = idesc_bf16(kBM, HD, 0, 1);
      const uint32_t sq = smem_u32(smem + LY::OFF_Q);
      const uint32_t sk = smem_u32(smem + LY::OFF_K);
      const uint32_t sv = smem_u32(smem + LY::OFF_V);
      int k_ready = -1, v_ready = -1;  // highest kv tile whose K / V wait is done
      bool ok = mbar_wait(&q_full, 0, &abort_flag);
      tc_fence_after();

      auto issue_s = [&](int t, int j) {
        const int st = j % STAGES;
        if (j > k_ready) {
          ok = ok && mbar_wait(&k_full[st], (j / STAGES) & 1, &abort_flag);
          k_ready = j;
          tc_fence_after();
        }
        const uint32_t d_tmem = tbase + t * LY::TILE_COLS + HD + (j % NS) * BN;
        const Desc qa = make_desc(sq + t * LY::Q_TILE_BYTES, 16, 1024);
        const Desc kb = make_desc(sk + st * LY::KV_TILE_BYTES, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks)
          mma_ss2(d_tmem, qa.at((ks / 4) * (kBM * 128) + (ks % 4) * 32), qa.hi,
                  kb.at((ks / 4) * (BN * 128) + (ks % 4) * 32), kb.hi, idesc_s, ks > 0 ? 1u : 0u);
        mma_commit(&s_full[t][j % NS]);
        if (t == NQ - 1) mma_commit(&k_empty[st]);
      };

      // prologue: the first NS score tiles of every query tile
      for (int j = 0; j < NS && ok; ++j)
        for (int t = 0; t < NQ; ++t)
          if (j < nt[t]) issue_s(t, j);

      for (int j = 0; j < nt_max && ok; ++j) {
        const int st = j % STAGES;
        for (int t = 0; t < NQ && ok; ++t) {
          if (j >= nt[t]) continue;
          const int sb = j % NS;
          ok = mbar_wait(&p_full[t][sb], (j / NS) & 1, &abort_flag);
          if (!ok) break;
          if (j > v_ready) {
            ok = mbar_wait(&v_full[st], (j / STAGES) & 1, &abort_flag);
            if (!ok) break;
            v_ready = j;
          }
          tc_fence_after();
          const uint32_t o_tmem = tbase + t * LY::TILE_COLS;
          const uint32_t p_tmem = o_tmem + HD + sb * BN;
          const Desc vb = make_desc(sv + st * LY::KV_TILE_BYTES, BN * 128, 1024);
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks)
            mma_ts2(o_tmem, p_tmem + ks * 8, vb.at(ks * 2048), vb.hi, idesc_o,
                    (j > 0 || ks > 0) ? 1u : 0u);
          mma_commit(&o_done[t]);
          if (j == nt[t] - 1) mma_commit(&o_final[t]);  // every PV of tile t issued
          if (t == NQ - 1) mma_commit(&v_empty[st]);
          if (j + NS < nt[t]) issue_s(t, j + NS);
        }
      }
      // all MMAs complete before TMEM can be released
      mma_commit(&mma_drain);
      mbar_wait_drain(&mma_drain, 0);
    }
  } else if (warp < 4 * NQ) {
    // ------------------------------------------------------------------ softmax warpgroups
    const int t = warp / 4;
    const int wl = warp % 4;
    const int r = wl * 32 + lane;  // row within the tile == TMEM lane
    const int i = m0 + t * kBM + r;
    const int ntt = nt[t];
    const int kmax_row = CAUSAL ? min(p.kl - 1, p.kl - p.ql + i) : p.kl - 1;  // last visible key
    const int tile_row0 = m0 + t * kBM;
    const float c2 = p.scale_log2;
    const uint32_t lane_base = tbase + ((uint32_t)(wl * 32) << 16);
    const uint32_t o_col = t * LY::TILE_COLS;
    const float* mrow = nullptr;
    if (HAS_MASK && i < p.ql) mrow = p.mask + ((size_t)bh * p.ql + i) * (size_t)p.kl;

    float m_used = -FLT_MAX / 2.0f;  // finite sentinel
    float l = 0.0f;
    bool ok = true;

    for (int j = 0; j < ntt; ++j) {
      const int sb = j % NS;
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t][sb], (j / NS) & 1, &abort_flag));
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_addr = lane_base + o_col + HD + sb * BN;
      uint32_t sr[BN / 32][32];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(s_addr + c * 32, sr[c]);
      tmem_wait_ld();

      const int n0 = j * BN;
      // does any element of this tile need masking (uniform over the warpgroup)?
      const bool edge = (n0 + BN > p.kl) || (CAUSAL && n0 + BN - 1 > p.kl - p.ql + tile_row0);
      const int lim = kmax_row - n0;  // element c visible iff c <= lim
      // scores in place of the loaded row: raw S, or (with a mask) the base-2 score; -inf
      // where the key is hidden. Tiles away from the diagonal and the key tail skip this.
      if (HAS_MASK || edge) {
#pragma unroll
        for (int c32 = 0; c32 < BN / 32; ++c32) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int c = c32 * 32 + e;
            float v = __uint_as_float(sr[c32][e]);
            if (HAS_MASK) {
              float mv = (mrow != nullptr && n0 + c < p.kl) ? mrow[n0 + c] : 0.0f;
              v = fmaf(v, c2, mv * kLog2e);
            }
            if (c > lim) v = -INFINITY;
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
      const float m_tile = HAS_MASK ? mx : mx * c2;
      const float m_new = fmaxf(m_used, m_tile);
      const bool need = m_new > m_used + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float factor = ex2(m_used - m_new);
        l *= factor;
        if (j > 0) {
          // O holds PV of tiles < j: wait for the last of them, then scale the row in place.
          // (S of tile j was committed after PV of tile j-NS, so at most NS-1 <= 1 phase of
          // o_done is outstanding here and the parity wait is exact.)
          ok = __all_sync(0xffffffffu, mbar_wait(&o_done[t], (j - 1) & 1, &abort_flag));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < HD; c += 32) {
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
          const uint64_t sv = HAS_MASK ? f2_add(xv, negm) : f2_fma(xv, c2v, negm);
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
      ok = __all_sync(0xffffffffu, mbar_wait(&o_final[t], 0, &abort_flag));
      tc_fence_after();
    }
    const bool live = ok && ntt > 0 && l > 0.0f;
    const float inv = live ? 1.0f / l : 0.0f;
    __nv_bfloat16* orow = p.o + ((size_t)bh * p.ql + (i < p.ql ? i : 0)) * HD;
#pragma unroll 1
    for (int c = 0; c < HD; c += 32) {
      uint32_t orr[32];
      if (ok && ntt > 0) {
        tmem_ld32(lane_base + o_col + c, orr);
        tmem_wait_ld();
      }
      uint32_t packed[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float a0 = live ? __uint_as_float(orr[2 * e]) * inv : 0.0f;
        float a1 = live ? __uint_as_float(orr[2 * e + 1]) * inv : 0.0f;
        packed[e] = pack_bf16(a0, a1);
      }
      if (i < p.ql) {
        uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)
          dst[v4] = make_uint4(packed[4 * v4], packed[4 * v4 + 1], packed[4 * v4 + 2],
                               packed[4 * v4 + 3]);
      }
    }
    if (i < p.ql) p.lse[(size_t)bh * p.ql + i] = live ? m_used * kLn2 + logf(l) : -INFINITY;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == LY::MMA_WARP) tmem_dealloc(tbase, LY::TMEM_COLS);
  if (threadIdx.x == 0) report_abort(&abort_flag, p.status);
}

int fwd_q_box_rows(int) { return kBM; }
int fwd_kv_box_rows(int d) {
  return d == 64 ? FwdTraits<64>::BN : d == 128 ? FwdTraits<128>::BN : FwdTraits<256>::BN;
}

template <int HD, bool CAUSAL, bool HAS_MASK>
static cudaError_t launch_fwd_t(const FwdArgs& a, const FwdMaps& m, cudaStream_t stream) {
  using LY = FwdLayout<HD>;
  auto kern = fwd_kernel<HD, CAUSAL, HAS_MASK>;
  static bool attr_set = false;  // per instantiation; the attribute is per device function
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  FwdKParams kp;
  kp.mask = a.mask;
  kp.o = reinterpret_cast<__nv_bfloat16*>(a.o);
  kp.lse = a.lse;
  kp.status = a.status;
  kp.H = a.H;
  kp.Hk = a.Hk;
  kp.ql = a.ql;
  kp.kl = a.kl;
  kp.n_mblk = (a.ql + FwdTraits<HD>::NQ * kBM - 1) / (FwdTraits<HD>::NQ * kBM);
  kp.scale_log2 = a.scale * kLog2e;
  dim3 grid(a.B * a.H, kp.n_mblk);
  profile_mark(kKernFwd, 0, stream);
  kern<<<grid, LY::THREADS, LY::SMEM_BYTES, stream>>>(m.q, m.k, m.v, kp);
  cudaError_t e = cudaGetLastError();
  profile_mark(kKernFwd, 1, stream);
  return e;
}

template <int HD>
static cudaError_t launch_fwd_d(const FwdArgs& a, const FwdMaps& m, cudaStream_t s) {
  if (a.causal) {
    return a.mask ? launch_fwd_t<HD, true, true>(a, m, s) : launch_fwd_t<HD, true, false>(a, m, s);
  }
  return a.mask ? launch_fwd_t<HD, false, true>(a, m, s) : launch_fwd_t<HD, false, false>(a, m, s);
}

cudaError_t launch_fwd(const FwdArgs& a, const FwdMaps& m, cudaStream_t stream) {
  switch (a.d) {
    case 64: return launch_fwd_d<64>(a, m, stream);
    case 128: return launch_fwd_d<128>(a, m, stream);
    case 256: return launch_fwd_d<256>(a, m, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa
