// fa_bwd_dq.cu -- deterministic dQ for the backward pass (sm_103a).
//
// The main backward pass (fa_bwd.cu) adds each kv tile's dQ contribution into an f32
// accumulator from many CTAs at once, so the order of the additions, and with it the rounding
// of dQ, changes from run to run. In deterministic mode that pass skips dQ and this kernel
// forms it instead, query-tile-major, with no atomics: one CTA owns 128 query rows of one
// (batch, head) and walks the kv tiles of its band in order, recomputing
//   S = Q K^T,  dP = dO V^T,  P = exp2(S * scale * log2(e) + mask * log2(e) - L * log2(e)),
//   dS = P o (dP - D),  dQ += dS K
// (the FlashAttention-2 backward equations of page "mlx-native tests/test_flash_attn_train.rs",
// `sdpa_backward_reference_f32`), and writes dQ = bf16(scale * dQ) once. The result depends
// only on the inputs.
//
// GB300 design: one warp streams K/V tiles (64 keys) with TMA through a ring; one warp issues
// the tcgen05 MMAs: S and dP into double-buffered TMEM (SS form, both operands K-major), then
// dQ += dS K with dS read from TMEM (written over S as packed bf16) and K MN-major; one
// warpgroup, thread = query row = TMEM lane, turns S and dP into dS. With a ring of two or
// more stages the next tile's S and dP are issued before this tile's dQ, so the tensor core
// works while the warpgroup computes dS.
#include <float.h>

#include "fa_band.cuh"
#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {

namespace {
constexpr float kLog2eQ = 1.4426950408889634f;
constexpr int kQM = 128;  // query rows per CTA (the MMA M)
constexpr int kQN = 64;   // keys per kv tile
}  // namespace

// STAGES: depth of the K/V ring (shared memory: Q and dO tiles + STAGES x (K + V) tiles).
template <int HD>
struct DqTraits;
template <>
struct DqTraits<64> {
  static constexpr int STAGES = 4;
};
template <>
struct DqTraits<128> {
  static constexpr int STAGES = 3;
};
template <>
struct DqTraits<256> {
  static constexpr int STAGES = 1;
};

template <int HD, int DV>
struct DqLayout {
  static constexpr int STAGES = DqTraits<HD>::STAGES;
  static constexpr bool LOOKAHEAD = STAGES >= 2;  // issue S, dP of tile j+1 before dQ of j
  static constexpr int KCH = HD / 64, VCH = DV / 64;
  static constexpr int Q_BYTES = kQM * HD * 2;
  static constexpr int DO_BYTES = kQM * DV * 2;
  static constexpr int K_BYTES = kQN * HD * 2;
  static constexpr int V_BYTES = kQN * DV * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + Q_BYTES;
  static constexpr int OFF_K = OFF_DO + DO_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * K_BYTES;
  static constexpr int OFF_END = OFF_V + STAGES * V_BYTES;
  static constexpr int SMEM_BYTES = OFF_END + 1024;
  // TMEM columns: S buffers 0, 1; dP buffers 0, 1; the dQ accumulator
  static constexpr int COL_S0 = 0;
  static constexpr int COL_DP0 = 2 * kQN;
  static constexpr int COL_DQ = 4 * kQN;
  static constexpr int TMEM_USED = COL_DQ + HD;
  static constexpr int TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
  static constexpr int THREADS = 192;  // warps 0-3: dS; warp 4: TMA; warp 5: MMA
  static constexpr int TMA_WARP = 4, MMA_WARP = 5;
  static_assert(TMEM_USED <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

struct DqKParams {
  const void* mask;         // additive f32 / bf16, or bool (uint8), addressed with the strides
  long long msb, msh, msq;  // mask strides (elements) of batch, head, query row
  const float* lse2;        // [B*H, ql_pad]: -L * log2(e) (-inf: the row sees nothing)
  const float* dvec;        // [B*H, ql_pad]: D
  __nv_bfloat16* dq;        // [B, H, ql, HD]
  int* status;
  const int32_t* cu_q;  // variable-length batch: sequence offsets, or nullptr
  const int32_t* cu_k;
  int total_q, total_k;
  int q_bshd, kv_bshd;  // 1: q, dO, dq / k, v are [batch, rows, heads, d] (tile maps 4-D)
  int H, Hk, ql, kl, ql_pad;
  int tiles_fast;  // 1: blockIdx.x = query tile, y = (batch, head); 0: swapped
  int lo_off, hi_off;
  float scale, scale_log2;
  unsigned long long wait_limit_ns;  // limit of one barrier wait
};

template <int MASKT>
__device__ __forceinline__ float dq_mask_log2(const void* mrow, long long j) {
  if constexpr (MASKT == 1) return reinterpret_cast<const float*>(mrow)[j] * kLog2eQ;
  if constexpr (MASKT == 2)
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(mrow)[j]) * kLog2eQ;
  if constexpr (MASKT == 3) return reinterpret_cast<const uint8_t*>(mrow)[j] ? 0.0f : -INFINITY;
  return 0.0f;
}

template <int HD, int DV, int BAND, int MASKT>
__global__ void __launch_bounds__(DqLayout<HD, DV>::THREADS, 1)
    bwd_dq_det_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                      const __grid_constant__ CUtensorMap mV,
                      const __grid_constant__ CUtensorMap mDO, const DqKParams p) {
  using LY = DqLayout<HD, DV>;
  constexpr int STAGES = LY::STAGES, KCH = LY::KCH, VCH = LY::VCH;
  constexpr bool WIN = BAND == kBandWindow;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ uint64_t q_full, kv_full[STAGES], kv_empty[STAGES];
  __shared__ uint64_t sdp_full[2], ds_ready[2], dq_final, mma_drain;
  __shared__ uint32_t tmem_base_s;
  __shared__ WaitCtl wctl;

  const int warp = warp_id(), lane = lane_id();
  // variable-length batch: the tiles of one (sequence, head) together (they share K, V in L2)
  const int bh = p.tiles_fast ? (int)blockIdx.y : (int)blockIdx.x;
  const int b = bh / p.H, h = bh % p.H;
  const int m0 = (int)(p.tiles_fast ? blockIdx.x : blockIdx.y) * kQM;
  // the rows of this problem: one (batch, head), or sequence b of a variable-length batch
  int ql = p.ql, kl = p.kl;
  const int kh = h / (p.H / p.Hk);
  int tb = b, qrow0 = 0, krow0 = 0;  // tb: batch coordinate of the tile loads
  int ob = bh / p.H, or0 = 0, orows = p.ql;  // dQ: batch, first row and rows of this problem
  if (p.cu_q != nullptr) {
    int qs, ks;
    varlen_seq(p.cu_q, b, p.total_q, p.ql, qs, ql);
    varlen_seq(p.cu_k, b, p.total_k, p.kl, ks, kl);
    tb = 0;
    qrow0 = qs;
    krow0 = ks;
    ob = 0;
    or0 = qs;
    orows = p.total_q;
  }
  if (m0 >= ql) return;  // a query tile past this sequence's rows (the whole CTA leaves)
  const int r1 = min(m0 + kQM, ql) - 1;
  int J0, J1;
  band_kv_tiles<kQN, BAND>(m0, r1, ql, kl, p.lo_off, p.hi_off, J0, J1);
  if (J0 < 0) J0 = J1 = 0;
  const int ntt = J1 - J0;  // kv tiles this CTA visits

  if (threadIdx.x == 0) {
    wait_ctl_init(&wctl, p.wait_limit_ns);
    mbar_init(&q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sdp_full[s], 1);
      mbar_init(&ds_ready[s], 128);
    }
    mbar_init(&dq_final, 1);
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
      tma_prefetch_desc(&mDO);
      int last[STAGES];
      for (int s = 0; s < STAGES; ++s) last[s] = -1;
      mbar_arrive_expect_tx(&q_full, LY::Q_BYTES + LY::DO_BYTES);
      for (int c = 0; c < KCH; ++c)
        tma_load_bh(smem + LY::OFF_Q + c * kQM * 128, &mQ, &q_full, c * 64, qrow0 + m0, h, tb,
                    p.H, p.q_bshd != 0);
      for (int c = 0; c < VCH; ++c)
        tma_load_bh(smem + LY::OFF_DO + c * kQM * 128, &mDO, &q_full, c * 64, qrow0 + m0, h, tb,
                    p.H, p.q_bshd != 0);
      const uint64_t pol = policy_evict_last();
      for (int jj = 0; jj < ntt; ++jj) {
        const int st = jj % STAGES;
        const uint32_t use = jj / STAGES;
        if (use > 0 && !mbar_wait(&kv_empty[st], (use - 1) & 1, &wctl)) break;
        const int n0 = (J0 + jj) * kQN;
        mbar_arrive_expect_tx(&kv_full[st], LY::K_BYTES + LY::V_BYTES);
        for (int c = 0; c < KCH; ++c)
          tma_load_bh_hint(smem + LY::OFF_K + st * LY::K_BYTES + c * kQN * 128, &mK, &kv_full[st],
                           c * 64, krow0 + n0, kh, tb, p.Hk, p.kv_bshd != 0, pol);
        for (int c = 0; c < VCH; ++c)
          tma_load_bh_hint(smem + LY::OFF_V + st * LY::V_BYTES + c * kQN * 128, &mV, &kv_full[st],
                           c * 64, krow0 + n0, kh, tb, p.Hk, p.kv_bshd != 0, pol);
        last[st] = jj;
      }
      mbar_wait_drain(&q_full, 0);
      for (int s = 0; s < STAGES; ++s)
        if (last[s] >= 0) mbar_wait_drain(&kv_full[s], (last[s] / STAGES) & 1);
    }
  } else if (warp == LY::MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      const uint32_t sq = smem_u32(smem + LY::OFF_Q), sdo = smem_u32(smem + LY::OFF_DO);
      const uint32_t sk = smem_u32(smem + LY::OFF_K), sv = smem_u32(smem + LY::OFF_V);
      const Desc qa = make_desc(sq, 16, 1024);    // Q, K-major
      const Desc da = make_desc(sdo, 16, 1024);   // dO, K-major
      const uint32_t id_s = idesc_bf16(kQM, kQN, 0, 0);  // S, dP: [q x kv]
      const uint32_t id_dq = idesc_bf16(kQM, HD, 0, 1);  // dQ: A = dS (tmem), B = K MN-major
      const uint32_t tDQ = tbase + LY::COL_DQ;
      bool ok = mbar_wait(&q_full, 0, &wctl);
      tc_fence_after();

      auto issue_sdp = [&](int jj) {  // S(jj) = Q K^T, dP(jj) = dO V^T into buffer jj % 2
        const int st = jj % STAGES;
        ok = ok && mbar_wait(&kv_full[st], (jj / STAGES) & 1, &wctl);
        if (!ok) return;
        tc_fence_after();
        const uint32_t tS = tbase + LY::COL_S0 + (jj % 2) * kQN;
        const uint32_t tDP = tbase + LY::COL_DP0 + (jj % 2) * kQN;
        const Desc kb = make_desc(sk + st * LY::K_BYTES, 16, 1024);
        const Desc vb = make_desc(sv + st * LY::V_BYTES, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks)
          mma_ss2(tS, qa.at((ks / 4) * (kQM * 128) + (ks % 4) * 32), qa.hi,
                  kb.at((ks / 4) * (kQN * 128) + (ks % 4) * 32), kb.hi, id_s, ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < DV / 16; ++ks)
          mma_ss2(tDP, da.at((ks / 4) * (kQM * 128) + (ks % 4) * 32), da.hi,
                  vb.at((ks / 4) * (kQN * 128) + (ks % 4) * 32), vb.hi, id_s, ks > 0 ? 1u : 0u);
        mma_commit(&sdp_full[jj % 2]);
      };

      if (ntt > 0 && ok) issue_sdp(0);
      for (int jj = 0; jj < ntt && ok; ++jj) {
        const int st = jj % STAGES;
        // S/dP of the next tile go to the other buffer, last read by dQ(jj - 1), which was
        // issued before them (MMAs from one thread run in order)
        if (LY::LOOKAHEAD && jj + 1 < ntt) {
          issue_sdp(jj + 1);
          if (!ok) break;
        }
        ok = mbar_wait(&ds_ready[jj % 2], (jj / 2) & 1, &wctl);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tS = tbase + LY::COL_S0 + (jj % 2) * kQN;
        const Desc kmn = make_desc(sk + st * LY::K_BYTES, kQN * 128, 1024);  // K, MN-major
#pragma unroll
        for (int ks = 0; ks < kQN / 16; ++ks)
          mma_ts2(tDQ, tS + ks * 8, kmn.at(ks * 2048), kmn.hi, id_dq, (jj > 0 || ks > 0) ? 1u : 0u);
        mma_commit(&kv_empty[st]);  // K and V of this tile are no longer needed
        if (!LY::LOOKAHEAD && jj + 1 < ntt) issue_sdp(jj + 1);
      }
      mma_commit(&dq_final);
      mma_commit(&mma_drain);
      mbar_wait_drain(&mma_drain, 0);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------------ dS warpgroup
    const int r = warp * 32 + lane;  // query row within the tile == TMEM lane
    const int i = m0 + r;
    const uint32_t lane_base = tbase + ((uint32_t)(warp * 32) << 16);
    const int off = kl - ql;
    const int hi_off = WIN ? p.hi_off : 0;
    // visible keys of this row: [klo_row, khi_row]; the tile bounds decide interior tiles
    const int klo_row = WIN ? off + i + p.lo_off : 0;
    const int khi_row = BAND != kBandNone ? min(kl - 1, off + i + hi_off) : kl - 1;
    const int klo_tile = WIN ? off + r1 + p.lo_off : 0;
    const int khi_tile = BAND != kBandNone ? min(kl - 1, off + m0 + hi_off) : kl - 1;
    const float nl2 = p.lse2[(size_t)bh * p.ql_pad + i];  // i < ql_pad: padding rows hold -inf
    const float Dr = p.dvec[(size_t)bh * p.ql_pad + i];
    const float c2 = p.scale_log2;
    const void* mrow = nullptr;
    if (MASKT != 0 && i < ql) {
      const size_t es = MASKT == 1 ? 4 : MASKT == 2 ? 2 : 1;
      mrow = reinterpret_cast<const uint8_t*>(p.mask) +
             (b * p.msb + (long long)h * p.msh + (long long)i * p.msq) * es;
    }
    bool ok = true;
    for (int jj = 0; jj < ntt; ++jj) {
      const uint32_t colS = LY::COL_S0 + (jj % 2) * kQN;
      const uint32_t colDP = LY::COL_DP0 + (jj % 2) * kQN;
      ok = __all_sync(0xffffffffu, mbar_wait(&sdp_full[jj % 2], (jj / 2) & 1, &wctl));
      if (!ok) break;
      tc_fence_after();
      uint32_t rs[2][32], rd[2][32];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        tmem_ld32(lane_base + colS + c * 32, rs[c]);
        tmem_ld32(lane_base + colDP + c * 32, rd[c]);
      }
      tmem_wait_ld();
      const int n0 = (J0 + jj) * kQN;
      const bool edge = (n0 + kQN - 1 > khi_tile) || (WIN && n0 < klo_tile);
      const int lim_lo = klo_row - n0, lim_hi = khi_row - n0;  // c visible iff lo <= c <= hi
#pragma unroll
      for (int c32 = 0; c32 < 2; ++c32) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float ds2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int c = c32 * 32 + 2 * e + u;
            float x = fmaf(__uint_as_float(rs[c32][2 * e + u]), c2, nl2);
            if (MASKT != 0)
              x += (mrow != nullptr && n0 + c < kl) ? dq_mask_log2<MASKT>(mrow, n0 + c) : 0.0f;
            float pv = ex2(x);
            if (edge && ((WIN && c < lim_lo) || c > lim_hi)) pv = 0.0f;
            ds2[u] = pv * (__uint_as_float(rd[c32][2 * e + u]) - Dr);
          }
          pk[e] = pack_bf16(ds2[0], ds2[1]);
        }
        tmem_st16(lane_base + colS + c32 * 16, pk);  // dS as bf16 over the S columns
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&ds_ready[jj % 2]);
    }
    // ---------------------------------------------------------------- epilogue
    bool have = false;
    if (ok && ntt > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&dq_final, 0, &wctl));
      tc_fence_after();
      have = ok;
    }
    __nv_bfloat16* out =
        p.dq + bhsd_offset(ob, bh % p.H, or0 + (i < ql ? i : 0), p.H, orows, HD, p.q_bshd != 0);
#pragma unroll 1
    for (int c = 0; c < HD; c += 32) {
      uint32_t rq[32];
      if (have) {
        tmem_ld32(lane_base + LY::COL_DQ + c, rq);
        tmem_wait_ld();
      }
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        pk[e] = have ? pack_bf16(__uint_as_float(rq[2 * e]) * p.scale,
                                 __uint_as_float(rq[2 * e + 1]) * p.scale)
                     : 0u;
      if (i < ql) {
        uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)
          dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == LY::MMA_WARP) tmem_dealloc(tbase, LY::TMEM_COLS);
  if (threadIdx.x == 0) report_abort(&wctl, p.status);
}

// ------------------------------------------------------------------------ host side
int dq_det_box_rows() { return kQN; }  // kv rows of a K / V box (Q and dO boxes: 128)

template <int HD, int DV, int BAND, int MASKT>
static cudaError_t launch_dq_det_t(const BwdArgs& a, const DqMaps& m, cudaStream_t s) {
  using LY = DqLayout<HD, DV>;
  auto kern = bwd_dq_det_kernel<HD, DV, BAND, MASKT>;
  static OncePerKey<> smem_attr;  // per instantiation and device
  {
    const cudaError_t e = set_smem_once(smem_attr, kern, LY::SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  DqKParams kp;
  kp.mask = a.mask;
  kp.msb = a.mask_stride_b;
  kp.msh = a.mask_stride_h;
  kp.msq = a.mask_stride_q;
  kp.lse2 = a.lse2;
  kp.dvec = a.dvec;
  kp.dq = reinterpret_cast<__nv_bfloat16*>(a.dq);
  kp.q_bshd = a.q_bshd;
  kp.kv_bshd = a.kv_bshd;
  kp.status = a.status;
  kp.wait_limit_ns = a.wait_limit_ns;
  kp.cu_q = a.cu_q;
  kp.cu_k = a.cu_k;
  kp.total_q = a.total_q;
  kp.total_k = a.total_k;
  kp.H = a.H;
  kp.Hk = a.Hk;
  kp.ql = a.ql;
  kp.kl = a.kl;
  kp.ql_pad = a.ql_pad;
  kp.lo_off = a.lo_off;
  kp.hi_off = a.hi_off;
  kp.scale = a.scale;
  kp.scale_log2 = a.scale * kLog2eQ;
  kp.tiles_fast = a.cu_q != nullptr && a.B * a.H <= 65535;
  const int mt = (a.ql + kQM - 1) / kQM;
  dim3 grid(kp.tiles_fast ? mt : a.B * a.H, kp.tiles_fast ? a.B * a.H : mt);
  kern<<<grid, LY::THREADS, LY::SMEM_BYTES, s>>>(m.q, m.k, m.v, m.dO, kp);
  return cudaGetLastError();
}

template <int HD, int DV, int BAND>
static cudaError_t launch_dq_det_m(const BwdArgs& a, const DqMaps& m, cudaStream_t s) {
  if (!a.mask) return launch_dq_det_t<HD, DV, BAND, 0>(a, m, s);
  switch (a.mask_type) {
    case 0: return launch_dq_det_t<HD, DV, BAND, 1>(a, m, s);
    case 1: return launch_dq_det_t<HD, DV, BAND, 2>(a, m, s);
    default: return launch_dq_det_t<HD, DV, BAND, 3>(a, m, s);
  }
}

template <int HD, int DV>
static cudaError_t launch_dq_det_d(const BwdArgs& a, const DqMaps& m, cudaStream_t s) {
  switch (a.band) {
    case kBandNone: return launch_dq_det_m<HD, DV, kBandNone>(a, m, s);
    case kBandCausal: return launch_dq_det_m<HD, DV, kBandCausal>(a, m, s);
    default: return launch_dq_det_m<HD, DV, kBandWindow>(a, m, s);
  }
}

cudaError_t launch_dq_det(const BwdArgs& a, const DqMaps& m, cudaStream_t s) {
  profile_mark(kKernBwdDqDet, 0, s);
  cudaError_t e = cudaErrorInvalidValue;
  if (a.d == 64 && a.dval == 64) e = launch_dq_det_d<64, 64>(a, m, s);
  else if (a.d == 128 && a.dval == 128) e = launch_dq_det_d<128, 128>(a, m, s);
  else if (a.d == 256 && a.dval == 256) e = launch_dq_det_d<256, 256>(a, m, s);
  else if (a.d == 128 && a.dval == 64) e = launch_dq_det_d<128, 64>(a, m, s);
  profile_mark(kKernBwdDqDet, 1, s);
  return e;
}

}  // namespace fa
