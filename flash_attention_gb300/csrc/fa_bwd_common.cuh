// fa_bwd_common.cuh -- pieces shared by the backward's kv-tile-major kernels (fa_bwd.cu: the
// single-CTA main pass at head_dim 64 and 128; fa_bwd_pair.cu: the CTA-pair main pass at
// head_dim 256): tile traits, the kernel parameter block, the query-tile range of a kv tile
// under the visibility band, mask reads and the 128-byte-swizzled row store.
#pragma once

#include <float.h>

#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {

constexpr float kLog2eB = 1.4426950408889634f;

// ------------------------------------------------------------------------ traits / layout
// BM query rows per tile; DSPLIT: slices of the head dimension (one CTA per slice);
// ST: depth of the Q/dO ring; NSB: score buffers (S^T) in TMEM; DQT: dQ formed transposed.
// Two dP^T buffers are always used; the dQ tile of iteration `it` is written into the dP^T
// buffer of `it` once dK has consumed the dS^T stored there. LOOKAHEAD: issue the next tile's
// dP^T before this tile's dK (needs ST >= 2), so the dS warpgroup is fed while the tensor core
// forms dV, dK and dQ.
template <int HD>
struct BwdTraits;
// DQ_BULK: the dQ tile is staged in shared memory (f32, in the accumulator's tile layout below)
// and added to the accumulator by one bulk reduction (every head dim of the main pass does so:
// at head_dim 128, adding the tile from registers with 16-byte vector reductions measured 721
// against 641 us on the 4k causal GQA shape, and at 64 scattered reductions 189 against 171 us).
// SPLIT_MMA: in the deterministic mode (no dQ MMAs here) two warps issue the MMAs, one S^T and
// dP^T, the other dV and dK, so that neither stream waits behind the other's barrier waits and
// the issuing thread is less often starved of issue slots by the busy compute warps that share
// its scheduler (measured on the d128 causal workload: 572 -> 484 us). With dQ MMAs the single
// issuer's order measured faster (661 vs 671 us).
template <>
struct BwdTraits<64> {
  // (a 2-deep Q/dO ring leaves room for the bulk dQ staging tile)
  static constexpr int BM = 128, DSPLIT = 1, ST = 2, NSB = 1;
  static constexpr bool DQT = false, LOOKAHEAD = true, DQ_BULK = true;  // dQ = dS K (M = BM)
  static constexpr bool SPLIT_MMA = false;
};
template <>
struct BwdTraits<128> {
  static constexpr int BM = 64, DSPLIT = 1, ST = 3, NSB = 2;
  // dQ^T = K^T dS^T (M = head-dim slice)
  static constexpr bool DQT = true, LOOKAHEAD = true, DQ_BULK = true;
  static constexpr bool SPLIT_MMA = true;
};
// head_dim 256 runs in the CTA-pair kernel of fa_bwd_pair.cu; only its query tile (BM) and
// Q/dO ring depth are used from here.
template <>
struct BwdTraits<256> {
  static constexpr int BM = 64, DSPLIT = 2, ST = 2, NSB = 2;
  static constexpr bool DQT = true, LOOKAHEAD = true, DQ_BULK = true;
  static constexpr bool SPLIT_MMA = false;
};

constexpr int kBN = 128;  // kv rows per CTA (the M of the kv-major MMAs)

// Bulk dQ path: with dQ^T formed (head_dim 128 and 256) the accumulator tile of one (batch,
// head, query tile) is stored transposed and chunk-major: the 16-byte chunk c (query rows
// 4c .. 4c+3) of head-dim row d at 16-byte position (d / 128) * 128 * kDqChunks + c * 128 +
// d % 128, so that 32 consecutive lanes (rows) write 512 contiguous bytes, whether they stage
// the tile for a bulk reduction or add it with vector reductions (at head_dim 256 each CTA of
// the pair adds one 128-row half). With dQ formed (head_dim 64) the tile keeps query rows of
// HD f32, the chunk c (head-dim 4c .. 4c+3) of row q at c ^ (q % kDqChunks), so that 8
// consecutive staging lanes store to 8 distinct bank groups.
constexpr int kDqChunks = 16;  // 16-byte chunks per staged row (64 f32)

struct BwdKParams {
  const void* mask;         // additive f32 / bf16, or bool (uint8), addressed with the strides
  long long msb, msh, msq;  // mask strides (elements) of batch, head, query row
  const float* lse2;
  const float* dvec;
  float* dqacc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int* status;
  int H, Hk, ql, kl, ql_pad;
  int lo_off, hi_off;  // key j is visible to query row i iff q_abs + lo_off <= j <= q_abs + hi_off
  int skip_dq;         // 1: dQ comes from the deterministic dQ kernel; no dQ work here
  int tiles_fast;      // 1: blockIdx.x = kv tile, y = (batch, kv head, slice); 0: swapped
  const int32_t* cu_q;  // variable-length batch: sequence offsets (VARLEN kernels)
  const int32_t* cu_k;
  int total_q, total_k;
  int q_bshd, kv_bshd;  // 1: dq / dk, dv are [batch, rows, heads, d] (else [batch, heads, rows, d])
  float scale, scale_log2;
  unsigned long long wait_limit_ns;  // limit of one barrier wait
};

// Kernel parameters of a backward launch (every field but tiles_fast).
inline BwdKParams make_bwd_kparams(const BwdArgs& a) {
  BwdKParams kp;
  kp.mask = a.mask;
  kp.msb = a.mask_stride_b;
  kp.msh = a.mask_stride_h;
  kp.msq = a.mask_stride_q;
  kp.lo_off = a.lo_off;
  kp.hi_off = a.hi_off;
  kp.skip_dq = a.deterministic ? 1 : 0;
  kp.cu_q = a.cu_q;
  kp.cu_k = a.cu_k;
  kp.total_q = a.total_q;
  kp.total_k = a.total_k;
  kp.q_bshd = a.q_bshd;
  kp.kv_bshd = a.kv_bshd;
  kp.lse2 = a.lse2;
  kp.dvec = a.dvec;
  kp.dqacc = a.dqacc;
  kp.dk = reinterpret_cast<__nv_bfloat16*>(a.dk);
  kp.dv = reinterpret_cast<__nv_bfloat16*>(a.dv);
  kp.status = a.status;
  kp.wait_limit_ns = a.wait_limit_ns;
  kp.H = a.H;
  kp.Hk = a.Hk;
  kp.ql = a.ql;
  kp.kl = a.kl;
  kp.ql_pad = a.ql_pad;
  kp.scale = a.scale;
  kp.scale_log2 = a.scale * kLog2eB;
  kp.tiles_fast = 0;
  return kp;
}

// Query tiles [first, last] whose rows see some key of the kv tile starting at n0: rows i with
// q_abs + lo_off <= j <= q_abs + hi_off for some j in the tile (q_abs = kl - ql + i). Under the
// causal band alone, key n0 is visible to the rows from n0 - (kl - ql) on, and to the last row.
template <int HD, int BAND>
__device__ __forceinline__ void bwd_mtile_range(int n0, const BwdKParams& p, int ql, int kl,
                                                int& first, int& last) {
  constexpr int BM = BwdTraits<HD>::BM;
  const int n_mt = (ql + BM - 1) / BM;
  if (BAND != kBandWindow) {
    first = 0;
    if (BAND == kBandCausal) {
      const int first_row = n0 - (kl - ql);
      first = first_row <= 0 ? 0 : first_row / BM;
    }
    last = n_mt - 1;
    return;
  }
  const long long off = (long long)kl - ql;
  const long long n1 = min(n0 + kBN, kl) - 1;
  const long long imin = max(0LL, (long long)n0 - off - p.hi_off);
  const long long imax = min((long long)ql - 1, n1 - off - p.lo_off);
  if (imax < imin) {
    first = 0;
    last = -1;
    return;
  }
  first = (int)(imin / BM);
  last = (int)(imax / BM);
}

// Mask value at element offset `e` from `base`, as a base-2 additive term.
template <int MASKT>
__device__ __forceinline__ float mask_log2_b(const void* base, long long e) {
  if constexpr (MASKT == 1) return reinterpret_cast<const float*>(base)[e] * kLog2eB;
  if constexpr (MASKT == 2)
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[e]) * kLog2eB;
  if constexpr (MASKT == 3) return reinterpret_cast<const uint8_t*>(base)[e] ? 0.0f : -INFINITY;
  return 0.0f;
}

// Writes 8 bf16 (one 16-byte granule g of row j) into a 128-byte-swizzled tile chunk.
__device__ __forceinline__ void st_swizzled(uint8_t* chunk, int j, int g, uint4 val) {
  *reinterpret_cast<uint4*>(chunk + j * 128 + ((g ^ (j & 7)) << 4)) = val;
}

}  // namespace fa
