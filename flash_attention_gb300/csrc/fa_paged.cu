// fa_paged.cu -- attention of a few new queries per sequence over a paged key/value cache
// (single-query decode, and the short causal prefill against a cache), sm_103a.
//
// Definition (page "nuvec-core tests/fast.rs", `paged_attention_equals_contiguous_attention`):
// the keys of sequence b are its first len_b cache positions; logical key j sits in page
// block_table[b][j / page_size], slot j % page_size, of caches [num_pages, Hk, page_size, d].
// The q_len queries are the sequence's last positions: with the causal mask query i sees key
// j iff j <= len_b - q_len + i. O = softmax(scale Q K^T) V and L = log sum exp per query. Page
// "tang src/compute/cuda.rs" (`kv_attention`) gives the decode (q_len = 1) and the cached
// prefill (len = cache_start + q_len) cases, and the nuvec-core test splits the keys into
// two passes above about 1024 of them.
//
// GB300 design. Decoding reads every key and value once and does 2 * G * q_len FLOPs per key
// element, so it is bound by HBM bandwidth, not by the tensor core:
//  * one CTA owns one (split, sequence, kv head) and up to 128 query rows: the G query heads
//    of the kv head times q_len queries are packed into the M = 128 rows of one tcgen05 tile
//    (Q viewed as [B * Hk, G * q_len, d]), so each K/V page is read once for all of them;
//  * one warp streams the pages with TMA through K and V rings (boxes of min(page_size, 64)
//    rows, 128-byte swizzle), the block-table entries staged in shared memory a chunk at a
//    time, and the box copies of a tile issued by all 32 lanes (small boxes issued by one
//    thread queue behind each other); a page the table does not name, or positions past the
//    sequence's end in a later page, are read as out-of-bounds boxes, which TMA fills with
//    zeros; before the last tile's P V the V rows past the sequence's end are zeroed, so
//    that whatever the cache holds there (NaN included) cannot reach O;
//  * one warp issues S = Q K^T into double-buffered TMEM as soon as its K tile has landed
//    (and frees that K stage when S is done); another issues O += P V with P read from TMEM
//    (and frees the V stage), so neither kind of MMA waits for the other's operands;
//  * one warpgroup (thread = query row = TMEM lane) runs the online softmax with the lazy
//    rescale of the training forward;
//  * with more than one split, each CTA writes its normalised partial O and its L, and a
//    combine kernel merges them: L = log sum_s exp(L_s), O = sum_s exp(L_s - L) O_s.
#include <float.h>

#include <algorithm>

#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {

namespace {
constexpr int kPM = 128;  // query rows per CTA (the MMA M)
constexpr int kPN = 64;   // keys per tile
constexpr float kLog2eP = 1.4426950408889634f;
constexpr float kLn2P = 0.6931471805599453f;
constexpr float kRescaleP = 8.0f;
constexpr int kPageChunk = 512;  // block-table entries staged in shared memory at a time
}  // namespace

template <int HD>
struct PagedLayout {
  // K/V ring depth; at head_dim <= 128 two CTAs fit on an SM (one streams while the other
  // starts or finishes)
  static constexpr int STAGES = HD == 64 ? 4 : 2;
  static constexpr int KCH = HD / 64;
  static constexpr int Q_BYTES = kPM * HD * 2;
  static constexpr int KV_BYTES = kPN * HD * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_END = OFF_V + STAGES * KV_BYTES;
  static constexpr int SMEM_BYTES = OFF_END + 1024;
  // TMEM columns: O, then two S buffers
  static constexpr int COL_O = 0;
  static constexpr int COL_S0 = HD;
  static constexpr int TMEM_USED = HD + 2 * kPN;
  static constexpr int TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
  // warps 0-3 softmax, warp 4 TMA, warp 5 issues S = Q K^T, warp 6 issues O += P V
  static constexpr int THREADS = 224;
  static constexpr int TMA_WARP = 4, S_WARP = 5, PV_WARP = 6;
  static_assert(TMEM_USED <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

struct PagedKParams {
  const int32_t* table;  // [B, max_pages]
  const int32_t* lens;   // [B]
  __nv_bfloat16* o;      // [B, H, lq, HD] (one split)
  float* lse;            // [B, H, lq] or nullptr (one split)
  float* o_part;         // [splits, B * Hk, rows, HD] (several splits)
  float* l_part;         // [splits, B * Hk, rows]
  int* status;
  int H, Hk, G, lq, rows, bs, max_pages, num_pages, kps, n_splits;
  float scale_log2;
  unsigned long long wait_limit_ns;  // limit of one barrier wait
};

template <int HD, bool CAUSAL>
__global__ void __launch_bounds__(PagedLayout<HD>::THREADS, 1)
    paged_attn_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                      const __grid_constant__ CUtensorMap mV, const PagedKParams p) {
  using LY = PagedLayout<HD>;
  constexpr int ST = LY::STAGES, KCH = LY::KCH;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ uint64_t q_full, k_full[ST], v_full[ST], k_empty[ST], v_empty[ST];
  __shared__ uint64_t s_full[2], p_full[2], pv_done[2], o_done, o_final, drain_s, drain_pv;
  __shared__ uint32_t tmem_base_s;
  __shared__ WaitCtl wctl;
  __shared__ int bad_input;
  __shared__ int page_s[kPageChunk];  // block-table entries [chunk_base, chunk_base + 512)

  const int warp = warp_id(), lane = lane_id();
  const int split = blockIdx.x;
  const int bkh = blockIdx.y;  // b * Hk + kh
  const int b = bkh / p.Hk, kh = bkh % p.Hk;
  const int r0 = (int)blockIdx.z * kPM;
  const int cap = p.max_pages * p.bs;
  const int raw_len = p.lens[b];
  const int len = raw_len < 0 ? 0 : (raw_len > cap ? cap : raw_len);
  const int k0 = split * p.kps;
  const int k1 = min(k0 + p.kps, len);
  const int ntt = k1 > k0 ? (k1 - k0 + kPN - 1) / kPN : 0;  // key tiles of this CTA
  // softmax warps that own at least one real query row (rows past G * q_len are padding of
  // the M = 128 tile: their P and O rows are never used, so their warps skip the work)
  const int live_warps = min(4, (min(p.rows - r0, kPM) + 31) / 32);

  if (threadIdx.x == 0) {
    wait_ctl_init(&wctl, p.wait_limit_ns);
    bad_input = raw_len != len;
    mbar_init(&q_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 32 * live_warps);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(&o_done, 1);
    mbar_init(&o_final, 1);
    mbar_init(&drain_s, 1);
    mbar_init(&drain_pv, 1);
    fence_barrier_init();
  }
  if (warp == LY::S_WARP) {
    tmem_alloc(&tmem_base_s, LY::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_s;

  if (warp == LY::TMA_WARP) {
    // ------------------------------------------------------------------ TMA producer: the
    // warp stages the block-table entries in shared memory (coalesced, a chunk at a time),
    // lane 0 issues the copies
    const bool leader = lane == 0;
    if (leader) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mV);
      if (ntt > 0) {
        mbar_arrive_expect_tx(&q_full, LY::Q_BYTES);
        for (int c = 0; c < KCH; ++c)
          tma_load_3d(smem + LY::OFF_Q + c * kPM * 128, &mQ, &q_full, c * 64, r0, bkh);
      }
    }
    const int box = p.bs < kPN ? p.bs : kPN;  // rows per TMA box
    const int nsub = kPN / box;                // boxes per key tile (<= 8)
    const int z_oob = p.num_pages * p.Hk;      // a page index past the cache: zero fill
    const int used_pages = (len + p.bs - 1) / p.bs;  // table entries of this sequence
    const int32_t* trow = p.table + (size_t)b * p.max_pages;
    int chunk_base = -1;  // first table entry held in page_s (-1: none)
    int last_k[ST], last_v[ST];
    for (int s = 0; s < ST; ++s) last_k[s] = last_v[s] = -1;
    // Makes page_s hold the table entries of tiles jt .. jt + 1 (warp-wide).
    auto stage_pages = [&](int jt) {
      const int p_first = (k0 + jt * kPN) / p.bs;
      const int p_last = min(used_pages - 1, (k0 + (jt + 2) * kPN - 1) / p.bs);
      if (chunk_base >= 0 && p_first >= chunk_base && p_last < chunk_base + kPageChunk) return;
      chunk_base = p_first;
      __syncwarp();  // the old chunk is no longer read
      for (int e = lane; e < kPageChunk; e += 32) {
        const int idx = chunk_base + e;
        int pg = -1;
        if (idx < used_pages) {  // < max_pages because len <= max_pages * page_size
          pg = trow[idx];
          if (pg < 0 || pg >= p.num_pages) {
            pg = -1;
            bad_input = 1;
          }
        }
        page_s[e] = pg;
      }
      __syncwarp();
    };
    // The copies of tile jt into stage jt % ST of the K (which = 0) or V ring (warp-wide): lane
    // 0 waits for the stage and sets the byte count, then the lanes issue the nsub * KCH box
    // copies in parallel (issued by one thread, small boxes queue behind each other).
    auto issue = [&](int jt, int which) -> bool {
      const int st = jt % ST;
      const uint32_t use = jt / ST;
      uint64_t* empty = which == 0 ? &k_empty[st] : &v_empty[st];
      uint64_t* full = which == 0 ? &k_full[st] : &v_full[st];
      bool ok = true;
      if (leader) {
        if (use > 0) ok = mbar_wait(empty, (use - 1) & 1, &wctl);
        if (ok) mbar_arrive_expect_tx(full, LY::KV_BYTES);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      const int n0 = k0 + jt * kPN;
      uint8_t* dst = smem + (which == 0 ? LY::OFF_K : LY::OFF_V) + st * LY::KV_BYTES;
      const CUtensorMap* map = which == 0 ? &mK : &mV;
      for (int e = lane; e < nsub * KCH; e += 32) {
        const int sub = e / KCH, c = e % KCH;
        const int key = n0 + sub * box;
        int z = z_oob, y = 0;
        if (key < len) {
          const int pg = page_s[key / p.bs - chunk_base];
          if (pg >= 0) {
            z = pg * p.Hk + kh;
            y = key % p.bs;
          }
        }
        tma_load_3d(dst + c * kPN * 128 + sub * box * 128, map, full, c * 64, y, z);
      }
      if (leader) (which == 0 ? last_k : last_v)[st] = jt;
      return true;
    };
    // K runs one tile ahead of V: S needs K earlier than P V needs V
    bool ok = true;
    if (ntt > 0) {
      stage_pages(0);
      ok = issue(0, 0);
    }
    for (int jj = 0; jj < ntt && ok; ++jj) {
      stage_pages(jj);
      if (jj + 1 < ntt) ok = issue(jj + 1, 0);
      if (ok) ok = issue(jj, 1);
    }
    if (leader) {
      if (ntt > 0) mbar_wait_drain(&q_full, 0);
      for (int s = 0; s < ST; ++s) {
        if (last_k[s] >= 0) mbar_wait_drain(&k_full[s], (last_k[s] / ST) & 1);
        if (last_v[s] >= 0) mbar_wait_drain(&v_full[s], (last_v[s] / ST) & 1);
      }
    }
  } else if (warp == LY::S_WARP) {
    // ------------------------------------------------------------------ S = Q K^T issuer: S(jj)
    // into buffer jj % 2 once K(jj) has landed and P V(jj - 2) has read that buffer; the K
    // stage is released as soon as S(jj) is done, so K loads run ahead of P V
    if (elect_one()) {
      const uint32_t sq = smem_u32(smem + LY::OFF_Q), sk = smem_u32(smem + LY::OFF_K);
      const uint32_t id_s = idesc_bf16(kPM, kPN, 0, 0);
      const Desc qa = make_desc(sq, 16, 1024);
      bool ok = ntt == 0 || mbar_wait(&q_full, 0, &wctl);
      tc_fence_after();
      for (int jj = 0; jj < ntt && ok; ++jj) {
        const int st = jj % ST;
        ok = mbar_wait(&k_full[st], (jj / ST) & 1, &wctl);
        if (ok && jj >= 2) ok = mbar_wait(&pv_done[jj % 2], ((jj - 2) / 2) & 1, &wctl);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tS = tbase + LY::COL_S0 + (jj % 2) * kPN;
        const Desc kb = make_desc(sk + st * LY::KV_BYTES, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks)
          mma_ss2(tS, qa.at((ks / 4) * (kPM * 128) + (ks % 4) * 32), qa.hi,
                  kb.at((ks / 4) * (kPN * 128) + (ks % 4) * 32), kb.hi, id_s, ks > 0 ? 1u : 0u);
        mma_commit(&s_full[jj % 2]);
        mma_commit(&k_empty[st]);
      }
      mma_commit(&drain_s);
      mbar_wait_drain(&drain_s, 0);
    }
  } else if (warp == LY::PV_WARP) {
    // ------------------------------------------------------------------ O += P V issuer (lane 0;
    // the whole warp zeroes the tail of the last V tile)
    const bool leader = lane == 0;
    const uint32_t sv = smem_u32(smem + LY::OFF_V);
    const uint32_t id_o = idesc_bf16(kPM, HD, 0, 1);
    const uint32_t tO = tbase + LY::COL_O;
    bool ok = true;
    for (int jj = 0; jj < ntt && ok; ++jj) {
      const int st = jj % ST;
      const int n0 = k0 + jj * kPN;
      ok = __all_sync(0xffffffffu, mbar_wait(&p_full[jj % 2], (jj / 2) & 1, &wctl));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&v_full[st], (jj / ST) & 1, &wctl));
      if (!ok) break;
      if (n0 + kPN > len) {
        // rows len - n0 .. kPN - 1 of this V tile hold no key of the sequence (the rest of the
        // page): zero all of their 128-byte rows
        uint8_t* vt = smem + LY::OFF_V + st * LY::KV_BYTES;
        const int r_first = len - n0;
        const int items = (kPN - r_first) * KCH * 8;  // 16-byte granules
        for (int e = lane; e < items; e += 32) {
          const int g = e % 8, c = (e / 8) % KCH, row = r_first + e / (8 * KCH);
          *reinterpret_cast<uint4*>(vt + c * kPN * 128 + row * 128 + g * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async();  // generic-proxy writes -> visible to the tensor core
        __syncwarp();
      }
      tc_fence_after();
      if (leader) {
        const uint32_t tP = tbase + LY::COL_S0 + (jj % 2) * kPN;
        const Desc vb = make_desc(sv + st * LY::KV_BYTES, kPN * 128, 1024);  // V, MN-major
#pragma unroll
        for (int ks = 0; ks < kPN / 16; ++ks)
          mma_ts2(tO, tP + ks * 8, vb.at(ks * 2048), vb.hi, id_o, (jj > 0 || ks > 0) ? 1u : 0u);
        mma_commit(&o_done);
        mma_commit(&pv_done[jj % 2]);
        if (jj == ntt - 1) mma_commit(&o_final);
        mma_commit(&v_empty[st]);
      }
      __syncwarp();
    }
    if (leader) {
      mma_commit(&drain_pv);
      mbar_wait_drain(&drain_pv, 0);
    }
    __syncwarp();
  } else if (warp < live_warps) {
    // ------------------------------------------------------------------ softmax warpgroup
    const int r = warp * 32 + lane;
    const int R = r0 + r;  // row of the (sequence, kv head) group: g * lq + i
    const bool valid = R < p.rows;
    const int g = valid ? R / p.lq : 0, i = valid ? R % p.lq : 0;
    const int h = kh * p.G + g;
    // visible keys of this row: [0, khi_row]; tiles past khi_tile need the per-key test
    const int q_abs = len - p.lq + i;
    const int khi_row = !valid ? -1 : (CAUSAL ? min(len - 1, q_abs) : len - 1);
    const int khi_tile = CAUSAL ? min(len - 1, len - p.lq) : len - 1;
    const uint32_t lane_base = tbase + ((uint32_t)(warp * 32) << 16);
    const float c2 = p.scale_log2;
    float m_used = -FLT_MAX / 2.0f;
    float l = 0.0f;
    bool ok = true;
    for (int jj = 0; jj < ntt; ++jj) {
      const uint32_t colS = LY::COL_S0 + (jj % 2) * kPN;
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[jj % 2], (jj / 2) & 1, &wctl));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[2][32];
      tmem_ld32(lane_base + colS, sr[0]);
      tmem_ld32(lane_base + colS + 32, sr[1]);
      tmem_wait_ld();
      const int n0 = k0 + jj * kPN;
      if (n0 + kPN - 1 > khi_tile || !valid) {
        const int lim = khi_row - n0;  // column c visible iff c <= lim
#pragma unroll
        for (int c32 = 0; c32 < 2; ++c32)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c32 * 32 + e > lim) sr[c32][e] = __float_as_uint(-INFINITY);
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c32 = 0; c32 < 2; ++c32)
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          mx = fmax3(mx, __uint_as_float(sr[c32][e]), __uint_as_float(sr[c32][e + 1]));
      const float m_new = fmaxf(m_used, mx * c2);
      const bool need = m_new > m_used + kRescaleP;
      if (__any_sync(0xffffffffu, need)) {
        const float factor = ex2(m_used - m_new);
        l *= factor;
        if (jj > 0) {
          // O holds P V of tiles < jj; S(jj) was issued after P V(jj - 2), so only the last
          // P V can be outstanding and the parity wait is exact
          ok = __all_sync(0xffffffffu, mbar_wait(&o_done, (jj - 1) & 1, &wctl));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < HD; c += 32) {
            uint32_t orr[32];
            tmem_ld32(lane_base + LY::COL_O + c, orr);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * factor);
            tmem_st32(lane_base + LY::COL_O + c, orr);
          }
          tmem_wait_st();
        }
        m_used = m_new;
      }
      float rs = 0.0f;
#pragma unroll
      for (int c32 = 0; c32 < 2; ++c32) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ex2(fmaf(__uint_as_float(sr[c32][2 * e]), c2, -m_used));
          const float p1 = ex2(fmaf(__uint_as_float(sr[c32][2 * e + 1]), c2, -m_used));
          rs += p0 + p1;
          pk[e] = pack_bf16(p0, p1);
        }
        tmem_st16(lane_base + colS + c32 * 16, pk);
      }
      l += rs;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[jj % 2]);
    }
    // ---------------------------------------------------------------- epilogue
    if (ok && ntt > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&o_final, 0, &wctl));
      tc_fence_after();
    }
    const bool have_o = ok && ntt > 0 && l > 0.0f;
    const float inv = have_o ? 1.0f / l : 0.0f;
    const float L = have_o ? m_used * kLn2P + logf(l) : -INFINITY;
    const bool one = p.n_splits == 1;
    const size_t orow = ((size_t)(b * p.H + h) * p.lq + i);                       // one split
    const size_t prow = ((size_t)split * gridDim.y + bkh) * (size_t)p.rows + R;  // partials
#pragma unroll 1
    for (int c = 0; c < HD; c += 32) {
      uint32_t orr[32];
      if (ok && ntt > 0) {
        tmem_ld32(lane_base + LY::COL_O + c, orr);
        tmem_wait_ld();
      }
      if (!valid) continue;
      if (one) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = have_o ? pack_bf16(__uint_as_float(orr[2 * e]) * inv,
                                     __uint_as_float(orr[2 * e + 1]) * inv)
                         : 0u;
        uint4* dst = reinterpret_cast<uint4*>(p.o + orow * HD + c);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)
          dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
      } else {
        float4* dst = reinterpret_cast<float4*>(p.o_part + prow * HD + c);
#pragma unroll
        for (int v4 = 0; v4 < 8; ++v4)
          dst[v4] = have_o ? make_float4(__uint_as_float(orr[4 * v4]) * inv,
                                         __uint_as_float(orr[4 * v4 + 1]) * inv,
                                         __uint_as_float(orr[4 * v4 + 2]) * inv,
                                         __uint_as_float(orr[4 * v4 + 3]) * inv)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (valid) {
      if (one) {
        if (p.lse) p.lse[orow] = L;
      } else {
        p.l_part[prow] = L;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == LY::S_WARP) tmem_dealloc(tbase, LY::TMEM_COLS);
  if (threadIdx.x == 0) {
    report_abort(&wctl, p.status);
    if (bad_input && p.status) atomicCAS(p.status, kStatusOk, kStatusBadInput);
  }
}

// Merges the splits of every query row: L = log sum_s exp(L_s), O = sum_s exp(L_s - L) O_s
// (O = 0 and L = -inf when no split saw a key). A group of HD / 8 threads owns one row.
template <int HD>
__global__ void __launch_bounds__(256) paged_combine_kernel(const float* __restrict__ o_part,
                                                            const float* __restrict__ l_part,
                                                            __nv_bfloat16* __restrict__ o,
                                                            float* __restrict__ lse, int n_splits,
                                                            int n_rows, int Hk, int G, int lq,
                                                            int H) {
  constexpr int TPR = HD / 8;
  const long long row = (long long)blockIdx.x * (256 / TPR) + threadIdx.x / TPR;
  const int c = (threadIdx.x % TPR) * 8;
  if (row >= n_rows) return;
  const int rows = G * lq;
  const long long bkh = row / rows;
  const int R = (int)(row % rows);
  const int b = (int)(bkh / Hk), kh = (int)(bkh % Hk);
  const int h = kh * G + R / lq, i = R % lq;
  float mx = -INFINITY;
  for (int s = 0; s < n_splits; ++s) mx = fmaxf(mx, l_part[(size_t)s * n_rows + row]);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float L = -INFINITY;
  if (mx != -INFINITY) {
    float z = 0.0f;
    for (int s = 0; s < n_splits; ++s) z += expf(l_part[(size_t)s * n_rows + row] - mx);
    L = mx + logf(z);
    for (int s = 0; s < n_splits; ++s) {
      const float ls = l_part[(size_t)s * n_rows + row];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - L);
      const float4* src = reinterpret_cast<const float4*>(o_part + ((size_t)s * n_rows + row) * HD + c);
      const float4 a = src[0], d = src[1];
      acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
      acc[4] += w * d.x; acc[5] += w * d.y; acc[6] += w * d.z; acc[7] += w * d.w;
    }
  }
  const size_t orow = (size_t)(b * H + h) * lq + i;
  uint4 out;
  out.x = pack_bf16(acc[0], acc[1]);
  out.y = pack_bf16(acc[2], acc[3]);
  out.z = pack_bf16(acc[4], acc[5]);
  out.w = pack_bf16(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(o + orow * HD + c) = out;
  if (lse && c == 0) lse[orow] = L;
}

// ------------------------------------------------------------------------ host side
int paged_key_box_rows(int page_size) { return page_size < kPN ? page_size : kPN; }
int paged_query_box_rows() { return kPM; }

int paged_splits(const PagedArgs& a) {
  const long long cap = (long long)a.max_pages * a.bs;
  if (a.num_splits > 0) return (int)std::min<long long>(a.num_splits, (cap + kPN - 1) / kPN);
  if (cap <= 1024) return 1;  // one pass
  // about 2048 keys per split (short enough to balance sequences of mixed lengths over the
  // SMs, long enough to amortise a CTA's start), and enough CTAs to fill the GPU
  const long long ctas = (long long)a.B * a.Hk * ((a.G * a.lq + kPM - 1) / kPM);
  long long s = std::max<long long>(2, (cap + 2047) / 2048);
  s = std::max<long long>(s, (2 * 152 + ctas - 1) / ctas);
  s = std::min<long long>(s, (cap + 255) / 256);  // at least 256 keys per split
  return (int)std::max<long long>(1, s);
}

size_t paged_workspace_bytes(const PagedArgs& a, int splits) {
  if (splits <= 1) return 0;
  const size_t rows = (size_t)a.B * a.Hk * a.G * a.lq;
  return ((size_t)splits * rows * a.d * 4 + 255) / 256 * 256 + (size_t)splits * rows * 4;
}

template <int HD, bool CAUSAL>
static cudaError_t launch_paged_t(const PagedArgs& a, const PagedMaps& m, int splits, void* ws,
                                  cudaStream_t s) {
  using LY = PagedLayout<HD>;
  auto kern = paged_attn_kernel<HD, CAUSAL>;
  static OncePerKey<> smem_attr;  // per instantiation and device
  {
    const cudaError_t e = set_smem_once(smem_attr, kern, LY::SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  const long long cap = (long long)a.max_pages * a.bs;
  const long long per = (cap + splits - 1) / splits;
  PagedKParams kp;
  kp.table = a.table;
  kp.lens = a.lens;
  kp.o = reinterpret_cast<__nv_bfloat16*>(a.o);
  kp.lse = a.lse;
  const size_t rows_all = (size_t)a.B * a.Hk * a.G * a.lq;
  kp.o_part = splits > 1 ? static_cast<float*>(ws) : nullptr;
  kp.l_part = splits > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                                    ((size_t)splits * rows_all * HD * 4 + 255) / 256 * 256)
                         : nullptr;
  kp.status = a.status;
  kp.wait_limit_ns = a.wait_limit_ns;
  kp.H = a.H;
  kp.Hk = a.Hk;
  kp.G = a.G;
  kp.lq = a.lq;
  kp.rows = a.G * a.lq;
  kp.bs = a.bs;
  kp.max_pages = a.max_pages;
  kp.num_pages = a.num_pages;
  kp.kps = (int)((per + kPN - 1) / kPN * kPN);
  kp.n_splits = splits;
  kp.scale_log2 = a.scale * kLog2eP;
  dim3 grid(splits, a.B * a.Hk, (kp.rows + kPM - 1) / kPM);
  profile_mark(kKernPaged, 0, s);
  kern<<<grid, LY::THREADS, LY::SMEM_BYTES, s>>>(m.q, m.k, m.v, kp);
  cudaError_t e = cudaGetLastError();
  profile_mark(kKernPaged, 1, s);
  if (e != cudaSuccess || splits == 1) return e;
  const int n_rows = (int)rows_all;
  const int rpb = 256 / (HD / 8);
  profile_mark(kKernPagedCombine, 0, s);
  paged_combine_kernel<HD><<<(n_rows + rpb - 1) / rpb, 256, 0, s>>>(
      kp.o_part, kp.l_part, kp.o, a.lse, splits, n_rows, a.Hk, a.G, a.lq, a.H);
  e = cudaGetLastError();
  profile_mark(kKernPagedCombine, 1, s);
  return e;
}

cudaError_t launch_paged(const PagedArgs& a, const PagedMaps& m, int splits, void* ws,
                         cudaStream_t s) {
  switch (a.d) {
    case 64: return a.causal ? launch_paged_t<64, true>(a, m, splits, ws, s)
                             : launch_paged_t<64, false>(a, m, splits, ws, s);
    case 128: return a.causal ? launch_paged_t<128, true>(a, m, splits, ws, s)
                              : launch_paged_t<128, false>(a, m, splits, ws, s);
    case 256: return a.causal ? launch_paged_t<256, true>(a, m, splits, ws, s)
                              : launch_paged_t<256, false>(a, m, splits, ws, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa
