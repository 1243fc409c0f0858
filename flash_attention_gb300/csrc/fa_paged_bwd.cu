// fa_paged_bwd.cu -- gradients through the paged key/value cache (sm_103a): dQ and the
// gradients of both caches, for the decode / cached-prefill attention of fa_paged.cu.
//
// Method: page "nuvec-core tests/fast.rs", `paged_attention_equals_contiguous_attention`, takes
// the gradients of the paged attention with respect to q and the caches ("paged grads"). Each
// sequence is the attention problem on the keys its block table names (its query i sees keys
// j <= length - q_len + i under the causal rule), so its gradients are the training
// backward's on those keys. The call turns the batch into a variable-length batch:
//   1. offsets: cu_k = prefix sums of the lengths, cu_q = b * rows per sequence;
//   2. gather: each sequence's used keys and values, page by page, into K, V packed head-major
//      without padding ([Hk, total keys, d]); every used page records which (sequence, table
//      slot) uses it; q, O, dO and L go into the packed head-major layout too. With decode
//      (q_len = 1) or without the causal rule no query row's keys depend on its position, so
//      the G query heads of a kv head become one sequence's G * q_len rows ("pack"): the
//      backward then reads each key tile once per kv head instead of once per query head;
//   3. the training backward on that batch (fa_bwd.cu, fa_bwd_pair.cu);
//   4. scatter: every cache slot gets its gradient from the packed dK, dV through its page's
//      owner, or 0 when no sequence reads it; dq goes back to [B, H, q_len, d].
// A page used by two sequences (or twice by one) would need the contributions summed; it gets
// a zero gradient and FA_ERR_BAD_INPUT is reported. With few query rows per kv head the
// decode path below replaces steps 1-4.
#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {

namespace {
__device__ __forceinline__ void report_bad(int* status) {
  if (status) atomicCAS(status, kStatusOk, kStatusBadInput);
}

__device__ __forceinline__ long long paged_cap(const PagedGradArgs& a) {
  return (long long)a.max_pages * a.ps;
}

// Query rows per sequence in the packed problem.
__device__ __forceinline__ int paged_rq(const PagedGradArgs& a) {
  return a.pack ? (a.H / a.Hk) * a.lq : a.lq;
}
}  // namespace

// One block of 1024 threads: cu_k (prefix sums of the lengths, each clamped to
// [0, capacity] with a report) and cu_q, 1024 sequences per pass.
__global__ void __launch_bounds__(1024) paged_index_kernel(PagedGradArgs a) {
  __shared__ int warp_sum[32];
  __shared__ int carry;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long cap = paged_cap(a);
  const int rq = paged_rq(a);
  if (threadIdx.x == 0) {
    carry = 0;
    a.cu_k[0] = 0;
    a.cu_q[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < a.B; base += 1024) {
    const int b = base + threadIdx.x;
    int len = 0;
    if (b < a.B) {
      len = a.lens[b];
      if (len < 0 || len > cap) {
        report_bad(a.status);
        len = len < 0 ? 0 : (int)cap;
      }
    }
    int v = len;  // inclusive scan within the warp, then over the warp totals
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += n;
    }
    if (lane == 31) warp_sum[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sum[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += n;
      }
      warp_sum[lane] = w;
    }
    __syncthreads();
    const int incl = carry + v + (warp > 0 ? warp_sum[warp - 1] : 0);
    if (b < a.B) {
      a.cu_k[b + 1] = incl;
      a.cu_q[b + 1] = (b + 1) * rq;
    }
    __syncthreads();  // every thread has read carry and warp_sum
    if (threadIdx.x == 1023) carry = incl;
    __syncthreads();
  }
}

// Grid (ceil(capacity * d / 8 / 256), batch * Hk); each thread moves one 16-byte chunk of one
// used key row of K and of V into the packed tensors. The first thread of each used
// (sequence, page slot) records the page's owner.
__global__ void __launch_bounds__(256) paged_gather_kernel(PagedGradArgs a) {
  const int bkh = blockIdx.y, b = bkh / a.Hk, kh = bkh % a.Hk;
  const int cpr = a.d / 8;  // 16-byte chunks per row
  const long long e = (long long)blockIdx.x * 256 + threadIdx.x;
  const long long r = e >> a.cpr_shift;
  const int c = (int)(e & (cpr - 1));
  const int k0 = a.cu_k[b], len = a.cu_k[b + 1] - k0;
  if (r >= len) return;
  const long long total_k = (long long)a.B * paged_cap(a);  // rows per head of k_pack
  const int slot = (int)(r >> a.ps_shift);
  const int in_page = (int)(r & (a.ps - 1));
  const int page = a.table[(size_t)b * a.max_pages + slot];
  const bool lead = kh == 0 && c == 0 && in_page == 0;
  uint4 kv = make_uint4(0, 0, 0, 0), vv = kv;
  if (page >= 0 && page < a.num_pages) {
    const size_t src = (((size_t)page * a.Hk + kh) * a.ps + in_page) * cpr + c;
    kv = reinterpret_cast<const uint4*>(a.k_cache)[src];
    vv = reinterpret_cast<const uint4*>(a.v_cache)[src];
    if (lead && atomicCAS(a.owner + page, -1, b * a.max_pages + slot) != -1) {
      atomicExch(a.owner + page, -2);  // a second user: no gradient for this page
      report_bad(a.status);
    }
  } else if (lead) {
    report_bad(a.status);  // a table entry outside the cache: read as zero keys
  }
  const size_t dst = ((size_t)kh * total_k + k0 + r) * cpr + c;
  reinterpret_cast<uint4*>(a.k_pack)[dst] = kv;
  reinterpret_cast<uint4*>(a.v_pack)[dst] = vv;
}

// Grid (kTailRows * d / 8 / 256, Hk): zeros in the kTailRows packed K, V rows after the last
// sequence's keys. A kv tile of the last sequence reads up to 127 rows past its end; the
// backward hides their scores, but a NaN left there by the allocator would still reach dQ
// through a zero-times-NaN product, so those rows must hold finite values (the rows past the
// other sequences' ends are the next sequence's keys).
constexpr int kTailRows = 256;
__global__ void __launch_bounds__(256) paged_tail_kernel(PagedGradArgs a) {
  const int kh = blockIdx.y;
  const int cpr = a.d / 8;
  const int e = blockIdx.x * 256 + threadIdx.x;  // < kTailRows * cpr
  const long long total_k = (long long)a.B * paged_cap(a);
  const long long row = (long long)a.cu_k[a.B] + e / cpr;
  if (row >= total_k) return;
  const size_t dst = ((size_t)kh * total_k + row) * cpr + e % cpr;
  reinterpret_cast<uint4*>(a.k_pack)[dst] = make_uint4(0, 0, 0, 0);
  reinterpret_cast<uint4*>(a.v_pack)[dst] = make_uint4(0, 0, 0, 0);
}

// Grid (ceil(B * H * lq * d / 8 / 256)): row (b, h, i) of the [B, H, lq, d] tensors <->
// packed row t of head hq. TO_PACK: q, O, dO and L in; else dq out.
template <bool TO_PACK>
__global__ void __launch_bounds__(256) paged_qside_kernel(PagedGradArgs a) {
  const int cpr = a.d / 8;
  const long long e = (long long)blockIdx.x * 256 + threadIdx.x;
  const long long rows = (long long)a.B * a.H * a.lq;
  if (e >= rows * cpr) return;
  const long long row = e / cpr;
  const int c = (int)(e % cpr);
  const int i = (int)(row % a.lq);
  const long long bh = row / a.lq;
  const int h = (int)(bh % a.H), b = (int)(bh / a.H);
  const int G = a.H / a.Hk, rq = paged_rq(a);
  const int hq = a.pack ? h / G : h;
  const long long t = (long long)b * rq + (a.pack ? (h % G) * a.lq + i : i);
  const long long total_q = (long long)a.B * rq;
  const size_t src = (size_t)row * cpr + c;
  const size_t dst = ((size_t)hq * total_q + t) * cpr + c;
  if constexpr (TO_PACK) {
    reinterpret_cast<uint4*>(a.q_pack)[dst] = reinterpret_cast<const uint4*>(a.q)[src];
    reinterpret_cast<uint4*>(a.o_pack)[dst] = reinterpret_cast<const uint4*>(a.o)[src];
    reinterpret_cast<uint4*>(a.do_pack)[dst] = reinterpret_cast<const uint4*>(a.dO)[src];
    if (c == 0) a.lse_pack[(size_t)hq * total_q + t] = a.lse[row];
  } else {
    reinterpret_cast<uint4*>(a.dq)[src] = reinterpret_cast<const uint4*>(a.dq_pack)[dst];
  }
}

// Grid (ceil(num_pages * page_size * d / 8 / 256), Hk): every 16-byte chunk of both cache
// gradients, from the packed dK, dV row of its page's owner, else 0.
__global__ void __launch_bounds__(256) paged_scatter_kernel(PagedGradArgs a) {
  const int kh = blockIdx.y;
  const int cpr = a.d / 8;
  const long long e = (long long)blockIdx.x * 256 + threadIdx.x;
  if (e >= (long long)a.num_pages * a.ps * cpr) return;
  const long long prow = e >> a.cpr_shift;  // page * ps + slot within the page
  const int c = (int)(e & (cpr - 1));
  const int page = (int)(prow >> a.ps_shift), s = (int)(prow & (a.ps - 1));
  uint4 gk = make_uint4(0, 0, 0, 0), gv = gk;
  const int own = a.owner[page];
  if (own >= 0) {
    const int b = own / a.max_pages;
    const long long r = (long long)(own % a.max_pages) * a.ps + s;
    const int k0 = a.cu_k[b], len = a.cu_k[b + 1] - k0;
    if (r < len) {
      const long long total_k = (long long)a.B * paged_cap(a);
      const size_t src = ((size_t)kh * total_k + k0 + r) * cpr + c;
      gk = reinterpret_cast<const uint4*>(a.dk_pack)[src];
      gv = reinterpret_cast<const uint4*>(a.dv_pack)[src];
    }
  }
  const size_t dst = (((size_t)page * a.Hk + kh) * a.ps + s) * cpr + c;
  reinterpret_cast<uint4*>(a.dk_cache)[dst] = gk;
  reinterpret_cast<uint4*>(a.dv_cache)[dst] = gv;
}

// ---------------------------------------------------------------- decode path
// With few query rows per kv head (G * q_len <= kDecRows: decode, short cached prefills) the
// gradients are HBM-bound: every used key and value is read once and its two gradient rows
// written once, against 5 * 2 * G * q_len FLOPs per key and head dim element. A tensor-core
// tile would hold at most kDecRows live rows of its 64 or 128, so these kernels run on the
// CUDA cores instead, read the keys through the block table, and write dK, dV straight into
// the cache gradients:
//   paged_owner_kernel     every used page records its (sequence, table slot);
//   paged_decode_bwd_kernel per (sequence, kv head, chunk of kDecKeys keys): P, dP, dS for
//                          the rows of the kv head's G query heads, dK and dV of each key, dQ
//                          partial sums;
//   paged_fill_kernel      zeros in every cache-gradient slot no sequence reads (and in pages
//                          used twice), then dq = bf16 of the f32 partial sums.
constexpr int kDecRows = 8;    // query rows per kv head of the decode path (G * q_len)
// keys per block of the decode kernel (on the decode workload 256 / 512 / 1024 keys measured
// 320 / 300 / 328 us: a block's set-up and dQ sums against the grid's tail)
constexpr int kDecKeys = 512;

namespace {
__device__ __forceinline__ int clamped_len(const PagedGradArgs& a, int b) {
  const int len = a.lens[b];
  const long long cap = paged_cap(a);
  return len < 0 ? 0 : (len > cap ? (int)cap : len);
}

// Recursive halving of N sums over the lanes of a 2*O-lane group: at each level (offsets O,
// O/2, ..., 1) a lane keeps the half of its C values that its lane bit selects and adds its
// partner's copy of that half, sending the other; once one value is left the remaining levels
// add the partner's value. The lane ends with halved_count(2*O, N) sums, those of value
// indices idx0 .. idx0 + halved_count - 1 (idx0 accumulates the kept halves' offsets).
__device__ __host__ constexpr int halved_count(int lanes, int n) {
  while (lanes > 1 && n > 1) {
    lanes /= 2;
    n /= 2;
  }
  return n;
}

// The lane (within its group) that ends with the sum of value index r (< n / 2).
__device__ __host__ constexpr int halved_holder(int r, int lanes, int n) {
  const int cf = halved_count(lanes, n);
  int rem = r - r % cf, holder = 0;
  for (int k = 1; (n >> (k + 1)) >= cf && (lanes >> (k + 1)) >= 1; ++k) {
    const int w = n >> (k + 1);  // the kept upper half at level k starts w values on
    if (rem >= w) {
      rem -= w;
      holder |= lanes >> (k + 1);
    }
  }
  return holder;
}

template <int O, int C, int N>
__device__ __forceinline__ void halve_sums(float (&v)[N], int lane, int& idx0) {
  if constexpr (O >= 1) {
    if constexpr (C > 1) {
      const bool up = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < C / 2; ++i) {
        const float send = up ? v[i] : v[C / 2 + i];
        const float keep = up ? v[C / 2 + i] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      if (up) idx0 += C / 2;
      halve_sums<O / 2, C / 2, N>(v, lane, idx0);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
      halve_sums<O / 2, 1, N>(v, lane, idx0);
    }
  }
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
}  // namespace

// Grid (ceil(max_pages / 256), B): table slot `slot` of sequence b, if it holds keys, claims
// its page (owner = b * max_pages + slot; -2 when the page is claimed twice).
__global__ void __launch_bounds__(256) paged_owner_kernel(PagedGradArgs a) {
  const int b = blockIdx.y;
  const int slot = blockIdx.x * 256 + threadIdx.x;
  const int len = a.lens[b];
  if (slot == 0 && (len < 0 || len > paged_cap(a))) report_bad(a.status);
  if (slot >= a.max_pages || (long long)slot * a.ps >= clamped_len(a, b)) return;
  const int page = a.table[(size_t)b * a.max_pages + slot];
  if (page < 0 || page >= a.num_pages) {
    report_bad(a.status);  // read as zero keys, no gradient written
    return;
  }
  if (atomicCAS(a.owner + page, -1, b * a.max_pages + slot) != -1) {
    atomicExch(a.owner + page, -2);
    report_bad(a.status);
  }
}

// Grid (ceil(capacity / kDecKeys), B * Hk), kDecThreads threads. Row r of a kv head is query
// head kh * G + r / q_len, query r % q_len; it sees keys j < length, and under the causal rule
// j <= length - q_len + r % q_len. A key row is LPK = D / 8 lanes (16 bytes, 8 elements
// each); a warp step takes KPW = 32 / LPK keys. A lane always holds the same 8 columns, so it
// keeps those columns of every row's q and dO in registers for the whole block. The dot
// products over a key row are summed across its lanes by recursive halving. RMAX: the row
// bound the registers are sized for (4 or kDecRows). The kernel is bound by latency and issue,
// not by HBM. Measured on the 16-sequence decode workload (d=128, 4 rows): 128-thread blocks
// at 3 per SM with q/dO in f32 registers took 369 us (325 us once the row sums were halved
// instead of butterflied); 256 threads at 1 per SM 573 us; q/dO read from shared memory at
// each key (256 threads, 2 per SM) 677 us; bf16 q/dO pairs at 4 blocks of 128 per SM
// (spilling) 427 us; two key steps in flight per warp instead of one 354 us; the block's
// page numbers and owners read into shared memory up front instead of the table at each key
// 333 against 320 us; keys streamed through a 4-stage cp.async ring in shared memory (each
// lane copying and reading back its own chunks) 296.8 against 299.7 us at 512 keys per block,
// not worth its code: the kernel is issue-bound once a step's loads overlap the previous
// step's arithmetic.
constexpr int kDecThreads = 128;
template <int D, int RMAX>
__global__ void __launch_bounds__(kDecThreads, RMAX <= 4 ? 3 : 1) paged_decode_bwd_kernel(
    PagedGradArgs a, float* dq_acc, float scale, float scale_log2) {
  constexpr int LPK = D / 8, KPW = 32 / LPK, NW = kDecThreads / 32;
  __shared__ __align__(16) float sq[RMAX][D];   // q rows
  __shared__ __align__(16) float sdo[RMAX][D];  // dO rows
  __shared__ __align__(16) float sdq[RMAX][D];  // the block's dQ sums (unscaled)
  __shared__ float sl2[RMAX], sdd[RMAX];        // L * log2(e) (-inf: no key), D = <dO, O>
  __shared__ int shi[RMAX];                     // keys j < shi[r] are visible to row r
  const int bkh = blockIdx.y, b = bkh / a.Hk, kh = bkh % a.Hk;
  const int G = a.H / a.Hk, R = G * a.lq;
  const int len = clamped_len(a, b);
  const int c0 = blockIdx.x * kDecKeys;
  if (c0 >= len) return;  // (block-uniform)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* o = static_cast<const __nv_bfloat16*>(a.o);
  const __nv_bfloat16* dO = static_cast<const __nv_bfloat16*>(a.dO);
  const size_t row0 = ((size_t)b * a.H + (size_t)kh * G) * a.lq;  // [B, H, lq] row of r = 0
  for (int x = tid; x < RMAX * D; x += kDecThreads) {
    const int r = x / D, e = x % D;
    float qv = 0.0f, dv = 0.0f;
    if (r < R) {
      qv = __bfloat162float(q[(row0 + r) * D + e]);
      dv = __bfloat162float(dO[(row0 + r) * D + e]);
    }
    sq[r][e] = qv;
    sdo[r][e] = dv;
    sdq[r][e] = 0.0f;
  }
  for (int r = warp; r < RMAX; r += NW) {  // one warp per row: D = <dO, O>, L, visibility
    float acc = 0.0f;
    if (r < R)
      for (int e = lane; e < D; e += 32)
        acc += __bfloat162float(o[(row0 + r) * D + e]) * __bfloat162float(dO[(row0 + r) * D + e]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      const float L = r < R ? a.lse[row0 + r] : -INFINITY;
      sdd[r] = acc;
      sl2[r] = L * 1.4426950408889634f;  // -inf stays -inf
      const int hi = a.causal ? len - a.lq + r % a.lq + 1 : len;
      shi[r] = r < R ? (hi < 0 ? 0 : hi) : 0;
    }
  }
  __syncthreads();

  const int sub = lane % LPK;  // 16-byte chunk of the key row: elements 8 * sub .. + 7
  const int kk = lane / LPK;   // key within the warp step
  const int e0 = sub * 8;
  const int c1 = min(c0 + kDecKeys, len);
  const long long total_kv = (long long)a.num_pages * a.Hk * a.ps;  // rows of each cache
  const uint4* K4 = static_cast<const uint4*>(a.k_cache);
  const uint4* V4 = static_cast<const uint4*>(a.v_cache);
  float dq[RMAX][8];
  float qr[RMAX][8], gr[RMAX][8];  // this lane's columns of q and dO
#pragma unroll
  for (int r = 0; r < RMAX; ++r)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      dq[r][e] = 0.0f;
      qr[r][e] = sq[r][e0 + e];
      gr[r][e] = sdo[r][e0 + e];
    }

  // key j's cache row (page * Hk + kh) * ps + j % ps, or -1 (past the end / outside the cache)
  auto key_row = [&](int j, int& slot, int& page) -> long long {
    slot = j >> a.ps_shift;
    page = j < c1 ? a.table[(size_t)b * a.max_pages + slot] : -1;
    if (page < 0 || page >= a.num_pages) return -1;
    return ((long long)page * a.Hk + kh) * a.ps + (j & (a.ps - 1));
  };
  const int step = NW * KPW;
  int j = c0 + warp * KPW + kk;
  int slot, page;
  long long kr = key_row(j, slot, page);
  uint4 kn = make_uint4(0, 0, 0, 0), vn = kn;
  if (kr >= 0 && kr < total_kv) {
    kn = K4[kr * LPK + sub];
    vn = V4[kr * LPK + sub];
  }
#pragma unroll 1
  for (int base = c0 + warp * KPW; base < c1; base += step) {  // (warp-uniform)
    const uint4 kc = kn, vc = vn;
    const int jc = j, slot_c = slot, page_c = page;
    const long long kr_c = kr;
    // the next step's loads go out before this step's arithmetic
    j += step;
    kr = key_row(j, slot, page);
    kn = make_uint4(0, 0, 0, 0);
    vn = kn;
    if (kr >= 0 && kr < total_kv) {
      kn = K4[kr * LPK + sub];
      vn = V4[kr * LPK + sub];
    }
    const bool live = jc < c1;
    const float kf[8] = {bf_lo(kc.x), bf_hi(kc.x), bf_lo(kc.y), bf_hi(kc.y),
                         bf_lo(kc.z), bf_hi(kc.z), bf_lo(kc.w), bf_hi(kc.w)};
    const float vf[8] = {bf_lo(vc.x), bf_hi(vc.x), bf_lo(vc.y), bf_hi(vc.y),
                         bf_lo(vc.z), bf_hi(vc.z), bf_lo(vc.w), bf_hi(vc.w)};
    float sv[RMAX], dpv[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      float s0 = 0.0f, d0 = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        s0 += qr[r][e] * kf[e];
        d0 += gr[r][e] * vf[e];
      }
      sv[r] = s0;
      dpv[r] = d0;
    }
    // the 2 * RMAX sums over the key row's LPK lanes by recursive halving: each lane ends with
    // CF of them (s or dP of rows idx0 .. idx0 + CF - 1 of its half), P and dS are formed once
    // per row, then every lane of the row gets all of them
    float hv[2 * RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      hv[r] = sv[r];
      hv[RMAX + r] = dpv[r];
    }
    int idx0 = 0;
    halve_sums<LPK / 2, 2 * RMAX, 2 * RMAX>(hv, lane, idx0);
    constexpr int CF = halved_count(LPK, 2 * RMAX);
    const bool dp_lane = (lane & (LPK / 2)) != 0;  // lanes of the upper half hold the dP sums
    const int r0 = dp_lane ? idx0 - RMAX : idx0;
    float p_own[CF], ds_own[CF];
#pragma unroll
    for (int i = 0; i < CF; ++i) {
      const float other = __shfl_xor_sync(0xffffffffu, hv[i], LPK / 2);
      const float s_r = dp_lane ? other : hv[i], dp_r = dp_lane ? hv[i] : other;
      const int r = r0 + i;
      const float l2 = sl2[r];
      const bool vis = live && r < R && jc < shi[r] && l2 != -INFINITY;
      p_own[i] = vis ? ex2(s_r * scale_log2 - l2) : 0.0f;
      ds_own[i] = p_own[i] * (dp_r - sdd[r]);
    }
    const int group = lane & ~(LPK - 1);
    float pr[RMAX], dsr[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      constexpr int cf = CF;
      const int src = group + halved_holder(r, LPK, 2 * RMAX);
      pr[r] = __shfl_sync(0xffffffffu, p_own[r % cf], src);
      dsr[r] = __shfl_sync(0xffffffffu, ds_own[r % cf], src);
    }
    float dk[8], dv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) dk[e] = dv[e] = 0.0f;
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        dk[e] += dsr[r] * qr[r][e];
        dv[e] += pr[r] * gr[r][e];
        dq[r][e] += dsr[r] * kf[e];
      }
    }
    // this sequence's own page only: a page claimed twice (or none) is zero-filled later
    if (kr_c >= 0 && kr_c < total_kv && a.owner[page_c] == b * a.max_pages + slot_c) {
      const uint4 wk = make_uint4(pack_bf16(dk[0] * scale, dk[1] * scale),
                                  pack_bf16(dk[2] * scale, dk[3] * scale),
                                  pack_bf16(dk[4] * scale, dk[5] * scale),
                                  pack_bf16(dk[6] * scale, dk[7] * scale));
      const uint4 wv = make_uint4(pack_bf16(dv[0], dv[1]), pack_bf16(dv[2], dv[3]),
                                  pack_bf16(dv[4], dv[5]), pack_bf16(dv[6], dv[7]));
      reinterpret_cast<uint4*>(a.dk_cache)[kr_c * LPK + sub] = wk;
      reinterpret_cast<uint4*>(a.dv_cache)[kr_c * LPK + sub] = wv;
    }
  }
  // dQ: the warp's keys (lanes of one chunk, different kk) summed, then the block's warps
  // in shared memory, then one global f32 sum per element
#pragma unroll
  for (int off = LPK; off < 32; off <<= 1)
#pragma unroll
    for (int r = 0; r < RMAX; ++r)
#pragma unroll
      for (int e = 0; e < 8; ++e) dq[r][e] += __shfl_xor_sync(0xffffffffu, dq[r][e], off);
  if (kk == 0) {
#pragma unroll
    for (int r = 0; r < RMAX; ++r)
      if (r < R)
#pragma unroll
        for (int e = 0; e < 8; ++e) atomicAdd(&sdq[r][e0 + e], dq[r][e]);
  }
  __syncthreads();
  for (int x = tid; x < R * D; x += kDecThreads) {
    const int r = x / D, e = x % D;
    atomicAdd(dq_acc + (row0 + r) * D + e, sdq[r][e] * scale);
  }
}

// Grid (ceil(num_pages * page_size * d / 8 / 256), Hk): zeros in every cache-gradient chunk
// whose slot holds no key of its page's one owner (the decode kernel wrote the others).
__global__ void __launch_bounds__(256) paged_fill_kernel(PagedGradArgs a) {
  const int kh = blockIdx.y;
  const int cpr = a.d / 8;
  const long long e = (long long)blockIdx.x * 256 + threadIdx.x;
  if (e >= (long long)a.num_pages * a.ps * cpr) return;
  const long long prow = e >> a.cpr_shift;
  const int c = (int)(e & (cpr - 1));
  const int page = (int)(prow >> a.ps_shift), s = (int)(prow & (a.ps - 1));
  const int own = a.owner[page];
  if (own >= 0 && (long long)(own % a.max_pages) * a.ps + s < clamped_len(a, own / a.max_pages))
    return;
  const size_t dst = (((size_t)page * a.Hk + kh) * a.ps + s) * cpr + c;
  reinterpret_cast<uint4*>(a.dk_cache)[dst] = make_uint4(0, 0, 0, 0);
  reinterpret_cast<uint4*>(a.dv_cache)[dst] = make_uint4(0, 0, 0, 0);
}

// Grid (ceil(B * H * lq * d / 8 / 256)): dq = bf16 of the f32 sums, 8 elements per thread.
__global__ void __launch_bounds__(256) paged_dq_convert_kernel(PagedGradArgs a,
                                                               const float* dq_acc) {
  const long long e = (long long)blockIdx.x * 256 + threadIdx.x;
  if (e >= (long long)a.B * a.H * a.lq * a.d / 8) return;
  const float4 x0 = reinterpret_cast<const float4*>(dq_acc)[2 * e];
  const float4 x1 = reinterpret_cast<const float4*>(dq_acc)[2 * e + 1];
  reinterpret_cast<uint4*>(a.dq)[e] =
      make_uint4(pack_bf16(x0.x, x0.y), pack_bf16(x0.z, x0.w), pack_bf16(x1.x, x1.y),
                 pack_bf16(x1.z, x1.w));
}

namespace {
unsigned blocks_of(long long n) { return (unsigned)((n + 255) / 256); }
}  // namespace

cudaError_t launch_paged_gather(const PagedGradArgs& a, cudaStream_t s) {
  const long long cap = (long long)a.max_pages * a.ps;
  const int cpr = a.d / 8;
  profile_mark(kKernPagedGather, 0, s);
  paged_index_kernel<<<1, 1024, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) {
    paged_gather_kernel<<<dim3(blocks_of(cap * cpr), a.B * a.Hk), 256, 0, s>>>(a);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    paged_tail_kernel<<<dim3(kTailRows * cpr / 256, a.Hk), 256, 0, s>>>(a);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    paged_qside_kernel<true><<<blocks_of((long long)a.B * a.H * a.lq * cpr), 256, 0, s>>>(a);
    e = cudaGetLastError();
  }
  profile_mark(kKernPagedGather, 1, s);
  return e;
}

cudaError_t launch_paged_scatter(const PagedGradArgs& a, cudaStream_t s) {
  const int cpr = a.d / 8;
  profile_mark(kKernPagedScatter, 0, s);
  paged_scatter_kernel<<<dim3(blocks_of((long long)a.num_pages * a.ps * cpr), a.Hk), 256, 0,
                         s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) {
    paged_qside_kernel<false><<<blocks_of((long long)a.B * a.H * a.lq * cpr), 256, 0, s>>>(a);
    e = cudaGetLastError();
  }
  profile_mark(kKernPagedScatter, 1, s);
  return e;
}

bool paged_decode_path(int G, int lq) { return (long long)G * lq <= kDecRows; }

cudaError_t launch_paged_decode_bwd(const PagedGradArgs& a, float* dq_acc, float scale,
                                    cudaStream_t s) {
  const long long cap = (long long)a.max_pages * a.ps;
  const int cpr = a.d / 8;
  const int R = (a.H / a.Hk) * a.lq;
  profile_mark(kKernPagedGather, 0, s);
  paged_owner_kernel<<<dim3(blocks_of(a.max_pages), a.B), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  profile_mark(kKernPagedGather, 1, s);
  if (e != cudaSuccess) return e;
  profile_mark(kKernPagedDecodeBwd, 0, s);
  const dim3 grid((unsigned)((cap + kDecKeys - 1) / kDecKeys), a.B * a.Hk);
  const float sl2 = scale * 1.4426950408889634f;
#define FA_DEC(DD)                                                                   \
  if (R <= 4)                                                                        \
    paged_decode_bwd_kernel<DD, 4><<<grid, kDecThreads, 0, s>>>(a, dq_acc, scale, sl2); \
  else                                                                               \
    paged_decode_bwd_kernel<DD, kDecRows><<<grid, kDecThreads, 0, s>>>(a, dq_acc, scale, sl2);
  if (a.d == 64) {
    FA_DEC(64)
  } else if (a.d == 128) {
    FA_DEC(128)
  } else {
    FA_DEC(256)
  }
#undef FA_DEC
  e = cudaGetLastError();
  profile_mark(kKernPagedDecodeBwd, 1, s);
  if (e != cudaSuccess) return e;
  profile_mark(kKernPagedScatter, 0, s);
  paged_fill_kernel<<<dim3(blocks_of((long long)a.num_pages * a.ps * cpr), a.Hk), 256, 0, s>>>(
      a);
  e = cudaGetLastError();
  if (e == cudaSuccess) {
    paged_dq_convert_kernel<<<blocks_of((long long)a.B * a.H * a.lq * cpr), 256, 0, s>>>(
        a, dq_acc);
    e = cudaGetLastError();
  }
  profile_mark(kKernPagedScatter, 1, s);
  return e;
}

}  // namespace fa
