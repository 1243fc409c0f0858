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
// a zero gradient and FA_ERR_BAD_INPUT is reported.
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
  const long long r = e / cpr;
  const int c = (int)(e % cpr);
  const int k0 = a.cu_k[b], len = a.cu_k[b + 1] - k0;
  if (r >= len) return;
  const long long total_k = (long long)a.B * paged_cap(a);  // rows per head of k_pack
  const int slot = (int)(r / a.ps);
  const int page = a.table[(size_t)b * a.max_pages + slot];
  const bool lead = kh == 0 && c == 0 && r % a.ps == 0;
  uint4 kv = make_uint4(0, 0, 0, 0), vv = kv;
  if (page >= 0 && page < a.num_pages) {
    const size_t src = (((size_t)page * a.Hk + kh) * a.ps + r % a.ps) * cpr + c;
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
  const long long prow = e / cpr;  // page * ps + slot within the page
  const int c = (int)(e % cpr);
  const int page = (int)(prow / a.ps), s = (int)(prow % a.ps);
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

}  // namespace fa
