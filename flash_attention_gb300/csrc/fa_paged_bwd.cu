// fa_paged_bwd.cu -- gradients through the paged key/value cache (sm_103a): dQ and the
// gradients of both caches, for the decode / cached-prefill attention of fa_paged.cu.
//
// Method: page "nuvec-core tests/fast.rs", `paged_attention_equals_contiguous_attention`, takes
// the gradients of the paged attention with respect to q and the caches ("paged grads"). Each
// sequence is the fixed-length attention problem on the keys its block table names, so its
// gradients are the training backward's on those keys. The call
//   1. gathers each sequence's keys and values from the pages into contiguous
//      [batch, kv heads, capacity, d] tensors (capacity = max_pages * page_size; slots past the
//      sequence's length are zero), counting how many times each page is named;
//   2. builds a bool mask [batch, q_len, capacity] that hides those slots and applies the
//      bottom-right causal rule of the forward;
//   3. runs the training backward (fa_bwd.cu, fa_bwd_pair.cu) on that problem;
//   4. scatters dK and dV back into the cache-shaped gradients, which start zeroed, so slots
//      no sequence reads keep a zero gradient.
// A page named by two sequences would need the two contributions summed; the scatter writes
// none for it and reports FA_ERR_BAD_INPUT.
// This moves each key and value three more times than a backward that reads the pages
// directly; it reuses the training backward's kernels unchanged.
#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {

namespace {
__device__ __forceinline__ void report_bad(int* status) {
  if (status) atomicCAS(status, kStatusOk, kStatusBadInput);
}

__device__ __forceinline__ int clamp_len(int len, long long cap, int* status, bool report) {
  if (len < 0 || len > cap) {
    if (report) report_bad(status);
    return len < 0 ? 0 : (int)cap;
  }
  return len;
}
}  // namespace

// Grid (ceil(capacity * d / 8 / 256), batch * Hk); each thread moves one 16-byte chunk of one
// row of K and of V.
__global__ void __launch_bounds__(256) paged_gather_kernel(PagedGradArgs a) {
  const int bkh = blockIdx.y, b = bkh / a.Hk, kh = bkh % a.Hk;
  const int cpr = a.d / 8;  // 16-byte chunks per row
  const long long cap = (long long)a.max_pages * a.ps;
  const long long e = (long long)blockIdx.x * 256 + threadIdx.x;
  if (e >= cap * cpr) return;
  const long long r = e / cpr;
  const int c = (int)(e % cpr);
  const bool lead = kh == 0 && c == 0 && r % a.ps == 0;  // one thread per (sequence, slot)
  const int len = clamp_len(a.lens[b], cap, a.status, lead && r == 0);
  uint4 kv = make_uint4(0, 0, 0, 0), vv = kv;
  if (r < len) {
    const int page = a.table[(size_t)b * a.max_pages + r / a.ps];
    if (page >= 0 && page < a.num_pages) {
      const size_t src = (((size_t)page * a.Hk + kh) * a.ps + r % a.ps) * cpr + c;
      kv = reinterpret_cast<const uint4*>(a.k_cache)[src];
      vv = reinterpret_cast<const uint4*>(a.v_cache)[src];
      if (lead) atomicAdd(a.uses + page, 1);
    } else if (lead) {
      report_bad(a.status);  // a table entry outside the cache: read as zero keys
    }
  }
  const size_t dst = ((size_t)bkh * cap + r) * cpr + c;
  reinterpret_cast<uint4*>(a.k_flat)[dst] = kv;
  reinterpret_cast<uint4*>(a.v_flat)[dst] = vv;
}

// Grid (ceil(capacity / 256), batch * q_len): mask[b, i, j] = 1 iff slot j holds a key query i
// sees (j < length, and with causal j <= length - q_len + i).
__global__ void __launch_bounds__(256) paged_mask_kernel(PagedGradArgs a) {
  const int b = blockIdx.y / a.lq, i = blockIdx.y % a.lq;
  const long long cap = (long long)a.max_pages * a.ps;
  const long long j = (long long)blockIdx.x * 256 + threadIdx.x;
  if (j >= cap) return;
  const int len = clamp_len(a.lens[b], cap, a.status, false);
  const bool vis = j < len && (!a.causal || j <= (long long)len - a.lq + i);
  a.mask[((size_t)b * a.lq + i) * cap + j] = vis ? 1 : 0;
}

// Same grid as the gather: rows of the pages a sequence uses go back to their pages.
__global__ void __launch_bounds__(256) paged_scatter_kernel(PagedGradArgs a) {
  const int bkh = blockIdx.y, b = bkh / a.Hk, kh = bkh % a.Hk;
  const int cpr = a.d / 8;
  const long long cap = (long long)a.max_pages * a.ps;
  const long long e = (long long)blockIdx.x * 256 + threadIdx.x;
  if (e >= cap * cpr) return;
  const long long r = e / cpr;
  const int c = (int)(e % cpr);
  const int len = clamp_len(a.lens[b], cap, nullptr, false);
  if (r >= (long long)(len + a.ps - 1) / a.ps * a.ps) return;  // past the last used page
  const int page = a.table[(size_t)b * a.max_pages + r / a.ps];
  if (page < 0 || page >= a.num_pages) return;
  if (a.uses[page] > 1) {  // named twice: the contributions would need a sum
    if (kh == 0 && c == 0 && r % a.ps == 0) report_bad(a.status);
    return;
  }
  const size_t src = ((size_t)bkh * cap + r) * cpr + c;
  const size_t dst = (((size_t)page * a.Hk + kh) * a.ps + r % a.ps) * cpr + c;
  reinterpret_cast<uint4*>(a.dk_cache)[dst] = reinterpret_cast<const uint4*>(a.dk_flat)[src];
  reinterpret_cast<uint4*>(a.dv_cache)[dst] = reinterpret_cast<const uint4*>(a.dv_flat)[src];
}

cudaError_t launch_paged_gather(const PagedGradArgs& a, cudaStream_t s) {
  const long long cap = (long long)a.max_pages * a.ps;
  const long long chunks = cap * (a.d / 8);
  profile_mark(kKernPagedGather, 0, s);
  paged_gather_kernel<<<dim3((unsigned)((chunks + 255) / 256), a.B * a.Hk), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) {
    paged_mask_kernel<<<dim3((unsigned)((cap + 255) / 256), a.B * a.lq), 256, 0, s>>>(a);
    e = cudaGetLastError();
  }
  profile_mark(kKernPagedGather, 1, s);
  return e;
}

cudaError_t launch_paged_scatter(const PagedGradArgs& a, cudaStream_t s) {
  const long long cap = (long long)a.max_pages * a.ps;
  const long long chunks = cap * (a.d / 8);
  profile_mark(kKernPagedScatter, 0, s);
  paged_scatter_kernel<<<dim3((unsigned)((chunks + 255) / 256), a.B * a.Hk), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  profile_mark(kKernPagedScatter, 1, s);
  return e;
}

}  // namespace fa
