// fa_launch.h -- internal interface between the C-ABI layer (fa_api.cu) and the kernel
// translation units. Host-side only; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fa_once.h"

namespace fa {

// Bounds of sequence b of a variable-length batch from its offsets: start and length, clamped
// to [0, total] and to `maxlen`. Returns true when the offsets were out of range.
__device__ __forceinline__ bool varlen_seq(const int32_t* cu, int b, int total, int maxlen,
                                           int& start, int& len) {
  int s = cu[b], e = cu[b + 1];
  const bool bad = s < 0 || e < s || e > total || e - s > maxlen;
  s = s < 0 ? 0 : (s > total ? total : s);
  e = e < s ? s : (e > total ? total : e);
  start = s;
  len = e - s < maxlen ? e - s : maxlen;
  return bad;
}

// Device-side status codes, written into the per-device status word the kernels are given (a
// device int owned by the library): kStatusTimeout when a bounded wait gave up (the kernel then
// winds down), kStatusBadInput when a paged kernel met a length or block-table entry out of
// range.
enum : int { kStatusOk = 0, kStatusTimeout = 1, kStatusBadInput = 2 };

// Default limit of one mbarrier wait in the kernels, in ns of %globaltimer. A legitimate wait
// lasts microseconds; reaching this means a pipeline bug, and the kernel then winds down
// instead of hanging the GPU. The host can set another limit (fa_set_wait_limit_ns); it reaches
// every kernel as a launch parameter.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Kernel ids of the timing facility (same values as FA_KERNEL_* in the public header).
enum KernelId {
  kKernFwd = 0,
  kKernBwdPrep = 1,
  kKernBwdMain = 2,
  kKernBwdDq = 3,
  kKernBwdDqDet = 4,
  kKernPaged = 5,
  kKernPagedCombine = 6,
  kKernPagedGather = 7,
  kKernPagedScatter = 8,
  kKernPagedDecodeBwd = 9,
  kNumKernels = 10
};

// Records a timing event before (end = 0) or after (end = 1) a launch on `s` when timing is
// enabled; does nothing otherwise. Defined in fa_api.cu.
void profile_mark(int kernel, int end, cudaStream_t s);

// A kernel launched with programmatic stream serialisation may start while the previous
// kernel of its stream still runs; grid_dep_wait() returns once that kernel has completed and
// its memory is visible (at once for a kernel launched without it). grid_dep_trigger() lets
// the next such kernel be scheduled once every CTA of this grid has issued it or exited.
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches `kernel` with programmatic stream serialisation: it may be scheduled before the
// previous kernel of `s` completes and must call grid_dep_wait() before it touches memory that
// kernel writes or reads.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Sets a kernel's dynamic shared-memory limit on the current device, once per device and
// thread-safely (the attribute belongs to a device context, so a process that drives several
// GPUs sets it on each).
template <class K>
inline cudaError_t set_smem_once(OncePerKey<>& once, K kern, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return once.run(dev, [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  });
}

// Visibility band of a row: key j is visible to query row i iff
//   q_abs + lo_off <= j <= q_abs + hi_off,  q_abs = kl - ql + i
// (plus j < kl). The kernels are compiled per band mode: kBandNone (no causal mask, no window:
// no per-element test), kBandCausal (the causal diagonal alone: hi_off = 0, lo unbounded) and
// kBandWindow (any other band; both bounds are runtime values and the kv ranges of the query
// tiles of one CTA may start at different tiles).
enum BandMode : int { kBandNone = 0, kBandCausal = 1, kBandWindow = 2 };
struct Band {
  int lo_off, hi_off;
  int mode;
};
constexpr int kUnbounded = 1 << 30;
inline Band make_band(int causal, int window_left, int window_right) {
  Band b;
  b.lo_off = window_left >= 0 ? -window_left : -kUnbounded;
  b.hi_off = window_right >= 0 ? window_right : kUnbounded;
  if (causal && b.hi_off > 0) b.hi_off = 0;
  if (!causal && window_left < 0 && window_right < 0)
    b.mode = kBandNone;
  else if (causal && window_left < 0)
    b.mode = kBandCausal;  // hi_off == 0 here
  else
    b.mode = kBandWindow;
  return b;
}

// Everything a forward launch needs besides the tensor maps.
struct FwdArgs {
  const void* mask;   // nullptr, or the mask in mask_type's element type
  int mask_type;      // 0 f32 additive, 1 bf16 additive, 2 bool (uint8, nonzero = visible)
  long long mask_stride_b, mask_stride_h, mask_stride_q;  // elements; keys contiguous
  void* o;            // bf16 [B, H, ql, dval] (see q_bshd)
  float* lse;         // [B, H, ql]
  const float* sinks; // [H] natural-log sink logits, or nullptr
  const int32_t* cu_q;  // variable-length batch: [B + 1] row offsets of the sequences, or nullptr
  const int32_t* cu_k;
  int total_q, total_k;  // rows per head of the packed q / k (variable-length batch)
  int q_bshd, kv_bshd;   // 1: q, o (and dO, dq) / k, v (and dk, dv) are [batch, rows, heads, d]
  int* status;        // device status word (nullable)
  uint64_t wait_limit_ns;  // limit of one barrier wait in the kernels (fa_set_wait_limit_ns)
  int B, H, Hk, ql, kl, d;  // ql, kl: the longest sequence in a variable-length batch
  int dval;           // value head dim (of v and o)
  float scale;
  int lo_off, hi_off;
  int band;  // BandMode
};

// Tensor maps of a forward launch (innermost first: d, rows, batch * heads, or 4-D d, rows,
// heads, batch for the bshd layout; 128-byte swizzle; box of 64 columns).
struct FwdMaps {
  CUtensorMap q, k, v;
};

// Rows per query tile and keys per kv tile the forward kernel of head_dim d uses (the tensor
// map boxes must match).
int fwd_q_box_rows(int d);
int fwd_kv_box_rows(int d);

cudaError_t launch_fwd(const FwdArgs& a, const FwdMaps& m, cudaStream_t stream);

// Backward.
struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const float* lse;
  const void* dO;
  const void* mask;
  int mask_type;
  long long mask_stride_b, mask_stride_h, mask_stride_q;
  void* dq;
  void* dk;
  void* dv;
  float* lse2;   // workspace [B*H, ql_pad]: -L * log2(e), -inf for fully masked rows
  float* dvec;   // workspace [B*H, ql_pad]: D = rowsum(dO * O)
  float* dqacc;  // workspace [B*H, ql_pad, d] f32 dQ accumulator
  const float* sinks;  // [H] sink logits, or nullptr
  const int32_t* cu_q;  // variable-length batch (see FwdArgs), or nullptr
  const int32_t* cu_k;
  int total_q, total_k;
  int q_bshd, kv_bshd;  // layouts, as in FwdArgs
  float* dsinks;       // [H] sink gradient output, or nullptr (then no sink partials)
  float* dsink_part;   // workspace [B*H, sink_chunks]: per-block partial sums of dsinks
  int* status;
  uint64_t wait_limit_ns;
  int B, H, Hk, ql, kl, d, ql_pad;
  int dval;  // value head dim (of v, o, dO, dV)
  int deterministic;  // 1: dQ from the query-tile-major kernel (no cross-CTA additions)
  float scale;
  int lo_off, hi_off;
  int band;  // BandMode
};

// Tensor maps of the deterministic dQ kernel (boxes: 128 query rows, dq_det_box_rows() keys).
struct DqMaps {
  CUtensorMap q, k, v, dO;
};

struct BwdMaps {
  CUtensorMap q, k, v, dO;
  DqMaps det;  // encoded only in deterministic mode
};

int bwd_q_box_rows(int d);
int bwd_kv_box_rows(int d);
int bwd_ql_pad(int ql);

// Workspace bytes of a backward call (lse2 + dvec + dqacc + the dsinks partials, each 256-byte
// aligned).
size_t bwd_workspace_bytes(int B, int H, int ql, int d);
void bwd_carve_workspace(void* base, int B, int H, int ql, int d, float** lse2, float** dvec,
                         float** dqacc, float** dsink_part);

cudaError_t launch_bwd(const BwdArgs& a, const BwdMaps& m, cudaStream_t stream);

// Backward main pass at head_dim 256 on CTA pairs (fa_bwd_pair.cu); needs the pre-pass's
// lse2, dvec (and the zeroed dQ accumulator unless deterministic).
cudaError_t launch_bwd_pair(const BwdArgs& a, const BwdMaps& m, cudaStream_t stream);

// Deterministic dQ (fa_bwd_dq.cu): needs lse2 and dvec from the pre-pass; writes a.dq (bf16).
int dq_det_box_rows();
cudaError_t launch_dq_det(const BwdArgs& a, const DqMaps& m, cudaStream_t stream);

// Fixed-size device scratch of fa_train_bwd_noalloc (defined in fa_bwd.cu): the first
// kNoAllocStatusBytes hold the status word of the calls that use it, the rest the backward's
// workspace. noalloc_scratch looks up the array's address on the current device (every call:
// nothing is cached, so nothing goes stale across a device reset); noalloc_status reads (and
// with clear != 0 zeroes) its status word, synchronously.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr size_t kNoAllocStatusBytes = 256;
cudaError_t noalloc_scratch(void** ptr);
cudaError_t noalloc_status(int clear, int* value);

// Diagnostics (fa_diag.cu): the softmax's exp2 forms on an array, and one bounded wait on a
// barrier that nothing completes (it runs out after `limit_ns`, records kStatusTimeout in
// `status` and writes the time it waited to `waited_ns` when that is not null).
cudaError_t launch_ex2_probe(const float* x, float* y_poly, float* y_mufu, float* y_ref,
                             long long n, cudaStream_t s);
cudaError_t launch_wait_probe(int* status, uint64_t limit_ns, unsigned long long* waited_ns,
                              cudaStream_t s);

// Paged key/value cache attention (fa_paged.cu).
struct PagedArgs {
  const int32_t* table;  // [B, max_pages] device
  const int32_t* lens;   // [B] device
  void* o;               // bf16 [B, H, lq, d]
  float* lse;            // [B, H, lq] or nullptr
  int* status;
  uint64_t wait_limit_ns;
  int B, H, Hk, G, lq, d, bs, max_pages, num_pages, causal, num_splits;
  float scale;
};
struct PagedMaps {
  CUtensorMap q, k, v;  // q as [B*Hk, G*lq, d]; caches as [num_pages*Hk, page_size, d]
};
int paged_key_box_rows(int page_size);
int paged_query_box_rows();
int paged_splits(const PagedArgs& a);
size_t paged_workspace_bytes(const PagedArgs& a, int splits);
cudaError_t launch_paged(const PagedArgs& a, const PagedMaps& m, int splits, void* ws,
                         cudaStream_t stream);

// Gradients through the paged cache (fa_paged_bwd.cu): the paged problem is turned into a
// variable-length batch (sequence b = its used keys, packed head-major without padding) for
// the training backward, and its gradients are put back into the pages and the [B, H, lq, d]
// layout. With `pack`, the G query heads of a kv head are one sequence's G * lq query rows
// (row g * lq + i), which the backward then treats as one head.
struct PagedGradArgs {
  const void* k_cache;   // bf16 [num_pages, Hk, page_size, d]
  const void* v_cache;
  const int32_t* table;  // [B, max_pages]
  const int32_t* lens;   // [B]
  const void* q;         // bf16 [B, H, lq, d]
  const void* o;
  const void* dO;
  const float* lse;      // f32 [B, H, lq]
  void* dq;              // output, bf16 [B, H, lq, d]
  void* dk_cache;        // outputs, bf16 like the caches, every element written
  void* dv_cache;
  void* k_pack;          // bf16 [Hk, B * capacity, d]: sequence b's keys at rows cu_k[b] ..
  void* v_pack;
  const void* dk_pack;   // the packed problem's dK, dV
  const void* dv_pack;
  void* q_pack;          // bf16 [Hq, B * rq, d] (Hq = Hk with pack, else H; rq = rows per
  void* o_pack;          // sequence, G * lq with pack, else lq)
  void* do_pack;
  const void* dq_pack;
  float* lse_pack;       // f32 [Hq, B * rq]
  int32_t* cu_q;         // [B + 1]: b * rq
  int32_t* cu_k;         // [B + 1]: prefix sums of the (clamped) lengths
  int32_t* owner;        // [num_pages]: b * max_pages + slot of the one table entry that uses
                         // the page; -1 (set before the gather) none, -2 two or more
  int* status;
  int B, H, Hk, lq, d, ps, max_pages, num_pages, pack, causal;
  int ps_shift, cpr_shift;  // log2 of page_size and of d / 8 (both powers of two)
};
// The offsets, the packed K, V (and the owner of every used page), the packed q-side tensors.
cudaError_t launch_paged_gather(const PagedGradArgs& a, cudaStream_t stream);
// Both cache gradients whole (zero where no sequence reads) and dq.
cudaError_t launch_paged_scatter(const PagedGradArgs& a, cudaStream_t stream);
// The decode path (G * q_len small: no packing, no training backward): page owners, the
// CUDA-core gradient kernel writing dK, dV into the cache gradients and f32 dQ sums into
// dq_acc (zeroed, [B, H, lq, d]), the zero fill of unread slots and dq. Uses q, o, dO, lse,
// dq, the caches, their gradients, table, lens, owner (set to -1) and status of `a`.
bool paged_decode_path(int G, int lq);
cudaError_t launch_paged_decode_bwd(const PagedGradArgs& a, float* dq_acc, float scale,
                                    cudaStream_t stream);

}  // namespace fa
