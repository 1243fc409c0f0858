// fa_api.cu -- the C ABI declared in include/fa_train.h: argument checks, TMA tensor-map
// encoding, workspace management and kernel dispatch on the caller's stream.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <cmath>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/fa_train.h"
#include "fa_launch.h"

namespace {

thread_local char g_last_cuda_error[256] = "";

int cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s (%d)", where,
           cudaGetErrorString(e), (int)e);
  return FA_ERR_CUDA;
}

// ---------------------------------------------------------------- driver entry point (TMA)
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

cudaError_t get_encoder() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) {
      g_encode_err = e;
    } else if (q != cudaDriverEntryPointSuccess || fn == nullptr) {
      g_encode_err = cudaErrorSymbolNotFound;
    } else {
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  });
  return g_encode_err;
}

// 4-D bf16 tensor map (d, rows, heads, batch) over a [batch, heads, rows, d] tensor stored as
// such or, with bshd, as [batch, rows, heads, d]; box (64, box_rows, 1, 1), 128-byte swizzle;
// reads outside [0, rows) fill with zeros.
bool encode_bf16_4d(CUtensorMap* m, const void* base, int d, int rows, int heads, int batch,
                    bool bshd, int box_rows) {
  const cuuint64_t row_b = (cuuint64_t)d * 2;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)heads, (cuuint64_t)batch};
  cuuint64_t strides[3];
  if (bshd) {
    strides[0] = row_b * heads;                    // next row
    strides[1] = row_b;                            // next head
    strides[2] = row_b * heads * (cuuint64_t)rows; // next batch
  } else {
    strides[0] = row_b;
    strides[1] = row_b * rows;
    strides[2] = row_b * rows * (cuuint64_t)heads;
  }
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D bf16 tensor map over a contiguous [bh, rows, d] tensor, box (64, box_rows, 1), 128-byte
// swizzle; reads outside [0, rows) fill with zeros (the paged caches and queries).
bool encode_bf16_3d(CUtensorMap* m, const void* base, int bh, int rows, int d, int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)bh};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows * (cuuint64_t)d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The tile map of a q-side or kv-side tensor: 3-D (d, rows, batch * heads) in the default
// layout, 4-D in the bshd layout (the kernels issue the matching load form).
bool encode_bf16_map(CUtensorMap* m, const void* base, int d, int rows, int heads, int batch,
                     bool bshd, int box_rows) {
  return bshd ? encode_bf16_4d(m, base, d, rows, heads, batch, true, box_rows)
              : encode_bf16_3d(m, base, heads * batch, rows, d, box_rows);
}

// ---------------------------------------------------------------- per-device status word
// One int in this file's device code: CUDA creates it, zeroed, with the module on each device,
// and again after a device reset. Its address is looked up on every call (cheap once the
// module is loaded, and nothing to go stale), as the no-allocation scratch's is.
__device__ int g_status_word;

cudaError_t device_status_word(int dev, int** out) {
  if (dev < 0) return cudaErrorInvalidDevice;
  return cudaGetSymbolAddress(reinterpret_cast<void**>(out), g_status_word);
}

// ---------------------------------------------------------------- bounded waits
// Limit of one barrier wait in the kernels launched from now on (fa_set_wait_limit_ns).
std::atomic<uint64_t> g_wait_limit_ns{fa::kWaitLimitNs};
constexpr uint64_t kMaxWaitLimitNs = 60ull * 1000000000ull;  // 60 s

// Devices on which fa_train_bwd_noalloc has been called (their fixed array's status word is
// then read by fa_device_status too).
std::atomic<uint64_t> g_noalloc_used{0};

// ---------------------------------------------------------------- argument checks
constexpr int kMaxLen = 1 << 22;  // keeps every grid dimension within its limit
constexpr int kPagedMaxRows = 128 * 65535;  // query rows per kv head (grid z of 128-row tiles)

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_params(const fa_params* p) {
  if (!p) return FA_ERR_INVALID;
  if (p->batch <= 0 || p->n_heads <= 0 || p->n_kv_heads <= 0 || p->ql <= 0 || p->kl <= 0)
    return FA_ERR_INVALID;
  if (p->n_heads % p->n_kv_heads != 0) return FA_ERR_INVALID;
  if (p->head_dim != 64 && p->head_dim != 128 && p->head_dim != 256) return FA_ERR_INVALID;
  if (!(isfinite(p->scale) && p->scale > 0.0f)) return FA_ERR_INVALID;
  if (p->causal != 0 && p->causal != 1) return FA_ERR_INVALID;
  if (p->ql > kMaxLen || p->kl > kMaxLen) return FA_ERR_INVALID;
  if ((int64_t)p->batch * p->n_heads > INT32_MAX / 2) return FA_ERR_INVALID;
  return FA_OK;
}

int check_bf16(const void* ptr) { return (ptr && aligned(ptr, 16)) ? FA_OK : FA_ERR_INVALID; }
int check_f32(const void* ptr) { return (ptr && aligned(ptr, 16)) ? FA_OK : FA_ERR_INVALID; }

// Options with the base entry points' meaning: no window, dense [B, H, ql, kl] f32 mask.
fa_options default_options(const fa_params* p) {
  fa_options o;
  o.window_left = -1;
  o.window_right = -1;
  o.mask_type = FA_MASK_F32;
  o.value_dim = 0;
  o.sinks = nullptr;
  o.dsinks = nullptr;
  o.deterministic = 0;
  o.layout = 0;
  o.cu_seqlens_q = nullptr;
  o.cu_seqlens_k = nullptr;
  o.total_q = 0;
  o.total_k = 0;
  o.mask_stride_q = p->kl;
  o.mask_stride_h = (int64_t)p->ql * p->kl;
  o.mask_stride_b = (int64_t)p->n_heads * p->ql * p->kl;
  return o;
}

// Option checks shared by both passes; `bwd` adds the dsinks rules. FA_ERR_INVALID comes before
// FA_ERR_UNSUPPORTED (a value head dim without kernels).
int check_options(const fa_options* o, const void* mask, const fa_params* p, bool bwd) {
  if (o->window_left < -1 || o->window_right < -1) return FA_ERR_INVALID;
  if (o->value_dim < 0) return FA_ERR_INVALID;
  if (o->deterministic != 0 && o->deterministic != 1) return FA_ERR_INVALID;
  if (o->layout & ~(FA_LAYOUT_Q_BSHD | FA_LAYOUT_KV_BSHD)) return FA_ERR_INVALID;
  if ((o->cu_seqlens_q == nullptr) != (o->cu_seqlens_k == nullptr)) return FA_ERR_INVALID;
  if (o->cu_seqlens_q) {
    if (!aligned(o->cu_seqlens_q, 4) || !aligned(o->cu_seqlens_k, 4)) return FA_ERR_INVALID;
    if (o->total_q < 1 || o->total_k < 1) return FA_ERR_INVALID;
    if ((int64_t)o->total_q * p->n_heads > INT32_MAX / 2 ||
        (int64_t)o->total_k * p->n_kv_heads > INT32_MAX / 2)
      return FA_ERR_INVALID;
    if (mask) return FA_ERR_UNSUPPORTED;  // a dense mask has no shape for packed sequences
  }
  if (o->sinks && !aligned(o->sinks, 4)) return FA_ERR_INVALID;
  if (bwd && o->dsinks && (!o->sinks || !aligned(o->dsinks, 4))) return FA_ERR_INVALID;
  if (o->mask_type != FA_MASK_F32 && o->mask_type != FA_MASK_BF16 && o->mask_type != FA_MASK_BOOL)
    return FA_ERR_INVALID;
  if (o->mask_stride_b < 0 || o->mask_stride_h < 0 || o->mask_stride_q < 0) return FA_ERR_INVALID;
  if (mask) {
    const uintptr_t es = o->mask_type == FA_MASK_F32 ? 4 : o->mask_type == FA_MASK_BF16 ? 2 : 1;
    if (!aligned(mask, es)) return FA_ERR_INVALID;
  }
  if (!fa_value_dim_supported(p->head_dim, o->value_dim ? o->value_dim : p->head_dim))
    return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

int check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0;
  e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  // the library holds sm_103a code only: any other device (sm_100 included) would fail at the
  // first launch with "no kernel image"
  if (major != 10 || minor != 3) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// ---------------------------------------------------------------- kernel timing
struct ProfRec {
  int kernel;
  cudaEvent_t start, stop;
};
std::atomic<int> g_prof_on{0};
std::mutex g_prof_mu;
std::vector<ProfRec> g_prof_recs;
std::vector<cudaEvent_t> g_prof_pool;
ProfRec g_prof_open[fa::kNumKernels];
bool g_prof_is_open[fa::kNumKernels] = {};

cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

}  // namespace

namespace fa {
void profile_mark(int kernel, int end, cudaStream_t s) {
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  if (kernel < 0 || kernel >= kNumKernels) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!end) {
    ProfRec r;
    r.kernel = kernel;
    r.start = prof_event();
    r.stop = prof_event();
    cudaEventRecord(r.start, s);
    g_prof_open[kernel] = r;
    g_prof_is_open[kernel] = true;
  } else if (g_prof_is_open[kernel]) {
    ProfRec r = g_prof_open[kernel];
    cudaEventRecord(r.stop, s);
    g_prof_recs.push_back(r);
    g_prof_is_open[kernel] = false;
  }
}
}  // namespace fa

extern "C" {

int fa_profile_enable(int on) {
  g_prof_on.store(on ? 1 : 0);
  return FA_OK;
}

int fa_profile_read(double* total_ms, int64_t* launches) {
  if (!total_ms || !launches) return FA_ERR_INVALID;
  for (int k = 0; k < fa::kNumKernels; ++k) {
    total_ms[k] = 0.0;
    launches[k] = 0;
  }
  std::lock_guard<std::mutex> lk(g_prof_mu);
  int rc = FA_OK;
  for (const ProfRec& r : g_prof_recs) {
    float ms = 0.0f;
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start, r.stop);
    if (e != cudaSuccess) {
      rc = cuda_fail(e, "fa_profile_read");
    } else {
      total_ms[r.kernel] += ms;
      launches[r.kernel] += 1;
    }
    g_prof_pool.push_back(r.start);
    g_prof_pool.push_back(r.stop);
  }
  g_prof_recs.clear();
  return rc;
}

const char* fa_kernel_name(int id) {
  switch (id) {
    case FA_KERNEL_FWD: return "fwd_kernel";
    case FA_KERNEL_BWD_PREP: return "bwd_prep_kernel";
    case FA_KERNEL_BWD_DQ_DET: return "bwd_dq_det_kernel";
    case FA_KERNEL_PAGED: return "paged_attn_kernel";
    case FA_KERNEL_PAGED_COMBINE: return "paged_combine_kernel";
    case FA_KERNEL_PAGED_GATHER: return "paged_gather_kernel";
    case FA_KERNEL_PAGED_SCATTER: return "paged_scatter_kernel";
    case FA_KERNEL_PAGED_DECODE_BWD: return "paged_decode_bwd_kernel";
    case FA_KERNEL_BWD_MAIN: return "bwd_main_kernel";
    case FA_KERNEL_BWD_DQ: return "bwd_dq_kernel";
    default: return "unknown";
  }
}

int fa_train_fwd_ex(const void* q, const void* k, const void* v, const void* mask, void* o,
                    float* lse, const fa_params* p, const fa_options* opt, void* stream) {
  int rc = check_params(p);
  if (rc) return rc;
  if ((rc = check_bf16(q)) || (rc = check_bf16(k)) || (rc = check_bf16(v)) ||
      (rc = check_bf16(o)) || (rc = check_f32(lse)))
    return rc;
  const fa_options o_def = default_options(p);
  const fa_options* op = opt ? opt : &o_def;
  if ((rc = check_options(op, mask, p, false))) return rc;
  if ((rc = check_device())) return rc;
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return cuda_fail(e, "cuTensorMapEncodeTiled entry point");
  int dev = 0;
  cudaGetDevice(&dev);
  fa::FwdArgs a;
  a.mask = mask;
  a.mask_type = op->mask_type;
  a.mask_stride_b = op->mask_stride_b;
  a.mask_stride_h = op->mask_stride_h;
  a.mask_stride_q = op->mask_stride_q;
  a.sinks = op->sinks;
  a.cu_q = op->cu_seqlens_q;
  a.cu_k = op->cu_seqlens_k;
  a.total_q = op->total_q;
  a.total_k = op->total_k;
  a.q_bshd = (op->layout & FA_LAYOUT_Q_BSHD) != 0;
  a.kv_bshd = (op->layout & FA_LAYOUT_KV_BSHD) != 0;
  a.o = o;
  a.lse = lse;
  if ((e = device_status_word(dev, &a.status)) != cudaSuccess) return cuda_fail(e, "status word");
  a.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  a.B = p->batch;
  a.H = p->n_heads;
  a.Hk = p->n_kv_heads;
  a.ql = p->ql;
  a.kl = p->kl;
  a.d = p->head_dim;
  a.dval = op->value_dim ? op->value_dim : p->head_dim;
  a.scale = p->scale;
  const fa::Band band = fa::make_band(p->causal, op->window_left, op->window_right);
  a.lo_off = band.lo_off;
  a.hi_off = band.hi_off;
  a.band = band.mode;
  fa::FwdMaps m;
  const int qrows = fa::fwd_q_box_rows(a.d), kvrows = fa::fwd_kv_box_rows(a.d);
  // tensor-map z and rows: (batch, head) slices of ql / kl rows, or for a variable-length
  // batch the heads of total_q / total_k packed rows
  const bool vl = a.cu_q != nullptr;
  const int nb = vl ? 1 : a.B;
  const int qr = vl ? a.total_q : a.ql, kr = vl ? a.total_k : a.kl;
  if (!encode_bf16_map(&m.q, q, a.d, qr, a.H, nb, a.q_bshd, qrows) ||
      !encode_bf16_map(&m.k, k, a.d, kr, a.Hk, nb, a.kv_bshd, kvrows) ||
      !encode_bf16_map(&m.v, v, a.dval, kr, a.Hk, nb, a.kv_bshd, kvrows))
    return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
  e = fa::launch_fwd(a, m, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return FA_OK;
}

int fa_train_fwd(const void* q, const void* k, const void* v, const float* mask, void* o,
                 float* lse, const fa_params* p, void* stream) {
  if (mask && !aligned(mask, 16)) return FA_ERR_INVALID;
  return fa_train_fwd_ex(q, k, v, mask, o, lse, p, nullptr, stream);
}

// Fills the backward arguments shared by the allocating and the no-allocation entry points.
static int prepare_bwd(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dO, const void* mask, void* dq, void* dk,
                       void* dv, const fa_params* p, const fa_options* opt, fa::BwdArgs* a,
                       fa::BwdMaps* m) {
  int rc = check_params(p);
  if (rc) return rc;
  if ((rc = check_bf16(q)) || (rc = check_bf16(k)) || (rc = check_bf16(v)) ||
      (rc = check_bf16(o)) || (rc = check_f32(lse)) || (rc = check_bf16(dO)) ||
      (rc = check_bf16(dq)) || (rc = check_bf16(dk)) || (rc = check_bf16(dv)))
    return rc;
  const fa_options o_def = default_options(p);
  const fa_options* op = opt ? opt : &o_def;
  if ((rc = check_options(op, mask, p, true))) return rc;
  a->q = q;
  a->k = k;
  a->v = v;
  a->o = o;
  a->lse = lse;
  a->dO = dO;
  a->mask = mask;
  a->mask_type = op->mask_type;
  a->mask_stride_b = op->mask_stride_b;
  a->mask_stride_h = op->mask_stride_h;
  a->mask_stride_q = op->mask_stride_q;
  a->sinks = op->sinks;
  a->dsinks = op->dsinks;
  a->dsink_part = nullptr;  // set with the workspace
  a->deterministic = op->deterministic;
  a->cu_q = op->cu_seqlens_q;
  a->cu_k = op->cu_seqlens_k;
  a->total_q = op->total_q;
  a->total_k = op->total_k;
  a->q_bshd = (op->layout & FA_LAYOUT_Q_BSHD) != 0;
  a->kv_bshd = (op->layout & FA_LAYOUT_KV_BSHD) != 0;
  a->dq = dq;
  a->dk = dk;
  a->dv = dv;
  a->B = p->batch;
  a->H = p->n_heads;
  a->Hk = p->n_kv_heads;
  a->ql = p->ql;
  a->kl = p->kl;
  a->d = p->head_dim;
  a->dval = op->value_dim ? op->value_dim : p->head_dim;
  a->ql_pad = fa::bwd_ql_pad(a->ql);
  a->scale = p->scale;
  const fa::Band band = fa::make_band(p->causal, op->window_left, op->window_right);
  a->lo_off = band.lo_off;
  a->hi_off = band.hi_off;
  a->band = band.mode;
  a->status = nullptr;
  a->wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  (void)m;
  return FA_OK;
}

static int encode_bwd_maps(const fa::BwdArgs& a, fa::BwdMaps* m) {
  const int qrows = fa::bwd_q_box_rows(a.d), kvrows = fa::bwd_kv_box_rows(a.d);
  const bool vl = a.cu_q != nullptr;  // variable-length batch: one batch of packed rows
  const int nb = vl ? 1 : a.B;
  const int qr = vl ? a.total_q : a.ql, kr = vl ? a.total_k : a.kl;
  const bool qs = a.q_bshd, ks = a.kv_bshd;
  if (!encode_bf16_map(&m->q, a.q, a.d, qr, a.H, nb, qs, qrows) ||
      !encode_bf16_map(&m->dO, a.dO, a.dval, qr, a.H, nb, qs, qrows) ||
      !encode_bf16_map(&m->k, a.k, a.d, kr, a.Hk, nb, ks, kvrows) ||
      !encode_bf16_map(&m->v, a.v, a.dval, kr, a.Hk, nb, ks, kvrows))
    return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
  if (a.deterministic) {
    const int drows = fa::dq_det_box_rows();
    if (!encode_bf16_map(&m->det.q, a.q, a.d, qr, a.H, nb, qs, 128) ||
        !encode_bf16_map(&m->det.dO, a.dO, a.dval, qr, a.H, nb, qs, 128) ||
        !encode_bf16_map(&m->det.k, a.k, a.d, kr, a.Hk, nb, ks, drows) ||
        !encode_bf16_map(&m->det.v, a.v, a.dval, kr, a.Hk, nb, ks, drows))
      return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
  }
  return FA_OK;
}

int fa_train_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, const void* mask, void* dq, void* dk, void* dv,
                    const fa_params* p, const fa_options* opt, void* stream) {
  fa::BwdArgs a;
  fa::BwdMaps m;
  int rc = prepare_bwd(q, k, v, o, lse, dO, mask, dq, dk, dv, p, opt, &a, &m);
  if (rc) return rc;
  if ((rc = check_device())) return rc;
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return cuda_fail(e, "cuTensorMapEncodeTiled entry point");
  int dev = 0;
  cudaGetDevice(&dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((e = device_status_word(dev, &a.status)) != cudaSuccess) return cuda_fail(e, "status word");
  if ((rc = encode_bwd_maps(a, &m))) return rc;

  const size_t ws_bytes = fa::bwd_workspace_bytes(a.B, a.H, a.ql, a.d);
  void* ws = nullptr;
  e = cudaMallocAsync(&ws, ws_bytes, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync (backward workspace)");
  fa::bwd_carve_workspace(ws, a.B, a.H, a.ql, a.d, &a.lse2, &a.dvec, &a.dqacc,
                          &a.dsink_part);
  e = fa::launch_bwd(a, m, s);
  cudaError_t e2 = cudaFreeAsync(ws, s);
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaFreeAsync (backward workspace)");
  return FA_OK;
}

int fa_train_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dO, const float* mask, void* dq, void* dk, void* dv,
                 const fa_params* p, void* stream) {
  if (mask && !aligned(mask, 16)) return FA_ERR_INVALID;
  return fa_train_bwd_ex(q, k, v, o, lse, dO, mask, dq, dk, dv, p, nullptr, stream);
}

int fa_train_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, const float* mask, void* dq, void* dk,
                         void* dv, const fa_params* p, void* stream) {
  if (mask && !aligned(mask, 16)) return FA_ERR_INVALID;
  fa::BwdArgs a;
  fa::BwdMaps m;
  int rc = prepare_bwd(q, k, v, o, lse, dO, mask, dq, dk, dv, p, nullptr, &a, &m);
  if (rc) return rc;
  const size_t ws_bytes = fa::bwd_workspace_bytes(a.B, a.H, a.ql, a.d);
  const size_t ws_max = fa::kNoAllocScratchBytes - fa::kNoAllocStatusBytes;
  if (ws_bytes > ws_max) {
    snprintf(g_last_cuda_error, sizeof(g_last_cuda_error),
             "fa_train_bwd_noalloc: needs %zu bytes of scratch, the fixed array holds %zu",
             ws_bytes, ws_max);
    return FA_ERR_TOO_LARGE;
  }
  if ((rc = check_device())) return rc;
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return cuda_fail(e, "cuTensorMapEncodeTiled entry point");
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  void* base = nullptr;
  if ((e = fa::noalloc_scratch(&base)) != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
  if ((rc = encode_bwd_maps(a, &m))) return rc;
  // the array's first bytes are this path's status word (a bounded wait that runs out is
  // recorded there, and fa_device_status reads it); the workspace follows. The pre-pass
  // rewrites L*log2(e) and D and zeroes the dQ accumulator for every row the main pass reads,
  // so the array's previous contents never reach a result
  a.status = static_cast<int*>(base);
  void* ws = static_cast<uint8_t*>(base) + fa::kNoAllocStatusBytes;
  if (dev >= 0 && dev < 64) g_noalloc_used.fetch_or(uint64_t(1) << dev);
  fa::bwd_carve_workspace(ws, a.B, a.H, a.ql, a.d, &a.lse2, &a.dvec, &a.dqacc,
                          &a.dsink_part);
  e = fa::launch_bwd(a, m, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  return FA_OK;
}

// Parameter and pointer checks shared by the paged forward and backward.
static int check_paged(const fa_paged_params* p, const void* q, const void* k_cache,
                       const void* v_cache, const int32_t* block_table, const int32_t* lengths) {
  if (!p) return FA_ERR_INVALID;
  const int ps = p->page_size;
  if (p->batch <= 0 || p->n_heads <= 0 || p->n_kv_heads <= 0 || p->q_len <= 0 ||
      p->max_pages <= 0 || p->num_pages <= 0 || p->n_heads % p->n_kv_heads)
    return FA_ERR_INVALID;
  if (p->head_dim != 64 && p->head_dim != 128 && p->head_dim != 256) return FA_ERR_INVALID;
  if (ps < 8 || ps > 256 || (ps & (ps - 1))) return FA_ERR_INVALID;
  if (!(p->scale > 0.0f) || !std::isfinite(p->scale)) return FA_ERR_INVALID;
  if ((p->causal != 0 && p->causal != 1) || p->reserved != 0) return FA_ERR_INVALID;
  if (p->num_splits < 0 || p->num_splits > 1024) return FA_ERR_INVALID;
  if ((int64_t)p->max_pages * ps > kMaxLen || p->q_len > kMaxLen) return FA_ERR_INVALID;
  if ((int64_t)p->num_pages * p->n_kv_heads > INT32_MAX / 2) return FA_ERR_INVALID;
  const int64_t G = p->n_heads / p->n_kv_heads;
  if (G * p->q_len > (int64_t)kPagedMaxRows) return FA_ERR_INVALID;
  if ((int64_t)p->batch * p->n_kv_heads > 65535) return FA_ERR_INVALID;  // grid y
  int rc;
  if ((rc = check_bf16(q)) || (rc = check_bf16(k_cache)) || (rc = check_bf16(v_cache))) return rc;
  if (!block_table || !lengths || !aligned(block_table, 4) || !aligned(lengths, 4))
    return FA_ERR_INVALID;
  return FA_OK;
}

int fa_paged_attention(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_table, const int32_t* lengths, void* o, float* lse,
                       const fa_paged_params* p, void* stream) {
  if (!p) return FA_ERR_INVALID;
  const int ps = p->page_size;
  const int64_t G = p->n_heads > 0 && p->n_kv_heads > 0 ? p->n_heads / p->n_kv_heads : 0;
  int rc;
  if ((rc = check_paged(p, q, k_cache, v_cache, block_table, lengths)) || (rc = check_bf16(o)))
    return rc;
  if (lse && !aligned(lse, 4)) return FA_ERR_INVALID;
  if ((rc = check_device())) return rc;
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return cuda_fail(e, "cuTensorMapEncodeTiled entry point");
  int dev = 0;
  cudaGetDevice(&dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  fa::PagedArgs a;
  a.table = block_table;
  a.lens = lengths;
  a.o = o;
  a.lse = lse;
  if ((e = device_status_word(dev, &a.status)) != cudaSuccess) return cuda_fail(e, "status word");
  a.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  a.B = p->batch;
  a.H = p->n_heads;
  a.Hk = p->n_kv_heads;
  a.G = (int)G;
  a.lq = p->q_len;
  a.d = p->head_dim;
  a.bs = ps;
  a.max_pages = p->max_pages;
  a.num_pages = p->num_pages;
  a.causal = p->causal;
  a.num_splits = p->num_splits;
  a.scale = p->scale;
  fa::PagedMaps m;
  const int rows = a.G * a.lq, kvrows = fa::paged_key_box_rows(ps);
  if (!encode_bf16_3d(&m.q, q, a.B * a.Hk, rows, a.d, fa::paged_query_box_rows()) ||
      !encode_bf16_3d(&m.k, k_cache, a.num_pages * a.Hk, ps, a.d, kvrows) ||
      !encode_bf16_3d(&m.v, v_cache, a.num_pages * a.Hk, ps, a.d, kvrows))
    return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
  const int splits = fa::paged_splits(a);
  const size_t ws_bytes = fa::paged_workspace_bytes(a, splits);
  void* ws = nullptr;
  if (ws_bytes) {
    e = cudaMallocAsync(&ws, ws_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync (paged workspace)");
  }
  e = fa::launch_paged(a, m, splits, ws, s);
  cudaError_t e2 = ws ? cudaFreeAsync(ws, s) : cudaSuccess;
  if (e != cudaSuccess) return cuda_fail(e, "paged attention launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaFreeAsync (paged workspace)");
  return FA_OK;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int fa_paged_attention_bwd(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_table, const int32_t* lengths, const void* o,
                           const float* lse, const void* dO, void* dq, void* dk_cache,
                           void* dv_cache, const fa_paged_params* p, void* stream) {
  int rc;
  if ((rc = check_paged(p, q, k_cache, v_cache, block_table, lengths))) return rc;
  if ((rc = check_bf16(o)) || (rc = check_bf16(dO)) || (rc = check_bf16(dq)) ||
      (rc = check_bf16(dk_cache)) || (rc = check_bf16(dv_cache)) || (rc = check_f32(lse)))
    return rc;
  const int B = p->batch, H = p->n_heads, Hk = p->n_kv_heads, lq = p->q_len, d = p->head_dim;
  const int G = H / Hk;
  const int64_t cap = (int64_t)p->max_pages * p->page_size;
  const int64_t chunks = d / 8;  // 16-byte chunks per row: grid x of the row kernels
  if ((int64_t)p->num_pages * p->page_size * chunks / 256 >= INT32_MAX ||
      (int64_t)B * H * lq * chunks / 256 >= INT32_MAX)
    return FA_ERR_INVALID;
  fa::PagedGradArgs g;
  g.k_cache = k_cache;
  g.v_cache = v_cache;
  g.table = block_table;
  g.lens = lengths;
  g.q = q;
  g.o = o;
  g.dO = dO;
  g.lse = lse;
  g.dq = dq;
  g.dk_cache = dk_cache;
  g.dv_cache = dv_cache;
  g.B = B;
  g.H = H;
  g.Hk = Hk;
  g.lq = lq;
  g.d = d;
  g.ps = p->page_size;
  g.max_pages = p->max_pages;
  g.num_pages = p->num_pages;
  g.causal = p->causal;
  g.ps_shift = 0;
  while ((1 << g.ps_shift) < p->page_size) ++g.ps_shift;
  g.cpr_shift = d == 64 ? 3 : d == 128 ? 4 : 5;
  if (fa::paged_decode_path(G, lq)) {
    // few query rows per kv head: the CUDA-core kernels read the pages directly
    if ((rc = check_device())) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t owner_bytes = align256((size_t)p->num_pages * 4);
    const size_t acc_bytes = align256((size_t)B * H * lq * d * 4);
    void* ws = nullptr;
    cudaError_t e = cudaMallocAsync(&ws, owner_bytes + acc_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync (paged backward workspace)");
    g.owner = static_cast<int32_t*>(ws);
    float* dq_acc = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + owner_bytes);
    if ((e = device_status_word(dev, &g.status)) != cudaSuccess ||
        (e = cudaMemsetAsync(g.owner, 0xFF, (size_t)p->num_pages * 4, s)) != cudaSuccess ||
        (e = cudaMemsetAsync(dq_acc, 0, (size_t)B * H * lq * d * 4, s)) != cudaSuccess ||
        (e = fa::launch_paged_decode_bwd(g, dq_acc, p->scale, s)) != cudaSuccess) {
      cudaFreeAsync(ws, s);
      return cuda_fail(e, "paged backward (decode path)");
    }
    if ((e = cudaFreeAsync(ws, s)) != cudaSuccess)
      return cuda_fail(e, "cudaFreeAsync (paged backward workspace)");
    return FA_OK;
  }
  // the packed problem: a variable-length batch of B sequences, one per sequence's used keys;
  // with `pack` the G query heads of a kv head are its G * lq rows (no row's keys depend on
  // its position: decode, or no causal rule)
  const bool pack = lq == 1 || !p->causal;
  const int Hq = pack ? Hk : H;
  const int64_t rq = pack ? (int64_t)G * lq : lq;
  const int64_t total_q = B * rq, total_k = B * cap;
  if (rq > kMaxLen || total_q * Hq > INT32_MAX / 2 || total_k * Hk > INT32_MAX / 2)
    return FA_ERR_INVALID;
  if ((rc = check_device())) return rc;
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return cuda_fail(e, "cuTensorMapEncodeTiled entry point");
  int dev = 0;
  cudaGetDevice(&dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  fa_params fp;
  fp.batch = B;
  fp.n_heads = Hq;
  fp.n_kv_heads = Hk;
  fp.ql = (int32_t)rq;
  fp.kl = (int32_t)cap;
  fp.head_dim = d;
  fp.scale = p->scale;
  fp.causal = pack ? 0 : 1;  // (bottom-right: query i of a sequence sees keys <= len - lq + i)
  fa_options fo = default_options(&fp);
  fo.total_q = (int32_t)total_q;
  fo.total_k = (int32_t)total_k;  // an upper bound: the keys used are cu_k[B] <= B * capacity
  const size_t kv_bytes = align256((size_t)Hk * total_k * d * 2);
  const size_t q_bytes = align256((size_t)B * H * lq * d * 2);
  const size_t lse_bytes = align256((size_t)B * H * lq * 4);
  const size_t cu_bytes = align256((size_t)(B + 1) * 4);
  const size_t owner_bytes = align256((size_t)p->num_pages * 4);
  const size_t bwd_bytes = fa::bwd_workspace_bytes(B, Hq, (int)rq, d);
  const size_t total =
      4 * kv_bytes + 4 * q_bytes + lse_bytes + 2 * cu_bytes + owner_bytes + bwd_bytes;
  void* ws = nullptr;
  e = cudaMallocAsync(&ws, total, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync (paged backward workspace)");
  uint8_t* w = static_cast<uint8_t*>(ws);
  auto take = [&w](size_t n) {
    uint8_t* r = w;
    w += n;
    return r;
  };
  g.k_pack = take(kv_bytes);
  g.v_pack = take(kv_bytes);
  g.dk_pack = take(kv_bytes);
  g.dv_pack = take(kv_bytes);
  g.q_pack = take(q_bytes);
  g.o_pack = take(q_bytes);
  g.do_pack = take(q_bytes);
  g.dq_pack = take(q_bytes);
  g.lse_pack = reinterpret_cast<float*>(take(lse_bytes));
  g.cu_q = reinterpret_cast<int32_t*>(take(cu_bytes));
  g.cu_k = reinterpret_cast<int32_t*>(take(cu_bytes));
  g.owner = reinterpret_cast<int32_t*>(take(owner_bytes));
  void* bwd_ws = take(bwd_bytes);
  g.pack = pack ? 1 : 0;
  fo.cu_seqlens_q = g.cu_q;
  fo.cu_seqlens_k = g.cu_k;
  fa::BwdArgs a;
  fa::BwdMaps m;
  if ((e = device_status_word(dev, &g.status)) != cudaSuccess ||
      (e = cudaMemsetAsync(g.owner, 0xFF, (size_t)p->num_pages * 4, s)) != cudaSuccess ||
      (e = fa::launch_paged_gather(g, s)) != cudaSuccess) {
    cudaFreeAsync(ws, s);
    return cuda_fail(e, "paged backward: gather");
  }
  rc = prepare_bwd(g.q_pack, g.k_pack, g.v_pack, g.o_pack, g.lse_pack, g.do_pack, nullptr,
                   const_cast<void*>(g.dq_pack), const_cast<void*>(g.dk_pack),
                   const_cast<void*>(g.dv_pack), &fp, &fo, &a, &m);
  if (!rc) {
    a.status = g.status;
    rc = encode_bwd_maps(a, &m);
  }
  if (rc) {
    cudaFreeAsync(ws, s);
    return rc;
  }
  fa::bwd_carve_workspace(bwd_ws, a.B, a.H, a.ql, a.d, &a.lse2, &a.dvec, &a.dqacc,
                          &a.dsink_part);
  if ((e = fa::launch_bwd(a, m, s)) != cudaSuccess ||
      (e = fa::launch_paged_scatter(g, s)) != cudaSuccess) {
    cudaFreeAsync(ws, s);
    return cuda_fail(e, "paged backward launch");
  }
  if ((e = cudaFreeAsync(ws, s)) != cudaSuccess)
    return cuda_fail(e, "cudaFreeAsync (paged backward workspace)");
  return FA_OK;
}

int fa_device_status(int clear) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int* w = nullptr;
  if ((e = device_status_word(dev, &w)) != cudaSuccess) return cuda_fail(e, "status word");
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  int v = 0;
  if ((e = cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "cudaMemcpy (status)");
  if (clear && v) {
    if ((e = cudaMemset(w, 0, sizeof(int))) != cudaSuccess) return cuda_fail(e, "cudaMemset");
  }
  if (dev < 64 && ((g_noalloc_used.load() >> dev) & 1u)) {  // the no-allocation path's word
    int v2 = 0;
    if ((e = fa::noalloc_status(clear, &v2)) != cudaSuccess)
      return cuda_fail(e, "no-allocation status word");
    if (v2 && (!v || v2 == fa::kStatusTimeout)) v = v2;
  }
  if (!v) return FA_OK;
  return v == fa::kStatusBadInput ? FA_ERR_BAD_INPUT : FA_ERR_DEVICE_TIMEOUT;
}

int fa_set_wait_limit_ns(uint64_t ns) {
  if (ns > kMaxWaitLimitNs) return FA_ERR_INVALID;
  g_wait_limit_ns.store(ns == 0 ? fa::kWaitLimitNs : ns);
  return FA_OK;
}

uint64_t fa_get_wait_limit_ns(void) { return g_wait_limit_ns.load(); }

int fa_debug_ex2(const float* x, float* y_poly, float* y_mufu, float* y_ref, int64_t n,
                 void* stream) {
  if (n < 0) return FA_ERR_INVALID;
  if (n > 0 && (!x || !y_poly || !y_mufu || !y_ref || !aligned(x, 4) || !aligned(y_poly, 4) ||
                !aligned(y_mufu, 4) || !aligned(y_ref, 4)))
    return FA_ERR_INVALID;
  int rc;
  if ((rc = check_device())) return rc;
  cudaError_t e = fa::launch_ex2_probe(x, y_poly, y_mufu, y_ref, (long long)n,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "exp2 probe launch");
}

int fa_debug_wait_timeout(uint64_t* waited_ns, void* stream) {
  if (waited_ns && !aligned(waited_ns, 8)) return FA_ERR_INVALID;
  int rc;
  if ((rc = check_device())) return rc;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int* status = nullptr;
  if ((e = device_status_word(dev, &status)) != cudaSuccess) return cuda_fail(e, "status word");
  e = fa::launch_wait_probe(status, g_wait_limit_ns.load(),
                            reinterpret_cast<unsigned long long*>(waited_ns),
                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "wait probe launch");
}

const char* fa_error_string(int code) {
  switch (code) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID: return "invalid argument (parameter, null or misaligned pointer)";
    case FA_ERR_CUDA: return "CUDA call or kernel launch failed";
    case FA_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait on the device";
    case FA_ERR_UNSUPPORTED:
      return "unsupported: the device is not compute capability 10.3 (the library holds sm_103a code only), or no kernel exists for this head-dim pair";
    case FA_ERR_TOO_LARGE: return "problem needs more scratch than the fixed no-allocation array holds";
    case FA_ERR_BAD_INPUT:
      return "a paged call met a sequence length or block-table entry out of range";
    default: return "unknown error code";
  }
}

const char* fa_last_cuda_error(void) { return g_last_cuda_error; }

const char* fa_version(void) { return "fa_gb300 0.1 (sm_103a, tcgen05)"; }

int fa_value_dim_supported(int head_dim, int value_dim) {
  if (value_dim == head_dim) return head_dim == 64 || head_dim == 128 || head_dim == 256;
  return head_dim == 128 && value_dim == 64;
}

}  // extern "C"
