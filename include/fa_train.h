/*
 * fa_train.h -- C ABI of libfa_gb300: exact scaled-dot-product attention for training on one
 * NVIDIA GB300 (sm_103a), forward and backward.
 *
 * The operation (page "mlx-native tests/test_flash_attn_train.rs", functions
 * `sdpa_reference_with_logsumexp` and `sdpa_backward_reference_f32`; causal alignment as in the
 * nuvec-core direct formula, page "nuvec-core tests/fast.rs",
 * `attention_fallback_matches_a_direct_formula`):
 *
 *   for batch b, query head h, query row i, kv head kh = h / (n_heads / n_kv_heads):
 *     visible(i, j) = !causal || j <= kl - ql + i          (bottom-right alignment, signed)
 *     s_ij = scale * <q_i, k_j> + mask[b,h,i,j]             (-inf where not visible)
 *     L_i  = log sum_j exp(s_ij)                            (natural log; -inf if no key)
 *     O_i  = sum_j exp(s_ij - L_i) v_j                      (0 if L_i = -inf)
 *
 *   backward, with dO the gradient of O and P_ij = exp(s_ij - L_i), D_i = <dO_i, O_i>:
 *     dS_ij = P_ij (<dO_i, v_j> - D_i)
 *     dQ_i  = scale * sum_j dS_ij k_j
 *     dK_j  = scale * sum_{h sharing kh} sum_i dS_ij q_i
 *     dV_j  =         sum_{h sharing kh} sum_i P_ij dO_i
 *
 * Internally the scores are taken to base 2: the f32 dot product is multiplied by
 * scale*log2(e), the mask by log2(e), the running row maximum starts at -FLT_MAX/2, and
 * L = max_2 * ln(2) + ln(sum) -- the conventions of the same mlx-native page.
 *
 * Layouts: every tensor is contiguous, row-major, on the current CUDA device.
 *   q, o, dO, dq          [batch, n_heads,    ql, head_dim]  bf16 (raw 16-bit patterns)
 *   k, v, dk, dv          [batch, n_kv_heads, kl, head_dim]  bf16
 *   lse                   [batch, n_heads,    ql]            f32, natural-log logsumexp L
 *   mask (optional)       [batch, n_heads,    ql, kl]        f32, natural-log additive; an
 *                                                            entry of -inf hides that key
 *
 * Ownership: the caller owns every buffer. Outputs are overwritten completely, never
 * accumulated into. The backward needs f32 scratch (a per-row D and a dQ accumulator); the
 * library takes it with cudaMallocAsync on `stream` and frees it with cudaFreeAsync on the same
 * stream inside the call.
 *
 * Streams: `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are
 * asynchronous: they return after the kernels are enqueued. Inputs must not be modified, and
 * outputs not read, until the stream reaches that point.
 *
 * Errors: a synchronous return code. Arguments are checked before anything is enqueued, so an
 * FA_ERR_INVALID call has no effect. FA_ERR_CUDA means a CUDA call or launch failed (the text
 * of the last such error is kept per thread, see fa_last_cuda_error). Kernel-side pipeline
 * stalls are bounded: a kernel that waited more than 2 s (see fa_set_wait_limit_ns) on one of
 * its own barriers gives up, returns, and leaves FA_ERR_DEVICE_TIMEOUT for fa_device_status to
 * report.
 *
 * Devices: the library holds sm_103a code only; every compute call first checks that the
 * current device has compute capability 10.3 (FA_ERR_UNSUPPORTED otherwise). Per-device state
 * (kernel attributes, the status word) is set up on each device at its first use, so one
 * process may drive several GPUs, from several host threads.
 */
#ifndef FA_TRAIN_H_
#define FA_TRAIN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Problem description. Mirrors the parameter block of the mlx-native dispatch functions
 * (`FlashAttnTrainParams` in the same test page, section "Run the training-forward kernel"). */
typedef struct fa_params {
  int32_t batch;      /* >= 1 */
  int32_t n_heads;    /* query heads, >= 1, a multiple of n_kv_heads */
  int32_t n_kv_heads; /* key/value heads, >= 1 */
  int32_t ql;         /* query length, >= 1 */
  int32_t kl;         /* key length, >= 1 */
  int32_t head_dim;   /* 64, 128 or 256 */
  float scale;        /* finite and > 0; a plain multiplier (not assumed to be 1/sqrt(d)) */
  int32_t causal;     /* 0 or 1: bottom-right causal mask (q_abs = kl - ql + i) */
} fa_params;

/* Return codes. */
#define FA_OK 0
#define FA_ERR_INVALID 1        /* bad parameter, null or misaligned pointer */
#define FA_ERR_CUDA 2           /* a CUDA runtime/driver call or a launch failed */
#define FA_ERR_DEVICE_TIMEOUT 3 /* a kernel gave up a bounded wait (see fa_device_status) */
#define FA_ERR_UNSUPPORTED 4    /* the device is not compute capability 10.3, or no kernel
                                   exists for the requested option */
#define FA_ERR_TOO_LARGE 5      /* the problem needs more scratch than fa_train_bwd_noalloc has */
#define FA_ERR_BAD_INPUT 6      /* (fa_device_status) a paged call met a sequence length or a
                                   block-table entry out of range; those keys were read as 0 */

/* Mask element types of fa_options.mask_type. */
#define FA_MASK_F32 0  /* additive, natural log, float (an entry -inf hides the key) */
#define FA_MASK_BF16 1 /* additive, natural log, bf16 */
#define FA_MASK_BOOL 2 /* uint8: nonzero = the key is visible, 0 = hidden */

/* Options beyond the pages' parameter block, for the *_ex entry points.
 *
 * Local (sliding-window) attention, the windowed form of the mlx-native SWA tests (sections 7
 * and 15 of the same page, which build it as an additive -inf mask): with
 * q_abs = kl - ql + i, key j is hidden from query row i when
 *   window_left  >= 0 and j < q_abs - window_left, or
 *   window_right >= 0 and j > q_abs + window_right
 * (-1 = unbounded on that side). It combines with `causal` (j > q_abs hidden) and the mask.
 * Kv tiles outside every row's window are neither loaded nor multiplied.
 *
 * Masks may be given in any of the FA_MASK_* element types and broadcast over batch, heads
 * and/or query rows: element (b, h, i, j) is read at
 *   mask + b*mask_stride_b + h*mask_stride_h + i*mask_stride_q + j      (in elements)
 * (keys contiguous; a zero stride broadcasts). The dense [B, H, ql, kl] f32 mask of the base
 * entry points is mask_type FA_MASK_F32 with strides (H*ql*kl, ql*kl, kl). The mask pointer
 * must be aligned to its element size.
 *
 * Attention sinks (page "nuvec-core tests/fast.rs", the per-head `sinks` input of the fused
 * attention in `attention_kernels_match_the_fallback`; the page gives only the shape, and the
 * reading taken is an extra logit with no value): sinks is NULL or a device array of n_heads
 * f32 natural-log logits, not scaled. sink_h joins the softmax normaliser of every row of
 * head h:  L = log(exp(sink_h) + sum_j exp(s_ij)),  O = sum_j exp(s_ij - L) v_j.
 * A row that sees no key then gives O = 0 and L = sink_h; a sink of -inf is no sink (values
 * must be finite or -inf). dsinks (backward only) is NULL or a device array of n_heads f32
 * that receives the gradient with respect to the sinks,
 *   dsinks[h] = -sum_b sum_i exp(sink_h - L_bhi) * D_bhi,   D = rowsum(dO * O),
 * overwritten (not accumulated) and summed in a fixed order, so it is bitwise reproducible.
 * dsinks requires sinks. The forward and the backward must be given the same sinks.
 *
 * Value head dim (same page: its shapes list (D, Dv) pairs with Dv != D): value_dim = 0 means
 * head_dim; otherwise v, dV are [B, Hk, kl, value_dim] and o, dO are [B, H, ql, value_dim]
 * while q, k, dQ, dK keep head_dim. Supported pairs (head_dim, value_dim) are listed by
 * fa_value_dim_supported; others give FA_ERR_UNSUPPORTED.
 *
 * Deterministic backward (the mlx-native page notes that its GPU backward reduces dQ in a
 * nondeterministic order): with deterministic = 1, dQ is formed query-tile-major by a
 * separate kernel that walks the kv tiles of each query tile in a fixed order, instead of
 * being added into an f32 accumulator by many CTAs at once. dK, dV and dsinks are always
 * reduced in a fixed order, so the whole backward then returns the same bits on every run.
 * It recomputes S and dP once more, which costs time. Ignored by the forward.
 *
 * Variable-length batch (no counterpart on the pages; each sequence is the fixed-length problem
 * above on its own rows): with cu_seqlens_q non-NULL, `batch` independent sequences are packed
 * head-major without padding: q, o, dO, dQ are [n_heads, total_q, d] (o, dO with value_dim),
 * k, v, dK, dV are [n_kv_heads, total_k, d], lse is [n_heads, total_q]. Sequence b owns rows
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1] of q and cu_seqlens_k[b] .. cu_seqlens_k[b+1] of k
 * (int32 device arrays of batch + 1 entries, 0 first, non-decreasing, the last = total_q /
 * total_k), and fa_params.ql / kl give the longest sequence (they size the grids). Causal and
 * window bands align bottom-right within each sequence. A sequence with no keys gives O = 0
 * and L = -inf (or its sink). Offsets out of range are clamped and reported by
 * fa_device_status (FA_ERR_BAD_INPUT). No mask may be given (FA_ERR_UNSUPPORTED).
 *
 * Layouts (page "nuvec-core tests/fast.rs", `attention_kernels_match_the_fallback`, passes K
 * and V as transposed views): by default every bf16 tensor is [batch, heads, rows, dim] in
 * memory. FA_LAYOUT_Q_BSHD makes q, o, dO and dQ [batch, ql, n_heads, dim] in memory, and
 * FA_LAYOUT_KV_BSHD makes k, v, dK and dV [batch, kl, n_kv_heads, dim]; a [batch, heads, rows,
 * dim] view of such a tensor is its transpose of dims 1 and 2. In a variable-length batch the
 * flags make them [total_q, n_heads, dim] / [total_k, n_kv_heads, dim]. The dim is contiguous
 * either way; lse keeps its layout. Outputs are written in the layout of their inputs. */
#define FA_LAYOUT_Q_BSHD 1  /* q, o, dO, dQ as [batch, ql, n_heads, dim] */
#define FA_LAYOUT_KV_BSHD 2 /* k, v, dK, dV as [batch, kl, n_kv_heads, dim] */
typedef struct fa_options {
  int32_t window_left;   /* -1, or >= 0 */
  int32_t window_right;  /* -1, or >= 0 */
  int32_t mask_type;     /* FA_MASK_* (ignored when the mask pointer is NULL) */
  int32_t value_dim;     /* 0 (= head_dim), or a supported value head dim */
  int64_t mask_stride_b; /* >= 0 */
  int64_t mask_stride_h; /* >= 0 */
  int64_t mask_stride_q; /* >= 0 */
  const float* sinks;    /* NULL, or [n_heads] f32 on the device, 4-byte aligned */
  float* dsinks;         /* backward only: NULL, or [n_heads] f32 output on the device */
  int32_t deterministic; /* 0 or 1 (backward only) */
  int32_t layout;        /* 0, or FA_LAYOUT_* flags */
  const int32_t* cu_seqlens_q; /* NULL, or the variable-length batch's query offsets [batch+1] */
  const int32_t* cu_seqlens_k; /* its key offsets [batch+1]; both or neither */
  int32_t total_q;       /* variable-length batch: rows per head of q (>= 1) */
  int32_t total_k;       /* rows per head of k and v (>= 1) */
} fa_options;

/* 1 if this build has kernels for the (head_dim, value_dim) pair, else 0. */
int fa_value_dim_supported(int head_dim, int value_dim);

/* Forward: O and L. Page "mlx-native tests/test_flash_attn_train.rs", sections 2-8 (forward
 * parity), function `sdpa_reference_with_logsumexp`.
 *   q, k, v : inputs (bf16, device, 16-byte aligned)
 *   mask    : NULL, or the f32 additive mask (device, 16-byte aligned)
 *   o       : output, bf16 [batch, n_heads, ql, head_dim]
 *   lse     : output, f32  [batch, n_heads, ql]
 *   p       : problem description (host pointer, read during the call only)
 *   stream  : cudaStream_t
 * A fully masked row gives O = 0 and L = -inf. */
int fa_train_fwd(const void* q, const void* k, const void* v, const float* mask, void* o,
                 float* lse, const fa_params* p, void* stream);

/* Forward with options (window, mask type and broadcast). opt == NULL gives the base
 * behaviour (no window; a mask, if any, dense [B, H, ql, kl] f32). Rows whose window and mask
 * leave no key give O = 0 and L = -inf. Errors as fa_train_fwd; FA_ERR_INVALID also for
 * window values below -1, an unknown mask type, unknown layout flags, a negative value_dim,
 * negative strides, a mask not aligned to its element size or a misaligned sinks pointer;
 * FA_ERR_UNSUPPORTED for a (head_dim, value_dim) pair without kernels. The forward ignores
 * dsinks. */
int fa_train_fwd_ex(const void* q, const void* k, const void* v, const void* mask, void* o,
                    float* lse, const fa_params* p, const fa_options* opt, void* stream);

/* Backward: dQ, dK, dV from the forward's O and L. Same page, sections 10-16 (backward parity),
 * function `sdpa_backward_reference_f32`; the kernel decomposition (a D_i = rowsum(dO * O)
 * pass, a kv-tile-major pass for dK/dV over the query heads that share a kv head, f32 dQ
 * accumulation) follows the flash backward of page "tang src/compute/cuda.rs",
 * `causal_attention_backward`.
 *   q, k, v, o, dO : inputs, bf16 (o is this library's forward output for q, k, v, mask)
 *   lse            : input, f32, the forward's L
 *   mask           : NULL, or the same mask as in the forward
 *   dq, dk, dv     : outputs, bf16, shapes of q, k, v
 * Rows with L = -inf (fully masked) contribute nothing and get dQ = 0. */
int fa_train_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dO, const float* mask, void* dq, void* dk, void* dv,
                 const fa_params* p, void* stream);

/* Kernel timing (a tracing aid). While enabled, each kernel launch of this library is
 * bracketed by two CUDA events recorded on the launch's own stream; fa_profile_read waits for
 * them, adds up the device time per kernel and clears the record. Kernel ids: */
#define FA_KERNEL_FWD 0      /* forward (O, L) */
#define FA_KERNEL_BWD_PREP 1 /* backward pre-pass: D = rowsum(dO * O), scratch zeroing */
#define FA_KERNEL_BWD_MAIN 2 /* backward main pass: dK, dV, dQ accumulation */
#define FA_KERNEL_BWD_DQ 3   /* backward dQ conversion to bf16 (and the dsinks sum) */
#define FA_KERNEL_BWD_DQ_DET 4 /* deterministic mode: query-tile-major dQ */
#define FA_KERNEL_PAGED 5      /* paged key/value cache attention */
#define FA_KERNEL_PAGED_COMBINE 6 /* merge of the key splits of fa_paged_attention */
#define FA_KERNEL_PAGED_GATHER 7  /* fa_paged_attention_bwd: packed K, V, q side / page owners */
#define FA_KERNEL_PAGED_SCATTER 8 /* fa_paged_attention_bwd: cache gradients completed, dq */
#define FA_KERNEL_PAGED_DECODE_BWD 9 /* fa_paged_attention_bwd, few rows: the gradient kernel */
#define FA_NUM_KERNELS 10

/* Turns timing on (1) or off (0). Returns FA_OK. */
int fa_profile_enable(int on);
/* Fills total_ms[FA_NUM_KERNELS] and launches[FA_NUM_KERNELS] (host arrays) with the device
 * time and number of launches recorded since the last read, then clears the record. */
int fa_profile_read(double* total_ms, int64_t* launches);
/* Name of a kernel id (static storage). */
const char* fa_kernel_name(int id);

/* Backward with options; `opt` (window, mask, value_dim, sinks) and `mask` must be those
 * given to the forward that produced o and lse. opt == NULL gives the base behaviour. With
 * opt->dsinks non-NULL the sink gradient is written too (FA_ERR_INVALID if opt->sinks is
 * NULL or either pointer is not 4-byte aligned). */
int fa_train_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, const void* mask, void* dq, void* dk, void* dv,
                    const fa_params* p, const fa_options* opt, void* stream);

/* Backward without any device allocation. The pages have no counterpart of this entry point.
 *
 * Some callers cannot let a library allocate device memory: processes whose GPU memory is
 * owned by a pool allocator that has already reserved the device (an allocation made behind
 * its back can fail or be invisible to its accounting), and step loops where an allocation is
 * not allowed because it may block or fail at an unpredictable moment. For them this call does
 * what fa_train_bwd does, with the same arguments, layouts and results, but takes its scratch
 * (the per-row D, L*log2(e) and the f32 dQ accumulator) from a fixed array compiled into the
 * library instead of cudaMallocAsync. It calls no cudaMalloc, cudaFree or other allocating
 * routine; the caller still provides every input and output.
 *
 * Limits and rules:
 *  - the array holds 64 MiB per GPU: its first 256 bytes are the status word of these calls (a
 *    bounded wait that runs out is recorded there and reported by fa_device_status, as for the
 *    other entry points), the rest is the backward's scratch. A problem whose scratch,
 *    4*B*H*ceil128(ql)*(head_dim + 2) bytes plus alignment, exceeds 64 MiB - 256 bytes returns
 *    FA_ERR_TOO_LARGE without touching the device;
 *  - the array is part of the library's device code, and CUDA creates it on a GPU when it
 *    loads that code there. With CUDA's default lazy loading this happens at the first call on
 *    that GPU of this entry point or of any backward entry point of the library, and that load
 *    does allocate device memory. So make one call (a warm-up) on each GPU before a pool
 *    allocator reserves the device, or run with CUDA_MODULE_LOADING=EAGER, which creates the
 *    array with the CUDA context. From then on the array stays until the process exits (or a
 *    cudaDeviceReset, after which the next call loads it again, as the first one did);
 *  - the first call on each GPU also sets the kernels' shared-memory attributes; make it
 *    before any stream capture;
 *  - every call looks up the array's address on the current device (cudaGetSymbolAddress,
 *    which allocates nothing once the array exists); nothing is cached between calls;
 *  - every call on a GPU shares that one array, and the array keeps the previous call's
 *    contents (each call rewrites or zeroes what it reads, so that does not leak into
 *    results); calls that overlap on the GPU (for example on two streams) race on it and give
 *    wrong results: serialise them. */
int fa_train_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, const float* mask, void* dq, void* dk,
                         void* dv, const fa_params* p, void* stream);

/* ------------------------------------------------------------------ paged key/value cache
 * Attention of a few new queries per sequence over a paged cache, for inference: single-query
 * decode (q_len = 1) and a causal prefill of q_len positions against a cache. Page
 * "nuvec-core tests/fast.rs", `paged_attention_equals_contiguous_attention` (layout, block
 * table, lengths; one pass below about 1024 keys, two above), and page "tang
 * src/compute/cuda.rs", `kv_attention` (decode, and the prefill with cache_start = len - q_len).
 *
 * The keys of sequence b are its first lengths[b] cache positions; logical key j is in page
 * block_table[b * max_pages + j / page_size], slot j % page_size. The q_len queries are the
 * sequence's last positions: with causal = 1, query i sees key j iff
 * j <= lengths[b] - q_len + i. O = softmax(scale * q k^T) v; L = natural-log logsumexp. A query
 * that sees no key gets O = 0 and L = -inf. Gradients: fa_paged_attention_bwd below. */
typedef struct fa_paged_params {
  int32_t batch;       /* sequences, >= 1 */
  int32_t n_heads;     /* query heads, a multiple of n_kv_heads */
  int32_t n_kv_heads;  /* >= 1 */
  int32_t q_len;       /* new positions per sequence, >= 1 */
  int32_t head_dim;    /* 64, 128 or 256 */
  int32_t page_size;   /* positions per page: a power of two in [8, 256] */
  int32_t max_pages;   /* columns of the block table; max_pages * page_size <= 2^22 */
  int32_t num_pages;   /* pages in each cache */
  float scale;         /* finite and > 0 */
  int32_t causal;      /* 0 or 1 */
  int32_t num_splits;  /* 0: chosen by the library; otherwise the key range is cut into this
                          many parts, each part one CTA, merged by a second kernel */
  int32_t reserved;    /* must be 0 */
} fa_paged_params;

/*   q            bf16 [batch, n_heads, q_len, head_dim] (device, 16-byte aligned)
 *   k_cache      bf16 [num_pages, n_kv_heads, page_size, head_dim] (device, 16-byte aligned)
 *   v_cache      same layout as k_cache
 *   block_table  int32 [batch, max_pages] (device, 4-byte aligned): page of each block of
 *                page_size positions; only the first ceil(lengths[b] / page_size) are read
 *   lengths      int32 [batch] (device): keys of each sequence, 0 .. max_pages * page_size
 *   o            output, bf16 [batch, n_heads, q_len, head_dim] (device, 16-byte aligned)
 *   lse          output or NULL: f32 [batch, n_heads, q_len]
 * The lengths and the table live on the device, so they are checked there: a length outside
 * [0, max_pages * page_size] is clamped and a table entry outside [0, num_pages) reads as zero
 * keys, and either makes fa_device_status return FA_ERR_BAD_INPUT. With more than one split
 * the call takes a small scratch buffer (splits * batch * n_heads * q_len * (head_dim + 1) f32)
 * with cudaMallocAsync on `stream`. Returns FA_OK, FA_ERR_INVALID (parameters, pointers),
 * FA_ERR_UNSUPPORTED or FA_ERR_CUDA. */
int fa_paged_attention(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_table, const int32_t* lengths, void* o, float* lse,
                       const fa_paged_params* p, void* stream);

/* Gradients through the paged cache: dQ and the gradients of both caches for the attention of
 * fa_paged_attention. Page "nuvec-core tests/fast.rs",
 * `paged_attention_equals_contiguous_attention`, checks the gradients for q and the caches
 * ("paged grads").
 *   q, k_cache, v_cache, block_table, lengths, p : as given to fa_paged_attention
 *   o, lse     : that call's outputs (lse required: f32 [batch, n_heads, q_len], 16-byte
 *                aligned)
 *   dO         : bf16 [batch, n_heads, q_len, head_dim], the gradient of the loss for o
 *   dq         : output, bf16 like q
 *   dk_cache, dv_cache : outputs, bf16 like the caches: every element is written; a slot
 *                that no (sequence, query) reads gets 0.
 * Each page may hold keys of one sequence only: a page named twice among the used table
 * entries (its gradient would be a sum) gets a zero gradient and makes fa_device_status return
 * FA_ERR_BAD_INPUT, as do lengths and table entries out of range (read as in the forward).
 * With at most 8 query rows per kv head ((n_heads / n_kv_heads) * q_len <= 8: decode and short
 * cached prefills) CUDA-core kernels read the keys through the block table and write dK, dV
 * into the cache gradients directly (scratch: num_pages * 4 + batch * n_heads * q_len *
 * head_dim * 4 bytes). Otherwise the call turns the batch into a variable-length batch of
 * each sequence's used keys, packed without padding, runs the training backward on it and
 * writes the gradients back; without the causal rule it takes the n_heads / n_kv_heads query
 * heads of a kv head as one sequence's rows (scratch: 4 * batch * n_kv_heads * max_pages *
 * page_size * head_dim * 2 bytes for the keys, 4 * batch * n_heads * q_len * (2 * head_dim +
 * 1) bytes for the query side, plus the backward's own). Scratch is taken with
 * cudaMallocAsync on `stream`.
 * p->num_splits is ignored. Returns FA_OK, FA_ERR_INVALID (parameters, pointers, a packed
 * problem past the size limits: batch * max_pages * page_size * n_kv_heads or
 * batch * n_heads * q_len at 2^30 or more), FA_ERR_UNSUPPORTED or FA_ERR_CUDA. */
int fa_paged_attention_bwd(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_table, const int32_t* lengths, const void* o,
                           const float* lse, const void* dO, void* dq, void* dk_cache,
                           void* dv_cache, const fa_paged_params* p, void* stream);

/* ------------------------------------------------------------------ bounded waits, diagnostics
 * Sets the limit of one barrier wait inside the kernels launched after this call, from any
 * thread (default 2 s; ns = 0 restores it; more than 60 s gives FA_ERR_INVALID). A wait that
 * lasts longer makes its kernel give up and return, with its outputs left undefined, and
 * fa_device_status then reports FA_ERR_DEVICE_TIMEOUT. A short limit makes legitimate waits
 * run out: it exists to test that path, not for normal use. No counterpart on the pages. */
int fa_set_wait_limit_ns(uint64_t ns);
/* The current limit, in ns. */
uint64_t fa_get_wait_limit_ns(void);

/* Test aid (no counterpart on the pages): evaluates, for the n floats of x (device), the two
 * base-2 exponentials the softmax uses -- the FMA-pipe polynomial into y_poly and the hardware
 * approximation into y_mufu -- and CUDA's exp2f into y_ref (device arrays of n floats, 4-byte
 * aligned). Asynchronous on `stream`. */
int fa_debug_ex2(const float* x, float* y_poly, float* y_mufu, float* y_ref, int64_t n,
                 void* stream);

/* Test aid (no counterpart on the pages): one kernel waits on a barrier that nothing ever
 * completes, using the current wait limit. The wait runs out, the kernel records
 * FA_ERR_DEVICE_TIMEOUT for fa_device_status and returns; with waited_ns non-NULL (device,
 * 8-byte aligned) it writes how long it waited, in ns. Asynchronous on `stream`. Set a short
 * limit first (fa_set_wait_limit_ns): with the default the kernel takes 2 s. */
int fa_debug_wait_timeout(uint64_t* waited_ns, void* stream);

/* Synchronises the current device, then returns FA_OK, FA_ERR_DEVICE_TIMEOUT if any kernel of
 * this library on it gave up a bounded wait, or FA_ERR_BAD_INPUT if a paged call met a length
 * or block-table entry out of range, since the last call with clear != 0. */
int fa_device_status(int clear);

/* Human-readable text of a return code (static storage). */
const char* fa_error_string(int code);

/* Text of the last CUDA error seen by this thread in a call that returned FA_ERR_CUDA. */
const char* fa_last_cuda_error(void);

/* Library version string (static storage). */
const char* fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_TRAIN_H_ */
