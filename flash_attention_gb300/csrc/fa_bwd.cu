// fa_bwd.cu -- backward of exact attention: dQ, dK, dV from Q, K, V, O, L and dO (sm_103a).
//
// Method: the FlashAttention-2 backward equations of page "mlx-native
// tests/test_flash_attn_train.rs" (`sdpa_backward_reference_f32`):
//   P = exp(S - L),  dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  dQ = scale dS K,
//   dK = scale dS^T Q,
// with D_i = rowsum(dO_i o O_i) taken from the stored forward output, and the split into
// kernels of the flash backward on page "tang src/compute/cuda.rs" (`causal_attention_backward`):
// a D pre-pass, a kv-tile-major main pass in which each CTA owns one kv tile and walks every
// query head that shares its kv head (so dK and dV are reduced in the CTA, without atomics),
// and dQ accumulated in f32 across CTAs. P is recomputed from L with base-2 exponentials:
// P = exp2(S * scale * log2(e) + mask * log2(e) - L * log2(e)); a row with L = -inf (no
// visible key) gets -inf in place of -L * log2(e), which makes its P exactly 0.
//
// Kernels:
//   bwd_prep_kernel  D_i, -L_i * log2(e), and zeroes the dQ accumulator (bandwidth bound)
//   bwd_main_kernel  per kv tile of 128 rows (and, for head_dim 256, per half of the head
//                    dimension): S^T = K Q^T and dP^T = V dO^T into TMEM; P^T and dS^T
//                    computed by one warpgroup (thread = kv row = TMEM lane) and written back
//                    to TMEM as bf16; dV += P^T dO and dK += dS^T Q with the A operand read
//                    from TMEM; dQ^T = K^T dS^T (head_dim >= 128) or dQ = dS K (head_dim 64)
//                    with dS^T staged in swizzled shared memory; a second warpgroup drains dQ
//                    from TMEM into the f32 accumulator with global reductions (head_dim 64
//                    and 128: one bulk reduction per tile staged in shared memory, at 128 kept
//                    transposed), and writes dK, dV at the end
//   bwd_dq_kernel    dQ = bf16(scale * accumulator); bwd_dq_tiles_kernel does the same from
//                    the transposed tiles of the head_dim-128 bulk path
#include <float.h>

#include "fa_bwd_common.cuh"
#include "fa_bwd_main.cuh"
#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {

// ------------------------------------------------------------------------ prep kernel
// D_i = <dO_i, O_i>, -L_i * log2(e) (-inf for padding rows and rows with L = -inf), and the
// dQ accumulator zeroed. Grid: x = chunk of RPB*ROWS rows within a head, y = head (strided).
// A group of HD/8 threads owns one row (16-byte loads of O and dO); each thread walks ROWS
// rows so that many loads are in flight; the chunk's accumulator rows are then zeroed with
// coalesced float4 stores.
// With sinks and a dsinks output, each block also sums the rows' sink-gradient terms
// -exp(sink_h - L_i) * D_i of its chunk in a fixed order into dsink_part[bh, chunk]; the dQ
// kernel adds those partials up per head (also in a fixed order).
constexpr int kPrepRowsMin = 32;  // fewest rows per prep block (head_dim 256): sizes the partials
template <int HD>
__host__ __device__ constexpr int prep_rows_per_block() {
  return (256 / (HD / 8)) * 4;
}

template <int HD, int DV>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                       const __nv_bfloat16* __restrict__ dO,
                                                       const float* __restrict__ lse,
                                                       float* __restrict__ lse2,
                                                       float* __restrict__ dvec,
                                                       float* __restrict__ dqacc,
                                                       const float* __restrict__ sinks,
                                                       float* __restrict__ dsink_part, int BH,
                                                       int H, int ql, int ql_pad, int zero_acc,
                                                       const int32_t* __restrict__ cu_q,
                                                       int total_q, int q_bshd) {
  constexpr int TPR = DV / 8;            // threads per O / dO row (8 bf16 = 16 bytes each)
  constexpr int RPB = 256 / TPR;         // rows per pass of the block
  constexpr int ROWS = 4;                // passes per block
  static_assert(RPB * ROWS == prep_rows_per_block<DV>(), "prep chunk");
  static_assert(RPB * ROWS >= kPrepRowsMin && RPB * ROWS <= 256, "sink partial layout");
  __shared__ float sink_terms[RPB * ROWS];
  grid_dep_wait();  // (launched to overlap the previous kernel's tail: O may be its output)
  grid_dep_trigger();
  const int sub = threadIdx.x % TPR;
  const int i0 = blockIdx.x * RPB * ROWS;  // first row of the chunk (ql_pad is a multiple)
  const bool want_dsink = dsink_part != nullptr;
  for (int bh = blockIdx.y; bh < BH; bh += gridDim.y) {
    // rows of this (batch, head): fixed length, or sequence b of a variable-length batch
    size_t rowbase = (size_t)bh * ql;            // L row of query 0
    int ob = bh / H, or0 = 0, orows = ql, qlen = ql;  // O / dO: batch, first row, rows
    if (cu_q != nullptr) {
      int qs;
      varlen_seq(cu_q, bh / H, total_q, ql, qs, qlen);
      rowbase = (size_t)(bh % H) * total_q + qs;
      ob = 0;
      or0 = qs;
      orows = total_q;
    }
    if (zero_acc) {  // (the deterministic mode has no accumulator) stores first: they overlap
                     // the loads below
      float4* z = reinterpret_cast<float4*>(dqacc + ((size_t)bh * ql_pad + i0) * HD);
#pragma unroll
      for (int c = threadIdx.x; c < RPB * ROWS * HD / 4; c += 256)
        z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    uint4 a[ROWS], g[ROWS];
    float Lr[ROWS];  // L of the rows this thread reduces (read by the first thread of a row)
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      const int i = i0 + r * RPB + threadIdx.x / TPR;
      a[r] = make_uint4(0, 0, 0, 0);
      g[r] = make_uint4(0, 0, 0, 0);
      Lr[r] = -INFINITY;
      if (i < qlen) {
        const size_t base = bhsd_offset(ob, bh % H, or0 + i, H, orows, DV, q_bshd != 0) + sub * 8;
        a[r] = *reinterpret_cast<const uint4*>(o + base);
        g[r] = *reinterpret_cast<const uint4*>(dO + base);
        if (sub == 0) Lr[r] = lse[rowbase + i];
      }
    }
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[r]);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g[r]);
      float acc = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        acc += __low2float(a2[e]) * __low2float(g2[e]) + __high2float(a2[e]) * __high2float(g2[e]);
#pragma unroll
      for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      const int i = i0 + r * RPB + threadIdx.x / TPR;
      if (sub == 0) {
        float nl2 = -INFINITY;  // padding rows and fully masked rows: P = exp2(s - inf) = 0
        float term = 0.0f;      // this row's share of dsinks[h]
        if (i < qlen) {
          const float L = Lr[r];
          if (L != -INFINITY) {
            nl2 = -L * kLog2eB;
            if (want_dsink) term = -expf(__ldg(sinks + bh % H) - L) * acc;
          }
        }
        lse2[(size_t)bh * ql_pad + i] = nl2;
        dvec[(size_t)bh * ql_pad + i] = i < qlen ? acc : 0.0f;
        if (want_dsink) sink_terms[r * RPB + threadIdx.x / TPR] = term;
      }
    }
    if (want_dsink) {  // block-uniform
      __syncthreads();
      if (threadIdx.x < 32) {
        float s = 0.0f;
        for (int k = threadIdx.x; k < RPB * ROWS; k += 32) s += sink_terms[k];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (threadIdx.x == 0) dsink_part[(size_t)bh * gridDim.x + blockIdx.x] = s;
      }
      __syncthreads();  // sink_terms is rewritten by the next head
    }
  }
}

// ------------------------------------------------------------------------ dQ convert
// dQ = bf16(scale * accumulator). Grid: x = chunk of 256 groups of 8 values within a head,
// y = head (strided). Each thread converts 8 consecutive values (two float4 loads, one 16-byte
// store).
// Blocks with x == 0 also finish dsinks[h] for h = y, y + gridDim.y, ...: the sum, in a fixed
// order, of the prep kernel's partials of every batch entry of head h. With convert = 0 (the
// deterministic mode, where dQ is written by its own kernel) only that sum is done.
// dsinks[h] for h = blockIdx.y, blockIdx.y + gridDim.y, ...: the prep kernel's partials of every
// batch entry of head h, summed in a fixed order (256 threads).
__device__ __forceinline__ void dsinks_sum(const float* __restrict__ dsink_part,
                                           float* __restrict__ dsinks, int B, int H,
                                           int sink_chunks) {
  __shared__ float red[256];
  const int n = B * sink_chunks;
  for (int h = blockIdx.y; h < H; h += gridDim.y) {
    float s = 0.0f;
    for (int k = threadIdx.x; k < n; k += 256)
      s += dsink_part[((size_t)(k / sink_chunks) * H + h) * sink_chunks + k % sink_chunks];
    red[threadIdx.x] = s;
    __syncthreads();
#pragma unroll
    for (int w = 128; w > 0; w >>= 1) {
      if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
      __syncthreads();
    }
    if (threadIdx.x == 0) dsinks[h] = red[0];
    __syncthreads();  // red is reused by the next head
  }
}

// SWZ: rows of the accumulator hold their 16-byte chunks XOR-rotated by (row % kDqChunks)
// (the bulk path at head_dim 64).
template <int HD, bool SWZ>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float* __restrict__ dqacc,
                                                     __nv_bfloat16* __restrict__ dq, int BH,
                                                     int ql, int ql_pad, float scale,
                                                     const float* __restrict__ dsink_part,
                                                     float* __restrict__ dsinks, int B, int H,
                                                     int sink_chunks, int convert,
                                                     const int32_t* __restrict__ cu_q,
                                                     int total_q, int q_bshd) {
  grid_dep_wait();  // the accumulator and the dsinks partials are the previous kernels' output
  if (dsinks != nullptr && blockIdx.x == 0) dsinks_sum(dsink_part, dsinks, B, H, sink_chunks);
  if (!convert) return;
  const int e = blockIdx.x * 256 + threadIdx.x;  // index of the 8-value group within a head
  const int i = e / (HD / 8), c = (e % (HD / 8)) * 8;
  if (i >= ql) return;
  for (int bh = blockIdx.y; bh < BH; bh += gridDim.y) {
    int ob = bh / H, or0 = 0, orows = ql;  // dQ: batch, first row and rows of this problem
    if (cu_q != nullptr) {  // sequence b of a variable-length batch
      int qs, qlen;
      varlen_seq(cu_q, bh / H, total_q, ql, qs, qlen);
      if (i >= qlen) continue;
      ob = 0;
      or0 = qs;
      orows = total_q;
    }
    const float4* srow = reinterpret_cast<const float4*>(dqacc + ((size_t)bh * ql_pad + i) * HD);
    const int c4 = c / 4, rot = SWZ ? (i % kDqChunks) : 0;  // (query tiles start at multiples of 16)
    const float4 v0 = __ldcs(srow + (c4 ^ rot)), v1 = __ldcs(srow + ((c4 + 1) ^ rot));
    uint4 out;
    out.x = pack_bf16(v0.x * scale, v0.y * scale);
    out.y = pack_bf16(v0.z * scale, v0.w * scale);
    out.z = pack_bf16(v1.x * scale, v1.y * scale);
    out.w = pack_bf16(v1.z * scale, v1.w * scale);
    __stcs(reinterpret_cast<uint4*>(dq + bhsd_offset(ob, bh % H, or0 + i, H, orows, HD,
                                                      q_bshd != 0) + c), out);
  }
}

// dQ = bf16(scale * accumulator) from the transposed, chunk-major accumulator tiles of the
// bulk path. Grid: x = (query tile of BM rows, 64-row slice of the head dimension), y =
// (batch, head) (strided); blocks with x == 0 also finish dsinks. A block reads its slice (64
// head-dim rows of BM f32) with all of its 16-byte loads in flight and transposes it through
// shared memory into [q][d] (rows padded to 65 floats, written conflict-free since a warp's
// loads cover one chunk of 32 consecutive rows); then four consecutive threads write one
// query row's 128 contiguous bytes of bf16. Both sides are touched once, so loads and stores
// are marked evict-first (35.1 against 37.6 us on the 4k GQA shape).
template <int HD, int BM>
__global__ void __launch_bounds__(256) bwd_dq_tiles_kernel(const float* __restrict__ dqacc,
                                                           __nv_bfloat16* __restrict__ dq,
                                                           int BH, int ql, int ql_pad,
                                                           float scale,
                                                           const float* __restrict__ dsink_part,
                                                           float* __restrict__ dsinks, int B,
                                                           int H, int sink_chunks,
                                                           const int32_t* __restrict__ cu_q,
                                                           int total_q, int q_bshd) {
  constexpr int DR = 64;                        // head-dim rows per block
  constexpr int NB = HD / DR;                   // blocks per query tile
  constexpr int NV = DR * kDqChunks / 256;      // 16-byte loads per thread
  static_assert(BM / 4 == kDqChunks && DR % kDqChunks == 0 && NV * 256 == DR * kDqChunks &&
                    BM * (DR / 16) == 256,
                "tile layout");
  grid_dep_wait();  // the accumulator and the dsinks partials are the previous kernels' output
  if (dsinks != nullptr && blockIdx.x == 0) dsinks_sum(dsink_part, dsinks, B, H, sink_chunks);
  __shared__ float tile[BM][DR + 1];
  const int q0 = (blockIdx.x / NB) * BM, d0 = (blockIdx.x % NB) * DR;
  for (int bh = blockIdx.y; bh < BH; bh += gridDim.y) {
    int ob = bh / H, or0 = 0, orows = ql, qlen = ql;  // dQ: batch, first row, rows
    if (cu_q != nullptr) {  // sequence b of a variable-length batch
      int qs;
      varlen_seq(cu_q, bh / H, total_q, ql, qs, qlen);
      ob = 0;
      or0 = qs;
      orows = total_q;
    }
    if (q0 >= qlen) continue;  // (block-uniform)
    const float4* tile4 = reinterpret_cast<const float4*>(dqacc + ((size_t)bh * ql_pad + q0) * HD);
    float4 v[NV];
    {
      // chunk-major (halves): chunk c of row d at (d / 128) * 128 * kDqChunks + c * 128 + d % 128
      const float4* src = tile4 + (d0 / 128) * 128 * kDqChunks + d0 % 128;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int f = threadIdx.x + 256 * k;
        v[k] = __ldcs(src + (f / DR) * 128 + f % DR);
      }
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int f = threadIdx.x + 256 * k;
        const int d = f % DR, q = 4 * (f / DR);
        tile[q][d] = v[k].x;
        tile[q + 1][d] = v[k].y;
        tile[q + 2][d] = v[k].z;
        tile[q + 3][d] = v[k].w;
      }
    }
    __syncthreads();
    const int q = threadIdx.x / (DR / 16), c = (threadIdx.x % (DR / 16)) * 16;
    if (q0 + q < qlen) {
      uint32_t w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        w[e] = pack_bf16(tile[q][c + 2 * e] * scale, tile[q][c + 2 * e + 1] * scale);
      uint4* dst = reinterpret_cast<uint4*>(
          dq + bhsd_offset(ob, bh % H, or0 + q0 + q, H, orows, HD, q_bshd != 0) + d0 + c);
      __stcs(dst, make_uint4(w[0], w[1], w[2], w[3]));
      __stcs(dst + 1, make_uint4(w[4], w[5], w[6], w[7]));
    }
    __syncthreads();  // the tile is rewritten for the next head
  }
}

// ------------------------------------------------------------------------ host side
int bwd_q_box_rows(int d) {
  return d == 64 ? BwdTraits<64>::BM : d == 128 ? BwdTraits<128>::BM : BwdTraits<256>::BM;
}
int bwd_kv_box_rows(int) { return kBN; }
int bwd_ql_pad(int ql) { return (ql + 127) / 128 * 128; }

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t bwd_workspace_bytes(int B, int H, int ql, int d) {
  const size_t rows = (size_t)B * H * bwd_ql_pad(ql);
  return align256(rows * 4) * 2 + align256(rows * d * 4) + align256(rows / kPrepRowsMin * 4);
}

void bwd_carve_workspace(void* base, int B, int H, int ql, int d, float** lse2, float** dvec,
                         float** dqacc, float** dsink_part) {
  const size_t rows = (size_t)B * H * bwd_ql_pad(ql);
  uint8_t* p = static_cast<uint8_t*>(base);
  *lse2 = reinterpret_cast<float*>(p);
  *dvec = reinterpret_cast<float*>(p + align256(rows * 4));
  *dqacc = reinterpret_cast<float*>(p + 2 * align256(rows * 4));
  *dsink_part = reinterpret_cast<float*>(p + 2 * align256(rows * 4) + align256(rows * d * 4));
}

template <int HD, int DV>
static cudaError_t launch_bwd_d(const BwdArgs& a, const BwdMaps& m, cudaStream_t s) {
  const int BH = a.B * a.H;
  constexpr int rows_per_block = prep_rows_per_block<DV>();  // divides 128, hence ql_pad
  const int sink_chunks = a.ql_pad / rows_per_block;
  float* dsink_part = a.dsinks != nullptr ? a.dsink_part : nullptr;
  {
    dim3 grid(sink_chunks, BH < 65535 ? BH : 65535);
    profile_mark(kKernBwdPrep, 0, s);
    cudaError_t e = launch_pdl(
        bwd_prep_kernel<HD, DV>, grid, dim3(256), 0, s,
        reinterpret_cast<const __nv_bfloat16*>(a.o), reinterpret_cast<const __nv_bfloat16*>(a.dO),
        a.lse, a.lse2, a.dvec, a.dqacc, a.sinks, dsink_part, BH, a.H, a.ql, a.ql_pad,
        a.deterministic ? 0 : 1, a.cu_q, a.total_q, a.q_bshd);
    profile_mark(kKernBwdPrep, 1, s);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e;
  if constexpr (HD == 256) {
    e = launch_bwd_pair(a, m, s);  // CTA pairs (fa_bwd_pair.cu)
  } else {
    e = (a.q_bshd || a.kv_bshd) ? launch_main_strided(a, m, s)
                                : launch_main_layout<HD, DV, false>(a, m, s);
  }
  if (e != cudaSuccess) return e;
  if (a.deterministic) {
    e = launch_dq_det(a, m.det, s);
    if (e != cudaSuccess) return e;
    if (a.dsinks != nullptr) {  // the dsinks sum alone
      profile_mark(kKernBwdDq, 0, s);
      bwd_dq_kernel<HD, false><<<dim3(1, a.H < 65535 ? a.H : 65535), 256, 0, s>>>(
          a.dqacc, reinterpret_cast<__nv_bfloat16*>(a.dq), BH, a.ql, a.ql_pad, a.scale,
          dsink_part, a.dsinks, a.B, a.H, sink_chunks, 0, a.cu_q, a.total_q, a.q_bshd);
      profile_mark(kKernBwdDq, 1, s);
    }
    return cudaGetLastError();
  }
  if constexpr (BwdTraits<HD>::DQT) {  // transposed accumulator tiles
    constexpr int BM = BwdTraits<HD>::BM;
    dim3 grid((unsigned)((a.ql + BM - 1) / BM * (HD / 64)), BH < 65535 ? BH : 65535);
    profile_mark(kKernBwdDq, 0, s);
    e = launch_pdl(bwd_dq_tiles_kernel<HD, BM>, grid, dim3(256), 0, s, a.dqacc,
                   reinterpret_cast<__nv_bfloat16*>(a.dq), BH, a.ql, a.ql_pad, a.scale,
                   dsink_part, a.dsinks, a.B, a.H, sink_chunks, a.cu_q, a.total_q, a.q_bshd);
    profile_mark(kKernBwdDq, 1, s);
    if (e != cudaSuccess) return e;
  } else {
    const long long groups = (long long)a.ql * (HD / 8);  // 8-value groups per head
    dim3 grid((unsigned)((groups + 255) / 256), BH < 65535 ? BH : 65535);
    profile_mark(kKernBwdDq, 0, s);
    e = launch_pdl(bwd_dq_kernel<HD, BwdTraits<HD>::DQ_BULK>, grid, dim3(256), 0, s, a.dqacc,
                   reinterpret_cast<__nv_bfloat16*>(a.dq), BH, a.ql, a.ql_pad, a.scale,
                   dsink_part, a.dsinks, a.B, a.H, sink_chunks, 1, a.cu_q, a.total_q,
                   a.q_bshd);
    profile_mark(kKernBwdDq, 1, s);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------------ fixed scratch
// Backward scratch for callers that must not allocate device memory (fa_train_bwd_noalloc).
// A file-scope device array: CUDA creates it when it loads this file's device code on a GPU
// (at context creation with eager module loading, else at the first use of one of its
// kernels or symbols), and it stays until the process exits. Host code cannot use the array's
// name as a device address, so the address is looked up with cudaGetSymbolAddress, on the
// current device, at every call (nothing cached: nothing goes stale across a device reset).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

cudaError_t noalloc_scratch(void** ptr) { return cudaGetSymbolAddress(ptr, g_noalloc_scratch); }

cudaError_t noalloc_status(int clear, int* value) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_noalloc_scratch, sizeof(int));
  if (e != cudaSuccess || !clear || *value == 0) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_noalloc_scratch, &zero, sizeof(int));
}

cudaError_t launch_bwd(const BwdArgs& a, const BwdMaps& m, cudaStream_t stream) {
  if (a.d == 64 && a.dval == 64) return launch_bwd_d<64, 64>(a, m, stream);
  if (a.d == 128 && a.dval == 128) return launch_bwd_d<128, 128>(a, m, stream);
  if (a.d == 256 && a.dval == 256) return launch_bwd_d<256, 256>(a, m, stream);
  if (a.d == 128 && a.dval == 64) return launch_bwd_d<128, 64>(a, m, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
