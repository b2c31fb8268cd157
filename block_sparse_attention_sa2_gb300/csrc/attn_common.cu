// Host-side TMA descriptors and the element-wise kernels around the attention kernels:
// fp16 copies of the token tensors, and the backward's preprocessing (fp16 dO, D =
// rowsum(dO * O) and log2(e) * LSE per row).
#include <algorithm>
#include <cstring>
#include <cudaTypedefs.h>

#include "sa2_internal.h"

namespace sa2 {

static PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// bf16 [B, H, N, d] viewed as a 4-D tensor (d, N, H, B); boxes of 64 channels x box_rows
// tokens with the 128-byte swizzle the tcgen05 descriptors expect.  Tokens past N read
// as zero.
bool make_token_map(CUtensorMap* map, const void* base, const ShapeArgs& s, int64_t sb, int64_t sh, int64_t sn,
                    int box_rows, bool f16) {
  auto enc = encode_tiled();
  if (!enc) return false;
  std::memset(map, 0, sizeof(*map));
  cuuint64_t dims[4] = {(cuuint64_t)s.d, (cuuint64_t)s.N, (cuuint64_t)s.H, (cuuint64_t)s.B};
  cuuint64_t strides[3] = {(cuuint64_t)sn * 2, (cuuint64_t)sh * 2, (cuuint64_t)sb * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                   const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename T>
__device__ __forceinline__ float4 ld4(const T* p);
template <>
__device__ __forceinline__ float4 ld4<float>(const float* p) { return *reinterpret_cast<const float4*>(p); }
template <>
__device__ __forceinline__ float4 ld4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                     __uint_as_float(w.y & 0xFFFF0000u));
}

// Token tensor (caller dtype and strides) -> contiguous fp16 [B, H, N, d].  bf16 values
// within the fp16 range convert exactly; a value of magnitude above 65504 is saturated and
// reported as a range error.  Each thread converts 8 consecutive channels of one token; for
// contiguous inputs the source offset is the destination offset.
template <typename T>
__device__ __forceinline__ void ld8(const T* p, float* v);
template <>
__device__ __forceinline__ void ld8<float>(const float* p, float* v) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <>
__device__ __forceinline__ void ld8<__nv_bfloat16>(const __nv_bfloat16* p, float* v) {
  const uint4 w = *reinterpret_cast<const uint4*>(p);
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(u[i] << 16);
    v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 to_f16x8(float* v, bool& bad) {
  const float lim = 65504.f;
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    bad |= !(fabsf(v[i]) <= lim);
    v[i] = fminf(fmaxf(v[i], -lim), lim);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = pack_f16x2(v[2 * i], v[2 * i + 1]);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// The low-order part of an fp32 -> fp16 rounding: fp16(v - hi) with hi the (saturated)
// fp16 value just stored, so that hi + lo carries about 22 significant bits.
__device__ __forceinline__ uint4 lo_f16x8(const float* v, uint4 hi) {
  const uint32_t h[4] = {hi.x, hi.y, hi.z, hi.w};
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 hh = *reinterpret_cast<const __half2*>(&h[i]);
    const float2 f = __half22float2(hh);
    // finite even for a saturated input (whose error is reported)
    w[i] = pack_f16x2(fminf(fmaxf(v[2 * i] - f.x, -65504.f), 65504.f),
                      fminf(fmaxf(v[2 * i + 1] - f.y, -65504.f), 65504.f));
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// fp16 copy of a token tensor (and, when dst_lo is not null, of its rounding residual)
template <typename T, bool CONTIG>
__global__ void __launch_bounds__(256) to_f16_kernel(const T* __restrict__ src, ShapeArgs s, __half* __restrict__ dst,
                                                     __half* __restrict__ dst_lo, unsigned* status) {
  const int64_t items = (int64_t)s.B * s.H * s.N * s.d / 8;
  const int per_row = s.d / 8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  bool bad = false;
  int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (CONTIG) {
    // four 16-byte loads in flight per thread before the first store
    for (; i0 + 3 * stride < items; i0 += 4 * stride) {
      float v[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u) ld8<T>(src + (i0 + u * stride) * 8, v[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float raw[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) raw[e] = v[u][e];
        const uint4 hi = to_f16x8(v[u], bad);
        *reinterpret_cast<uint4*>(dst + (i0 + u * stride) * 8) = hi;
        if (dst_lo) *reinterpret_cast<uint4*>(dst_lo + (i0 + u * stride) * 8) = lo_f16x8(raw, hi);
      }
    }
  }
  for (int64_t i = i0; i < items; i += stride) {
    const int64_t e = i * 8;
    int64_t off = e;
    if (!CONTIG) {
      const int64_t row = i / per_row;
      const int c = (int)(i - row * per_row) * 8;
      const int64_t bh = row / s.N;
      const int n = (int)(row - bh * s.N);
      off = (bh / s.H) * s.sb + (bh % s.H) * s.sh + (int64_t)n * s.sn + c;
    }
    float v[8], raw[8];
    ld8<T>(src + off, v);
#pragma unroll
    for (int u = 0; u < 8; ++u) raw[u] = v[u];
    const uint4 hi = to_f16x8(v, bad);
    *reinterpret_cast<uint4*>(dst + e) = hi;
    if (dst_lo) *reinterpret_cast<uint4*>(dst_lo + e) = lo_f16x8(raw, hi);
  }
  if (bad) report_error(status, kDevErrRange);
}

static bool contiguous(const ShapeArgs& s) {
  return s.sn == s.d && s.sh == (int64_t)s.N * s.d && s.sb == (int64_t)s.H * s.N * s.d;
}

static int grid_for(int64_t items) { return (int)std::min<int64_t>((items + 255) / 256, 152 * 8); }

namespace {

// The launch order of the query blocks.  Heads stay in order, each head's blocks by descending
// list length, so the items in flight at any time come from one or two heads and share their
// K / V blocks in L2.  A head's long lists would end after everything else when that head
// comes late, so a list of head h longer than the work the heads from h on leave per slot,
// (heads - h) * W_h / slots blocks with W_h the head's total, is taken out of its head and
// put into one list in front, all heads' long lists together by descending length (the
// longest-processing-time-first rule).  Two passes of one CTA per head: the first sets the
// head's threshold and counts its long lists into a global histogram, the second places the
// long lists from the global histogram and the rest of the head behind the long list and the
// earlier heads.  Histograms are counting sorts over Tk - length in shared memory.
constexpr int kOrderThreads = 1024;

struct OrderScratch {
  int* hist;    // [Tk + 1] long lists of all heads by Tk - length (zeroed before the first pass)
  int* cur;     // [Tk + 1] cursors into hist's bins (zeroed before the first pass)
  int* thr;     // [heads] a list is long when its length is above this
  int* nshort;  // [heads] the lists of the head that are not long
};

__device__ __forceinline__ int clamped_len(const int32_t* row_cnt, int64_t x, int Tk) {
  const int n = row_cnt[x];
  return n < 0 ? 0 : (n > Tk ? Tk : n);
}

__global__ void __launch_bounds__(kOrderThreads) item_split_kernel(const int32_t* __restrict__ row_cnt, int Tq,
                                                                   int Tk, int slots, OrderScratch o) {
  __shared__ unsigned long long work;
  __shared__ int nlong;
  const int tid = threadIdx.x, h = blockIdx.x;
  const int64_t x0 = (int64_t)h * Tq;
  if (tid == 0) {
    work = 0;
    nlong = 0;
  }
  __syncthreads();
  unsigned long long w = 0;
  for (int i = tid; i < Tq; i += kOrderThreads) w += (unsigned long long)clamped_len(row_cnt, x0 + i, Tk);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) w += __shfl_xor_sync(0xffffffffu, w, off);
  if ((tid & 31) == 0) atomicAdd(&work, w);
  __syncthreads();
  const unsigned long long later = (unsigned long long)(gridDim.x - h) * work;
  const unsigned long long t = (later + (unsigned long long)slots - 1) / (unsigned long long)slots;
  const int thr = t > (unsigned long long)Tk ? Tk : (int)t;
  int mine = 0;
  for (int i = tid; i < Tq; i += kOrderThreads) {
    const int n = clamped_len(row_cnt, x0 + i, Tk);
    if (n > thr) {
      atomicAdd(&o.hist[Tk - n], 1);
      ++mine;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, off);
  if ((tid & 31) == 0 && mine) atomicAdd(&nlong, mine);
  __syncthreads();
  if (tid == 0) {
    o.thr[h] = thr;
    o.nshort[h] = Tq - nlong;
  }
}

// In-place exclusive scan of bins[0, nb) by the whole block; returns the total to every thread.
__device__ int scan_bins(int* bins, int nb, int* warp_sum) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // each thread sums a contiguous run of bins, the runs are scanned across the block, then
  // each run is rewritten as offsets
  const int per = (nb + kOrderThreads - 1) / kOrderThreads;
  const int b0 = min(nb, tid * per), b1 = min(nb, b0 + per);
  int run = 0;
  for (int i = b0; i < b1; ++i) run += bins[i];
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    warp_sum[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  int base = incl - run + (warp > 0 ? warp_sum[warp - 1] : 0);
  for (int i = b0; i < b1; ++i) {
    const int c = bins[i];
    bins[i] = base;
    base += c;
  }
  const int total = warp_sum[kOrderThreads / 32 - 1];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kOrderThreads) item_order_kernel(const int32_t* __restrict__ row_cnt, int Tq,
                                                                   int Tk, int32_t* __restrict__ order,
                                                                   OrderScratch o, int* __restrict__ work_ctr) {
  extern __shared__ int bins[];  // Tk + 1
  __shared__ int warp_sum[kOrderThreads / 32];
  __shared__ int earlier;
  const int tid = threadIdx.x, h = blockIdx.x;
  const int64_t x0 = (int64_t)h * Tq;
  const int nb = Tk + 1;
  const int thr = o.thr[h];
  // the long lists of every head: global offsets from the global histogram
  for (int i = tid; i < nb; i += kOrderThreads) bins[i] = o.hist[i];
  if (tid == 0) earlier = 0;
  __syncthreads();
  const int nlong_all = scan_bins(bins, nb, warp_sum);
  for (int i = tid; i < Tq; i += kOrderThreads) {
    const int n = clamped_len(row_cnt, x0 + i, Tk);
    if (n > thr) order[bins[Tk - n] + atomicAdd(&o.cur[Tk - n], 1)] = (int32_t)(x0 + i);
  }
  // the rest of this head, behind the long lists and the rest of the earlier heads
  int e = 0;
  for (int g = tid; g < h; g += kOrderThreads) e += o.nshort[g];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) e += __shfl_xor_sync(0xffffffffu, e, off);
  __syncthreads();
  if ((tid & 31) == 0 && e) atomicAdd(&earlier, e);
  for (int i = tid; i < nb; i += kOrderThreads) bins[i] = 0;
  __syncthreads();
  for (int i = tid; i < Tq; i += kOrderThreads) {
    const int n = clamped_len(row_cnt, x0 + i, Tk);
    if (n <= thr) atomicAdd(&bins[Tk - n], 1);
  }
  __syncthreads();
  scan_bins(bins, nb, warp_sum);
  const int base = nlong_all + earlier;
  for (int i = tid; i < Tq; i += kOrderThreads) {
    const int n = clamped_len(row_cnt, x0 + i, Tk);
    if (n <= thr) order[base + atomicAdd(&bins[Tk - n], 1)] = (int32_t)(x0 + i);
  }
  if (work_ctr && h == 0 && tid == 0) *work_ctr = 0;
}

}  // namespace

size_t item_order_ints(int heads, int Tq, int Tk) {
  return (size_t)heads * Tq + 2 * ((size_t)Tk + 1) + 2 * (size_t)heads;
}

cudaError_t launch_item_order(const int32_t* row_cnt, int heads, int Tq, int Tk, int slots, int32_t* order,
                              int* work_ctr, cudaStream_t st) {
  const size_t smem = (size_t)(Tk + 1) * sizeof(int);
  if (smem > 48 * 1024) return cudaErrorInvalidValue;  // Tk <= 12287
  if (heads <= 0 || Tq <= 0) return cudaSuccess;
  OrderScratch o;
  o.hist = order + (size_t)heads * Tq;
  o.cur = o.hist + (Tk + 1);
  o.thr = o.cur + (Tk + 1);
  o.nshort = o.thr + heads;
  prof_start(st, kItemOrder);
  cudaError_t e = cudaMemsetAsync(o.hist, 0, sizeof(int) * 2 * ((size_t)Tk + 1), st);
  if (e == cudaSuccess) {
    item_split_kernel<<<heads, kOrderThreads, 0, st>>>(row_cnt, Tq, Tk, slots < 1 ? 1 : slots, o);
    item_order_kernel<<<heads, kOrderThreads, smem, st>>>(row_cnt, Tq, Tk, order, o, work_ctr);
    e = cudaGetLastError();
  }
  prof_stop(st, kItemOrder);
  return e;
}

cudaError_t launch_to_f16(const void* src, const ShapeArgs& s, __half* dst, unsigned* status, cudaStream_t st,
                          __half* dst_lo) {
  const int blocks = grid_for((int64_t)s.B * s.H * s.N * s.d / 8);
  const bool c = contiguous(s);
  prof_start(st, kToF16);
  if (s.dtype == 0) {
    auto p = static_cast<const __nv_bfloat16*>(src);
    if (c)
      to_f16_kernel<__nv_bfloat16, true><<<blocks, 256, 0, st>>>(p, s, dst, dst_lo, status);
    else
      to_f16_kernel<__nv_bfloat16, false><<<blocks, 256, 0, st>>>(p, s, dst, dst_lo, status);
  } else {
    auto p = static_cast<const float*>(src);
    if (c)
      to_f16_kernel<float, true><<<blocks, 256, 0, st>>>(p, s, dst, dst_lo, status);
    else
      to_f16_kernel<float, false><<<blocks, 256, 0, st>>>(p, s, dst, dst_lo, status);
  }
  prof_stop(st, kToF16);
  return cudaGetLastError();
}

// Backward preparation of dO, one pass: the contiguous fp16 copy of dO the MMAs read and
// D = sum_c dO16[c] * (O[c] + O_lo[c]) in fp32, so that D matches the dO of dP = dO V^T.
// Sixteen threads per token (8 channels each, d = 128) or eight (d = 64).
template <typename T>
__global__ void __launch_bounds__(256) do_prep_kernel(const T* __restrict__ dO, const T* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ o_lo,
                                                      const float* __restrict__ lse, ShapeArgs s,
                                                      __half* __restrict__ dO16, float* __restrict__ stats,
                                                      unsigned* status) {
  // grid: x = b*H + h, y over the tokens of one head (per_row threads of 8 channels each);
  // a warp covers whole tokens (per_row = 16 or 8 divides 32), so the shuffles below stay
  // inside a token and every lane takes part in them
  const int shift = s.d == 128 ? 4 : 3;  // log2(per_row)
  const int per_row = 1 << shift;
  const int bh = blockIdx.x;
  const int b = bh / s.H, h = bh - b * s.H;
  const int Tsub = s.Tq * (s.bq / 64);
  const int idx = blockIdx.y * blockDim.x + threadIdx.x;
  const int n = idx >> shift;
  const int c = (idx & (per_row - 1)) * 8;
  const bool live = n < s.N;
  bool bad = false;
  float acc = 0.f;
  if (live) {
    const int64_t off = (int64_t)b * s.sb + (int64_t)h * s.sh + (int64_t)n * s.sn + c;
    float g[8], ov[8];
    ld8<T>(dO + off, g);
    ld8<T>(o + off, ov);
    if (o_lo) {
      float lo[8];
      ld8<__nv_bfloat16>(o_lo + off, lo);
#pragma unroll
      for (int k = 0; k < 8; ++k) ov[k] += lo[k];
    }
    const uint4 hv = to_f16x8(g, bad);
    *reinterpret_cast<uint4*>(dO16 + ((int64_t)bh * s.N + n) * s.d + c) = hv;
    const __half* hh = reinterpret_cast<const __half*>(&hv);
#pragma unroll
    for (int k = 0; k < 8; ++k) acc += __half2float(hh[k]) * ov[k];
  }
  for (int w = per_row / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
  if (live && c == 0) {
    float* rec = stats + ((int64_t)bh * Tsub + (n >> 6)) * 128 + (n & 63);
    rec[0] = lse[(int64_t)bh * s.N + n] * 1.4426950408889634f;
    rec[64] = acc;
  }
  // rows of the last sub-tiles past N: +inf makes their P exactly 0
  if (blockIdx.y == 0) {
    const int pad = Tsub * 64 - s.N;
    for (int i = threadIdx.x; i < pad; i += blockDim.x) {
      const int np = s.N + i;
      float* rec = stats + ((int64_t)bh * Tsub + (np >> 6)) * 128 + (np & 63);
      rec[0] = __int_as_float(0x7f800000);
      rec[64] = 0.f;
    }
  }
  if (bad) report_error(status, kDevErrRange);
}

cudaError_t launch_do_prep(const ShapeArgs& s, const void* dO, const void* o, const void* o_lo, const float* lse,
                           __half* dO16, float* stats, unsigned* status, cudaStream_t st) {
  const int64_t per_head = (int64_t)s.N * (s.d / 8);
  // y <= 491520 tokens x 16 / 256 = 30720 blocks, within the 65535 limit of gridDim.y
  const dim3 grid((unsigned)(s.B * s.H), (unsigned)((per_head + 255) / 256));
  prof_start(st, kBwdPre);
  if (s.dtype == 0)
    do_prep_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(dO),
                                                        static_cast<const __nv_bfloat16*>(o),
                                                        static_cast<const __nv_bfloat16*>(o_lo), lse, s, dO16,
                                                        stats, status);
  else
    do_prep_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(dO), static_cast<const float*>(o),
                                                nullptr, lse, s, dO16, stats, status);
  prof_stop(st, kBwdPre);
  return cudaGetLastError();
}

// ------------------------------------------------------------- distillation loss (toy)
//
// gist.science explainer of SpargeAttention2, section 2.B: the fine-tuning loss is the
// squared L2 distance between the sparse and the full-attention velocity; on one attention
// block its output stands in for the velocity.  loss = sum (O_s - O_t)^2, dO = 2 (O_s - O_t).
// The difference is formed as (hi_s - hi_t) + (lo_s - lo_t): both partial differences are
// exact in fp32 for bf16 parts, so the only rounding is their sum.  Each CTA leaves its fp64
// partial sum; one CTA adds the partials in index order, so the loss is deterministic.

template <typename T>
__device__ __forceinline__ void st8(T* p, const float* v);
template <>
__device__ __forceinline__ void st8<float>(float* p, const float* v) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}
template <>
__device__ __forceinline__ void st8<__nv_bfloat16>(__nv_bfloat16* p, const float* v) {
  *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                            pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}

template <typename T>
__global__ void __launch_bounds__(256) vd_loss_kernel(const T* __restrict__ os, const __nv_bfloat16* __restrict__ os_lo,
                                                      const T* __restrict__ ot, const __nv_bfloat16* __restrict__ ot_lo,
                                                      ShapeArgs s, T* __restrict__ d_o, double* __restrict__ partial) {
  __shared__ double red[8];
  const int per_row = s.d / 8;
  const int64_t items = (int64_t)s.B * s.H * s.N * per_row;
  double acc = 0.0;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < items; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / per_row;
    const int c = (int)(i - row * per_row) * 8;
    const int64_t bh = row / s.N;
    const int n = (int)(row - bh * s.N);
    const int64_t off = (bh / s.H) * s.sb + (bh % s.H) * s.sh + (int64_t)n * s.sn + c;
    float a[8], b[8], g[8];
    ld8<T>(os + off, a);
    ld8<T>(ot + off, b);
#pragma unroll
    for (int k = 0; k < 8; ++k) g[k] = a[k] - b[k];
    if (os_lo && ot_lo) {
      ld8<__nv_bfloat16>(os_lo + off, a);
      ld8<__nv_bfloat16>(ot_lo + off, b);
#pragma unroll
      for (int k = 0; k < 8; ++k) g[k] += a[k] - b[k];
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      acc += (double)g[k] * (double)g[k];
      g[k] *= 2.f;
    }
    st8<T>(d_o + off, g);
  }
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < 8; ++w) t += red[w];
    partial[blockIdx.x] = t;
  }
}

__global__ void __launch_bounds__(256) vd_loss_sum_kernel(const double* __restrict__ partial, int n,
                                                          double* __restrict__ loss) {
  __shared__ double red[256];
  double t = 0.0;
  for (int i = threadIdx.x; i < n; i += 256) t += partial[i];
  red[threadIdx.x] = t;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = red[0];
}

size_t vd_loss_workspace_bytes() { return sizeof(double) * 152 * 8; }

cudaError_t launch_vd_loss(const ShapeArgs& s, const void* os, const void* os_lo, const void* ot, const void* ot_lo,
                           void* d_o, double* loss, double* partial, cudaStream_t st) {
  const int blocks = grid_for((int64_t)s.B * s.H * s.N * (s.d / 8));  // <= 152 * 8 partials
  prof_start(st, kVdLoss);
  if (s.dtype == 0)
    vd_loss_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(os), static_cast<const __nv_bfloat16*>(os_lo),
        static_cast<const __nv_bfloat16*>(ot), static_cast<const __nv_bfloat16*>(ot_lo), s,
        static_cast<__nv_bfloat16*>(d_o), partial);
  else
    vd_loss_kernel<float><<<blocks, 256, 0, st>>>(static_cast<const float*>(os), nullptr,
                                                  static_cast<const float*>(ot), nullptr, s,
                                                  static_cast<float*>(d_o), partial);
  vd_loss_sum_kernel<<<1, 256, 0, st>>>(partial, blocks, loss);
  prof_stop(st, kVdLoss);
  return cudaGetLastError();
}

}  // namespace sa2
