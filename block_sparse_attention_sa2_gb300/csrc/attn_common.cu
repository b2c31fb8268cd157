// Host-side TMA descriptors and the element-wise kernels around the attention kernels:
// fp32 -> bf16 staging of SA2_FP32 inputs, the backward's preprocessing
// (D = rowsum(dO * O), zeroed fp32 dQ accumulator) and the dQ conversion.
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
// reported as a range error.
template <typename T>
__global__ void to_f16_kernel(const T* __restrict__ src, ShapeArgs s, __half* __restrict__ dst, unsigned* status) {
  const int64_t n4 = (int64_t)s.B * s.H * s.N * s.d / 4;
  bool bad = false;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = i * 4;
    const int c = (int)(e % s.d);
    const int64_t t = e / s.d;
    const int n = (int)(t % s.N);
    const int64_t bh = t / s.N;
    const int h = (int)(bh % s.H), b = (int)(bh / s.H);
    float4 v = ld4<T>(src + b * s.sb + h * s.sh + (int64_t)n * s.sn + c);
    const float lim = 65504.f;
    bad |= !(fabsf(v.x) <= lim && fabsf(v.y) <= lim && fabsf(v.z) <= lim && fabsf(v.w) <= lim);
    v.x = fminf(fmaxf(v.x, -lim), lim);
    v.y = fminf(fmaxf(v.y, -lim), lim);
    v.z = fminf(fmaxf(v.z, -lim), lim);
    v.w = fminf(fmaxf(v.w, -lim), lim);
    uint2 w;
    w.x = pack_f16x2(v.x, v.y);
    w.y = pack_f16x2(v.z, v.w);
    *reinterpret_cast<uint2*>(dst + e) = w;
  }
  if (bad) report_error(status, kDevErrRange);
}

cudaError_t launch_to_f16(const void* src, const ShapeArgs& s, __half* dst, unsigned* status, cudaStream_t st) {
  const int64_t n4 = (int64_t)s.B * s.H * s.N * s.d / 4;
  const int blocks = (int)std::min<int64_t>((n4 + 255) / 256, 152 * 16);
  prof_start(st, kToF16);
  if (s.dtype == 0)
    to_f16_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(src), s, dst, status);
  else
    to_f16_kernel<float><<<blocks, 256, 0, st>>>(static_cast<const float*>(src), s, dst, status);
  prof_stop(st, kToF16);
  return cudaGetLastError();
}

template <typename T>
__device__ __forceinline__ float ld_elem(const T* p);
template <>
__device__ __forceinline__ float ld_elem<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_elem<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }
template <>
__device__ __forceinline__ float ld_elem<__half>(const __half* p) { return __half2float(*p); }

// One warp per token row: D = sum_c dO[c] * (O[c] + O_lo[c]) (fp32).  O has the call's
// dtype and strides; dO is the contiguous fp16 copy the MMAs read, so that D matches the dO
// of dP = dO V^T.
template <typename TO>
__global__ void bwd_preprocess_kernel(const TO* __restrict__ o, const __nv_bfloat16* __restrict__ o_lo,
                                      const __half* __restrict__ dO, ShapeArgs s, float* __restrict__ Dvec) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)s.B * s.H * s.N;
  for (int64_t row = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / 32; row < rows;
       row += (int64_t)gridDim.x * blockDim.x / 32) {
    const int n = (int)(row % s.N);
    const int64_t bh = row / s.N;
    const int h = (int)(bh % s.H), b = (int)(bh / s.H);
    const int64_t off = b * s.sb + h * s.sh + (int64_t)n * s.sn;
    const __half* drow = dO + row * s.d;
    float acc = 0.f;
    for (int c = lane; c < s.d; c += 32) {
      const float ov = ld_elem<TO>(o + off + c) + (o_lo ? __bfloat162float(o_lo[off + c]) : 0.f);
      acc += ov * __half2float(drow[c]);
    }
#pragma unroll
    for (int w = 16; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
    if (lane == 0) Dvec[row] = acc;
  }
}

cudaError_t launch_bwd_preprocess(const ShapeArgs& s, const void* o, const void* o_lo, const __half* dO16,
                                  float* Dvec, cudaStream_t st) {
  const __nv_bfloat16* lo = s.dtype == 0 ? static_cast<const __nv_bfloat16*>(o_lo) : nullptr;
  const int64_t rows = (int64_t)s.B * s.H * s.N;
  const int blocks = (int)std::min<int64_t>((rows * 32 + 255) / 256, 152 * 16);
  prof_start(st, kBwdPre);
  if (s.dtype == 0)
    bwd_preprocess_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(o), lo, dO16,
                                                                 s, Dvec);
  else
    bwd_preprocess_kernel<float><<<blocks, 256, 0, st>>>(static_cast<const float*>(o), nullptr, dO16, s, Dvec);
  prof_stop(st, kBwdPre);
  return cudaGetLastError();
}

}  // namespace sa2
