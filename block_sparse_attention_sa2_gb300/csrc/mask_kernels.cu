// Hybrid Top-k + Top-p block mask on sm_103a.
//
// gist.science explainer of SpargeAttention2 (arXiv 2602.13515), section 2.A: the rows of
// the block-pooled attention map P-bar are masked with the union of their Top-k% and
// Top-p% sets; section 1 defines Top-k (the k largest entries) and Top-p (the smallest set
// whose cumulative probability reaches p).
//
// Three kernels:
//   pool_kernel          mean of Q and K over each block (fp32), written transposed
//                        ([B*H, d, T]) for the score kernel.  HBM-bound streaming read.
//   score_select_kernel  one CTA per (b*h, RQ query blocks): fp32 pooled scores against all
//                        key blocks, row softmax, and the hybrid selection by a bisection on
//                        the fp32 bit patterns of P-bar; emits the row lists and the u8 mask.
//   csc_kernel           transposes the u8 mask into the per-key-block lists (ascending).
#include "sa2_internal.h"

namespace sa2 {

// ------------------------------------------------------------------------------ pooling

template <typename T>
__device__ __forceinline__ void load_vec(const T* p, float* out);

template <>
__device__ __forceinline__ void load_vec<__nv_bfloat16>(const __nv_bfloat16* p, float* out) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    out[2 * i] = __uint_as_float(w[i] << 16);
    out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <>
__device__ __forceinline__ void load_vec<float>(const float* p, float* out) {
  const float4 v = __ldg(reinterpret_cast<const float4*>(p));
  out[0] = v.x;
  out[1] = v.y;
  out[2] = v.z;
  out[3] = v.w;
}

// One CTA (256 threads) pools one block of one head.  blockIdx.x enumerates, per head,
// the Tq query blocks then the Tk key blocks; blockIdx.y is b*H + h.
template <typename T>
__global__ void __launch_bounds__(256) pool_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                   ShapeArgs s, int tq_pad, int tk_pad, float* __restrict__ qbarT,
                                                   float* __restrict__ kbarT) {
  constexpr int VEC = 16 / sizeof(T);
  __shared__ float part[256 * VEC];
  const int bh = blockIdx.y;
  const int b = bh / s.H, h = bh % s.H;
  int blk = blockIdx.x;
  const bool is_q = blk < s.Tq;
  if (!is_q) blk -= s.Tq;
  const int bsz = is_q ? s.bq : s.bk;
  const T* base = (is_q ? q : k) + (int64_t)b * s.sb + (int64_t)h * s.sh;
  const int t0 = blk * bsz;
  const int nrows = min(bsz, s.N - t0);
  const int vpr = s.d / VEC;  // vectors per token row
  const int rpp = 256 / vpr;  // rows per pass
  const int tid = threadIdx.x;
  const int vc = tid % vpr, r0 = tid / vpr;
  float acc[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) acc[i] = 0.f;
#pragma unroll 4
  for (int r = r0; r < nrows; r += rpp) {
    float v[VEC];
    load_vec<T>(base + (int64_t)(t0 + r) * s.sn + vc * VEC, v);
#pragma unroll
    for (int i = 0; i < VEC; ++i) acc[i] += v[i];
  }
  // part[r0][vc*VEC + i]
#pragma unroll
  for (int i = 0; i < VEC; ++i) part[r0 * s.d + vc * VEC + i] = acc[i];
  __syncthreads();
  if (tid < s.d) {
    float sum = 0.f;
    for (int r = 0; r < rpp; ++r) sum += part[r * s.d + tid];
    const float mean = sum / static_cast<float>(nrows);
    const int pitch = is_q ? tq_pad : tk_pad;
    float* out = (is_q ? qbarT : kbarT) + ((int64_t)bh * s.d + tid) * pitch + blk;
    *out = mean;
  }
}

// ------------------------------------------------------------------ scores + selection

constexpr int kScoreThreads = 256;
constexpr int kKeyChunk = 128;

// Fixed-point mass of a non-negative fp32 probability given by its bit pattern:
// floor(P * 2^60), from the exponent and mantissa with integer shifts (P <= 1, so the
// result fits in 61 bits).  Exact for P >= 2^-37; smaller values lose less than 2^-60.
__device__ __forceinline__ unsigned long long mass_fix(uint32_t key) {
  const int e = (int)(key >> 23);  // biased exponent; sign bit is 0
  if (e == 0) return 0ull;         // zero or subnormal: below 2^-126
  const unsigned long long m = (unsigned long long)((key & 0x7FFFFFu) | 0x800000u);
  const int sh = e - 90;           // P * 2^60 = m * 2^(e - 127 - 23 + 60)
  return sh >= 0 ? (m << sh) : (sh > -64 ? (m >> (-sh)) : 0ull);
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct Predicate {
  uint32_t cnt;
  unsigned long long mass;
};

// Count and fixed-point mass of the row's entries whose key is >= t (ge) or > t (gt).
__device__ __forceinline__ Predicate count_mass(const uint32_t* keys, int Tk, uint32_t t, bool strictly) {
  const int lane = threadIdx.x & 31;
  uint32_t c = 0;
  unsigned long long m = 0;
  for (int j = lane; j < Tk; j += 32) {
    const uint32_t key = keys[j];
    const bool in = strictly ? key > t : key >= t;
    if (in) {
      ++c;
      m += mass_fix(key);
    }
  }
  Predicate p;
  p.cnt = __reduce_add_sync(0xffffffffu, c);
  p.mass = warp_sum_u64(m);
  return p;
}

// Keys per lane held in registers by the selection when Tk <= 32 * kRegKeys.
constexpr int kRegKeys = 40;

// The hybrid selection of one row (one warp), with the row's keys and their fixed-point
// masses in registers: the same bisection as the shared-memory path below, without its
// loads.  Sets keep_all when the row's mass never reaches p; otherwise the threshold t and
// the number of entries equal to t to take.
__device__ __forceinline__ void select_in_registers(const uint32_t* keys, int Tk, const SelectArgs& sel,
                                                    bool& keep_all, uint32_t& t, int& take) {
  const int lane = threadIdx.x & 31;
  uint32_t k[kRegKeys];
  unsigned long long mf[kRegKeys];
  unsigned long long msum = 0;
#pragma unroll
  for (int i = 0; i < kRegKeys; ++i) {
    const int j = lane + 32 * i;
    k[i] = j < Tk ? keys[j] : 0u;
    mf[i] = mass_fix(k[i]);
    msum += mf[i];
  }
  const bool use_mass = sel.p_mode == 0;
  if (use_mass && warp_sum_u64(msum) < sel.p_fix) {
    keep_all = true;
    return;
  }
  // largest t with count(>= t) >= K and mass(>= t) >= p; the lanes' padding keys are 0 and
  // every tested t is >= 1, so padding is never counted
  uint32_t lo = 0, hi = 0x3F800001u;
  while (hi - lo > 1) {
    const uint32_t mid = lo + (hi - lo) / 2;
    uint32_t c = 0;
#pragma unroll
    for (int i = 0; i < kRegKeys; ++i) c += k[i] >= mid ? 1u : 0u;
    bool ok = __reduce_add_sync(0xffffffffu, c) >= (uint32_t)sel.K;  // same in every lane
    if (ok && use_mass) {
      unsigned long long m = 0;
#pragma unroll
      for (int i = 0; i < kRegKeys; ++i) m += k[i] >= mid ? mf[i] : 0ull;
      ok = warp_sum_u64(m) >= sel.p_fix;
    }
    if (ok)
      lo = mid;
    else
      hi = mid;
  }
  t = lo;
  uint32_t c = 0;
  unsigned long long m = 0;
#pragma unroll
  for (int i = 0; i < kRegKeys; ++i) {
    c += k[i] > t ? 1u : 0u;
    m += k[i] > t ? mf[i] : 0ull;
  }
  c = __reduce_add_sync(0xffffffffu, c);
  m = warp_sum_u64(m);
  const int r_k = sel.K - (int)c;
  int r_m = 0;
  if (use_mass && m < sel.p_fix) {
    const unsigned long long vfix = mass_fix(t);
    r_m = vfix ? (int)((sel.p_fix - m + vfix - 1) / vfix) : 0;
  }
  take = max(max(r_k, r_m), 0);
}

__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// RQ query blocks per CTA; NBUF k-bar chunk buffers (2: the next chunk streams in while the
// current one is used).
template <int RQ, int NBUF>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_select_kernel(const float* __restrict__ qbarT, const float* __restrict__ kbarT, ShapeArgs s, int tq_pad,
                        int tk_pad, SelectArgs sel, MaskOut out) {
  extern __shared__ __align__(16) float smem[];
  const int Tk = s.Tk;
  const int Tk_pad = tk_pad;  // multiple of kKeyChunk; pooled keys past Tk are never read back
  float* qs = smem;                    // [d][RQ]
  float* ks = qs + s.d * RQ;           // NBUF x [d][kKeyChunk]
  float* S = ks + NBUF * s.d * kKeyChunk;  // [RQ][Tk_pad]
  const int bh = blockIdx.y;
  const int i0 = blockIdx.x * RQ;
  const int nrow = min(RQ, s.Tq - i0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // q-bar tile, transposed: qs[c][r] (rows past Tq hold padding and are never used)
  constexpr int QV = RQ / 4;  // float4 per channel row of the tile
  for (int idx = tid; idx < s.d * QV; idx += kScoreThreads) {
    const int c = idx / QV, r4 = idx % QV;
    reinterpret_cast<float4*>(qs)[idx] =
        *reinterpret_cast<const float4*>(qbarT + ((int64_t)bh * s.d + c) * tq_pad + i0 + 4 * r4);
  }
  // ---- pooled scores S[r][j] = (q-bar_r . k-bar_j) / sqrt(d), fp32 FMA in channel order
  constexpr int RPT = RQ / 4;  // rows per thread
  const int tr = tid / 64, tj = tid % 64;  // keys 2 tj, 2 tj + 1 of each chunk
  const float* kbase = kbarT + (int64_t)bh * s.d * Tk_pad;
  const int nchunks = (Tk + kKeyChunk - 1) / kKeyChunk;
  // chunk ci (d x 128 floats = d*32 float4, d/8 per thread) into buffer ci % NBUF
  auto fetch = [&](int ci) {
    float* dst = ks + (ci % NBUF) * s.d * kKeyChunk;
    const int j0 = ci * kKeyChunk;
    for (int idx = tid; idx < s.d * 32; idx += kScoreThreads) {
      const int c = idx >> 5, j4 = idx & 31;
      cp_async16(dst + 4 * idx, kbase + (int64_t)c * Tk_pad + j0 + 4 * j4);
    }
    cp_async_commit();
  };
  if (NBUF == 2) fetch(0);
  for (int ci = 0; ci < nchunks; ++ci) {
    const int j0 = ci * kKeyChunk;
    if (NBUF == 2) {
      // buffer (ci + 1) % 2 was last read by chunk ci - 1, which every thread has finished
      if (ci + 1 < nchunks) {
        fetch(ci + 1);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
    } else {
      fetch(ci);
      cp_async_wait<0>();
    }
    __syncthreads();
    const float* kc = ks + (ci % NBUF) * s.d * kKeyChunk;
    float acc[RPT][2];
#pragma unroll
    for (int a = 0; a < RPT; ++a) acc[a][0] = acc[a][1] = 0.f;
#pragma unroll 4
    for (int c = 0; c < s.d; ++c) {
      const float2 kk = *reinterpret_cast<const float2*>(kc + c * kKeyChunk + 2 * tj);
      float qv[RPT];
      if constexpr (RPT == 4) {
        const float4 t = *reinterpret_cast<const float4*>(qs + c * RQ + tr * 4);
        qv[0] = t.x; qv[1] = t.y; qv[2] = t.z; qv[3] = t.w;
      } else if constexpr (RPT == 2) {
        const float2 t = *reinterpret_cast<const float2*>(qs + c * RQ + tr * 2);
        qv[0] = t.x; qv[1] = t.y;
      } else {
        qv[0] = qs[c * RQ + tr];
      }
#pragma unroll
      for (int a = 0; a < RPT; ++a) {
        acc[a][0] = fmaf(qv[a], kk.x, acc[a][0]);
        acc[a][1] = fmaf(qv[a], kk.y, acc[a][1]);
      }
    }
#pragma unroll
    for (int a = 0; a < RPT; ++a)
      *reinterpret_cast<float2*>(S + (tr * RPT + a) * Tk_pad + j0 + 2 * tj) =
          make_float2(acc[a][0] * sel.inv_sqrt_d, acc[a][1] * sel.inv_sqrt_d);
    // every thread is done with this chunk's buffer before it is refilled
    __syncthreads();
  }
  __syncthreads();

  // ---- per row (one warp per row): softmax, hybrid selection, emit
  for (int r = warp; r < nrow; r += kScoreThreads / 32) {
    float* row = S + r * Tk_pad;
    uint32_t* keys = reinterpret_cast<uint32_t*>(row);
    const int i = i0 + r;
    const int64_t rowid = (int64_t)bh * s.Tq + i;
    float mx = -INFINITY;
    for (int j = lane; j < Tk; j += 32) mx = fmaxf(mx, row[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
    for (int j = lane; j < Tk; j += 32) {
      const float e = expf(row[j] - mx);
      row[j] = e;
      sum += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    for (int j = lane; j < Tk; j += 32) row[j] = __fdiv_rn(row[j], sum);
    __syncwarp();

    // Selection: keep every key > t, and the first `take` keys == t (ascending index).
    // keep_all / keep_none cover K >= Tk, p >= 1, and K = 0 with p <= 0.
    bool keep_all = sel.K >= Tk || sel.p_mode == 2;
    const bool keep_none = !keep_all && sel.K == 0 && sel.p_mode == 1;
    uint32_t t = 0;
    int take = 0;
    if (!keep_all && !keep_none && Tk <= 32 * kRegKeys) {
      select_in_registers(keys, Tk, sel, keep_all, t, take);
    } else if (!keep_all && !keep_none) {
      const bool use_mass = sel.p_mode == 0;
      if (use_mass) {
        const Predicate tot = count_mass(keys, Tk, 0u, false);
        if (tot.mass < sel.p_fix) keep_all = true;  // the row's mass never reaches p
      }
      if (!keep_all) {
        // largest t with count(>= t) >= K and mass(>= t) >= p: the key of the last kept entry
        uint32_t lo = 0, hi = 0x3F800001u;
        while (hi - lo > 1) {
          const uint32_t mid = lo + (hi - lo) / 2;
          const Predicate pr = count_mass(keys, Tk, mid, false);
          const bool ok = pr.cnt >= (uint32_t)sel.K && (!use_mass || pr.mass >= sel.p_fix);
          if (ok)
            lo = mid;
          else
            hi = mid;
        }
        t = lo;
        const Predicate gt = count_mass(keys, Tk, t, true);
        int r_k = sel.K - (int)gt.cnt;
        int r_m = 0;
        if (use_mass && gt.mass < sel.p_fix) {
          const unsigned long long vfix = mass_fix(t);
          r_m = vfix ? (int)((sel.p_fix - gt.mass + vfix - 1) / vfix) : 0;
        }
        take = max(max(r_k, r_m), 0);
      }
    }
    // emit: ascending kept indices, u8 mask, pooled probabilities
    int kept = 0, ties_seen = 0;
    int32_t* ridx = out.row_idx + rowid * Tk;
    uint8_t* mrow = out.mask + rowid * Tk;
    float* prow = out.pooled_p ? out.pooled_p + rowid * Tk : nullptr;
    const unsigned lt = (1u << lane) - 1u;
    for (int j0 = 0; j0 < Tk; j0 += 32) {
      const int j = j0 + lane;
      const bool valid = j < Tk;
      const uint32_t key = valid ? keys[j] : 0u;
      bool keep;
      if (keep_all)
        keep = valid;
      else if (keep_none)
        keep = false;
      else {
        const bool eq = valid && key == t;
        const unsigned eqm = __ballot_sync(0xffffffffu, eq);
        const int tie_rank = ties_seen + __popc(eqm & lt);
        ties_seen += __popc(eqm);
        keep = valid && (key > t || (eq && tie_rank < take));
      }
      const unsigned km = __ballot_sync(0xffffffffu, keep);
      if (keep) ridx[kept + __popc(km & lt)] = j;
      kept += __popc(km);
      if (valid) {
        mrow[j] = keep ? 1 : 0;
        if (prow) prow[j] = __uint_as_float(key);
      }
    }
    if (lane == 0) out.row_cnt[rowid] = kept;
    __syncwarp();
  }
}

// One thread per key block: walks the column of the u8 mask, appends the query blocks
// that keep it (ascending).
__global__ void __launch_bounds__(128) csc_kernel(ShapeArgs s, const uint8_t* __restrict__ mask,
                                                  int32_t* __restrict__ col_cnt, int32_t* __restrict__ col_idx) {
  const int bh = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= s.Tk) return;
  const uint8_t* m = mask + (int64_t)bh * s.Tq * s.Tk + j;
  int32_t* out = col_idx + ((int64_t)bh * s.Tk + j) * s.Tq;
  int cnt = 0;
  int i = 0;
  for (; i + 4 <= s.Tq; i += 4) {
    const uint8_t a = m[(int64_t)i * s.Tk], b = m[(int64_t)(i + 1) * s.Tk], c = m[(int64_t)(i + 2) * s.Tk],
                  d = m[(int64_t)(i + 3) * s.Tk];
    if (a) out[cnt++] = i;
    if (b) out[cnt++] = i + 1;
    if (c) out[cnt++] = i + 2;
    if (d) out[cnt++] = i + 3;
  }
  for (; i < s.Tq; ++i)
    if (m[(int64_t)i * s.Tk]) out[cnt++] = i;
  col_cnt[(int64_t)bh * s.Tk + j] = cnt;
}

// ------------------------------------------------------------------------------- host

int mask_tq_pad(int Tq) { return (Tq + 15) / 16 * 16; }
int mask_tk_pad(int Tk) { return (Tk + kKeyChunk - 1) / kKeyChunk * kKeyChunk; }

size_t mask_pooled_bytes(const ShapeArgs& s, size_t* kbar_offset) {
  const size_t q = (sizeof(float) * (size_t)s.B * s.H * s.d * mask_tq_pad(s.Tq) + 255) / 256 * 256;
  const size_t k = sizeof(float) * (size_t)s.B * s.H * s.d * mask_tk_pad(s.Tk);
  if (kbar_offset) *kbar_offset = q;
  return q + k;
}

static size_t score_smem_bytes(int rq, int nbuf, int Tk, int d) {
  return sizeof(float) * ((size_t)d * rq + (size_t)nbuf * d * kKeyChunk + (size_t)rq * mask_tk_pad(Tk));
}

int score_rows_per_cta(int Tk, int d) {
  for (int rq : {16, 8, 4})
    if (score_smem_bytes(rq, 1, Tk, d) <= kMaxDynSmem) return rq;
  return 0;
}

// chunk buffers for rq rows per CTA: two when they fit beside the score rows
static int score_chunk_buffers(int rq, int Tk, int d) {
  return score_smem_bytes(rq, 2, Tk, d) <= kMaxDynSmem ? 2 : 1;
}

template <int RQ, int NBUF>
static cudaError_t launch_score(const float* qbarT, const float* kbarT, const ShapeArgs& s, const SelectArgs& sel,
                                const MaskOut& out, cudaStream_t st) {
  const size_t smem = score_smem_bytes(RQ, NBUF, s.Tk, s.d);
  auto kern = score_select_kernel<RQ, NBUF>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((s.Tq + RQ - 1) / RQ, s.B * s.H);
  prof_start(st, kScoreSelect);
  kern<<<grid, kScoreThreads, smem, st>>>(qbarT, kbarT, s, mask_tq_pad(s.Tq), mask_tk_pad(s.Tk), sel, out);
  prof_stop(st, kScoreSelect);
  return cudaGetLastError();
}

template <int RQ>
static cudaError_t launch_score(const float* qbarT, const float* kbarT, const ShapeArgs& s, const SelectArgs& sel,
                                const MaskOut& out, cudaStream_t st) {
  return score_chunk_buffers(RQ, s.Tk, s.d) == 2 ? launch_score<RQ, 2>(qbarT, kbarT, s, sel, out, st)
                                                 : launch_score<RQ, 1>(qbarT, kbarT, s, sel, out, st);
}

cudaError_t launch_build_mask(const ShapeArgs& s, const void* q, const void* k, const SelectArgs& sel,
                              void* pooled, const MaskOut& out, cudaStream_t st) {
  size_t koff = 0;
  mask_pooled_bytes(s, &koff);
  float* qbarT = static_cast<float*>(pooled);
  float* kbarT = reinterpret_cast<float*>(static_cast<uint8_t*>(pooled) + koff);
  const int tqp = mask_tq_pad(s.Tq), tkp = mask_tk_pad(s.Tk);
  dim3 pgrid(s.Tq + s.Tk, s.B * s.H);
  prof_start(st, kPool);
  if (s.dtype == 0)
    pool_kernel<__nv_bfloat16><<<pgrid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(q),
                                                       static_cast<const __nv_bfloat16*>(k), s, tqp, tkp, qbarT,
                                                       kbarT);
  else
    pool_kernel<float><<<pgrid, 256, 0, st>>>(static_cast<const float*>(q), static_cast<const float*>(k), s, tqp, tkp,
                                              qbarT, kbarT);
  prof_stop(st, kPool);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int rq = score_rows_per_cta(s.Tk, s.d);
  if (rq == 16)
    e = launch_score<16>(qbarT, kbarT, s, sel, out, st);
  else if (rq == 8)
    e = launch_score<8>(qbarT, kbarT, s, sel, out, st);
  else
    e = launch_score<4>(qbarT, kbarT, s, sel, out, st);
  if (e != cudaSuccess) return e;
  dim3 cgrid((s.Tk + 127) / 128, s.B * s.H);
  prof_start(st, kCsc);
  csc_kernel<<<cgrid, 128, 0, st>>>(s, out.mask, out.col_cnt, out.col_idx);
  prof_stop(st, kCsc);
  return cudaGetLastError();
}

}  // namespace sa2
