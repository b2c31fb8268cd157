// Block-sparse attention backward, dK / dV part, on sm_103a (tcgen05 + TMEM + TMA).
//
// The abstract of SpargeAttention2 (arXiv 2602.13515), contribution (ii), calls the sparse
// attention trainable; the pages do not spell out its backward, so this is the gradient of
// the forward with the block mask held fixed:
//   P = exp(s - LSE), dV = P^T dO, dP = dO V^T, dS = P * (dP - D), D = rowsum(dO * O),
//   dK = scale dS^T Q   (dQ = scale dS K is the job of attn_bwd_dq.cu),
// computed over kept tiles only (gist.science explainer, section 2.C: skipped tiles cost
// nothing).
//
// Each CTA owns one key block j (64 tokens) and walks the list of query blocks that keep
// it (the column list of the mask).  Every GEMM has M = 128:
//   S   = Q_i K_j^T      M = 128 query rows, N = 64 keys, K = d     (A, B K-major)
//   dP  = dO_i V_j^T     M = 128, N = 64, K = d                      (A, B K-major)
//   dV^T += dO_i^T P     M = d, N = 64, K = 128 query rows           (A, B MN-major)
//   dK^T += Q_i^T dS     M = d, N = 64, K = 128                      (A, B MN-major)
// dV^T and dK^T accumulate in TMEM across the whole list and are written once at the end,
// so the kernel needs no cross-CTA reduction.
//
// Roles (192 threads, 1 CTA per SM): warp 0 TMA producer (K_j, V_j once; Q_i, dO_i per list
// entry into 2 stages), warp 1 TMEM owner and MMA issuer, warps 2..5 one query row per
// thread: P and dS from S, dP, LSE and D (prefetched one list entry ahead), written as fp16
// into 128-byte-swizzled shared tiles; finally dK, dV out of TMEM (one channel per thread).
//
// All operands are fp16: the call's Q, K, V, dO arrive as fp16 copies (exact for bf16
// inputs within the fp16 range) and P, dS are written as fp16, which keeps 11 significant
// bits of P and dS against bf16's 8.
//
// The tiles are always 128 channels wide: for d = 64 the second channel panel is read past
// the end of the tensor map and arrives as zeros, and the extra rows of the results are not
// stored.
#include "sa2_internal.h"

namespace sa2 {
namespace {

constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
// TMEM columns
constexpr uint32_t kColS = 0;     // 2 x 64
constexpr uint32_t kColDP = 128;  // 2 x 64
constexpr uint32_t kColDV = 256;  // 64 (lanes = channels)
constexpr uint32_t kColDK = 320;  // 64

// shared memory (bytes from the 1024-aligned base)
constexpr int kOffK = 0;                  // 64 rows x 2 panels of 128 B = 16 KB
constexpr int kOffV = 16384;              // 16 KB
constexpr int kOffStage = 32768;          // 2 stages x (Q 32 KB + dO 32 KB)
constexpr int kStageBytes = 65536;
constexpr int kOffP = kOffStage + 2 * kStageBytes;  // 128 rows x 128 B (swizzled) = 16 KB
constexpr int kOffDS = kOffP + 16384;
constexpr int kOffBar = kOffDS + 16384;
constexpr int kSmemBytes = kOffBar + 256 + 1024;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Row r of a 128-row tile with 128-byte rows in the 128-byte swizzle: 16-byte chunk c lands
// at chunk c ^ (r % 8).
__device__ __forceinline__ void st_swizzled_row(uint8_t* tile, int r, const uint4 (&v)[8]) {
  uint8_t* row = tile + r * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) = v[c];
}

template <typename T>
__device__ __forceinline__ void store_elem(T* p, float v);
template <>
__device__ __forceinline__ void store_elem<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_elem<__nv_bfloat16>(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

template <typename GT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo, ShapeArgs s,
                    BwdArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  const uint32_t bar_kv = smem_u32(&bars[0]);
  auto bar_full = [&](int st) { return smem_u32(&bars[1 + st]); };
  auto bar_empty = [&](int st) { return smem_u32(&bars[3 + st]); };
  auto bar_sfull = [&](int b) { return smem_u32(&bars[5 + b]); };
  const uint32_t bar_pready = smem_u32(&bars[7]);
  const uint32_t bar_pdsfree = smem_u32(&bars[8]);  // the MMAs that read P / dS have completed
  const uint32_t bar_drain = smem_u32(&bars[9]);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 192);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x / s.Tk;
  const int kj = blockIdx.x % s.Tk;
  const int b = bh / s.H, h = bh % s.H;
  const int64_t colid = (int64_t)bh * s.Tk + kj;
  int nq = a.col_cnt[colid];
  if (nq < 0 || nq > s.Tq) {
    if (tid == 0) report_error(a.status, kDevErrBounds);
    nq = nq < 0 ? 0 : s.Tq;
  }
  const int32_t* list = a.col_idx + colid * s.Tq;
  const int kv_valid = min(64, s.N - kj * 64);

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bar_kv, 1);
    for (int st = 0; st < 2; ++st) {
      mbar_init(bar_full(st), 1);
      mbar_init(bar_empty(st), 1);
      mbar_init(bar_sfull(st), 1);
    }
    mbar_init(bar_pready, 128);
    mbar_init(bar_pdsfree, 1);
    mbar_init(bar_drain, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && nq > 0) {
      tma_prefetch_map(&mq);
      tma_prefetch_map(&mdo);
      mbar_arrive_expect_tx(bar_kv, 32768);
      for (int p = 0; p < 2; ++p) {
        tma_load_4d(sbase + kOffK + p * 8192, &mk, bar_kv, p * 64, kj * 64, h, b);
        tma_load_4d(sbase + kOffV + p * 8192, &mv, bar_kv, p * 64, kj * 64, h, b);
      }
      for (int t = 0; t < nq; ++t) {
        const int st = t & 1;
        if (t >= 2 && !mbar_wait(bar_empty(st), ((t >> 1) - 1) & 1, abort_flag)) break;
        int qi = list[t];
        if (qi < 0 || qi >= s.Tq) {
          report_error(a.status, kDevErrBounds);
          qi = 0;
        }
        const uint32_t stg = sbase + kOffStage + st * kStageBytes;
        mbar_arrive_expect_tx(bar_full(st), kStageBytes);
        for (int p = 0; p < 2; ++p) {
          tma_load_4d(stg + p * 16384, &mq, bar_full(st), p * 64, qi * s.bq, h, b);
          tma_load_4d(stg + 32768 + p * 16384, &mdo, bar_full(st), p * 64, qi * s.bq, h, b);
        }
      }
      const int first = nq > 2 ? nq - 2 : 0;
      for (int t = first; t < nq; ++t) mbar_wait(bar_full(t & 1), (t >> 1) & 1, abort_flag);
      mbar_wait(bar_kv, 0, abort_flag);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------------- MMA issuer
    if (lane == 0 && nq > 0) {
      constexpr uint32_t idS = idesc_f16_f32(128, 64, false, false);
      constexpr uint32_t idT = idesc_f16_f32(128, 64, true, true);
      bool ok = mbar_wait(bar_kv, 0, abort_flag);
      for (int t = 0; ok && t <= nq; ++t) {
        if (t < nq) {
          const int st = t & 1;
          if (!mbar_wait(bar_full(st), (t >> 1) & 1, abort_flag)) break;
          tc_fence_after();
          const uint32_t qs = sbase + kOffStage + st * kStageBytes, dos = qs + 32768;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            const uint32_t koff = (kk >> 2) * 8192 + (kk & 3) * 32;
            umma_ss(tmem + kColS + st * 64, smem_desc(qs + off, 16, 1024), smem_desc(sbase + kOffK + koff, 16, 1024),
                    idS, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            const uint32_t koff = (kk >> 2) * 8192 + (kk & 3) * 32;
            umma_ss(tmem + kColDP + st * 64, smem_desc(dos + off, 16, 1024),
                    smem_desc(sbase + kOffV + koff, 16, 1024), idS, kk > 0);
          }
          umma_commit(bar_sfull(st));
        }
        if (t >= 1) {
          const int u = t - 1;
          const int st = u & 1;
          if (!mbar_wait(bar_pready, u & 1, abort_flag)) break;
          tc_fence_after();
          const uint32_t qs = sbase + kOffStage + st * kStageBytes, dos = qs + 32768;
          // dV^T += dO^T P and dK^T += Q^T dS: K = 128 query rows in steps of 16
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t adesc = smem_desc(dos + kk * 2048, 16384, 1024);
            const uint64_t bdesc = smem_desc(sbase + kOffP + kk * 2048, 1024, 1024);
            umma_ss(tmem + kColDV, adesc, bdesc, idT, (u > 0 || kk > 0) ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t adesc = smem_desc(qs + kk * 2048, 16384, 1024);
            const uint64_t bdesc = smem_desc(sbase + kOffDS + kk * 2048, 1024, 1024);
            umma_ss(tmem + kColDK, adesc, bdesc, idT, (u > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(bar_empty(st));
          umma_commit(bar_pdsfree);
        }
      }
      umma_commit(bar_drain);
      mbar_wait(bar_drain, 0, abort_flag);
    }
  } else {
    // -------------------------------------------------------------- query-row threads
    const int sub = warp & 3;
    const int r = 32 * sub + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * sub) << 16);
    const float lse_scale = 1.4426950408889634f;
    // LSE and D of this thread's row for list entry t are loaded one entry ahead, and the
    // query block of entry t two entries ahead, so no dependent global load sits on the path
    // from one tile to the next
    auto row_stats = [&](int t, int qi, float& lse2, float& Dr, bool& valid) {
      qi = (qi < 0 || qi >= s.Tq) ? 0 : qi;
      const int64_t tok = (int64_t)qi * s.bq + r;
      valid = t < nq && r < s.bq && tok < s.N;
      lse2 = valid ? a.lse[(int64_t)bh * s.N + tok] * lse_scale : 0.f;
      Dr = valid ? a.Dvec[(int64_t)bh * s.N + tok] : 0.f;
    };
    float n_lse2, n_D;
    bool n_valid;
    row_stats(0, nq > 0 ? list[0] : 0, n_lse2, n_D, n_valid);
    int qi_ahead = nq > 1 ? list[1] : 0;
    bool ok = true;
    for (int t = 0; t < nq; ++t) {
      const float lse2 = n_lse2, Dr = n_D;
      const bool row_valid = n_valid;
      const int qi_next = qi_ahead;
      qi_ahead = t + 2 < nq ? list[t + 2] : 0;
      row_stats(t + 1, qi_next, n_lse2, n_D, n_valid);
      uint4 pk[8], dk[8];
      const int st = t & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_sfull(st), (t >> 1) & 1, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t sv[32], dv[32];
        tmem_ld32(trow + kColS + st * 64 + half * 32, sv);
        tmem_ld32(trow + kColDP + st * 64 + half * 32, dv);
        tmem_ld_wait(sv);
        tmem_ld_wait(dv);
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          uint32_t pw[4], dw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float pv[2], ds[2];
#pragma unroll
            for (int z = 0; z < 2; ++z) {
              const int c = c8 * 8 + e * 2 + z;
              const bool cv = row_valid && (half * 32 + c) < kv_valid;
              const float p = cv ? ex2(__uint_as_float(sv[c]) * a.scale_log2 - lse2) : 0.f;
              pv[z] = p;
              ds[z] = p * (__uint_as_float(dv[c]) - Dr);
            }
            pw[e] = pack_f16x2(pv[0], pv[1]);
            dw[e] = pack_f16x2(ds[0], ds[1]);
          }
          pk[half * 4 + c8] = make_uint4(pw[0], pw[1], pw[2], pw[3]);
          dk[half * 4 + c8] = make_uint4(dw[0], dw[1], dw[2], dw[3]);
        }
      }
      // the MMAs that read the previous P / dS tiles must have completed
      if (t >= 1 && !__all_sync(0xffffffffu, mbar_wait(bar_pdsfree, (t - 1) & 1, abort_flag))) {
        ok = false;
        break;
      }
      st_swizzled_row(smem + kOffP, r, pk);
      st_swizzled_row(smem + kOffDS, r, dk);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_pready);
    }
    if (ok && nq > 0) ok = __all_sync(0xffffffffu, mbar_wait(bar_pdsfree, (nq - 1) & 1, abort_flag));
    // ---- dK, dV of this key block: thread = channel (TMEM lane), columns = keys
    const int c = r;
    GT* dkp = reinterpret_cast<GT*>(a.dk) + (int64_t)b * a.g_sb + (int64_t)h * a.g_sh + c;
    GT* dvp = reinterpret_cast<GT*>(a.dv) + (int64_t)b * a.g_sb + (int64_t)h * a.g_sh + c;
    if (nq == 0) {
      if (c < s.d)
        for (int kv = 0; kv < kv_valid; ++kv) {
          store_elem<GT>(dkp + (int64_t)(kj * 64 + kv) * a.g_sn, 0.f);
          store_elem<GT>(dvp + (int64_t)(kj * 64 + kv) * a.g_sn, 0.f);
        }
    } else if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t kvv[32], vvv[32];
        tmem_ld32(trow + kColDK + half * 32, kvv);
        tmem_ld32(trow + kColDV + half * 32, vvv);
        tmem_ld_wait(kvv);
        tmem_ld_wait(vvv);
        if (c < s.d) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int kv = half * 32 + e;
            if (kv < kv_valid) {
              store_elem<GT>(dkp + (int64_t)(kj * 64 + kv) * a.g_sn, __uint_as_float(kvv[e]) * a.scale);
              store_elem<GT>(dvp + (int64_t)(kj * 64 + kv) * a.g_sn, __uint_as_float(vvv[e]));
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) report_error(a.status, kDevErrTimeout);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename GT>
cudaError_t launch_bwd_t(const ShapeArgs& s, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mdo, const BwdArgs& a, cudaStream_t st) {
  auto kern = attn_bwd_dkdv_kernel<GT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)s.B * s.H * s.Tk;
  prof_start(st, kAttnBwd);
  kern<<<(unsigned)grid, kThreads, kSmemBytes, st>>>(mq, mk, mv, mdo, s, a);
  prof_stop(st, kAttnBwd);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd(const ShapeArgs& s, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            const CUtensorMap& mdo, const BwdArgs& a, cudaStream_t st) {
  return s.dtype == 0 ? launch_bwd_t<__nv_bfloat16>(s, mq, mk, mv, mdo, a, st)
                      : launch_bwd_t<float>(s, mq, mk, mv, mdo, a, st);
}

}  // namespace sa2
