// Hybrid Top-k + Top-p block mask on sm_103a.
//
// gist.science explainer of SpargeAttention2 (arXiv 2602.13515), section 2.A: the rows of
// the block-pooled attention map P-bar are masked with the union of their Top-k% and
// Top-p% sets; section 1 defines Top-k (the k largest entries) and Top-p (the smallest set
// whose cumulative probability reaches p).
//
// Four kernels:
//   pool_kernel      persistent; streams Q and K through a ring of shared-memory stages
//                    with TMA and writes the block means (fp32) as a TF32 pair hi + lo,
//                    row-major [2][B*H][T][d].  The HBM-bound part of the builder.
//   score_tc_kernel  pooled scores S-bar = q-bar k-bar^T / sqrt(d) of a 128-row x 256-key
//                    tile on the tensor cores (tcgen05, kind::tf32) as the three products
//                    hi.hi + hi.lo + lo.hi -- about fp32 accuracy -- accumulated in tensor
//                    memory and written to a scratch tile.
//   select_kernel    one warp per row: row softmax in fp32, the hybrid selection by a
//                    bisection on the fp32 bit patterns of P-bar with the mass in 2^-60
//                    fixed point, and the emit of the row list and the u8 mask.
//   csc_kernel       transposes the u8 mask into the per-key-block lists (ascending).
// The scores run in chunks of heads whose scratch tiles stay small enough for L2.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <utility>

#include "sa2_internal.h"

namespace sa2 {

namespace {

constexpr int kChunkTokens = 128;           // tokens per pooling chunk
constexpr int kScoreRows = 128;             // MMA M: query blocks per tile
constexpr int kScoreKeys = 256;             // MMA N: key blocks per tile
constexpr int kSelectThreads = 256;
constexpr size_t kScoreChunkBudget = 24u << 20;  // bytes of scratch tiles per head chunk

// ---------------------------------------------------------------------------- helpers

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// TMA load with an L2 eviction-priority policy (evict_first for data streamed once).
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                                 int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ----------------------------------------------------------------------------- pooling

// One pooling item: a chunk of 128 tokens of Q or K of one head (1 or 2 blocks), read by one
// warp.  A lane owns one 16-byte channel group and every RS-th token of the chunk (RS =
// tokens per load instruction: the 32 lanes cover RS whole token rows, so every load of the
// warp reads RS contiguous rows); it sums each 64-token half in fp32 in token order, keeping
// up to 16 loads in flight.  The RS lanes of a channel group are combined with shuffles and
// the lane holding the sum divides by the block's valid tokens and stores hi = tf32(mean),
// lo = tf32(mean - hi).  Items run head by head over the heads [bh0, bh0 + nbh): Q chunks,
// then K chunks; warp w of the grid takes items w, w + (warps in the grid), ...
struct PoolArgs {
  float* qbar;  // [2][B*H][Tq][d]
  float* kbar;  // [2][B*H][Tk][d]
  int bh0, nbh;
};
constexpr int kPoolThreads = 256;

template <typename T, int D>
__global__ void __launch_bounds__(kPoolThreads, 4) pool_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                             ShapeArgs s, PoolArgs a) {
  constexpr int kEsz = sizeof(T);
  constexpr int VE = 16 / kEsz;          // elements per 16-byte group
  constexpr int G = D * kEsz / 16;       // groups per token row: 8, 16 or 32
  constexpr int RS = 32 / G;             // token rows per warp load: 4, 2 or 1
  constexpr int PER_HALF = 64 / RS;      // loads per lane per 64-token half
  constexpr int BATCH = PER_HALF < 8 ? PER_HALF : 8;  // loads in flight per lane
  const int lane = threadIdx.x & 31;
  const int g = lane % G, rs = lane / G;
  const int nc = (s.N + kChunkTokens - 1) / kChunkTokens;
  const long long items = (long long)a.nbh * 2 * nc;
  const long long nwarps = (long long)gridDim.x * (kPoolThreads / 32);
  for (long long x = (long long)blockIdx.x * (kPoolThreads / 32) + (threadIdx.x >> 5); x < items; x += nwarps) {
    const int z = (int)(x / (2 * nc));
    const int r = (int)(x - (long long)z * 2 * nc);
    const bool isk = r >= nc;
    const int c = isk ? r - nc : r;
    const int bh = a.bh0 + z, b = bh / s.H, h = bh - b * s.H;
    const T* src = (isk ? k : q) + (int64_t)b * s.sb + (int64_t)h * s.sh + g * VE;
    const int t0 = c * kChunkTokens;
    float acc[2][VE];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
#pragma unroll
      for (int e = 0; e < VE; ++e) acc[u][e] = 0.f;
#pragma unroll 1
      for (int i0 = 0; i0 < PER_HALF; i0 += BATCH) {
        uint4 v[BATCH];
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
          const int tok = t0 + 64 * u + (i0 + i) * RS + rs;
          v[i] = tok < s.N ? __ldcs(reinterpret_cast<const uint4*>(src + (int64_t)tok * s.sn)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
          if constexpr (kEsz == 2) {
            const uint32_t ww[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc[u][2 * e] += __uint_as_float(ww[e] << 16);
              acc[u][2 * e + 1] += __uint_as_float(ww[e] & 0xFFFF0000u);
            }
          } else {
            acc[u][0] += __uint_as_float(v[i].x);
            acc[u][1] += __uint_as_float(v[i].y);
            acc[u][2] += __uint_as_float(v[i].z);
            acc[u][3] += __uint_as_float(v[i].w);
          }
        }
      }
    }
    // combine the RS lanes of each channel group (lanes g, g + G, g + 2G, ...)
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int e = 0; e < VE; ++e)
#pragma unroll
        for (int o = G; o < 32; o <<= 1) acc[u][e] += __shfl_xor_sync(0xffffffffu, acc[u][e], o);
    if (rs != 0) continue;
    const int bsz = isk ? s.bk : s.bq;
    const int nblk = bsz == 128 ? 1 : 2;
    const int nT = isk ? s.Tk : s.Tq;
    float* out = isk ? a.kbar : a.qbar;
    const size_t plane = (size_t)s.B * s.H * nT * s.d;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (u >= nblk) break;
      const int blk = c * nblk + u;
      if (blk >= nT) break;
      const int valid = min(bsz, s.N - blk * bsz);
      const float inv = 1.f / static_cast<float>(valid);
      float hi[VE], lo[VE];
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        // a block of 128 tokens spans both halves of the chunk
        const float sum = nblk == 1 ? acc[0][e] + acc[1][e] : acc[u][e];
        const float mean = sum * inv;
        hi[e] = tf32_rna(mean);
        lo[e] = tf32_rna(mean - hi[e]);
      }
      float* dst = out + ((size_t)bh * nT + blk) * s.d + g * VE;
#pragma unroll
      for (int e = 0; e < VE; e += 4) {
        *reinterpret_cast<float4*>(dst + e) = make_float4(hi[e], hi[e + 1], hi[e + 2], hi[e + 3]);
        *reinterpret_cast<float4*>(dst + plane + e) = make_float4(lo[e], lo[e + 1], lo[e + 2], lo[e + 3]);
      }
    }
  }
}

// ------------------------------------------------------------------------ TC scores

// One tile: 128 query blocks (TMEM lanes) x 256 key blocks (columns) of one head.  The
// channels arrive in panels of 32 (128 bytes, the TF32 K-major 128-byte-swizzled layout),
// two panels in flight: per panel the hi and lo parts of both operands (96 KB).
// S = Ahi Bhi + Ahi Blo + Alo Bhi over 8-channel k-steps; the epilogue scales by 1/sqrt(d)
// and writes the tile rows to the scratch [chunk heads][Tq_pad][Tk_pad].
constexpr int kAPanelBytes = kScoreRows * 128;  // 16 KB
constexpr int kBPanelBytes = kScoreKeys * 128;  // 32 KB
constexpr int kScoreStageBytes = 2 * kAPanelBytes + 2 * kBPanelBytes;
constexpr int kScoreSmem = 2 * kScoreStageBytes + 256 + 1024;

__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  // D fp32, A and B tf32 (format 2), both K-major
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct ScoreArgs {
  float* sbar;   // scratch tiles of the head chunk
  int bh0;       // first head of the chunk
  int nbh;       // heads of the chunk
  int tq_pad, tk_pad;
  float inv_sqrt_d;
  unsigned* status;
};

// Persistent: CTA c takes tiles c, c + gridDim.x, ... (key chunk fastest, then row tile,
// then head).  Warp 0 streams the panels of its tiles through a two-stage ring without
// stopping between tiles, warp 1 owns tensor memory (two 256-column accumulators) and issues
// the MMAs, warps 2..5 read each finished accumulator out (thread = tile row = TMEM lane),
// so the write-out of tile i overlaps the products of tile i + 1.
constexpr int kScoreThreadsP = 192;

template <int D>
__global__ void __launch_bounds__(kScoreThreadsP, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap mqb, const __grid_constant__ CUtensorMap mkb, ShapeArgs s,
                    ScoreArgs a) {
  constexpr int P = D / 32;  // channel panels per tile
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kScoreStageBytes);
  auto bar_full = [&](int i) { return smem_u32(&bars[i]); };
  auto bar_empty = [&](int i) { return smem_u32(&bars[2 + i]); };
  auto bar_acc = [&](int i) { return smem_u32(&bars[4 + i]); };   // accumulator i complete
  auto bar_free = [&](int i) { return smem_u32(&bars[6 + i]); };  // accumulator i read out
  const uint32_t bar_drain = smem_u32(&bars[8]);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[10]);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&bars[11]);
  const WaitCtl wc{abort_flag, s.wait_ns};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nkc = a.tk_pad / kScoreKeys, nrt = a.tq_pad / kScoreRows;
  const int tiles = a.nbh * nrt * nkc;
  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_full(i), 1);
      mbar_init(bar_empty(i), 1);
      mbar_init(bar_acc(i), 1);
      mbar_init(bar_free(i), 4);  // one arrival per epilogue warp
    }
    mbar_init(bar_drain, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 2 * kScoreKeys);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_map(&mqb);
      tma_prefetch_map(&mkb);
      uint32_t issued = 0;
      bool ok = true;
      for (int ti = blockIdx.x; ti < tiles && ok; ti += gridDim.x) {
        const int kc = ti % nkc, rt = (ti / nkc) % nrt, z = ti / (nkc * nrt);
        for (int p = 0; p < P; ++p, ++issued) {
          const int st = issued & 1;
          if (issued >= 2 && !mbar_wait(bar_empty(st), ((issued >> 1) - 1) & 1, wc)) {
            ok = false;
            break;
          }
          const uint32_t stg = sbase + st * kScoreStageBytes;
          mbar_arrive_expect_tx(bar_full(st), kScoreStageBytes);
          for (int hl = 0; hl < 2; ++hl) {
            tma_load_4d(stg + hl * kAPanelBytes, &mqb, bar_full(st), p * 32, rt * kScoreRows, a.bh0 + z, hl);
            tma_load_4d(stg + 2 * kAPanelBytes + hl * kBPanelBytes, &mkb, bar_full(st), p * 32, kc * kScoreKeys,
                        a.bh0 + z, hl);
          }
        }
      }
      // no copy may still be in flight when the CTA exits
      for (uint32_t v = issued > 2 ? issued - 2 : 0; v < issued; ++v)
        mbar_drain(bar_full(v & 1), (v >> 1) & 1, abort_flag);
    }
  } else if (warp == 1) {
    constexpr uint32_t idS = idesc_tf32(kScoreRows, kScoreKeys);
    bool ok = true;
    uint32_t used = 0, n = 0;  // panels consumed, tiles issued
    for (int ti = blockIdx.x; ti < tiles && ok; ti += gridDim.x, ++n) {
      const int tb = n & 1;
      // accumulator tb was read out by the epilogue of tile n - 2
      if (n >= 2 && !__all_sync(0xffffffffu, mbar_wait(bar_free(tb), ((n >> 1) - 1) & 1, wc))) break;
      tc_fence_after();
      const uint32_t acc = tmem + tb * kScoreKeys;
      for (int p = 0; p < P; ++p, ++used) {
        const int st = used & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar_full(st), (used >> 1) & 1, wc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t stg = sbase + st * kScoreStageBytes;
        const uint64_t ahi = smem_desc(stg, 16, 1024), alo = smem_desc(stg + kAPanelBytes, 16, 1024);
        const uint64_t bhi = smem_desc(stg + 2 * kAPanelBytes, 16, 1024);
        const uint64_t blo = smem_desc(stg + 2 * kAPanelBytes + kBPanelBytes, 16, 1024);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ka = kmajor_kstep(kk, kScoreRows), kb = kmajor_kstep(kk, kScoreKeys);
            umma_tf32(acc, ahi + ka, bhi + kb, idS, (p > 0 || kk > 0) ? 1u : 0u);
            umma_tf32(acc, ahi + ka, blo + kb, idS, 1u);
            umma_tf32(acc, alo + ka, bhi + kb, idS, 1u);
          }
          umma_commit(bar_empty(st));
          if (p == P - 1) umma_commit(bar_acc(tb));
        }
        __syncwarp();
      }
    }
    // every MMA completed (on the abort path too) before tensor memory is freed
    if (elect_one()) umma_commit(bar_drain);
    __syncwarp();
    mbar_drain(bar_drain, 0, abort_flag);
  } else {
    const int q4 = warp & 3;  // TMEM lane quarter of this warp (warps 2..5: 2, 3, 0, 1)
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    uint32_t n = 0;
    for (int ti = blockIdx.x; ti < tiles; ti += gridDim.x, ++n) {
      const int tb = n & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_acc(tb), (n >> 1) & 1, wc))) break;
      tc_fence_after();
      const int kc = ti % nkc, rt = (ti / nkc) % nrt, z = ti / (nkc * nrt);
      const int row = rt * kScoreRows + 32 * q4 + lane;
      float* dst = a.sbar + ((size_t)z * a.tq_pad + row) * a.tk_pad + (size_t)kc * kScoreKeys;
#pragma unroll 1
      for (int c0 = 0; c0 < kScoreKeys; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(trow + tb * kScoreKeys + c0, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          reinterpret_cast<float4*>(dst + c0)[i] =
              make_float4(__uint_as_float(r[4 * i]) * a.inv_sqrt_d, __uint_as_float(r[4 * i + 1]) * a.inv_sqrt_d,
                          __uint_as_float(r[4 * i + 2]) * a.inv_sqrt_d, __uint_as_float(r[4 * i + 3]) * a.inv_sqrt_d);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_free(tb));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) report_error(a.status, kDevErrTimeout);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kScoreKeys);
  }
}

// ----------------------------------------------------------------------- selection

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

// Count and fixed-point mass of the row's entries whose key is >= t (or > t, strictly).
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

// The hybrid selection of one row (one warp) with the row's keys in registers (lane holds
// entries lane, lane + 32, ...; padding keys are 0).  The kept set is every key > t and the
// first `take` keys == t in index order, where t is the largest value with
// count(>= t) >= K and mass(>= t) >= p; keep_all when the row's mass never reaches p.
//
// Masses are compared in 2^-60 fixed point, exactly.  Each lane keeps a coarse 32-bit mass
// per key, c = floor(P * 2^31) = floor(P * 2^60) / 2^29 rounded down; the row's coarse sum S
// stays below 2^32, and over n keys the exact sum lies in [S 2^29, (S + n) 2^29).  A test
// against p is decided by that bracket unless p falls inside it; only then is the exact sum
// formed (from the keys themselves).
__device__ __forceinline__ bool mass_at_least(const uint32_t (&k)[kRegKeys], const uint32_t (&c31)[kRegKeys],
                                              uint32_t t, bool strictly, uint32_t n, unsigned long long p_fix) {
  uint32_t s0 = 0, s1 = 0, s2 = 0, s3 = 0;
#pragma unroll
  for (int i = 0; i < kRegKeys; i += 4) {
    s0 += (strictly ? k[i] > t : k[i] >= t) ? c31[i] : 0u;
    s1 += (strictly ? k[i + 1] > t : k[i + 1] >= t) ? c31[i + 1] : 0u;
    s2 += (strictly ? k[i + 2] > t : k[i + 2] >= t) ? c31[i + 2] : 0u;
    s3 += (strictly ? k[i + 3] > t : k[i + 3] >= t) ? c31[i + 3] : 0u;
  }
  const unsigned long long S = __reduce_add_sync(0xffffffffu, (s0 + s1) + (s2 + s3));
  if ((S << 29) >= p_fix) return true;
  if (((S + n) << 29) <= p_fix) return false;
  unsigned long long m = 0;
#pragma unroll
  for (int i = 0; i < kRegKeys; ++i) m += (strictly ? k[i] > t : k[i] >= t) ? mass_fix(k[i]) : 0ull;
  return warp_sum_u64(m) >= p_fix;
}

__device__ __forceinline__ unsigned long long mass_exact(const uint32_t (&k)[kRegKeys], uint32_t t) {
  unsigned long long m = 0;
#pragma unroll
  for (int i = 0; i < kRegKeys; ++i) m += k[i] > t ? mass_fix(k[i]) : 0ull;
  return warp_sum_u64(m);
}

__device__ __forceinline__ void select_in_registers(const uint32_t (&k)[kRegKeys], const SelectArgs& sel,
                                                    bool& keep_all, uint32_t& t, int& take) {
  const bool use_mass = sel.p_mode == 0;
  uint32_t c31[kRegKeys];
#pragma unroll
  for (int i = 0; i < kRegKeys; ++i) c31[i] = (uint32_t)(mass_fix(k[i]) >> 29);
  // every real key is >= 1 (P > 0 after the softmax; a key of 0 is padding or an
  // underflowed probability, whose mass is 0 as well)
  if (use_mass && !mass_at_least(k, c31, 1u, false, 32u * kRegKeys, sel.p_fix)) {
    keep_all = true;
    return;
  }
  // every tested t is >= 1, so the padding keys (0) are never counted
  uint32_t lo = 0, hi = 0x3F800001u;
  while (hi - lo > 1) {
    const uint32_t mid = lo + (hi - lo) / 2;
    uint32_t c0 = 0, c1 = 0, c2 = 0, c3 = 0;
#pragma unroll
    for (int i = 0; i < kRegKeys; i += 4) {
      c0 += k[i] >= mid ? 1u : 0u;
      c1 += k[i + 1] >= mid ? 1u : 0u;
      c2 += k[i + 2] >= mid ? 1u : 0u;
      c3 += k[i + 3] >= mid ? 1u : 0u;
    }
    const uint32_t n = __reduce_add_sync(0xffffffffu, (c0 + c1) + (c2 + c3));  // same in every lane
    bool ok = n >= (uint32_t)sel.K;
    if (ok && use_mass) ok = mass_at_least(k, c31, mid, false, n, sel.p_fix);
    if (ok)
      lo = mid;
    else
      hi = mid;
  }
  t = lo;
  uint32_t c = 0;
#pragma unroll
  for (int i = 0; i < kRegKeys; ++i) c += k[i] > t ? 1u : 0u;
  c = __reduce_add_sync(0xffffffffu, c);
  const int r_k = sel.K - (int)c;
  int r_m = 0;
  if (use_mass) {
    const unsigned long long m = mass_exact(k, t);
    if (m < sel.p_fix) {
      const unsigned long long vfix = mass_fix(t);
      r_m = vfix ? (int)((sel.p_fix - m + vfix - 1) / vfix) : 0;
    }
  }
  take = max(max(r_k, r_m), 0);
}

// The same selection with the keys in memory (rows longer than 32 * kRegKeys).
__device__ __forceinline__ void select_in_memory(const uint32_t* keys, int Tk, const SelectArgs& sel, bool& keep_all,
                                                 uint32_t& t, int& take) {
  const bool use_mass = sel.p_mode == 0;
  if (use_mass) {
    const Predicate tot = count_mass(keys, Tk, 0u, false);
    if (tot.mass < sel.p_fix) {
      keep_all = true;
      return;
    }
  }
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
  const int r_k = sel.K - (int)gt.cnt;
  int r_m = 0;
  if (use_mass && gt.mass < sel.p_fix) {
    const unsigned long long vfix = mass_fix(t);
    r_m = vfix ? (int)((sel.p_fix - gt.mass + vfix - 1) / vfix) : 0;
  }
  take = max(max(r_k, r_m), 0);
}

// Sorting network for the kRegKeys keys of a lane, descending: K. E. Batcher's odd-even
// merge sort (1968) for 64 inputs, generated at compile time, keeping only the comparators
// whose two positions are below kRegKeys (positions kRegKeys..63 would hold zeros, the
// minimum, which no comparator moves).
// Comparator `idx` of the network (its first or second position), or the number of
// comparators when idx < 0; evaluated by the compiler only.
constexpr int sort_net(int idx, bool second) {
  int n = 0;
  for (int p = 1; p < 64; p *= 2)
    for (int k = p; k >= 1; k /= 2)
      for (int j = k % p; j + k < 64; j += 2 * k)
        for (int i = 0; i < k && i + j + k < 64; ++i)
          if ((i + j) / (2 * p) == (i + j + k) / (2 * p) && i + j + k < kRegKeys) {
            if (n == idx) return second ? i + j + k : i + j;
            ++n;
          }
  return n;
}
constexpr int kSortNetSize = sort_net(-1, false);

template <int C>
__device__ __forceinline__ void sort_cmp(uint32_t (&k)[kRegKeys]) {
  constexpr int a = sort_net(C, false), b = sort_net(C, true);
  const uint32_t x = k[a], y = k[b];
  k[a] = max(x, y);
  k[b] = min(x, y);
}

template <int... C>
__device__ __forceinline__ void sort_all(uint32_t (&k)[kRegKeys], std::integer_sequence<int, C...>) {
  (sort_cmp<C>(k), ...);
}

__device__ __forceinline__ void sort_desc(uint32_t (&k)[kRegKeys]) {
  sort_all(k, std::make_integer_sequence<int, kSortNetSize>{});
}

constexpr int kWalkMax = 128;  // longest walk before the bisection takes over

// The hybrid selection by walking the row in descending order: each lane sorts its keys and
// parks them in shared memory (column `lane`), the warp repeatedly takes the largest head
// (all lanes holding that value advance), and counts and masses (2^-60 fixed point, exact)
// accumulate until count >= K and mass >= p.  The value reached is the threshold t; the
// counts and masses of the keys strictly above it give `take` exactly as the bisection
// does.  Returns false when the walk needs more than kWalkMax steps (the row is then
// left to the bisection; k is sorted but its values are intact).
__device__ __forceinline__ bool select_by_walk(uint32_t (&k)[kRegKeys], uint32_t* col, const SelectArgs& sel,
                                               uint32_t& t, int& take) {
  const int lane = threadIdx.x & 31;
  const bool use_mass = sel.p_mode == 0;
  sort_desc(k);
#pragma unroll
  for (int i = 0; i < kRegKeys; ++i) col[i * 32 + lane] = k[i];
  __syncwarp();
  int cur = 0;
  uint32_t head = k[0];
  uint32_t count = 0, cnt_gt = 0, val = 0xFFFFFFFFu;
  unsigned long long mass = 0, mass_gt = 0;
  for (int step = 0; step < kWalkMax; ++step) {
    const uint32_t mx = __reduce_max_sync(0xffffffffu, head);
    if (mx == 0u) return false;  // every key consumed (not reached when K <= Tk and the mass reaches p)
    if (mx != val) {  // a new value: the keys counted so far are all above it
      val = mx;
      cnt_gt = count;
      mass_gt = mass;
    }
    const bool adv = head == mx;  // every lane holding the value advances
    const uint32_t n_eq = __popc(__ballot_sync(0xffffffffu, adv));
    count += n_eq;
    mass += (unsigned long long)n_eq * mass_fix(mx);
    if (count >= (uint32_t)sel.K && (!use_mass || mass >= sel.p_fix)) {
      t = mx;
      const int r_k = sel.K - (int)cnt_gt;
      int r_m = 0;
      if (use_mass && mass_gt < sel.p_fix) {
        const unsigned long long vfix = mass_fix(t);
        r_m = vfix ? (int)((sel.p_fix - mass_gt + vfix - 1) / vfix) : 0;
      }
      take = max(max(r_k, r_m), 0);
      return true;
    }
    // branch-free advance: every lane stays on the warp-wide reductions' path
    const int nc = cur + (adv ? 1 : 0);
    const uint32_t nxt = nc < kRegKeys ? col[nc * 32 + lane] : 0u;
    head = adv ? nxt : head;
    cur = nc;
  }
  return false;
}

struct SelArgs {
  float* sbar;  // scratch tiles of the head chunk; rows past 32 * kRegKeys keys are
                // overwritten in place by their P-bar bit patterns
  int bh0, nbh;
  int tq_pad, tk_pad;
};

// One warp per row: softmax of the pooled scores in fp32 (exponentials by the ex2
// instruction, one correctly rounded reciprocal of the row sum), the hybrid selection (the
// walk, or the bisection for long walks and long rows), and the emit of the ascending kept
// indices, the u8 mask and, when asked, P-bar.
constexpr int kSelectWarps = kSelectThreads / 32;
constexpr int kSelectSmem = kSelectWarps * 2 * kRegKeys * 32 * 4;  // 80 KB

__global__ void __launch_bounds__(kSelectThreads, 2) select_kernel(ShapeArgs s, SelectArgs sel, SelArgs a,
                                                                   MaskOut out) {
  // per warp: the sorted keys of the walk, and the keys in index order for the emit
  extern __shared__ __align__(16) uint32_t sel_smem[];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  uint32_t* walk_col = sel_smem + wib * (2 * kRegKeys * 32);
  uint32_t* row_keys = walk_col + kRegKeys * 32;
  const long long gw = (long long)blockIdx.x * kSelectWarps + wib;
  if (gw >= (long long)a.nbh * s.Tq) return;  // whole warps only
  const int z = (int)(gw / s.Tq), i = (int)(gw - (long long)z * s.Tq);
  const int Tk = s.Tk;
  float* row = a.sbar + ((size_t)z * a.tq_pad + i) * a.tk_pad;
  const int64_t rowid = (int64_t)(a.bh0 + z) * s.Tq + i;
  const bool in_regs = Tk <= 32 * kRegKeys;

  // row softmax
  float mx = -INFINITY, inv = 0.f;
  uint32_t k[kRegKeys];
  if (in_regs) {
    float v[kRegKeys];
#pragma unroll
    for (int t = 0; t < kRegKeys; ++t) {
      const int j = lane + 32 * t;
      v[t] = j < Tk ? row[j] : -INFINITY;
      mx = fmaxf(mx, v[t]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int t = 0; t < kRegKeys; ++t) {
      v[t] = lane + 32 * t < Tk ? ex2_approx((v[t] - mx) * kLog2e) : 0.f;
      if (t & 1)
        s1 += v[t];
      else
        s0 += v[t];
    }
    float sum = s0 + s1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    inv = __frcp_rn(sum);
#pragma unroll
    for (int t = 0; t < kRegKeys; ++t) {
      k[t] = lane + 32 * t < Tk ? __float_as_uint(v[t] * inv) : 0u;
      row_keys[t * 32 + lane] = k[t];  // entry lane + 32 t: the emit reads these keys
    }
    __syncwarp();
  } else {
    for (int j = lane; j < Tk; j += 32) mx = fmaxf(mx, row[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
    for (int j = lane; j < Tk; j += 32) sum += ex2_approx((row[j] - mx) * kLog2e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    inv = __frcp_rn(sum);
    __syncwarp();
    for (int j = lane; j < Tk; j += 32) row[j] = ex2_approx((row[j] - mx) * kLog2e) * inv;
    __syncwarp();
  }
  const uint32_t* mkeys = reinterpret_cast<const uint32_t*>(row);

  // selection: keep every key > t, and the first `take` keys == t (ascending index);
  // keep_all / keep_none cover K >= Tk, p >= 1, and K = 0 with p <= 0
  bool keep_all = sel.K >= Tk || sel.p_mode == 2;
  const bool keep_none = !keep_all && sel.K == 0 && sel.p_mode == 1;
  uint32_t t = 0;
  int take = 0;
  if (!keep_all && !keep_none) {
    if (in_regs) {
      // the row's mass may never reach p (rounding): then every block is kept
      if (sel.p_mode == 0) {
        uint32_t c31[kRegKeys];
#pragma unroll
        for (int q = 0; q < kRegKeys; ++q) c31[q] = (uint32_t)(mass_fix(k[q]) >> 29);
        keep_all = !mass_at_least(k, c31, 1u, false, 32u * kRegKeys, sel.p_fix);
      }
      if (!keep_all && !select_by_walk(k, walk_col, sel, t, take))
        select_in_registers(k, sel, keep_all, t, take);
    } else {
      select_in_memory(mkeys, Tk, sel, keep_all, t, take);
    }
  }
  // emit: ascending kept indices (ballot-compacted), the u8 mask and P-bar, from the very keys
  // the selection used (entry j = j0 + lane is key j0 / 32 of the lane)
  int kept = 0, ties_seen = 0;
  int32_t* ridx = out.row_idx + rowid * Tk;
  uint8_t* mrow = out.mask + rowid * Tk;
  float* prow = out.pooled_p ? out.pooled_p + rowid * Tk : nullptr;
  const unsigned lt = (1u << lane) - 1u;
  for (int j0 = 0; j0 < Tk; j0 += 32) {
    const int j = j0 + lane;
    const bool valid = j < Tk;
    const uint32_t key = !valid ? 0u : (in_regs ? row_keys[j0 + lane] : mkeys[j]);
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
}

// Column lists from the u8 mask.  A CTA takes 32 consecutive key blocks of one head (lane =
// key block) and its 8 warps split the query blocks into ranges: each warp reads its rows'
// 32-byte segments (coalesced, 32 loads in flight), keeps the kept-bits of its lane's column
// in shared memory, then the per-warp counts are prefix-summed and every lane writes its
// column's query blocks in ascending order.  blockIdx.y is the head within [bh0, ...).
constexpr int kCscWarps = 8;
constexpr int kCscMaxWords = 30;  // Tq <= 7680 (bq >= 64, N <= 7680 * 64): 960 rows per warp

__global__ void __launch_bounds__(32 * kCscWarps) csc_kernel(ShapeArgs s, int bh0, const uint8_t* __restrict__ mask,
                                                             int32_t* __restrict__ col_cnt,
                                                             int32_t* __restrict__ col_idx) {
  __shared__ uint32_t bits[kCscWarps][kCscMaxWords][32];
  __shared__ int cnt[kCscWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = bh0 + blockIdx.y;
  const int j = blockIdx.x * 32 + lane;
  const bool col_ok = j < s.Tk;
  const int R = (s.Tq + kCscWarps - 1) / kCscWarps;  // rows per warp (<= 32 * kCscMaxWords)
  const int i0 = warp * R, i1 = min(s.Tq, i0 + R);
  const uint8_t* m = mask + (int64_t)bh * s.Tq * s.Tk + min(j, s.Tk - 1);
  int c = 0;
  for (int w = 0; w * 32 < R; ++w) {
    uint8_t v[32];
#pragma unroll
    for (int b = 0; b < 32; ++b) v[b] = m[(int64_t)min(i0 + w * 32 + b, s.Tq - 1) * s.Tk];
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 32; ++b)
      if (v[b] && i0 + w * 32 + b < i1) word |= 1u << b;
    if (!col_ok) word = 0;
    bits[warp][w][lane] = word;
    c += __popc(word);
  }
  cnt[warp][lane] = c;
  __syncthreads();
  int base = 0, total = 0;
  for (int q = 0; q < kCscWarps; ++q) {
    if (q < warp) base += cnt[q][lane];
    total += cnt[q][lane];
  }
  if (!col_ok) return;
  int32_t* out = col_idx + ((int64_t)bh * s.Tk + j) * s.Tq + base;
  for (int w = 0; w * 32 < R; ++w) {
    uint32_t word = bits[warp][w][lane];
    while (word) {
      const int b = __ffs(word) - 1;
      word &= word - 1;
      *out++ = i0 + w * 32 + b;
    }
  }
  if (warp == 0) col_cnt[(int64_t)bh * s.Tk + j] = total;
}

// ------------------------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// Pooled pairs [2][B*H][T][d] fp32 as a 4-D map (d, T, B*H, 2), boxes of 32 channels x
// `rows` blocks, 128-byte swizzle (the TF32 K-major operand layout); rows past T read as zero.
bool make_pooled_map(CUtensorMap* map, const float* base, const ShapeArgs& s, int T, int rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  std::memset(map, 0, sizeof(*map));
  const cuuint64_t BH = (cuuint64_t)s.B * s.H;
  cuuint64_t dims[4] = {(cuuint64_t)s.d, (cuuint64_t)T, BH, 2};
  cuuint64_t strides[3] = {(cuuint64_t)s.d * 4, (cuuint64_t)T * s.d * 4, BH * T * s.d * 4};
  cuuint32_t box[4] = {32, (cuuint32_t)rows, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct MaskLayout {
  size_t qbar, kbar, sbar, total;
  int tq_pad, tk_pad, hc;  // padded tile extents; heads per score chunk
};

MaskLayout mask_layout(const ShapeArgs& s, size_t sbar_budget) {
  MaskLayout L;
  const size_t BH = (size_t)s.B * s.H;
  auto al = [](size_t x) { return (x + 1023) / 1024 * 1024; };
  L.tq_pad = (s.Tq + kScoreRows - 1) / kScoreRows * kScoreRows;
  L.tk_pad = (s.Tk + kScoreKeys - 1) / kScoreKeys * kScoreKeys;
  const size_t per_head = (size_t)L.tq_pad * L.tk_pad * 4;
  L.hc = (int)std::max<size_t>(1, std::min<size_t>(BH, sbar_budget / per_head));
  L.qbar = 0;
  L.kbar = al(2 * BH * s.Tq * s.d * 4);
  L.sbar = L.kbar + al(2 * BH * s.Tk * s.d * 4);
  L.total = L.sbar + al((size_t)L.hc * per_head);
  return L;
}

// A second stream per device on which the scores, the selection and the column lists of a
// chunk of heads run while the caller's stream pools the next chunk; the caller's stream
// waits for it at the end of the call.  Set up on the first build on a device.
struct AuxStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t pooled = nullptr, done = nullptr;
  cudaError_t err = cudaSuccess;
  std::mutex mu;  // one enqueue sequence at a time per device
};
constexpr int kMaxAuxDevices = 64;
AuxStream g_aux[kMaxAuxDevices];
std::once_flag g_aux_once[kMaxAuxDevices];

AuxStream* aux_stream(int dev) {
  if (dev < 0 || dev >= kMaxAuxDevices) return nullptr;
  std::call_once(g_aux_once[dev], [dev]() {
    AuxStream& a = g_aux[dev];
    a.err = cudaStreamCreateWithFlags(&a.stream, cudaStreamNonBlocking);
    if (a.err == cudaSuccess) a.err = cudaEventCreateWithFlags(&a.pooled, cudaEventDisableTiming);
    if (a.err == cudaSuccess) a.err = cudaEventCreateWithFlags(&a.done, cudaEventDisableTiming);
  });
  return g_aux[dev].err == cudaSuccess ? &g_aux[dev] : nullptr;
}

}  // namespace

int score_rows_per_cta(int Tk, int d) { return Tk >= 1 && (d == 64 || d == 128) ? kScoreRows : 0; }

size_t mask_scratch_bytes(const ShapeArgs& s, size_t budget) {
  if (budget == 0) return mask_layout(s, kScoreChunkBudget).total;
  // the largest head chunk that fits the budget (at least one head)
  const MaskLayout one = mask_layout(s, 0);
  if (one.total > budget) return one.total;
  return mask_layout(s, budget - one.sbar).total;
}

cudaError_t launch_build_mask(const ShapeArgs& s, const void* q, const void* k, const SelectArgs& sel, void* scratch,
                              size_t scratch_bytes, const MaskOut& out, cudaStream_t st) {
  const MaskLayout L0 = mask_layout(s, 0);
  if (scratch_bytes != 0 && scratch_bytes < L0.total) return cudaErrorInvalidValue;
  const MaskLayout L = scratch_bytes == 0 ? mask_layout(s, kScoreChunkBudget)
                                          : mask_layout(s, std::min(kScoreChunkBudget, scratch_bytes - L0.sbar));
  uint8_t* base = static_cast<uint8_t*>(scratch);
  float* qbar = reinterpret_cast<float*>(base + L.qbar);
  float* kbar = reinterpret_cast<float*>(base + L.kbar);
  float* sbar = reinterpret_cast<float*>(base + L.sbar);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  AuxStream* aux = aux_stream(dev);
  if (!aux) return cudaErrorUnknown;

  CUtensorMap mqb, mkb;
  if (!make_pooled_map(&mqb, qbar, s, s.Tq, kScoreRows) || !make_pooled_map(&mkb, kbar, s, s.Tk, kScoreKeys))
    return cudaErrorInvalidValue;
  auto score = s.d == 128 ? score_tc_kernel<128> : score_tc_kernel<64>;
  e = cudaFuncSetAttribute(score, cudaFuncAttributeMaxDynamicSharedMemorySize, kScoreSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelectSmem);
  if (e != cudaSuccess) return e;
  const void* pool = s.dtype == 0
                         ? (s.d == 128 ? (const void*)pool_kernel<__nv_bfloat16, 128> : (const void*)pool_kernel<__nv_bfloat16, 64>)
                         : (s.d == 128 ? (const void*)pool_kernel<float, 128> : (const void*)pool_kernel<float, 64>);
  int pool_occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&pool_occ, pool, kPoolThreads, 0);
  if (e != cudaSuccess) return e;
  // a third of the SMs' pooling capacity per chunk: the other kernels of the previous chunk
  // run beside it
  const int pool_blocks = std::max(1, sms * std::max(1, pool_occ) / 2);

  std::lock_guard<std::mutex> lock(aux->mu);
  const int BH = s.B * s.H;
  const int nc = (s.N + kChunkTokens - 1) / kChunkTokens;
  for (int bh0 = 0; bh0 < BH; bh0 += L.hc) {
    const int nbh = std::min(L.hc, BH - bh0);
    // ---- pooling of the chunk, on the caller's stream
    PoolArgs pa;
    pa.qbar = qbar;
    pa.kbar = kbar;
    pa.bh0 = bh0;
    pa.nbh = nbh;
    const long long pool_warps = (long long)nbh * 2 * nc;
    const int pgrid = (int)std::min<long long>((pool_warps + 7) / 8, pool_blocks);
    prof_start(st, kPool);
    if (s.dtype == 0) {
      auto qq = static_cast<const __nv_bfloat16*>(q);
      auto kk = static_cast<const __nv_bfloat16*>(k);
      if (s.d == 128)
        pool_kernel<__nv_bfloat16, 128><<<pgrid, kPoolThreads, 0, st>>>(qq, kk, s, pa);
      else
        pool_kernel<__nv_bfloat16, 64><<<pgrid, kPoolThreads, 0, st>>>(qq, kk, s, pa);
    } else {
      auto qq = static_cast<const float*>(q);
      auto kk = static_cast<const float*>(k);
      if (s.d == 128)
        pool_kernel<float, 128><<<pgrid, kPoolThreads, 0, st>>>(qq, kk, s, pa);
      else
        pool_kernel<float, 64><<<pgrid, kPoolThreads, 0, st>>>(qq, kk, s, pa);
    }
    prof_stop(st, kPool);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaEventRecord(aux->pooled, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(aux->stream, aux->pooled, 0);
    if (e != cudaSuccess) return e;
    // ---- scores, selection and column lists of the chunk, on the second stream
    cudaStream_t st2 = aux->stream;
    ScoreArgs sa;
    sa.sbar = sbar;
    sa.bh0 = bh0;
    sa.nbh = nbh;
    sa.tq_pad = L.tq_pad;
    sa.tk_pad = L.tk_pad;
    sa.inv_sqrt_d = sel.inv_sqrt_d;
    sa.status = out.status;
    const int tiles = nbh * (L.tq_pad / kScoreRows) * (L.tk_pad / kScoreKeys);
    prof_start(st2, kScoreTc);
    score<<<std::min(tiles, sms), kScoreThreadsP, kScoreSmem, st2>>>(mqb, mkb, s, sa);
    prof_stop(st2, kScoreTc);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    SelArgs ca;
    ca.sbar = sbar;
    ca.bh0 = bh0;
    ca.nbh = nbh;
    ca.tq_pad = L.tq_pad;
    ca.tk_pad = L.tk_pad;
    const long long rows = (long long)nbh * s.Tq;
    prof_start(st2, kScoreSelect);
    select_kernel<<<(unsigned)((rows + kSelectWarps - 1) / kSelectWarps), kSelectThreads, kSelectSmem, st2>>>(
        s, sel, ca, out);
    prof_stop(st2, kScoreSelect);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 cgrid((s.Tk + 31) / 32, nbh);
    prof_start(st2, kCsc);
    csc_kernel<<<cgrid, 32 * kCscWarps, 0, st2>>>(s, bh0, out.mask, out.col_cnt, out.col_idx);
    prof_stop(st2, kCsc);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  e = cudaEventRecord(aux->done, aux->stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, aux->done, 0);
  return e;
}

}  // namespace sa2
