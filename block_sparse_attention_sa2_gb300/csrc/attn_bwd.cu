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
// A work item is a pair of adjacent key blocks (2m, 2m+1: 128 keys); the CTA that takes it
// walks the union of their two column lists (built by pair_union_kernel below) in sub-tiles
// of 64 query rows and writes the pair's dK, dV once.
// The products are formed transposed, keys along the 128 TMEM lanes:
//   S^T  = K Q_u^T    M = 128 keys, N = 64 queries, K = d   (A, B from shared memory)
//   dP^T = V dO_u^T   M = 128, N = 64, K = d
//   dV  += P^T dO_u   M = 128 keys, N = d, K = 64 queries   (A = P^T from TMEM)
//   dK  += dS^T Q_u   M = 128, N = d, K = 64                 (A = dS^T from TMEM)
// so P^T and dS^T never go through shared memory: the element-wise warps read S^T and dP^T
// out of TMEM and write P^T and dS^T back into TMEM as fp16.  For a query block kept by
// only one of the two key blocks the other block's 64 key rows get P = 0 (a warp-uniform
// choice: they are whole warps), which is the price of the pairing -- about a fifth more
// MMA work on the Wan-like masks -- against a tensor-core step that is twice as wide.
//
// TMEM (512 columns): S^T and dP^T (64 columns each; single at d = 128, double-buffered at
// d = 64), P^T and dS^T as fp16 pairs (32 columns each, double-buffered), dV and dK
// accumulators (d columns each, lanes = keys, columns = channels).  S^T / dP^T are free
// again as soon as the element-wise warps hold them in registers, so the next sub-tile's
// S^T, dP^T MMAs never wait for the dV, dK MMAs to complete: the tensor pipe runs S/dP(u+1)
// behind dV/dK(u-1) without draining (at d = 64, S/dP(u+1) need not even wait for sub-tile
// u to be read out).  Shared memory: K and V of the pair (16 KB per 64-channel panel each)
// and a 4-deep ring of query sub-tiles (Q and dO, 8 KB per panel each, and the sub-tile's
// log2(e)*LSE and D vectors, 512 B).
//
// Roles (352 threads, 1 CTA per SM): warp 0 TMA producer, warp 1 TMEM owner and issuer
// of the S^T / dP^T MMAs, warp 2 issuer of the dV / dK MMAs (each converged, one
// elect.sync lane issuing), warps 3..10 element-wise (thread = key row; warps 3-6 take
// query columns 0-31 of the sub-tile, warps 7-10 columns 32-63), then the dK / dV
// epilogue.
//
// The CTAs are persistent, one per SM, and take key-block pairs from a counter until none
// is left.  The producer publishes each pair in a two-slot ring in shared memory that every
// role reads; all barrier phases count sub-tiles and pairs over the CTA's whole run.  So the
// set-up (barriers, TMEM allocation) is paid once per SM, the next pair's K and V load as
// soon as the current pair's S^T / dP^T MMAs have completed, and its first S^T / dP^T
// MMAs run while the element-wise warps store the current pair's dK and dV.
//
// All operands are fp16: the call's Q, K, V, dO arrive as fp16 copies (exact for bf16
// inputs within the fp16 range) and P, dS are written as fp16, which keeps 11 significant
// bits of P and dS against bf16's 8.
//
// The channel dimension is a template parameter: d = 128 tiles hold two 64-channel panels,
// d = 64 tiles one, so that a d = 64 call runs half the k-steps of Sᵀ / dPᵀ and dV / dK
// products of N = 64 (the accumulators keep their 128 columns, half of them unused).
#include "sa2_internal.h"

namespace sa2 {
namespace {

constexpr int kThreads = 352;
constexpr int kItemReaders = 10;  // warps reading the item slot: 1, 2 and the 8 element-wise warps
constexpr uint32_t kTmemCols = 512;
// TMEM columns
// TMEM columns.  d = 128: S^T and dP^T once (64 each), P^T and dS^T as fp16 pairs
// double-buffered (2 x 32 each), dV and dK (128 each).  d = 64: the accumulators take 64
// columns each, which leaves room to double-buffer S^T and dP^T as well (buffer b of S^T at
// 128 b, of dP^T at 128 b + 64), so that S^T(u+1) does not wait for the element-wise warps to
// have read S^T(u) out.
template <int D>
struct DkdvCols {
  static constexpr int kSBuf = D == 64 ? 2 : 1;  // S^T / dP^T buffers
  static constexpr uint32_t S(int b) { return 128u * b; }
  static constexpr uint32_t DP(int b) { return 128u * b + 64u; }
  static constexpr uint32_t P = 128u * kSBuf, DS = P + 64u;  // 2 x 32 each, after the S^T / dP^T buffers
  static constexpr uint32_t DV = DS + 64u, DK = DV + (uint32_t)D;
  static_assert(DK + D <= 512, "TMEM columns");
  static_assert(D != 128 || (P == 128 && DV == 256 && DK == 384), "the d = 128 layout");
  static_assert(D != 64 || (P == 256 && DV == 384 && DK == 448), "the d = 64 layout");
};

// Shared memory (bytes from the 1024-aligned base).  SPLIT (fp32 calls): K and Q also as
// fp16 residuals lo = fp16(x - hi) for the split product S^T = Khi Qhi^T + Khi Qlo^T +
// Klo Qhi^T, with a 2-deep sub-tile ring to fit.
template <bool SPLIT, int D>
struct DkdvSmem {
  static constexpr int kPanels = D / 64;          // 64-channel panels of 128 B rows
  static constexpr int kStages = SPLIT ? 2 : 4;
  static constexpr int kShift = SPLIT ? 1 : 2;  // log2(kStages)
  static constexpr int kKVBytes = 128 * 128 * kPanels;  // 128 key rows x panels (panel = 16 KB)
  static constexpr int kOffK = 0;
  static constexpr int kOffKlo = kKVBytes;  // (SPLIT)
  static constexpr int kOffV = SPLIT ? 2 * kKVBytes : kKVBytes;
  static constexpr int kOffStage = kOffV + kKVBytes;  // stage: Q (panels x 64 rows x 128 B), dO (same), stats
  static constexpr int kTileBytes = 64 * 128 * kPanels;
  static constexpr int kStageQ = 0, kStageDO = kTileBytes, kStageStats = 2 * kTileBytes;
  static constexpr int kStageQlo = 2 * kTileBytes + 1024;  // (SPLIT)
  static constexpr int kStageBytes = SPLIT ? kStageQlo + kTileBytes : 2 * kTileBytes + 1024;
  static constexpr uint32_t kStageTx = (SPLIT ? 3 : 2) * kTileBytes + 512;
  static constexpr int kOffBar = kOffStage + kStages * kStageBytes;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;
  static_assert(kSmemBytes <= (int)kMaxDynSmem, "shared memory");
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename GT>
__device__ __forceinline__ void store_row64(GT* p, const uint32_t (&x)[32], const uint32_t (&y)[32], float mul);
template <>
__device__ __forceinline__ void store_row64<__nv_bfloat16>(__nv_bfloat16* p, const uint32_t (&x)[32],
                                                           const uint32_t (&y)[32], float mul) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 w;
    w.x = pack_bf16x2(__uint_as_float(x[8 * c + 0]) * mul, __uint_as_float(x[8 * c + 1]) * mul);
    w.y = pack_bf16x2(__uint_as_float(x[8 * c + 2]) * mul, __uint_as_float(x[8 * c + 3]) * mul);
    w.z = pack_bf16x2(__uint_as_float(x[8 * c + 4]) * mul, __uint_as_float(x[8 * c + 5]) * mul);
    w.w = pack_bf16x2(__uint_as_float(x[8 * c + 6]) * mul, __uint_as_float(x[8 * c + 7]) * mul);
    *reinterpret_cast<uint4*>(p + 8 * c) = w;
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 w;
    w.x = pack_bf16x2(__uint_as_float(y[8 * c + 0]) * mul, __uint_as_float(y[8 * c + 1]) * mul);
    w.y = pack_bf16x2(__uint_as_float(y[8 * c + 2]) * mul, __uint_as_float(y[8 * c + 3]) * mul);
    w.z = pack_bf16x2(__uint_as_float(y[8 * c + 4]) * mul, __uint_as_float(y[8 * c + 5]) * mul);
    w.w = pack_bf16x2(__uint_as_float(y[8 * c + 6]) * mul, __uint_as_float(y[8 * c + 7]) * mul);
    *reinterpret_cast<uint4*>(p + 32 + 8 * c) = w;
  }
}
template <>
__device__ __forceinline__ void store_row64<float>(float* p, const uint32_t (&x)[32], const uint32_t (&y)[32],
                                                   float mul) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<float4*>(p + 4 * c) =
        make_float4(__uint_as_float(x[4 * c]) * mul, __uint_as_float(x[4 * c + 1]) * mul,
                    __uint_as_float(x[4 * c + 2]) * mul, __uint_as_float(x[4 * c + 3]) * mul);
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<float4*>(p + 32 + 4 * c) =
        make_float4(__uint_as_float(y[4 * c]) * mul, __uint_as_float(y[4 * c + 1]) * mul,
                    __uint_as_float(y[4 * c + 2]) * mul, __uint_as_float(y[4 * c + 3]) * mul);
}

template <typename GT>
__device__ __forceinline__ void zero_row64(GT* p) {
  constexpr int kVec = 16 / sizeof(GT);
#pragma unroll
  for (int c = 0; c < 64 / kVec; ++c) *reinterpret_cast<uint4*>(p + kVec * c) = make_uint4(0, 0, 0, 0);
}

template <typename GT, bool SPLIT, int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                         const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                         const __grid_constant__ CUtensorMap mql, const __grid_constant__ CUtensorMap mkl,
                         ShapeArgs s, BwdArgs a) {
  using L = DkdvSmem<SPLIT, D>;
  constexpr int kStages = L::kStages, kStShift = L::kShift;
  constexpr int kOffK = L::kOffK, kOffKlo = L::kOffKlo, kOffV = L::kOffV, kOffStage = L::kOffStage;
  constexpr int kStageQ = L::kStageQ, kStageDO = L::kStageDO, kStageStats = L::kStageStats, kStageQlo = L::kStageQlo;
  constexpr int kStageBytes = L::kStageBytes, kOffBar = L::kOffBar;
  constexpr uint32_t kStageTx = L::kStageTx;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  const uint32_t bar_kv = smem_u32(&bars[0]);  // K, V of the current pair landed
  auto bar_full = [&](int st) { return smem_u32(&bars[1 + st]); };
  auto bar_empty = [&](int st) { return smem_u32(&bars[5 + st]); };
  using C = DkdvCols<D>;
  constexpr int kSBuf = C::kSBuf;
  // S^T, dP^T of a sub-tile in TMEM buffer b, and read out by the element-wise warps
  auto bar_sfull = [&](int b) { return smem_u32(&bars[b == 0 ? 9 : 23]); };
  auto bar_sfree = [&](int b) { return smem_u32(&bars[b == 0 ? 10 : 24]); };
  auto bar_pready = [&](int b) { return smem_u32(&bars[11 + b]); };  // P^T, dS^T buffer b written
  auto bar_pfree = [&](int b) { return smem_u32(&bars[13 + b]); };   // MMAs reading buffer b done
  const uint32_t bar_drain = smem_u32(&bars[15]);   // every dV / dK MMA of the pair completed
  const uint32_t bar_sdrain = smem_u32(&bars[16]);  // every S^T / dP^T MMA of the CTA completed
  const uint32_t bar_kvfree = smem_u32(&bars[17]);  // every S^T / dP^T MMA of the pair completed
  const uint32_t bar_gdrain = smem_u32(&bars[18]);  // every dV / dK MMA of the CTA completed
  auto bar_item_full = [&](int i) { return smem_u32(&bars[19 + i]); };  // item slot i written
  auto bar_item_free = [&](int i) { return smem_u32(&bars[21 + i]); };  // ... and read by every role
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 224);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 232);
  volatile int* item_slot = reinterpret_cast<volatile int*>(smem + kOffBar + 240);
  const WaitCtl wc{abort_flag, s.wait_ns};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Work items are key-block pairs in pair-major order (item x: pair m = x / BH of head
  // x % BH), so the pairs holding the first key blocks of every head, where attention sinks
  // and so the longest lists usually sit, start first.  Each CTA stays resident and takes
  // items from a counter: its first is blockIdx.x, the next gridDim.x + (counter value).
  const int BH = s.B * s.H;
  const int Tp = (s.Tk + 1) >> 1;
  const int num_items = BH * Tp;
  const int sub_shift = s.bq == 128 ? 1 : 0;  // 64-row sub-tiles per query block: 2 or 1
  const int Tsub = s.Tq << sub_shift;
  // union length of item x, clamped to [0, Tq] (the producer reports a bad value)
  auto item_len = [&](int x, bool report) {
    const int m = x / BH, bh = x - m * BH;
    int nu = a.pair_cnt[(int64_t)bh * Tp + m];
    if (nu < 0 || nu > s.Tq) {
      if (report) report_error(a.status, kDevErrBounds);
      nu = nu < 0 ? 0 : s.Tq;
    }
    return nu;
  };
  // a consumer warp takes item n from its slot and hands the slot back; -1 ends the loop
  auto take_item = [&](int n, bool& ok) {
    const int slot = n & 1;
    if (!__all_sync(0xffffffffu, mbar_wait(bar_item_full(slot), (n >> 1) & 1, wc))) {
      ok = false;
      return -1;
    }
    const int x = item_slot[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_item_free(slot));
    return x;
  };

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bar_kv, 1);
    for (int st = 0; st < kStages; ++st) {
      mbar_init(bar_full(st), 1);
      mbar_init(bar_empty(st), 1);
    }
    for (int sb = 0; sb < kSBuf; ++sb) {
      mbar_init(bar_sfull(sb), 1);
      mbar_init(bar_sfree(sb), 256);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_pready(i), 256);
      mbar_init(bar_pfree(i), 1);
      mbar_init(bar_item_full(i), 1);
      mbar_init(bar_item_free(i), kItemReaders);
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_sdrain, 1);
    mbar_init(bar_kvfree, 1);
    mbar_init(bar_gdrain, 1);
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

  // Barrier phases count sub-tiles (U, W) and pairs with a non-empty list (kvn, an) over
  // all items of the CTA, so every ring runs on across item boundaries.
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_map(&mq);
      tma_prefetch_map(&mdo);
      tma_prefetch_map(&mk);
      tma_prefetch_map(&mv);
    }
    bool ok = true;
    uint32_t U = 0, kvn = 0;
    int x = blockIdx.x;
    for (int n = 0; ok; ++n) {
      const int slot = n & 1;
      if (n >= 2 && !__all_sync(0xffffffffu, mbar_wait(bar_item_free(slot), ((n >> 1) - 1) & 1, wc))) {
        ok = false;
        break;
      }
      const bool done = x >= num_items;
      int xn = 0;
      if (lane == 0) {
        item_slot[slot] = done ? -1 : x;
        mbar_arrive(bar_item_full(slot));
        if (!done) xn = (int)gridDim.x + atomicAdd(a.work_ctr, 1);  // the item after this one
      }
      if (done) break;
      const int nu = item_len(x, lane == 0);
      const int nsub = nu << sub_shift;
      if (nsub > 0) {
        const int m = x / BH, bh = x - m * BH, b = bh / s.H, h = bh - b * s.H;
        const uint32_t* list = a.pair_idx + ((int64_t)bh * Tp + m) * s.Tq;
        // K, V of the previous pair are free once its S^T / dP^T MMAs completed
        if (kvn >= 1 && !__all_sync(0xffffffffu, mbar_wait(bar_kvfree, (kvn - 1) & 1, wc))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_kv, (SPLIT ? 3 : 2) * L::kKVBytes);
          for (int p = 0; p < L::kPanels; ++p)
            for (int r = 0; r < 2; ++r) {
              tma_load_4d(sbase + kOffK + p * 16384 + r * 8192, &mk, bar_kv, p * 64, m * 128 + r * 64, h, b);
              if constexpr (SPLIT)
                tma_load_4d(sbase + kOffKlo + p * 16384 + r * 8192, &mkl, bar_kv, p * 64, m * 128 + r * 64, h, b);
              tma_load_4d(sbase + kOffV + p * 16384 + r * 8192, &mv, bar_kv, p * 64, m * 128 + r * 64, h, b);
            }
        }
        ++kvn;
        uint32_t chunk = 0;  // list entries t0 + lane of the current 32-entry chunk
        for (int u = 0; u < nsub; ++u, ++U) {
          const int t = u >> sub_shift, hh = u & sub_shift;
          if ((t & 31) == 0 && hh == 0) chunk = t + lane < nu ? list[t + lane] : 0u;
          int qi = (int)(__shfl_sync(0xffffffffu, chunk, t & 31) & 0x3FFFFFFFu);
          if (qi >= s.Tq) {
            if (lane == 0) report_error(a.status, kDevErrBounds);
            qi = 0;
          }
          const int st = U & (kStages - 1);
          if (U >= kStages &&
              !__all_sync(0xffffffffu, mbar_wait(bar_empty(st), ((U >> kStShift) - 1) & 1, wc))) {
            ok = false;
            break;
          }
          if (lane == 0) {
            const uint32_t stg = sbase + kOffStage + st * kStageBytes;
            const int row = (qi << sub_shift) + hh;  // 64-row sub-tile index within the head
            mbar_arrive_expect_tx(bar_full(st), kStageTx);
            for (int p = 0; p < L::kPanels; ++p) {
              tma_load_4d(stg + kStageQ + p * 8192, &mq, bar_full(st), p * 64, row * 64, h, b);
              if constexpr (SPLIT) tma_load_4d(stg + kStageQlo + p * 8192, &mql, bar_full(st), p * 64, row * 64, h, b);
              tma_load_4d(stg + kStageDO + p * 8192, &mdo, bar_full(st), p * 64, row * 64, h, b);
            }
            bulk_load(stg + kStageStats, a.stats + ((int64_t)bh * Tsub + row) * 128, 512, bar_full(st));
          }
          __syncwarp();
        }
      }
      x = __shfl_sync(0xffffffffu, xn, 0);
    }
    // No copy may still be in flight when the CTA exits, whether the loop ran to its end or
    // gave up: U and kvn count the loads issued, so drain the last load of each stage and the
    // last K / V load (each is its barrier's latest phase).
    if (lane == 0) {
      for (uint32_t v = U > kStages ? U - kStages : 0; v < U; ++v)
        mbar_drain(bar_full(v & (kStages - 1)), (v >> kStShift) & 1, abort_flag);
      if (kvn > 0) mbar_drain(bar_kv, (kvn - 1) & 1, abort_flag);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- S^T, dP^T issuer (warp 1)
    // The whole warp runs the loop and one elected lane issues.  tcgen05.mma issue stalls
    // while the MMA queue is full, so a single issuer that also waits on barriers between
    // its groups lets the tensor pipe drain; with S/dP and dV/dK issued by two warps, one
    // of them is always queued behind the other's MMAs.
    constexpr uint32_t idS = idesc_f16_f32(128, 64, false, false);
    const uint64_t kd = smem_desc(sbase + kOffK, 16, 1024), vd = smem_desc(sbase + kOffV, 16, 1024);
    bool ok = true;
    uint32_t U = 0, kvn = 0;
    for (int n = 0; ok; ++n) {
      const int x = take_item(n, ok);
      if (x < 0) break;
      const int nsub = item_len(x, false) << sub_shift;
      if (nsub == 0) continue;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_kv, kvn & 1, wc))) {
        ok = false;
        break;
      }
      ++kvn;
      for (int u = 0; u < nsub; ++u, ++U) {
        const int st = U & (kStages - 1);
        const int sb = (int)(U % kSBuf);
        // the stage landed, and S^T / dP^T of sub-tile U - kSBuf were read out of buffer sb
        if (!__all_sync(0xffffffffu,
                        mbar_wait(bar_full(st), (U >> kStShift) & 1, wc) &&
                            (U < (uint32_t)kSBuf || mbar_wait(bar_sfree(sb), ((U / kSBuf) - 1) & 1, wc)))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t stg = sbase + kOffStage + st * kStageBytes;
        const uint64_t qd = smem_desc(stg + kStageQ, 16, 1024), dod = smem_desc(stg + kStageDO, 16, 1024);
        if (elect_one()) {
          mma_ss_kmajor<idS, 128, 64, D / 16>(tmem + C::S(sb), kd, qd);
          if constexpr (SPLIT) {
            const uint64_t kld = smem_desc(sbase + kOffKlo, 16, 1024), qld = smem_desc(stg + kStageQlo, 16, 1024);
            mma_ss_kmajor_acc<idS, 128, 64, D / 16>(tmem + C::S(sb), kd, qld);
            mma_ss_kmajor_acc<idS, 128, 64, D / 16>(tmem + C::S(sb), kld, qd);
          }
          mma_ss_kmajor<idS, 128, 64, D / 16>(tmem + C::DP(sb), vd, dod);
          umma_commit(bar_sfull(sb));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) umma_commit(bar_kvfree);
      __syncwarp();
    }
    // no MMA of this warp may still run when TMEM is released, on the abort path too
    if (elect_one()) umma_commit(bar_sdrain);
    __syncwarp();
    mbar_drain(bar_sdrain, 0, abort_flag);
  } else if (warp == 2) {
    // --------------------------------------------------------- dV, dK issuer (warp 2)
    constexpr uint32_t idG = idesc_f16_f32(128, D, false, true);
    bool ok = true;
    uint32_t W = 0;
    for (int n = 0; ok; ++n) {
      const int x = take_item(n, ok);
      if (x < 0) break;
      const int nsub = item_len(x, false) << sub_shift;
      for (int w = 0; w < nsub; ++w, ++W) {
        const int st = W & (kStages - 1), bb = W & 1;
        // P^T / dS^T of sub-tile W written (the stage's load completed long before).  For
        // the first sub-tile of a pair this also orders the overwrite of the dV, dK
        // accumulators after the previous pair's epilogue: every element-wise thread read
        // them out before it wrote this P^T / dS^T.
        if (!__all_sync(0xffffffffu, mbar_wait(bar_pready(bb), (W >> 1) & 1, wc) &&
                                         mbar_wait(bar_full(st), (W >> kStShift) & 1, wc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t stg = sbase + kOffStage + st * kStageBytes;
        // B = dO_w / Q_w read MN-major: 16 query rows (2048 B) per k-step, channel panels
        // 8 KB apart; A = P^T / dS^T of buffer bb, 8 columns (16 queries) per k-step
        const uint64_t dod = smem_desc(stg + kStageDO, 8192, 1024), qd = smem_desc(stg + kStageQ, 8192, 1024);
        if (elect_one()) {
          mma_ts_bmn<idG, 4>(tmem + C::DV, tmem + C::P + bb * 32, dod, w == 0);
          mma_ts_bmn<idG, 4>(tmem + C::DK, tmem + C::DS + bb * 32, qd, w == 0);
          umma_commit(bar_empty(st));
          umma_commit(bar_pfree(bb));
        }
        __syncwarp();
      }
      if (!ok) break;
      // the pair's S^T / dP^T MMAs all completed before its last P^T was written, so this
      // commit covers every MMA of the pair
      if (nsub > 0 && elect_one()) umma_commit(bar_drain);
      __syncwarp();
    }
    if (elect_one()) umma_commit(bar_gdrain);
    __syncwarp();
    mbar_drain(bar_gdrain, 0, abort_flag);
  } else {
    // ------------------------------------------------------------- element-wise warps
    if (s.stall_ns && blockIdx.x == 0) stall_for(s.stall_ns);  // failure-path test hook
    const int q4 = warp & 3;          // TMEM lane quarter
    const int g = (warp - 3) >> 2;    // query columns 32g .. 32g+31 of each sub-tile
    const int r = 32 * q4 + lane;     // key row of the pair
    const int half = r >> 6;          // 0: key block 2m, 1: key block 2m+1
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    const int c0 = 64 * g;            // epilogue: channels 64g .. 64g+63 of the key row
    bool ok = true;
    uint32_t U = 0, an = 0;
    for (int n = 0; ok; ++n) {
      const int x = take_item(n, ok);
      if (x < 0) break;
      const int nu = item_len(x, false);
      const int nsub = nu << sub_shift;
      const int m = x / BH, bh = x - m * BH, b = bh / s.H, h = bh - b * s.H;
      const uint32_t* list = a.pair_idx + ((int64_t)bh * Tp + m) * s.Tq;
      const int key = m * 128 + r;
      const bool key_valid = key < s.N;
      uint32_t e_next = nu > 0 ? list[0] : 0u;
      uint32_t e = 0;
      for (int u = 0; u < nsub; ++u, ++U) {
        const int t = u >> sub_shift;
        if ((u & sub_shift) == 0) {
          e = e_next;
          e_next = t + 1 < nu ? list[t + 1] : 0u;
        }
        const bool keep = ((e >> (30 + half)) & 1u) != 0;  // same for the whole warp
        const int st = U & (kStages - 1), bb = U & 1, sb = (int)(U % kSBuf);
        if (!__all_sync(0xffffffffu, mbar_wait(bar_sfull(sb), (U / kSBuf) & 1, wc) &&
                                         mbar_wait(bar_full(st), (U >> kStShift) & 1, wc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sv[32], dv[32];
        tmem_ld32(trow + C::S(sb) + 32 * g, sv);
        tmem_ld32(trow + C::DP(sb) + 32 * g, dv);
        const float4* l4 =
            reinterpret_cast<const float4*>(smem + kOffStage + st * kStageBytes + kStageStats) + 8 * g;
        const float4* d4 = l4 + 16;
        tmem_ld_wait(sv);
        tmem_ld_wait(dv);
        tc_fence_before();
        mbar_arrive(bar_sfree(sb));
        uint32_t pw[16], dw[16];
        if (keep) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 L = l4[j], D = d4[j];
            const float lv[4] = {L.x, L.y, L.z, L.w}, Dv[4] = {D.x, D.y, D.z, D.w};
            float pv[4], ds[4];
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
              const int c = 4 * j + e4;
              const float p = key_valid ? ex2(fmaf(__uint_as_float(sv[c]), a.scale_log2, -lv[e4])) : 0.f;
              pv[e4] = p;
              ds[e4] = p * (__uint_as_float(dv[c]) - Dv[e4]);
            }
            pw[2 * j] = pack_f16x2(pv[0], pv[1]);
            pw[2 * j + 1] = pack_f16x2(pv[2], pv[3]);
            dw[2 * j] = pack_f16x2(ds[0], ds[1]);
            dw[2 * j + 1] = pack_f16x2(ds[2], ds[3]);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) pw[j] = dw[j] = 0u;
        }
        // buffer bb was last read by the dV / dK MMAs of sub-tile U - 2
        if (U >= 2 && !__all_sync(0xffffffffu, mbar_wait(bar_pfree(bb), ((U >> 1) - 1) & 1, wc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st16(trow + C::P + bb * 32 + 16 * g, pw);
        tmem_st16(trow + C::DS + bb * 32 + 16 * g, dw);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_pready(bb));
      }
      if (!ok) break;
      // ---- dK, dV of the pair: thread = key row, 64 channels 64g .. 64g+63
      GT* dkp = reinterpret_cast<GT*>(a.dk) + (int64_t)b * a.g_sb + (int64_t)h * a.g_sh + (int64_t)key * a.g_sn + c0;
      GT* dvp = reinterpret_cast<GT*>(a.dv) + (int64_t)b * a.g_sb + (int64_t)h * a.g_sh + (int64_t)key * a.g_sn + c0;
      const bool store = key_valid && c0 < s.d;
      if (nsub == 0) {
        if (store) {
          zero_row64<GT>(dkp);
          zero_row64<GT>(dvp);
        }
        continue;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar_drain, an & 1, wc))) {
        ok = false;
        break;
      }
      ++an;
      tc_fence_after();
      if (c0 < D) {  // (warp-uniform; at d = 64 the second group has no channels and no columns)
        uint32_t xv[32], yv[32];
        tmem_ld32(trow + C::DK + c0, xv);
        tmem_ld32(trow + C::DK + c0 + 32, yv);
        tmem_ld_wait(xv);
        tmem_ld_wait(yv);
        if (store) store_row64<GT>(dkp, xv, yv, a.scale);
        tmem_ld32(trow + C::DV + c0, xv);
        tmem_ld32(trow + C::DV + c0 + 32, yv);
        tmem_ld_wait(xv);
        tmem_ld_wait(yv);
        if (store) store_row64<GT>(dvp, xv, yv, 1.f);
      }
      tc_fence_before();
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

// Union of the column lists of key blocks 2m and 2m+1, one warp per pair: the query blocks
// are marked in two bitmaps and read back in ascending order, each entry tagged with the
// blocks that keep it (bit 30: block 2m, bit 31: block 2m+1).
constexpr int kUnionWarps = 4;
constexpr int kMaxTqWords = 240;  // Tq <= 7680

__global__ void __launch_bounds__(32 * kUnionWarps) pair_union_kernel(const int32_t* __restrict__ col_cnt,
                                                                     const int32_t* __restrict__ col_idx, ShapeArgs s,
                                                                     int32_t* __restrict__ pair_cnt,
                                                                     uint32_t* __restrict__ pair_idx,
                                                                     int* __restrict__ work_ctr,
                                                                     unsigned* status) {
  __shared__ uint32_t bits[kUnionWarps][2][kMaxTqWords];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the work counters of the two persistent backward kernels that run after this pass
  if (blockIdx.x == 0 && threadIdx.x < kBwdWorkCounters) work_ctr[threadIdx.x] = 0;
  const int Tp = (s.Tk + 1) >> 1;
  const int64_t pid = (int64_t)blockIdx.x * kUnionWarps + warp;
  if (pid >= (int64_t)s.B * s.H * Tp) return;  // whole warps only; no block-wide barrier below
  const int64_t bh = pid / Tp;
  const int m = (int)(pid - bh * Tp);
  const int nw = (s.Tq + 31) >> 5;
  for (int w = lane; w < nw; w += 32) bits[warp][0][w] = bits[warp][1][w] = 0u;
  __syncwarp();
  bool bad = false;
  for (int half = 0; half < 2; ++half) {
    const int j = 2 * m + half;
    if (j >= s.Tk) break;
    const int64_t col = bh * s.Tk + j;
    int cnt = col_cnt[col];
    if (cnt < 0 || cnt > s.Tq) {
      bad = true;
      cnt = cnt < 0 ? 0 : s.Tq;
    }
    const int32_t* li = col_idx + col * s.Tq;
    for (int i = lane; i < cnt; i += 32) {
      const int qi = li[i];
      if (qi < 0 || qi >= s.Tq) {
        bad = true;
        continue;
      }
      atomicOr(&bits[warp][half][qi >> 5], 1u << (qi & 31));
    }
  }
  __syncwarp();
  uint32_t* out = pair_idx + pid * s.Tq;
  int base = 0;
  for (int w0 = 0; w0 < nw; w0 += 32) {
    const int w = w0 + lane;
    const uint32_t x = w < nw ? bits[warp][0][w] : 0u, y = w < nw ? bits[warp][1][w] : 0u;
    uint32_t un = x | y;
    const int n = __popc(un);
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int pos = base + incl - n;
    while (un) {
      const int bit = __ffs(un) - 1;
      un &= un - 1;
      out[pos++] = (uint32_t)(w * 32 + bit) | (((x >> bit) & 1u) << 30) | (((y >> bit) & 1u) << 31);
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) pair_cnt[pid] = base;
  if (bad) report_error(status, kDevErrBounds);
}

template <typename GT, bool SPLIT, int D>
cudaError_t launch_bwd_t(const ShapeArgs& s, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mdo, const CUtensorMap& mql, const CUtensorMap& mkl, const BwdArgs& a,
                         cudaStream_t st) {
  constexpr int kSmemBytes = DkdvSmem<SPLIT, D>::kSmemBytes;
  const long long pairs = (long long)s.B * s.H * ((s.Tk + 1) / 2);
  prof_start(st, kBwdPairs);
  pair_union_kernel<<<(unsigned)((pairs + kUnionWarps - 1) / kUnionWarps), 32 * kUnionWarps, 0, st>>>(
      a.col_cnt, a.col_idx, s, a.pair_cnt, a.pair_idx, a.work_ctr, a.status);
  prof_stop(st, kBwdPairs);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kern = attn_bwd_dkdv_kernel<GT, SPLIT, D>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long grid = pairs < sms ? pairs : sms;  // persistent: one CTA per SM
  prof_start(st, kAttnBwd);
  kern<<<(unsigned)grid, kThreads, kSmemBytes, st>>>(mq, mk, mv, mdo, mql, mkl, s, a);
  prof_stop(st, kAttnBwd);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_pair_entries(const ShapeArgs& s) { return (size_t)s.B * s.H * ((s.Tk + 1) / 2) * s.Tq; }

cudaError_t launch_attn_bwd(const ShapeArgs& s, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            const CUtensorMap& mdo, const CUtensorMap* mql, const CUtensorMap* mkl, const BwdArgs& a,
                            cudaStream_t st) {
  if (s.Tq > 32 * kMaxTqWords || (long long)s.B * s.H * ((s.Tk + 1) / 2) > INT32_MAX) return cudaErrorInvalidValue;
  // fp32 calls take the split S product
  if (s.dtype != 0 && (!mql || !mkl)) return cudaErrorInvalidValue;
  if (s.d == 128)
    return s.dtype == 0 ? launch_bwd_t<__nv_bfloat16, false, 128>(s, mq, mk, mv, mdo, mq, mk, a, st)
                        : launch_bwd_t<float, true, 128>(s, mq, mk, mv, mdo, *mql, *mkl, a, st);
  return s.dtype == 0 ? launch_bwd_t<__nv_bfloat16, false, 64>(s, mq, mk, mv, mdo, mq, mk, a, st)
                      : launch_bwd_t<float, true, 64>(s, mq, mk, mv, mdo, *mql, *mkl, a, st);
}

}  // namespace sa2
