// Hybrid Top-k + Top-p block mask on sm_103a.
//
// gist.science explainer of SpargeAttention2 (arXiv 2602.13515), section 2.A: the rows of
// the block-pooled attention map P-bar are masked with the union of their Top-k% and
// Top-p% sets; section 1 defines Top-k (the k largest entries) and Top-p (the smallest set
// whose cumulative probability reaches p).
//
// Four kernels:
//   pool_tc_kernel   (bf16 inputs) persistent; 128-token chunks of Q and K streamed by TMA
//                    and summed per 64-token half on the tensor cores (D = X^T Sel with a 0/1
//                    selector), the block means written as a TF32 pair hi + lo, row-major
//                    [2][B*H][T][d].  The HBM-bound part.
//   pool_kernel      (fp32 inputs) the same with one warp per chunk: plain streaming loads
//                    and fp32 sums in token order.
//   score_tc_kernel  pooled scores S-bar = q-bar k-bar^T / sqrt(d) of a 128-row x 128-key
//                    tile on the tensor cores (tcgen05, kind::tf32) as the three products
//                    hi.hi + hi.lo + lo.hi -- about fp32 accuracy -- accumulated in tensor
//                    memory and written to a scratch row in a lane-friendly permuted order.
//   select_kernel    one warp per row: row softmax in fp32, the hybrid selection with the
//                    mass in 2^-60 fixed point (a warp-wide sort of each lane's largest
//                    keys, or a bisection on the fp32 bit patterns of P-bar), and the emit
//                    of the row list, the u8 mask and the row's kept bits.
//   csc_kernel       transposes the kept bits into the per-key-block lists (ascending).
// The heads run in chunks: the caller's stream pools chunk after chunk while kChains more
// streams take the scores, the selection and the column lists of successive chunks in turn,
// each with its own scratch buffer, which stays mostly in L2 between the kernels of a chain.
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
constexpr int kScoreKeys = 128;             // MMA N: key blocks per tile
constexpr int kRowPad = 256;                // score rows are padded to a multiple of this
constexpr int kSelectThreads = 256;
constexpr int kChains = 2;                       // head chunks whose score / select / lists run at once
// bytes of the kChains head-chunk buffers: 64 MB (config 3: five chunks of up to 9 heads) measured
// 0.44 ms for the whole build against 0.49 ms at 32 MB (ten chunks of 4), 0.55 ms at 16 MB and
// 0.45 ms at 96 or 128 MB
constexpr size_t kScoreChunkBudget = 64u << 20;

// ---------------------------------------------------------------------------- helpers

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

__device__ __forceinline__ float tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
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
  int* ctr;     // chunk counter of this launch (zeroed on the stream before it; TC pooling)
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

// ------------------------------------------------------------------- pooling on the TC

// Pooling of bf16 Q and K as a product on the tensor cores.  A 128-token chunk X
// [tokens x d channels] lands in shared memory by TMA (64-channel panels, 128-byte swizzle)
// and is read as the MN-major A operand of D = X^T Sel: M = 128 channel rows (a d = 64 chunk
// leaves the upper 64 rows unused), K = 128 tokens, N = 16 columns, where the selector Sel
// (K-major, 4 KB) has column 0 = ones on tokens 0..63 and column 1 = ones on tokens
// 64..127.  So D[c][0], D[c][1] are the sums of channel c over the two 64-token halves:
// products by 1 are exact and the sums accumulate in fp32.  The SMs' ALUs stay free for
// the kernels that run beside the pooling.
// Persistent: the CTAs take the chunks of the head chunk (Q chunks, then K chunks, head by
// head) from a counter, so a CTA that starts late (its SM busy with the kernels beside the
// pooling) takes fewer.  Warp 0 fetches them and streams them through a kPoolStages-deep
// ring, publishing each chunk's index in a ring of item slots that the other roles read in
// order; warp 1 owns tensor memory (two 16-column accumulators) and issues one 8-k-step MMA
// per chunk, warps 2..5 read the accumulators out (thread = channel = TMEM lane), form the
// block means (fp32, divided by the valid tokens) and store them as TF32 pairs, a warp's 32
// channels as one 128-byte row segment.
constexpr int kPoolStages = 2;
constexpr int kPoolStageBytes = 128 * 128 * 2;  // two 64-channel panels of 128 tokens x 128 B
constexpr int kPoolSelBytes = 2 * 16 * 128;     // Sel: 16 rows x 2 panels of 64 tokens
constexpr int kPoolTcThreads = 192;
constexpr int kPoolItems = 8;  // item slots in flight (>= stages + accumulators)
constexpr int kPoolTcSmem = kPoolStages * kPoolStageBytes + kPoolSelBytes + 512 + 1024;

__device__ __forceinline__ void tmem_ld2(uint32_t taddr, uint32_t& r0, uint32_t& r1) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait2(uint32_t& r0, uint32_t& r1) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r0), "+r"(r1)::"memory");
}

template <int D>
__global__ void __launch_bounds__(kPoolTcThreads, 1)
    pool_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk, ShapeArgs s,
                   PoolArgs a, unsigned* status) {
  constexpr int kPanels = D / 64;
  constexpr uint32_t kCols = 32;  // two accumulators of 16 columns
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t ssel = sbase + kPoolStages * kPoolStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPoolStages * kPoolStageBytes + kPoolSelBytes);
  auto bar_full = [&](int st) { return smem_u32(&bars[st]); };
  auto bar_empty = [&](int st) { return smem_u32(&bars[kPoolStages + st]); };
  auto bar_acc = [&](int b) { return smem_u32(&bars[2 * kPoolStages + b]); };          // accumulator b complete
  auto bar_accfree = [&](int b) { return smem_u32(&bars[2 * kPoolStages + 2 + b]); };  // ... read out
  const uint32_t bar_drain = smem_u32(&bars[2 * kPoolStages + 4]);
  auto bar_item_full = [&](int i) { return smem_u32(&bars[2 * kPoolStages + 5 + i]); };  // slot i written
  auto bar_item_free = [&](int i) { return smem_u32(&bars[2 * kPoolStages + 5 + kPoolItems + i]); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[2 * kPoolStages + 5 + 2 * kPoolItems]);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&bars[2 * kPoolStages + 6 + 2 * kPoolItems]);
  volatile int* item_slot = reinterpret_cast<volatile int*>(&bars[2 * kPoolStages + 7 + 2 * kPoolItems]);
  const WaitCtl wc{abort_flag, s.wait_ns};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nc = (s.N + kChunkTokens - 1) / kChunkTokens;
  const int items = a.nbh * 2 * nc;
  // a consumer warp takes item n from its slot and hands the slot back; -1 ends the loop
  auto take_item = [&](uint32_t n, bool& ok) {
    const int slot = n % kPoolItems;
    if (!__all_sync(0xffffffffu, mbar_wait(bar_item_full(slot), (n / kPoolItems) & 1, wc))) {
      ok = false;
      return -1;
    }
    const int x = item_slot[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_item_free(slot));
    return x;
  };
  // the selector: row j of panel p is 128 bytes of bf16 ones when token half p is column j
  // (j = p for j < 2), zeros otherwise; rows of ones or zeros are swizzle-invariant
  {
    uint32_t* sel = reinterpret_cast<uint32_t*>(smem + kPoolStages * kPoolStageBytes);
    for (int i = tid; i < kPoolSelBytes / 4; i += kPoolTcThreads) {
      const int p = i / (16 * 32), row = (i / 32) % 16;
      sel[i] = row == p ? 0x3F803F80u : 0u;
    }
  }
  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kPoolStages; ++i) {
      mbar_init(bar_full(i), 1);
      mbar_init(bar_empty(i), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_acc(b), 1);
      mbar_init(bar_accfree(b), 4);  // one arrival per epilogue warp
    }
    for (int i = 0; i < kPoolItems; ++i) {
      mbar_init(bar_item_full(i), 1);
      mbar_init(bar_item_free(i), 5);  // the MMA warp and the four epilogue warps
    }
    mbar_init(bar_drain, 1);
    fence_barrier_init();
  }
  fence_proxy_async();  // the selector's generic stores, before the tensor core reads them
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_map(&mq);
      tma_prefetch_map(&mk);
      const uint64_t stream_policy = policy_evict_first();
      uint32_t n = 0, loads = 0;  // items published, chunk loads issued
      for (bool ok = true; ok; ++n) {
        const int slot = n % kPoolItems;
        if (n >= kPoolItems && !mbar_wait(bar_item_free(slot), ((n / kPoolItems) - 1) & 1, wc)) break;
        const int x = atomicAdd(a.ctr, 1);
        const bool done = x >= items;
        item_slot[slot] = done ? -1 : x;
        mbar_arrive(bar_item_full(slot));
        if (done) break;
        const int z = x / (2 * nc), r2 = x - z * 2 * nc;
        const bool isk = r2 >= nc;
        const int c = isk ? r2 - nc : r2;
        const int bh = a.bh0 + z, b = bh / s.H, h = bh - b * s.H;
        const int st = n % kPoolStages;
        if (n >= kPoolStages && !mbar_wait(bar_empty(st), ((n / kPoolStages) - 1) & 1, wc)) break;
        mbar_arrive_expect_tx(bar_full(st), kPanels * 16384);
        // Q and K are read once: evict them first, so that the chains' score rows and kept
        // bits stay in L2
        for (int p = 0; p < kPanels; ++p)
          tma_load_4d_hint(sbase + st * kPoolStageBytes + p * 16384, isk ? &mk : &mq, bar_full(st), p * 64,
                           c * kChunkTokens, h, b, stream_policy);
        ++loads;
      }
      // no copy may still be in flight when the CTA exits
      for (uint32_t v = loads > kPoolStages ? loads - kPoolStages : 0; v < loads; ++v)
        mbar_drain(bar_full(v % kPoolStages), (v / kPoolStages) & 1, abort_flag);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA issuer
    constexpr uint32_t idP = idesc_bf16_f32(128, 16, true, false);
    // Sel as the K-major B operand (16 rows); X as the MN-major A operand: M = 128 channels
    // (64-channel groups 16 KB apart), 16 tokens (2048 B) per k-step
    const uint64_t seld = smem_desc(ssel, 16, 1024);
    bool ok = true;
    for (uint32_t n = 0; ok; ++n) {
      if (take_item(n, ok) < 0) break;
      const int st = n % kPoolStages, ab = n & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_full(st), (n / kPoolStages) & 1, wc) &&
                                       (n < 2 || mbar_wait(bar_accfree(ab), ((n >> 1) - 1) & 1, wc))))
        break;
      tc_fence_after();
      const uint64_t xd = smem_desc(sbase + st * kPoolStageBytes, 16384, 1024);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + ab * 16, xd + (uint64_t)(kk * 128), seld + kmajor_kstep(kk, 16), idP, kk > 0 ? 1u : 0u);
        umma_commit(bar_empty(st));
        umma_commit(bar_acc(ab));
      }
      __syncwarp();
    }
    // every MMA completed (on the abort path too) before tensor memory is freed
    if (elect_one()) umma_commit(bar_drain);
    __syncwarp();
    mbar_drain(bar_drain, 0, abort_flag);
  } else {
    // ------------------------------------------ epilogue: thread = channel = TMEM lane
    const int q4 = warp & 3;  // warps 2..5: lane quarters 2, 3, 0, 1
    const int ch = 32 * q4 + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    bool ok = true;
    for (uint32_t n = 0; ok; ++n) {
      const int x = take_item(n, ok);
      if (x < 0) break;
      const int ab = n & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_acc(ab), (n >> 1) & 1, wc))) break;
      tc_fence_after();
      uint32_t u0 = 0, u1 = 0;
      tmem_ld2(trow + ab * 16, u0, u1);
      tmem_ld_wait2(u0, u1);
      // accumulator ab read out: the MMA of chunk n + 2 may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_accfree(ab));
      if (ch >= D) continue;  // (d = 64: the upper lanes hold no channel)
      const int z = x / (2 * nc), r2 = x - z * 2 * nc;
      const bool isk = r2 >= nc;
      const int c = isk ? r2 - nc : r2;
      const int bh = a.bh0 + z;
      const int bsz = isk ? s.bk : s.bq;
      const int nT = isk ? s.Tk : s.Tq;
      float* out = isk ? a.kbar : a.qbar;
      const size_t plane = (size_t)s.B * s.H * nT * s.d;
      const float s0 = __uint_as_float(u0), s1 = __uint_as_float(u1);
      const int nblk = bsz == 128 ? 1 : 2;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (u >= nblk) break;
        const int blk = c * nblk + u;
        if (blk >= nT) break;
        const int valid = min(bsz, s.N - blk * bsz);
        const float inv = 1.f / static_cast<float>(valid);
        // a block of 128 tokens spans both halves of the chunk
        const float sum = nblk == 1 ? s0 + s1 : (u == 0 ? s0 : s1);
        const float mean = sum * inv;
        const float hi = tf32_rna(mean);
        float* dst = out + ((size_t)bh * nT + blk) * s.d + ch;
        dst[0] = hi;
        dst[plane] = tf32_rna(mean - hi);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) report_error(status, kDevErrTimeout);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// ------------------------------------------------------------------------ TC scores

// One tile: 128 query blocks (TMEM lanes) x 128 key blocks (columns) of one head.  The
// channels arrive in panels of 32 (128 bytes, the TF32 K-major 128-byte-swizzled layout),
// two panels in flight: per panel the hi and lo parts of both operands (64 KB, so that a
// pooling CTA fits beside the two stages on an SM).
// S = Ahi Bhi + Ahi Blo + Alo Bhi over 8-channel k-steps; the epilogue scales by 1/sqrt(d)
// and writes the tile rows to the scratch [chunk heads][Tq_pad][Tk_pad].
constexpr int kAPanelBytes = kScoreRows * 128;  // 16 KB
constexpr int kBPanelBytes = kScoreKeys * 128;  // 16 KB
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
// stopping between tiles, warp 1 owns tensor memory (two 128-column accumulators) and issues
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
      // rows are stored permuted per 128-key chunk (key 128 c + 32 i + l at 128 c + 4 l + i),
      // keys past Tk as -inf
#pragma unroll 1
      for (int g = 0; g < kScoreKeys; g += 128) {
        uint32_t r[4][32];
#pragma unroll
        for (int i = 0; i < 4; ++i) tmem_ld32(trow + tb * kScoreKeys + g + 32 * i, r[i]);
        tmem_ld_wait(r[0]);
        tmem_ld_wait(r[1]);
        tmem_ld_wait(r[2]);
        tmem_ld_wait(r[3]);
        const int j0 = kc * kScoreKeys + g;
#pragma unroll
        for (int l = 0; l < 32; ++l) {
          float v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            v[i] = j0 + 32 * i + l < s.Tk ? __uint_as_float(r[i][l]) * a.inv_sqrt_d : -INFINITY;
          reinterpret_cast<float4*>(dst + g)[l] = make_float4(v[0], v[1], v[2], v[3]);
        }
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

// Coarse mass floor(P * 2^31) of a key, equal to mass_fix(key) >> 29: the scaling by 2^31 is
// exact in fp32 and the conversion rounds down.
__device__ __forceinline__ uint32_t mass_c31(uint32_t key) {
  return __float2uint_rd(__uint_as_float(key) * 2147483648.0f);
}

// Scratch rows of scores (and, for rows in memory, of keys) are stored permuted within each
// 128-entry chunk: entry 128 c + 32 i + l sits at position 128 c + 4 l + i, so that one
// 16-byte load gives lane l the entries l, l + 32, l + 64, l + 96 of chunk c.  A lane then
// holds every 32nd entry of the row (neighbouring key blocks sit in neighbouring lanes), and
// a ballot over the lanes for a fixed i covers 32 consecutive entries.  Positions past Tk
// hold -inf scores, hence zero keys.

// The hybrid selection of one row (one warp) keeps every key > t and the first `take` keys
// == t in index order, where t is the largest value with count(>= t) >= K and
// mass(>= t) >= p; keep_all when the row's mass never reaches p.  Masses are compared in
// 2^-60 fixed point, exactly.

// `take` from the count and the exact mass of the keys strictly above t.
__device__ __forceinline__ int ties_to_take(const SelectArgs& sel, uint32_t t, uint32_t cnt_gt,
                                            unsigned long long mass_gt) {
  const int r_k = sel.K - (int)cnt_gt;
  int r_m = 0;
  if (sel.p_mode == 0 && mass_gt < sel.p_fix) {
    const unsigned long long vfix = mass_fix(t);
    r_m = vfix ? (int)((sel.p_fix - mass_gt + vfix - 1) / vfix) : 0;
  }
  return max(max(r_k, r_m), 0);
}

// Whether the n keys in memory that are >= t number at least K (when with_count) and reach
// the mass p (when with_mass).  Each lane sums a coarse 32-bit mass per key,
// c = floor(P * 2^31); the row's coarse sum S stays below 2^32, and over m keys the exact sum
// lies in [S 2^29, (S + m) 2^29).  The test against p is decided by that bracket unless p
// falls inside it; only then is the exact sum formed.
__device__ __forceinline__ bool keys_reach(const uint32_t* keys, int n, uint32_t t, const SelectArgs& sel,
                                           bool with_count, bool with_mass) {
  const int lane = threadIdx.x & 31;
  uint32_t c = 0, S = 0;
  for (int j = lane; j < n; j += 32) {
    const uint32_t key = keys[j];
    const bool in = key >= t;
    c += in ? 1u : 0u;
    S += in ? mass_c31(key) : 0u;
  }
  c = __reduce_add_sync(0xffffffffu, c);
  if (with_count && c < (uint32_t)sel.K) return false;
  if (!with_mass) return true;
  const unsigned long long St = __reduce_add_sync(0xffffffffu, S);
  if ((St << 29) >= sel.p_fix) return true;
  if (((St + c) << 29) <= sel.p_fix) return false;
  unsigned long long m = 0;
  for (int j = lane; j < n; j += 32) {
    const uint32_t key = keys[j];
    m += key >= t ? mass_fix(key) : 0ull;
  }
  return warp_sum_u64(m) >= sel.p_fix;
}

// The selection by bisection over the fp32 bit patterns, with the row's n keys in memory
// (shared or global; padding keys 0).  Sets keep_all when the row's mass never reaches p,
// else t, take and n_eq (the number of keys == t, padding zeros included when t = 0).
__device__ __forceinline__ void select_in_memory(const uint32_t* keys, int n, const SelectArgs& sel, bool& keep_all,
                                                 uint32_t& t, int& take, int& n_eq) {
  const bool use_mass = sel.p_mode == 0;
  // every real key is >= 1 (P > 0 after the softmax; a key of 0 is padding or an
  // underflowed probability, whose mass is 0 as well), so every tested t is >= 1
  if (use_mass && !keys_reach(keys, n, 1u, sel, false, true)) {
    keep_all = true;
    return;
  }
  uint32_t lo = 0, hi = 0x3F800001u;
  while (hi - lo > 1) {
    const uint32_t mid = lo + (hi - lo) / 2;
    if (keys_reach(keys, n, mid, sel, true, use_mass))
      lo = mid;
    else
      hi = mid;
  }
  t = lo;
  const Predicate gt = count_mass(keys, n, t, true);
  const Predicate ge = count_mass(keys, n, t, false);
  n_eq = (int)(ge.cnt - gt.cnt);
  take = ties_to_take(sel, t, gt.cnt, gt.mass);
}

// Sorting network for N keys, descending: K. E. Batcher's odd-even merge sort (1968) for the
// next power of two P2 >= N inputs, generated at compile time, keeping only the comparators
// whose two positions are below N (positions N..P2-1 would hold zeros, the minimum, which no
// comparator moves).  sort_net<N>(idx, second) is comparator idx's first or second position,
// or the number of comparators when idx < 0; evaluated by the compiler only.
template <int N>
__host__ __device__ constexpr int sort_net(int idx, bool second) {
  int P2 = 1;
  while (P2 < N) P2 *= 2;
  int n = 0;
  for (int p = 1; p < P2; p *= 2)
    for (int k = p; k >= 1; k /= 2)
      for (int j = k % p; j + k < P2; j += 2 * k)
        for (int i = 0; i < k && i + j + k < P2; ++i)
          if ((i + j) / (2 * p) == (i + j + k) / (2 * p) && i + j + k < N) {
            if (n == idx) return second ? i + j + k : i + j;
            ++n;
          }
  return n;
}

// Comparator C of the N-key network applied to k[O .. O + N).
template <int N, int O, int C, int L>
__device__ __forceinline__ void sort_cmp(uint32_t (&k)[L]) {
  constexpr int a = O + sort_net<N>(C, false), b = O + sort_net<N>(C, true);
  const uint32_t x = k[a], y = k[b];
  k[a] = max(x, y);
  k[b] = min(x, y);
}

template <int N, int O, int L, int... C>
__device__ __forceinline__ void sort_all(uint32_t (&k)[L], std::integer_sequence<int, C...>) {
  (sort_cmp<N, O, C>(k), ...);
}

// Sorts k[O .. O + N) descending.
template <int N, int O = 0, int L>
__device__ __forceinline__ void sort_desc(uint32_t (&k)[L]) {
  static_assert(O + N <= L, "slice out of range");
  sort_all<N, O>(k, std::make_integer_sequence<int, sort_net<N>(-1, false)>{});
}

template <int L, int... G>
__device__ __forceinline__ void sort_groups8(uint32_t (&k)[L], std::integer_sequence<int, G...>) {
  (sort_desc<8, 8 * G>(k), ...);
}

// Leaves the 8 largest of the lane's KPL keys in k[0..7], descending, and returns the
// largest of the others.  Each group of 8 is sorted; then group g is folded into group 0 by
// comparing k[i] with the group's (7 - i)-th key: the larger of each pair are the 8 largest
// of the 16 (in bitonic order, sorted by three half-cleaner steps), the smaller are out of
// the running for good, and the largest of those is tracked.
template <int KPL>
__device__ __forceinline__ uint32_t top8_desc(uint32_t (&k)[KPL]) {
  static_assert(KPL % 8 == 0 && KPL >= 16, "groups of 8");
  sort_groups8(k, std::make_integer_sequence<int, KPL / 8>{});
  uint32_t H = 0;
#pragma unroll
  for (int g = 1; g < KPL / 8; ++g) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t x = k[i], y = k[8 * g + 7 - i];
      k[i] = max(x, y);
      H = max(H, min(x, y));
    }
#pragma unroll
    for (int dist = 4; dist >= 1; dist /= 2)
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if ((i & dist) == 0) {
          const uint32_t x = k[i], y = k[i + dist];
          k[i] = max(x, y);
          k[i + dist] = min(x, y);
        }
  }
  return H;
}

// Bitonic merge across the warp: on entry every lane holds M keys in descending order in
// k[0..M-1]; on exit the 32 M keys are in descending order lane after lane (lane 0 holds
// the M largest).  Level m merges pairs of sorted runs of 2^m lanes: the first step
// compares each key of the first run with its mirror image in the second (lane ^ (2^(m+1) -
// 1), position M - 1 - r), which leaves two bitonic halves with every key of the first
// above every key of the second; half-cleaners at lane distances 2^(m-1) .. 1 and then at
// register distances M/2 .. 1 sort each half.
template <int M, int N>
__device__ __forceinline__ void warp_merge_runs(uint32_t (&k)[N], int lane) {
#pragma unroll
  for (int m = 0; m < 5; ++m) {
    {
      const bool upper = (lane >> m) & 1;
      uint32_t o[M];
#pragma unroll
      for (int r = 0; r < M; ++r) o[r] = __shfl_xor_sync(0xffffffffu, k[M - 1 - r], (2 << m) - 1);
#pragma unroll
      for (int r = 0; r < M; ++r) k[r] = upper ? min(k[r], o[r]) : max(k[r], o[r]);
    }
#pragma unroll
    for (int d = m - 1; d >= 0; --d) {
      const bool upper = (lane >> d) & 1;
#pragma unroll
      for (int r = 0; r < M; ++r) {
        const uint32_t o = __shfl_xor_sync(0xffffffffu, k[r], 1 << d);
        k[r] = upper ? min(k[r], o) : max(k[r], o);
      }
    }
#pragma unroll
    for (int dist = M / 2; dist >= 1; dist /= 2)
#pragma unroll
      for (int r = 0; r < M; ++r)
        if ((r & dist) == 0) {
          const uint32_t x = k[r], y = k[r + dist];
          k[r] = max(x, y);
          k[r + dist] = min(x, y);
        }
  }
}

// The selection by sorting.  The M0 largest keys of every lane (or all of them when a lane
// holds fewer) are the candidates, merged into one descending order across the warp.
// Position e of that order has count e + 1 and the exact prefix mass of positions 0..e
// (lane-local prefix plus a warp scan); the first position where count >= K and mass >= p
// holds t.  That order is the row's own order for every value above H, the largest key left
// out of the candidates, so the result is the row's whenever t > H (or no key was left
// out).  Returns false when it is not (or when no position qualifies): a second pass with
// more candidates, or the bisection, then decides the row.  k is clobbered.
template <int KPL, int M0>
__device__ __forceinline__ bool select_by_sort(uint32_t (&k)[KPL], const SelectArgs& sel, uint32_t& t, int& take,
                                               int& n_eq) {
  constexpr int M = KPL < M0 ? KPL : M0;
  const int lane = threadIdx.x & 31;
  const bool use_mass = sel.p_mode == 0;
  uint32_t H = 0;
  if constexpr (KPL == M) {
    sort_desc<KPL>(k);
  } else if constexpr (M == 8) {
    H = __reduce_max_sync(0xffffffffu, top8_desc(k));
  } else {
    sort_desc<KPL>(k);
    H = __reduce_max_sync(0xffffffffu, k[M]);
  }
  warp_merge_runs<M>(k, lane);
  unsigned long long lp[M];  // lane-local inclusive prefix masses
  unsigned long long run = 0;
#pragma unroll
  for (int r = 0; r < M; ++r) {
    run += mass_fix(k[r]);
    lp[r] = run;
  }
  unsigned long long base = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long v = __shfl_up_sync(0xffffffffu, base, o);
    if (lane >= o) base += v;
  }
  base -= run;  // mass of the lanes before this one
  const int e0 = lane * M;
  int first = M;
#pragma unroll
  for (int r = M - 1; r >= 0; --r) {
    const bool ok = e0 + r + 1 >= sel.K && (!use_mass || base + lp[r] >= sel.p_fix);
    first = ok ? r : first;
  }
  const unsigned found = __ballot_sync(0xffffffffu, first < M);
  if (found == 0u) return false;
  uint32_t tv = 0;
#pragma unroll
  for (int r = 0; r < M; ++r) tv = r == first ? k[r] : tv;
  t = __shfl_sync(0xffffffffu, tv, __ffs(found) - 1);
  if (KPL > M && t <= H) return false;
  uint32_t c = 0, ce = 0;
#pragma unroll
  for (int r = 0; r < M; ++r) {
    c += k[r] > t ? 1u : 0u;
    ce += k[r] == t ? 1u : 0u;
  }
  const uint32_t cnt_gt = __reduce_add_sync(0xffffffffu, c);
  n_eq = (int)__reduce_add_sync(0xffffffffu, ce);
  unsigned long long mass_gt = 0;
  if (cnt_gt > 0) {  // the prefix mass at position cnt_gt - 1
    const int pos = (int)cnt_gt - 1, rr = pos % M;
    unsigned long long v = 0;
#pragma unroll
    for (int r = 0; r < M; ++r) v = r == rr ? lp[r] : v;
    mass_gt = __shfl_sync(0xffffffffu, base + v, pos / M);
  }
  take = ties_to_take(sel, t, cnt_gt, mass_gt);
  return true;
}

struct SelArgs {
  float* sbar;     // permuted score rows of the head chunk; rows past 32 * kMaxKeysPerLane
                   // keys are overwritten in place by their keys
  uint32_t* bits;  // kept bits of the head chunk's rows, [nbh][Tq][W]
  int bh0, nbh;
  int tq_pad, tk_pad;
  int W;           // 32-bit words per row: ceil(Tk / 32)
};

// Writes a row's outputs from its keys in the permuted order (one 16-byte read per lane per
// 128-entry chunk): for each quarter i of the chunk the 32 lanes hold 32 consecutive entries,
// so one ballot gives the kept bits of a 32-entry word and compacts the ascending kept
// indices; the u8 mask and P-bar (when asked) are written entry by entry.
__device__ __forceinline__ void emit_row(const uint4* keys4, int Tk, const MaskOut& out, int64_t rowid,
                                         uint32_t* bits_row, int W, bool keep_all, bool keep_none, bool tie_order,
                                         uint32_t t, int take) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  int kept = 0, ties_seen = 0;
  int32_t* ridx = out.row_idx + rowid * Tk;
  uint8_t* mrow = out.mask ? out.mask + rowid * Tk : nullptr;
  float* prow = out.pooled_p ? out.pooled_p + rowid * Tk : nullptr;
  const int nch = (Tk + 127) / 128;
  for (int c = 0; c < nch; ++c) {
    const uint4 kv = keys4[c * 32 + lane];
    const uint32_t key[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = c * 128 + 32 * i + lane;
      const bool valid = j < Tk;
      bool keep;
      if (keep_all || keep_none || !tie_order) {
        keep = valid && (keep_all || (!keep_none && key[i] >= t));
      } else {  // only `take` of the keys == t, in ascending index order
        const bool eq = valid && key[i] == t;
        const unsigned eqm = __ballot_sync(0xffffffffu, eq);
        keep = valid && (key[i] > t || (eq && ties_seen + __popc(eqm & lt) < take));
        ties_seen += __popc(eqm);
      }
      const unsigned km = __ballot_sync(0xffffffffu, keep);
      if (keep) ridx[kept + __popc(km & lt)] = j;
      kept += __popc(km);
      if (lane == 0 && 4 * c + i < W) bits_row[4 * c + i] = km;
      if (valid) {
        if (mrow) mrow[j] = keep ? 1 : 0;
        if (prow) prow[j] = __uint_as_float(key[i]);
      }
    }
  }
  if (lane == 0) out.row_cnt[rowid] = kept;
}

// Rows of up to 32 * KPL keys: one warp per row, the warps of the grid striding over the
// rows of the head chunk.  Row softmax in fp32 (exponentials by the ex2 instruction, one
// correctly rounded reciprocal of the row sum), the selection by sorting (the bisection
// where that cannot decide), and the emit from the keys parked in shared memory.
constexpr int kSelectWarps = kSelectThreads / 32;
constexpr int kMaxKeysPerLane = 40;

template <int KPL>
constexpr int select_smem_bytes() {
  return kSelectWarps * KPL * 32 * 4;
}

template <int KPL>
__global__ void __launch_bounds__(kSelectThreads, KPL >= 16 ? 3 : 4)
    select_kernel(ShapeArgs s, SelectArgs sel, SelArgs a, MaskOut out) {
  extern __shared__ __align__(16) uint4 sel_smem4[];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  uint4* row_keys = sel_smem4 + wib * (KPL / 4) * 32;
  const int Tk = s.Tk;
  const long long rows = (long long)a.nbh * s.Tq;
  const long long nwarps = (long long)gridDim.x * kSelectWarps;
  for (long long gw = (long long)blockIdx.x * kSelectWarps + wib; gw < rows; gw += nwarps) {
    const int z = (int)(gw / s.Tq), i = (int)(gw - (long long)z * s.Tq);
    const float4* row4 = reinterpret_cast<const float4*>(a.sbar + ((size_t)z * a.tq_pad + i) * a.tk_pad);
    const int64_t rowid = (int64_t)(a.bh0 + z) * s.Tq + i;
    uint32_t k[KPL];
    {
      float v[KPL];
#pragma unroll
      for (int c = 0; c < KPL / 4; ++c) {
        const float4 x = row4[c * 32 + lane];
        v[4 * c] = x.x;
        v[4 * c + 1] = x.y;
        v[4 * c + 2] = x.z;
        v[4 * c + 3] = x.w;
      }
      // the row maximum and the row sum as 4-way trees (short dependency chains)
      float m4[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
      for (int r = 4; r < KPL; ++r) m4[r & 3] = fmaxf(m4[r & 3], v[r]);
      float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float mb = mx * kLog2e;
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int r = 0; r < KPL; ++r) {
        v[r] = ex2_approx(fmaf(v[r], kLog2e, -mb));  // -inf padding: 0
        s4[r & 3] += v[r];
      }
      float sum = (s4[0] + s4[1]) + (s4[2] + s4[3]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      const float inv = __frcp_rn(sum);
#pragma unroll
      for (int r = 0; r < KPL; ++r) k[r] = __float_as_uint(v[r] * inv);
#pragma unroll
      for (int c = 0; c < KPL / 4; ++c)
        row_keys[c * 32 + lane] = make_uint4(k[4 * c], k[4 * c + 1], k[4 * c + 2], k[4 * c + 3]);
    }
    __syncwarp();
    // keep_all / keep_none cover K >= Tk, p >= 1, and K = 0 with p <= 0
    bool keep_all = sel.K >= Tk || sel.p_mode == 2;
    const bool keep_none = !keep_all && sel.K == 0 && sel.p_mode == 1;
    uint32_t t = 0;
    int take = 0, n_eq = 0;
    if (!keep_all && !keep_none && !select_by_sort<KPL, 8>(k, sel, t, take, n_eq)) {
      bool done = false;
      if constexpr (KPL > 8) {  // the 16 largest keys of every lane
#pragma unroll
        for (int c = 0; c < KPL / 4; ++c) {
          const uint4 x = row_keys[c * 32 + lane];
          k[4 * c] = x.x;
          k[4 * c + 1] = x.y;
          k[4 * c + 2] = x.z;
          k[4 * c + 3] = x.w;
        }
        done = select_by_sort<KPL, 16>(k, sel, t, take, n_eq);
      }
      if (!done)
        select_in_memory(reinterpret_cast<const uint32_t*>(row_keys), 32 * KPL, sel, keep_all, t, take, n_eq);
    }
    emit_row(row_keys, Tk, out, rowid, a.bits + ((size_t)z * s.Tq + i) * a.W, a.W, keep_all, keep_none, take < n_eq,
             t, take);
    __syncwarp();
  }
}

// Rows longer than 32 * kMaxKeysPerLane keys: the softmax overwrites the scratch row with
// its keys (same permuted positions), the bisection runs over memory.
__global__ void __launch_bounds__(kSelectThreads) select_mem_kernel(ShapeArgs s, SelectArgs sel, SelArgs a,
                                                                    MaskOut out) {
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int Tk = s.Tk, n = a.tk_pad;
  const long long rows = (long long)a.nbh * s.Tq;
  const long long nwarps = (long long)gridDim.x * kSelectWarps;
  for (long long gw = (long long)blockIdx.x * kSelectWarps + wib; gw < rows; gw += nwarps) {
    const int z = (int)(gw / s.Tq), i = (int)(gw - (long long)z * s.Tq);
    float* row = a.sbar + ((size_t)z * a.tq_pad + i) * a.tk_pad;
    const int64_t rowid = (int64_t)(a.bh0 + z) * s.Tq + i;
    float mx = -INFINITY;
    for (int j = lane; j < n; j += 32) mx = fmaxf(mx, row[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
    for (int j = lane; j < n; j += 32) sum += ex2_approx((row[j] - mx) * kLog2e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float inv = __frcp_rn(sum);
    __syncwarp();
    for (int j = lane; j < n; j += 32) row[j] = ex2_approx((row[j] - mx) * kLog2e) * inv;
    __syncwarp();
    const uint32_t* keys = reinterpret_cast<const uint32_t*>(row);
    bool keep_all = sel.K >= Tk || sel.p_mode == 2;
    const bool keep_none = !keep_all && sel.K == 0 && sel.p_mode == 1;
    uint32_t t = 0;
    int take = 0, n_eq = 0;
    if (!keep_all && !keep_none) select_in_memory(keys, n, sel, keep_all, t, take, n_eq);
    emit_row(reinterpret_cast<const uint4*>(row), Tk, out, rowid, a.bits + ((size_t)z * s.Tq + i) * a.W, a.W,
             keep_all, keep_none, take < n_eq, t, take);
    __syncwarp();
  }
}

// Column lists from the rows' kept bits.  A CTA takes one 32-bit word of the rows (32
// consecutive key blocks, lane = key block) of one head, and its 8 warps split the query
// blocks into ranges: per 32 rows a warp loads one word per row (lane = row) and transposes
// the 32 x 32 bit block with ballots, so that lane j holds its column's kept bits; the per-warp
// counts are then prefix-summed and every lane writes its column's query blocks in ascending
// order.  blockIdx.y is the head within the chunk.
constexpr int kCscWarps = 8;
constexpr int kCscMaxWords = 30;  // Tq <= 7680 (bq >= 64, N <= 7680 * 64): 960 rows per warp

__global__ void __launch_bounds__(32 * kCscWarps) csc_kernel(ShapeArgs s, int bh0, int W,
                                                             const uint32_t* __restrict__ bits,
                                                             int32_t* __restrict__ col_cnt,
                                                             int32_t* __restrict__ col_idx) {
  __shared__ uint32_t cbits[kCscWarps][kCscMaxWords][32];
  __shared__ int cnt[kCscWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int z = blockIdx.y, bh = bh0 + z;
  const int j = blockIdx.x * 32 + lane;
  const int R = (s.Tq + kCscWarps - 1) / kCscWarps;  // rows per warp (<= 32 * kCscMaxWords)
  const int i0 = warp * R, i1 = min(s.Tq, i0 + R);
  const uint32_t* b = bits + (size_t)z * s.Tq * W + blockIdx.x;
  int c = 0;
  for (int g = 0; g * 32 < R; ++g) {
    const int i = i0 + g * 32 + lane;
    const uint32_t word = i < i1 ? b[(size_t)i * W] : 0u;
    uint32_t mine = 0;
#pragma unroll
    for (int q = 0; q < 32; ++q) {
      const unsigned m = __ballot_sync(0xffffffffu, (word >> q) & 1u);
      mine = lane == q ? m : mine;
    }
    cbits[warp][g][lane] = mine;  // bit r: query block i0 + 32 g + r keeps key block j
    c += __popc(mine);
  }
  cnt[warp][lane] = c;
  __syncthreads();
  int base = 0, total = 0;
  for (int q = 0; q < kCscWarps; ++q) {
    if (q < warp) base += cnt[q][lane];
    total += cnt[q][lane];
  }
  if (j >= s.Tk) return;
  int32_t* o = col_idx + ((int64_t)bh * s.Tk + j) * s.Tq + base;
  for (int g = 0; g * 32 < R; ++g) {
    uint32_t word = cbits[warp][g][lane];
    while (word) {
      const int q = __ffs(word) - 1;
      word &= word - 1;
      *o++ = i0 + g * 32 + q;
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
  size_t qbar, kbar, sbar, bits, ctr, total;
  size_t sbar_buf, bits_buf;  // bytes of one buffer of each
  int tq_pad, tk_pad, hc;     // padded tile extents; heads per chunk
  int W;                      // 32-bit words of kept bits per row
};

// The pooled pairs of all heads, then kChains buffers (one per head chunk in flight) of the
// chunk's score tiles and of its rows' kept bits.  chunk_budget bounds the bytes of all the
// buffers together; a chunk holds at least one head.
MaskLayout mask_layout(const ShapeArgs& s, size_t chunk_budget) {
  MaskLayout L;
  const size_t BH = (size_t)s.B * s.H;
  auto al = [](size_t x) { return (x + 1023) / 1024 * 1024; };
  L.tq_pad = (s.Tq + kScoreRows - 1) / kScoreRows * kScoreRows;
  L.tk_pad = (s.Tk + kRowPad - 1) / kRowPad * kRowPad;
  L.W = (s.Tk + 31) / 32;
  const size_t tile_head = (size_t)L.tq_pad * L.tk_pad * 4, bits_head = (size_t)s.Tq * L.W * 4;
  L.hc = (int)std::max<size_t>(1, std::min<size_t>(BH, chunk_budget / (kChains * (tile_head + bits_head) + 4096)));
  L.sbar_buf = al((size_t)L.hc * tile_head);
  L.bits_buf = al((size_t)L.hc * bits_head);
  L.qbar = 0;
  L.kbar = al(2 * BH * s.Tq * s.d * 4);
  L.sbar = L.kbar + al(2 * BH * s.Tk * s.d * 4);
  L.bits = L.sbar + kChains * L.sbar_buf;
  L.ctr = L.bits + kChains * L.bits_buf;  // the pooling's chunk counters, one per head chunk
  L.total = L.ctr + al(BH * sizeof(int));
  return L;
}

// kChains more streams per device, of the highest priority.  The scores, the selection and
// the column lists of head chunk c run on stream c % kChains (with buffer c % kChains) while
// the caller's stream pools the next chunks, so that the chains of several chunks overlap;
// the caller's stream waits for all of them at the end of the call.  Set up on the first
// build on a device.
struct AuxStream {
  cudaStream_t stream[kChains] = {};
  cudaEvent_t pooled = nullptr, done[kChains] = {};
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
    // the chains are latency-bound and the pooling streams in the background: the chains'
    // blocks go first where both wait for an SM
    int lo = 0, hi = 0;
    a.err = cudaDeviceGetStreamPriorityRange(&lo, &hi);
    for (int i = 0; i < kChains && a.err == cudaSuccess; ++i) {
      a.err = cudaStreamCreateWithPriority(&a.stream[i], cudaStreamNonBlocking, hi);
      if (a.err == cudaSuccess) a.err = cudaEventCreateWithFlags(&a.done[i], cudaEventDisableTiming);
    }
    if (a.err == cudaSuccess) a.err = cudaEventCreateWithFlags(&a.pooled, cudaEventDisableTiming);
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
  int* pool_ctr = reinterpret_cast<int*>(base + L.ctr);
  float* qbar = reinterpret_cast<float*>(base + L.qbar);
  float* kbar = reinterpret_cast<float*>(base + L.kbar);
  float* sbar_buf[kChains];
  uint32_t* bits_buf[kChains];
  for (int i = 0; i < kChains; ++i) {
    sbar_buf[i] = reinterpret_cast<float*>(base + L.sbar + i * L.sbar_buf);
    bits_buf[i] = reinterpret_cast<uint32_t*>(base + L.bits + i * L.bits_buf);
  }
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
  // the selection: keys per lane by row length, or the rows in memory
  const void* select = nullptr;
  int sel_smem = 0;
  auto pick = [&](auto kernel, int bytes) {
    select = (const void*)kernel;
    sel_smem = bytes;
  };
  if (s.Tk <= 128)
    pick(select_kernel<4>, select_smem_bytes<4>());
  else if (s.Tk <= 256)
    pick(select_kernel<8>, select_smem_bytes<8>());
  else if (s.Tk <= 512)
    pick(select_kernel<16>, select_smem_bytes<16>());
  else if (s.Tk <= 768)
    pick(select_kernel<24>, select_smem_bytes<24>());
  else if (s.Tk <= 1024)
    pick(select_kernel<32>, select_smem_bytes<32>());
  else if (s.Tk <= 32 * kMaxKeysPerLane)
    pick(select_kernel<kMaxKeysPerLane>, select_smem_bytes<kMaxKeysPerLane>());
  else
    pick(select_mem_kernel, 0);
  // a register row reads 32 * (keys per lane) entries of its scratch row: never past tk_pad
  if (sel_smem > 0 && sel_smem / (kSelectWarps * 4) > L.tk_pad) return cudaErrorInvalidValue;
  if (e == cudaSuccess && sel_smem > 0)
    e = cudaFuncSetAttribute(select, cudaFuncAttributeMaxDynamicSharedMemorySize, sel_smem);
  int sel_occ = 0;
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&sel_occ, select, kSelectThreads, sel_smem);
  if (e != cudaSuccess) return e;
  const void* pool = s.d == 128 ? (const void*)pool_kernel<float, 128> : (const void*)pool_kernel<float, 64>;
  int pool_occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&pool_occ, pool, kPoolThreads, 0);
  if (e != cudaSuccess) return e;
  // bf16 inputs: the tensor-core pooling over token tensor maps (128-token boxes)
  CUtensorMap mqt, mkt;
  auto pool_tc = s.d == 128 ? pool_tc_kernel<128> : pool_tc_kernel<64>;
  if (s.dtype == 0) {
    if (!make_token_map(&mqt, q, s, s.sb, s.sh, s.sn, kChunkTokens, false) ||
        !make_token_map(&mkt, k, s, s.sb, s.sh, s.sn, kChunkTokens, false))
      return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(pool_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kPoolTcSmem);
    if (e != cudaSuccess) return e;
  }
  // a third of the SMs' pooling capacity per chunk: the other kernels of the previous chunk
  // run beside it
  const int pool_blocks = std::max(1, sms * std::max(1, pool_occ) / 2);

  std::lock_guard<std::mutex> lock(aux->mu);
  const int BH = s.B * s.H;
  if (s.dtype == 0) {
    e = cudaMemsetAsync(pool_ctr, 0, (size_t)((BH + L.hc - 1) / L.hc) * sizeof(int), st);
    if (e != cudaSuccess) return e;
  }
  const int nc = (s.N + kChunkTokens - 1) / kChunkTokens;
  for (int bh0 = 0, ci = 0; bh0 < BH; bh0 += L.hc, ++ci) {
    const int nbh = std::min(L.hc, BH - bh0);
    const int chain = ci % kChains;
    float* sbar = sbar_buf[chain];
    uint32_t* bits = bits_buf[chain];
    // ---- pooling of the chunk, on the caller's stream
    PoolArgs pa;
    pa.qbar = qbar;
    pa.kbar = kbar;
    pa.bh0 = bh0;
    pa.nbh = nbh;
    pa.ctr = pool_ctr + ci;
    const long long pool_warps = (long long)nbh * 2 * nc;
    const int pgrid = (int)std::min<long long>((pool_warps + 7) / 8, pool_blocks);
    prof_start(st, kPool);
    if (s.dtype == 0) {
      const int tgrid = (int)std::min<long long>(pool_warps, sms);
      pool_tc<<<tgrid, kPoolTcThreads, kPoolTcSmem, st>>>(mqt, mkt, s, pa, out.status);
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
    if (e == cudaSuccess) e = cudaStreamWaitEvent(aux->stream[chain], aux->pooled, 0);
    if (e != cudaSuccess) return e;
    // ---- scores, selection and column lists of the chunk, on the second stream
    cudaStream_t st2 = aux->stream[chain];
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
    ca.bits = bits;
    ca.bh0 = bh0;
    ca.nbh = nbh;
    ca.tq_pad = L.tq_pad;
    ca.tk_pad = L.tk_pad;
    ca.W = L.W;
    const long long rows = (long long)nbh * s.Tq;
    const int sgrid = (int)std::min<long long>((rows + kSelectWarps - 1) / kSelectWarps,
                                               (long long)sms * std::max(1, sel_occ));
    prof_start(st2, kScoreSelect);
    {
      SelectArgs sl = sel;
      MaskOut mo = out;
      void* args[] = {(void*)&s, (void*)&sl, (void*)&ca, (void*)&mo};
      e = cudaLaunchKernel(select, dim3(sgrid), dim3(kSelectThreads), args, (size_t)sel_smem, st2);
    }
    prof_stop(st2, kScoreSelect);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 cgrid(L.W, nbh);
    prof_start(st2, kCsc);
    csc_kernel<<<cgrid, 32 * kCscWarps, 0, st2>>>(s, bh0, L.W, bits, out.col_cnt, out.col_idx);
    prof_stop(st2, kCsc);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // join the chains that took a chunk back into the caller's stream (only those: under stream
  // capture a chain stream that took no work is not part of the capture, and waiting on an
  // event recorded there would break it)
  const int used = std::min(kChains, (BH + L.hc - 1) / L.hc);
  for (int i = 0; i < used && e == cudaSuccess; ++i) {
    e = cudaEventRecord(aux->done[i], aux->stream[i]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, aux->done[i], 0);
  }
  return e;
}

}  // namespace sa2
