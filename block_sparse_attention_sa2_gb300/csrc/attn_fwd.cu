// Block-sparse attention forward on sm_103a (tcgen05 + TMEM + TMA).
//
// gist.science explainer of SpargeAttention2 (arXiv 2602.13515), section 2.C: a
// FlashAttention-style block-sparse kernel in which whole tiles are kept or skipped, and
// skipped tiles cost neither matmul nor softmax.  Here each CTA owns one query block of
// 128 rows and walks that block's list of kept 64-token key blocks.
//
// Roles (224 threads, 2 CTAs per SM):
//   warp 0      TMA producer: Q once, then K_j / V_j per kept key block into NS stages
//   warp 1      TMEM owner and issuer of S_j = Q K_j^T into a double-buffered TMEM tile
//   warp 2      issuer of O += P_j V_j with P_j read from TMEM (two issuing warps, each
//               converged with one elect.sync lane issuing, keep the MMA queue fed while
//               either waits on a barrier)
//   warps 3..6  softmax: each thread owns one query row (its TMEM lane); online softmax in
//               fp32 with exp2, P_j (fp16) written back over S_j in TMEM; epilogue O / l
//
// Operand types: S = Q K^T in bf16 (bf16 calls) or, for fp32 calls, as three fp16 products
// of the inputs' hi = fp16(x) and lo = fp16(x - hi) parts, Qhi Khi^T + Qhi Klo^T + Qlo Khi^T
// (about 22 bits: the fp32 scores to within ~2^-21 relative); P V always in fp16 with an
// fp16 copy of V: P lies in [0, 1], where fp16 keeps 11 significant bits against bf16's 8,
// and bf16 V converts to fp16 exactly.
//
// TMEM columns: S buffers at 0 and 64 (fp32, 64 columns each; P_j as packed fp16 pairs in
// the first 32 columns of its S buffer), O at 128 (D columns).
#include "sa2_internal.h"

namespace sa2 {
namespace {

constexpr int kThreads = 224;
constexpr int kNumStages = 2;  // also the number of S/P buffers in TMEM (the waits rely on it)
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColO = 128;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: O and l are rescaled only past 2^8

// SPLIT (fp32 calls): Q and K also as fp16 residuals, lo = fp16(x - hi), behind their hi
// tiles; S = Qhi Khi^T + Qhi Klo^T + Qlo Khi^T carries ~22 bits of the fp32 inputs.
template <int D, bool SPLIT>
struct FwdSmem {
  static constexpr int kPanels = D / 64;
  static constexpr int kQBytes = 128 * 128 * kPanels;   // 128 rows x 128 B per panel
  static constexpr int kKVBytes = 64 * 128 * kPanels;   // 64 rows x 128 B per panel
  static constexpr int kParts = SPLIT ? 2 : 1;          // hi (and lo) of Q and K
  static constexpr int kOffQ = 0;
  static constexpr int kOffQlo = kOffQ + kQBytes;
  static constexpr int kOffK = kOffQ + kParts * kQBytes;
  static constexpr int kOffKlo = kOffK + kNumStages * kKVBytes;
  static constexpr int kOffV = kOffK + kParts * kNumStages * kKVBytes;
  static constexpr int kOffBar = kOffV + kNumStages * kKVBytes;
  // barriers, TMEM slot and alignment slack; at least 80 KB so that no more than two CTAs
  // (2 x 256 TMEM columns) share an SM
  static constexpr int kBytes = (kOffBar + 256 + 1024) > 80 * 1024 ? (kOffBar + 256 + 1024) : 80 * 1024;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename OutT>
__device__ __forceinline__ void store_row_chunk(OutT* dst, const float* v);

template <>
__device__ __forceinline__ void store_row_chunk<__nv_bfloat16>(__nv_bfloat16* dst, const float* v) {
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
    w.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
    w.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
    w.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
    p[i] = w;
  }
}

// Low-order part of a bf16 rounding: bf16(v - bf16(v)), so that hi + lo carries ~16 bits.
__device__ __forceinline__ void store_residual_chunk(__nv_bfloat16* dst, const float* v) {
  float r[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) r[c] = v[c] - __bfloat162float(__float2bfloat16_rn(v[c]));
  store_row_chunk<__nv_bfloat16>(dst, r);
}

template <>
__device__ __forceinline__ void store_row_chunk<float>(float* dst, const float* v) {
  float4* p = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i) p[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

template <int D, typename OutT, bool S_F16, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 2)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mql,
                    const __grid_constant__ CUtensorMap mkl, ShapeArgs s, FwdArgs a) {
  using L = FwdSmem<D, SPLIT>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  // barrier slots
  const uint32_t bar_q = smem_u32(&bars[0]);
  // K_j is released as soon as S_j has been computed, V_j only after P_j V_j: separate
  // rings keep the K loads running ahead of the softmax
  auto bar_kfull = [&](int st) { return smem_u32(&bars[1 + st]); };
  auto bar_vfull = [&](int st) { return smem_u32(&bars[1 + kNumStages + st]); };
  auto bar_kempty = [&](int st) { return smem_u32(&bars[1 + 2 * kNumStages + st]); };
  auto bar_vempty = [&](int st) { return smem_u32(&bars[1 + 3 * kNumStages + st]); };
  auto bar_sfull = [&](int b) { return smem_u32(&bars[1 + 4 * kNumStages + b]); };
  auto bar_pfull = [&](int b) { return smem_u32(&bars[3 + 4 * kNumStages + b]); };
  const uint32_t bar_odone = smem_u32(&bars[5 + 4 * kNumStages]);
  const uint32_t bar_drain = smem_u32(&bars[6 + 4 * kNumStages]);   // every P V MMA completed
  const uint32_t bar_sdrain = smem_u32(&bars[7 + 4 * kNumStages]);  // every S MMA completed
  // 16 barriers occupy the first 128 bytes of the 256-byte barrier area
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffBar + 160);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffBar + 192);
  const WaitCtl wc{abort_flag, s.wait_ns};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // CTAs launch in the order of launch_item_order: head by head, within a head longest list
  // first, so the CTAs in flight share their heads' K / V in L2 and the last wave holds short
  // lists; the lists too long to start late launch first of all
  const int x = a.order[blockIdx.x];
  const int bh = x / s.Tq;
  const int qi = x % s.Tq;
  const int b = bh / s.H, h = bh % s.H;
  const int64_t rowid = (int64_t)bh * s.Tq + qi;
  int nkv = a.row_cnt[rowid];
  if (nkv < 0 || nkv > s.Tk) {
    if (tid == 0) report_error(a.status, kDevErrBounds);
    nkv = nkv < 0 ? 0 : s.Tk;
  }
  const int32_t* list = a.row_idx + rowid * s.Tk;

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bar_q, 1);
    for (int st = 0; st < kNumStages; ++st) {
      mbar_init(bar_kfull(st), 1);
      mbar_init(bar_vfull(st), 1);
      mbar_init(bar_kempty(st), 1);
      mbar_init(bar_vempty(st), 1);
    }
    for (int bb = 0; bb < 2; ++bb) {
      mbar_init(bar_sfull(bb), 1);
      mbar_init(bar_pfull(bb), 128);
    }
    mbar_init(bar_odone, 1);
    mbar_init(bar_drain, 1);
    mbar_init(bar_sdrain, 1);
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
    if (lane == 0 && nkv > 0) {
      tma_prefetch_map(&mq);
      tma_prefetch_map(&mk);
      tma_prefetch_map(&mv);
      if constexpr (SPLIT) {
        tma_prefetch_map(&mql);
        tma_prefetch_map(&mkl);
      }
      mbar_arrive_expect_tx(bar_q, L::kParts * L::kQBytes);
      for (int p = 0; p < L::kPanels; ++p) {
        tma_load_4d(sbase + L::kOffQ + p * 16384, &mq, bar_q, p * 64, qi * s.bq, h, b);
        if constexpr (SPLIT) tma_load_4d(sbase + L::kOffQlo + p * 16384, &mql, bar_q, p * 64, qi * s.bq, h, b);
      }
      int nk = 0, nv = 0;  // K and V loads issued
      for (int j = 0; j < nkv; ++j) {
        const int st = j % kNumStages;
        const uint32_t ph = ((j / kNumStages) - 1) & 1;
        int kb = list[j];
        if (kb < 0 || kb >= s.Tk) {
          report_error(a.status, kDevErrBounds);
          kb = 0;
        }
        if (j >= kNumStages && !mbar_wait(bar_kempty(st), ph, wc)) break;
        mbar_arrive_expect_tx(bar_kfull(st), L::kParts * L::kKVBytes);
        for (int p = 0; p < L::kPanels; ++p) {
          tma_load_4d(sbase + L::kOffK + st * L::kKVBytes + p * 8192, &mk, bar_kfull(st), p * 64, kb * 64, h, b);
          if constexpr (SPLIT)
            tma_load_4d(sbase + L::kOffKlo + st * L::kKVBytes + p * 8192, &mkl, bar_kfull(st), p * 64, kb * 64, h,
                        b);
        }
        ++nk;
        if (j >= kNumStages && !mbar_wait(bar_vempty(st), ph, wc)) break;
        mbar_arrive_expect_tx(bar_vfull(st), L::kKVBytes);
        for (int p = 0; p < L::kPanels; ++p)
          tma_load_4d(sbase + L::kOffV + st * L::kKVBytes + p * 8192, &mv, bar_vfull(st), p * 64, kb * 64, h, b);
        ++nv;
      }
      // No copy may still be in flight when the CTA exits, whether the loop ran to its end or
      // gave up: drain Q and the last load of each stage (each is that stage's latest phase).
      mbar_drain(bar_q, 0, abort_flag);
      for (int j = nk > kNumStages ? nk - kNumStages : 0; j < nk; ++j)
        mbar_drain(bar_kfull(j % kNumStages), (j / kNumStages) & 1, abort_flag);
      for (int j = nv > kNumStages ? nv - kNumStages : 0; j < nv; ++j)
        mbar_drain(bar_vfull(j % kNumStages), (j / kNumStages) & 1, abort_flag);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ S_j issuer
    if (nkv > 0) {
      constexpr uint32_t idS = idesc_f32acc(128, 64, false, false, !S_F16);
      const uint64_t qd = smem_desc(sbase + L::kOffQ, 16, 1024);
      bool ok = __all_sync(0xffffffffu, mbar_wait(bar_q, 0, wc));
      for (int j = 0; ok && j < nkv; ++j) {
        const int st = j % kNumStages;
        if (!__all_sync(0xffffffffu, mbar_wait(bar_kfull(st), (j / kNumStages) & 1, wc))) break;
        // S_j overwrites the TMEM buffer whose P_{j-2} the MMA P_{j-2} V_{j-2} read: a
        // later tcgen05.mma is not ordered after an earlier one's TMEM operand reads, so
        // wait for that MMA to complete (its commit also releases V_{j-2}; buffer and
        // V stage have the same index, both rings being 2 deep)
        if (j >= 2 &&
            !__all_sync(0xffffffffu, mbar_wait(bar_vempty(st), ((j - 2) / kNumStages) & 1, wc)))
          break;
        tc_fence_after();
        const uint64_t kd = smem_desc(sbase + L::kOffK + st * L::kKVBytes, 16, 1024);
        if (elect_one()) {
          mma_ss_kmajor<idS, 128, 64, D / 16>(tmem + (j & 1) * 64, qd, kd);
          if constexpr (SPLIT) {
            const uint64_t kld = smem_desc(sbase + L::kOffKlo + st * L::kKVBytes, 16, 1024);
            const uint64_t qld = smem_desc(sbase + L::kOffQlo, 16, 1024);
            mma_ss_kmajor_acc<idS, 128, 64, D / 16>(tmem + (j & 1) * 64, qd, kld);
            mma_ss_kmajor_acc<idS, 128, 64, D / 16>(tmem + (j & 1) * 64, qld, kd);
          }
          umma_commit(bar_sfull(j & 1));
          umma_commit(bar_kempty(st));
        }
        __syncwarp();
      }
      // no MMA of this warp may still run when TMEM is released, on the abort path too
      if (elect_one()) umma_commit(bar_sdrain);
      __syncwarp();
      mbar_drain(bar_sdrain, 0, abort_flag);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- P_j V_j issuer
    if (nkv > 0) {
      constexpr uint32_t idO = idesc_f16_f32(128, D, false, true);
      for (int jj = 0; jj < nkv; ++jj) {
        const int st = jj % kNumStages;
        if (!__all_sync(0xffffffffu, mbar_wait(bar_pfull(jj & 1), (jj >> 1) & 1, wc) &&
                                         mbar_wait(bar_vfull(st), (jj / kNumStages) & 1, wc)))
          break;
        tc_fence_after();
        // V as the MN-major B operand: N = D (64-element groups 8 KB apart), K = 16 rows
        const uint64_t vd = smem_desc(sbase + L::kOffV + st * L::kKVBytes, 8192, 1024);
        if (elect_one()) {
          mma_ts_bmn<idO, 4>(tmem + kColO, tmem + (jj & 1) * 64, vd, jj == 0);
          umma_commit(bar_vempty(st));
          umma_commit(bar_odone);
        }
        __syncwarp();
      }
      // the S MMAs all completed before the last P was written: this commit covers every
      // MMA of the CTA
      if (elect_one()) umma_commit(bar_drain);
      __syncwarp();
      mbar_drain(bar_drain, 0, abort_flag);
    }
  } else {
    // ------------------------------------------------------------------ softmax rows
    if (s.stall_ns && blockIdx.x == 0) stall_for(s.stall_ns);  // failure-path test hook
    const int sub = warp & 3;  // TMEM lane quarter this warp may access
    const int r = 32 * sub + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * sub) << 16);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    // tcgen05.ld / st are warp-collective (.sync.aligned): every branch around them is
    // decided uniformly per warp (__all_sync / __any_sync).
    int next_kb = nkv > 0 ? list[0] : 0;  // key block of the next entry, loaded one entry ahead
    for (int j = 0; j < nkv; ++j) {
      const int bsel = j & 1;
      int kb = next_kb;
      if (j + 1 < nkv) next_kb = list[j + 1];
      if (!__all_sync(0xffffffffu, mbar_wait(bar_sfull(bsel), (j >> 1) & 1, wc))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t u0[32], u1[32];
      tmem_ld32(trow + bsel * 64, u0);
      tmem_ld32(trow + bsel * 64 + 32, u1);
      tmem_ld_wait(u0);
      tmem_ld_wait(u1);
      kb = (kb < 0 || kb >= s.Tk) ? 0 : kb;
      // raw scores; the scale (> 0) is folded into the exponent's FMA below
      float x[64];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        x[c] = __uint_as_float(u0[c]);
        x[c + 32] = __uint_as_float(u1[c]);
      }
      const int valid = min(64, s.N - kb * 64);
      if (valid < 64) {  // the ragged last key block (the same for the whole CTA)
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = c < valid ? x[c] : -INFINITY;
      }
      // row maximum and (below) row sum as 8- and 4-way trees: short dependency chains
      float m8[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) m8[c] = x[c];
#pragma unroll
      for (int c = 8; c < 64; ++c) m8[c & 7] = fmaxf(m8[c & 7], x[c]);
      const float mr = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      const float mx = mr * a.scale_log2;
      if (j == 0) {
        m_used = mx;
      } else {
        const bool need = mx > m_used + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          // O must hold P_0..P_{j-1} V before it is rescaled; lanes that keep their max
          // multiply by 1
          const float alpha = need ? ex2(m_used - mx) : 1.f;
          // S_j was issued only after P_{j-2} V_{j-2} completed, so o_done is at most one
          // phase behind j - 1 here and the parity wait is exact
          if (!__all_sync(0xffffffffu, mbar_wait(bar_odone, (j - 1) & 1, wc))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(trow + kColO + c0, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st32(trow + kColO + c0, o);
          }
          tmem_st_wait();
          if (need) {
            l *= alpha;
            m_used = mx;
          }
        }
      }
      uint32_t pk[32];
      float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = ex2(fmaf(x[2 * c], a.scale_log2, -m_used));
        const float p1 = ex2(fmaf(x[2 * c + 1], a.scale_log2, -m_used));
        l4[c & 3] += p0 + p1;
        pk[c] = pack_f16x2(p0, p1);
      }
      l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
      tmem_st32(trow + bsel * 64, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_pfull(bsel));
    }
    // ---- epilogue
    const int64_t tok = (int64_t)qi * s.bq + r;
    const bool row_valid = r < s.bq && tok < s.N;
    OutT* orow = reinterpret_cast<OutT*>(a.o) + (int64_t)b * a.o_sb + (int64_t)h * a.o_sh + tok * a.o_sn;
    if (nkv == 0) {
      if (row_valid) {
        float z[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) z[c] = 0.f;
        for (int c0 = 0; c0 < D; c0 += 32) {
          store_row_chunk<OutT>(orow + c0, z);
          if constexpr (sizeof(OutT) == 2) {
            if (a.o_lo) store_row_chunk<__nv_bfloat16>(reinterpret_cast<__nv_bfloat16*>(a.o_lo) + (int64_t)b * a.o_sb +
                                                           (int64_t)h * a.o_sh + tok * a.o_sn + c0,
                                                       z);
          }
        }
        a.lse[(int64_t)bh * s.N + tok] = -INFINITY;
      }
    } else if (__all_sync(0xffffffffu, ok && mbar_wait(bar_drain, 0, wc) && !*abort_flag)) {
      // bar_drain completes once, after the last MMA.  (A parity wait on o_done is only
      // valid while that barrier is at most one phase behind the awaited phase; here the
      // last two P V MMAs may both still be pending.)  On the abort path the P V issuer
      // completes it after fewer products: the flag is up then, and nothing is written.
      tc_fence_after();
      const float inv_l = 1.f / l;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(trow + kColO + c0, o);
        tmem_ld_wait(o);
        float v[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] = __uint_as_float(o[c]) * inv_l;
        if (row_valid) {
          store_row_chunk<OutT>(orow + c0, v);
          if constexpr (sizeof(OutT) == 2) {
            if (a.o_lo) store_residual_chunk(reinterpret_cast<__nv_bfloat16*>(a.o_lo) +
                                                 (int64_t)b * a.o_sb + (int64_t)h * a.o_sh + tok * a.o_sn + c0,
                                             v);
          }
        }
      }
      if (row_valid) a.lse[(int64_t)bh * s.N + tok] = (m_used + __log2f(l)) * 0.69314718055994531f;
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

template <int D, typename OutT, bool S_F16, bool SPLIT>
cudaError_t launch_fwd_t(const ShapeArgs& s, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mql, const CUtensorMap& mkl, const FwdArgs& a, cudaStream_t st) {
  const int smem = FwdSmem<D, SPLIT>::kBytes;
  auto kern = attn_fwd_kernel<D, OutT, S_F16, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)s.B * s.H * s.Tq;
  e = launch_item_order(a.row_cnt, s.B * s.H, s.Tq, s.Tk, sms * (per_sm > 0 ? per_sm : 1), a.order, nullptr, st);
  prof_start(st, kAttnFwd);
  if (e == cudaSuccess) kern<<<(unsigned)grid, kThreads, smem, st>>>(mq, mk, mv, mql, mkl, s, a);
  prof_stop(st, kAttnFwd);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace

cudaError_t launch_attn_fwd(const ShapeArgs& s, bool s_f16, const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& mv, const CUtensorMap* mql, const CUtensorMap* mkl, const FwdArgs& a,
                            cudaStream_t st) {
  // bf16 calls: bf16 S, bf16 output; fp32 calls: the split fp16 S product, fp32 output
  if (!s_f16)
    return s.d == 128 ? launch_fwd_t<128, __nv_bfloat16, false, false>(s, mq, mk, mv, mq, mk, a, st)
                      : launch_fwd_t<64, __nv_bfloat16, false, false>(s, mq, mk, mv, mq, mk, a, st);
  if (!mql || !mkl) return cudaErrorInvalidValue;
  return s.d == 128 ? launch_fwd_t<128, float, true, true>(s, mq, mk, mv, *mql, *mkl, a, st)
                    : launch_fwd_t<64, float, true, true>(s, mq, mk, mv, *mql, *mkl, a, st);
}

}  // namespace sa2
