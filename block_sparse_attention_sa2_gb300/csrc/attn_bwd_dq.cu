// Block-sparse attention backward, dQ part, on sm_103a (tcgen05 + TMEM + TMA).
//
// dQ = scale * dS K with dS = P * (dP - D), P = exp(s - LSE), dP = dO V^T: the gradient of
// the block-sparse forward with respect to Q (the abstract of SpargeAttention2, arXiv
// 2602.13515, contribution (ii): trainable sparse attention; gist.science explainer,
// section 2.C: whole tiles kept or skipped).  A work item is one query block of 128 rows;
// the CTA that takes it walks that block's list of kept key blocks -- the forward's
// traversal -- so dQ accumulates in TMEM over the whole list and is written once: no
// cross-CTA reduction.
//
// Roles (352 threads, 1 CTA per SM): warp 0 TMA (Q and dO once per query block, K_j / V_j
// per kept block into 4 / 2 stages), warp 1 TMEM owner and issuer of the S_j / dP_j MMAs,
// warp 2 issuer of the dQ MMAs (each converged, one elect.sync lane issuing: two issuers keep the MMA queue
// fed while either waits on a barrier), and two row warpgroups (warps 3..6 and 7..10) that
// both work on every list entry (TMEM buffers j % 2), one query row per thread, group g on
// key columns 32g .. 32g+31 of the entry, so that each entry's dS is ready in half the time.
// Per kept key block j:
//   S_j  = Q K_j^T     M = 128, N = 64, K = d     (A = Q from TMEM, B = K_j K-major, fp16)
//   dP_j = dO V_j^T    M = 128, N = 64, K = d     (A, B K-major, fp16)
//   row threads: P = exp2(S * scale*log2e - LSE*log2e), dS = P (dP - D), dS as fp16 pairs
//                into their own TMEM buffer
//   dQ  += dS_j K_j    M = 128, N = d, K = 64     (A = dS from TMEM, B = K_j MN-major)
// TMEM columns: S at 0 / 64, dP at 128 / 192, dS at 256 / 288 (all double-buffered), the
// query block's Q at 320 (d / 2 columns of fp16 pairs), dQ at 384 (d columns).  S_j / dP_j
// may overwrite their buffers as soon as the row threads have read S_{j-2} / dP_{j-2} out;
// only the row threads wait for dQ_{j-2} to complete before writing dS_j, so the tensor pipe
// never drains to let an MMA overwrite an operand.
//
// Q sits in TMEM as the A operand of S_j because an M128 N64 product with both operands in
// shared memory reads 6 KB per k-step, more than shared memory delivers in the 32 cycles of
// the k-step's math; with A in TMEM it reads only the 2 KB of K_j.  The row threads copy
// each query block's Q out of its shared-memory slot into TMEM (thread = row = TMEM lane),
// which they do for the next block as soon as the current block's last S_j has been read,
// before the current block's epilogue.  Q and dO load into a two-slot ring, so the next
// block's tiles are in shared memory well before it starts.  fp32 calls (the split S
// product reads Q's fp16 residual too) keep Q in shared memory and a one-slot ring.
//
// The CTAs are persistent, one per SM, and take query blocks from a counter until none is
// left, in the order of launch_item_order (head by head, longest list first within a head,
// lists too long to start late in front).  The producer publishes each block in a two-slot
// ring in shared memory that every role reads; the K / V rings and the TMEM buffers run on across blocks.  So the set-up is
// paid once per SM, the next block's K_j / V_j stream in behind the current block's, its
// Q and dO load as soon as the current block's S_j / dP_j MMAs have completed, and its
// first S_j / dP_j MMAs run while the row threads store the current block's dQ.
#include "sa2_internal.h"

namespace sa2 {
namespace {

constexpr int kThreads = 352;
constexpr int kItemReaders = 10;  // warps reading the item slot: 1, 2 and the 8 row warps
// K_j feeds S_j and, after the softmax, dQ += dS_j K_j, so its ring is deep; V_j only feeds
// dP_j and is released right after it
constexpr int kKStages = 4;
constexpr int kVStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColDS = 256, kColQ = 320, kColDQ = 384;

// SPLIT (fp32 calls): Q and K also as fp16 residuals lo = fp16(x - hi) for the split S
// product Qhi Khi^T + Qhi Klo^T + Qlo Khi^T; the K ring is then 2 deep to fit.
template <int D, bool SPLIT>
struct DqSmem {
  static constexpr bool kQInTmem = !SPLIT;           // Q as the TMEM A operand of S_j
  static constexpr int kQBuf = SPLIT ? 1 : 2;        // Q / dO ring depth
  static constexpr int kKSt = SPLIT ? 2 : kKStages;  // K ring depth
  static constexpr int kPanels = D / 64;
  static constexpr int kQBytes = 128 * 128 * kPanels;  // 128 rows x 128 B per panel
  static constexpr int kKVBytes = 64 * 128 * kPanels;
  static constexpr int kParts = SPLIT ? 2 : 1;
  // a Q / dO slot: Q, (Qlo,) dO
  static constexpr int kQSlot = (kParts + 1) * kQBytes;
  static constexpr int kSlotQ = 0, kSlotQlo = kQBytes, kSlotDO = kParts * kQBytes;
  static constexpr int kOffK = kQBuf * kQSlot;
  static constexpr int kOffKlo = kOffK + kKSt * kKVBytes;
  static constexpr int kOffV = kOffK + kParts * kKSt * kKVBytes;
  static constexpr int kOffBar = kOffV + kVStages * kKVBytes;
  static constexpr int kBytes = kOffBar + 512 + 1024;
  static_assert(kBytes <= (int)kMaxDynSmem, "shared memory");
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename OutT>
__device__ __forceinline__ void store_chunk(OutT* dst, const float* v);
template <>
__device__ __forceinline__ void store_chunk<__nv_bfloat16>(__nv_bfloat16* dst, const float* v) {
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    p[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                      pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
}
template <>
__device__ __forceinline__ void store_chunk<float>(float* dst, const float* v) {
  float4* p = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i) p[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

template <int D, typename OutT, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                       const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                       const __grid_constant__ CUtensorMap mql, const __grid_constant__ CUtensorMap mkl, ShapeArgs s,
                       DqArgs a) {
  using L = DqSmem<D, SPLIT>;
  constexpr int kKStages = L::kKSt;  // the K ring of this variant
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  auto bar_q = [&](int qs) { return smem_u32(&bars[qs == 0 ? 0 : 29]); };  // Q, dO of slot qs landed
  auto bar_kfull = [&](int st) { return smem_u32(&bars[1 + st]); };
  auto bar_kempty = [&](int st) { return smem_u32(&bars[5 + st]); };
  auto bar_vfull = [&](int st) { return smem_u32(&bars[9 + st]); };
  auto bar_vempty = [&](int st) { return smem_u32(&bars[11 + st]); };
  auto bar_sfull = [&](int b) { return smem_u32(&bars[13 + b]); };   // S_j, dP_j in TMEM
  auto bar_sfree = [&](int b) { return smem_u32(&bars[15 + b]); };   // ... read out by the rows
  auto bar_pready = [&](int b) { return smem_u32(&bars[17 + b]); };  // dS_j written
  auto bar_pfree = [&](int b) { return smem_u32(&bars[19 + b]); };   // dQ MMA reading dS_j done
  const uint32_t bar_dq = smem_u32(&bars[21]);      // every dQ MMA of the query block completed
  const uint32_t bar_gdrain = smem_u32(&bars[22]);  // every dQ MMA of the CTA completed
  const uint32_t bar_sdrain = smem_u32(&bars[23]);  // every S_j / dP_j MMA of the CTA completed
  // every S_j / dP_j MMA of the query block in slot qs completed
  auto bar_qfree = [&](int qs) { return smem_u32(&bars[qs == 0 ? 24 : 30]); };
  auto bar_item_full = [&](int i) { return smem_u32(&bars[25 + i]); };  // item slot i written
  auto bar_item_free = [&](int i) { return smem_u32(&bars[27 + i]); };  // ... and read by every role
  const uint32_t bar_qt = smem_u32(&bars[31]);  // the query block's Q copied into TMEM
  // 32 barriers occupy the first 256 bytes of the 512-byte barrier area
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffBar + 384);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffBar + 392);
  volatile int* item_slot = reinterpret_cast<volatile int*>(smem + L::kOffBar + 400);
  const WaitCtl wc{abort_flag, s.wait_ns};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Work items are query blocks (block x: block x % Tq of head x / Tq), taken in the order of
  // launch_item_order: each CTA stays resident and takes items from a counter over that
  // order, its first being order[blockIdx.x], the next order[gridDim.x + (counter value)].
  const int num_items = s.B * s.H * s.Tq;
  // list length of item x, clamped to [0, Tk] (the producer reports a bad value)
  auto item_len = [&](int x, bool report) {
    int nkv = a.row_cnt[x];
    if (nkv < 0 || nkv > s.Tk) {
      if (report) report_error(a.status, kDevErrBounds);
      nkv = nkv < 0 ? 0 : s.Tk;
    }
    return nkv;
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
    for (int qs = 0; qs < L::kQBuf; ++qs) {
      mbar_init(bar_q(qs), 1);
      mbar_init(bar_qfree(qs), 1);
    }
    mbar_init(bar_qt, 256);
    for (int st = 0; st < kKStages; ++st) {
      mbar_init(bar_kfull(st), 1);
      mbar_init(bar_kempty(st), 1);
    }
    for (int st = 0; st < kVStages; ++st) {
      mbar_init(bar_vfull(st), 1);
      mbar_init(bar_vempty(st), 1);
    }
    for (int bb = 0; bb < 2; ++bb) {
      mbar_init(bar_sfull(bb), 1);
      mbar_init(bar_sfree(bb), 256);
      mbar_init(bar_pready(bb), 256);
      mbar_init(bar_pfree(bb), 1);
      mbar_init(bar_item_full(bb), 1);
      mbar_init(bar_item_free(bb), kItemReaders);
    }
    mbar_init(bar_dq, 1);
    mbar_init(bar_gdrain, 1);
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

  // Barrier phases count list entries (J) and query blocks with a non-empty list (qn, an)
  // over all items of the CTA, so every ring runs on across item boundaries.
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_map(&mq);
      tma_prefetch_map(&mdo);
      tma_prefetch_map(&mk);
      tma_prefetch_map(&mv);
      bool ok = true;
      uint32_t J = 0, qn = 0;
      uint32_t nk = 0, nv = 0;  // K and V loads issued (J can lag one of them on the abort path)
      int x = blockIdx.x;
      for (int n = 0; ok; ++n) {
        const int slot = n & 1;
        if (n >= 2 && !mbar_wait(bar_item_free(slot), ((n >> 1) - 1) & 1, wc)) {
          ok = false;
          break;
        }
        const bool done = x >= num_items;
        int qb = done ? -1 : a.order[x];
        if (!done && (qb < 0 || qb >= num_items)) {
          report_error(a.status, kDevErrBounds);
          qb = 0;
        }
        item_slot[slot] = qb;
        mbar_arrive(bar_item_full(slot));
        if (done) break;
        const int xn = (int)gridDim.x + atomicAdd(a.work_ctr, 1);  // the item after this one
        const int nkv = item_len(qb, true);
        if (nkv > 0) {
          const int bh = qb / s.Tq, qi = qb - bh * s.Tq, b = bh / s.H, h = bh - b * s.H;
          const int32_t* list = a.row_idx + (int64_t)qb * s.Tk;
          // slot qs last held Q, dO of query block qn - kQBuf: free once its S_j / dP_j MMAs
          // completed (the row threads copied that Q into TMEM before its first S_j)
          const int qs = (int)(qn % L::kQBuf);
          if (qn >= (uint32_t)L::kQBuf && !mbar_wait(bar_qfree(qs), ((qn / L::kQBuf) - 1) & 1, wc)) {
            ok = false;
            break;
          }
          ++qn;
          const uint32_t slot_base = sbase + qs * L::kQSlot;
          mbar_arrive_expect_tx(bar_q(qs), L::kQSlot);
          for (int p = 0; p < L::kPanels; ++p) {
            tma_load_4d(slot_base + L::kSlotQ + p * 16384, &mq, bar_q(qs), p * 64, qi * s.bq, h, b);
            if constexpr (SPLIT)
              tma_load_4d(slot_base + L::kSlotQlo + p * 16384, &mql, bar_q(qs), p * 64, qi * s.bq, h, b);
            tma_load_4d(slot_base + L::kSlotDO + p * 16384, &mdo, bar_q(qs), p * 64, qi * s.bq, h, b);
          }
          for (int j = 0; j < nkv; ++j, ++J) {
            const int ks = J % kKStages, vs = J % kVStages;
            int kb = list[j];
            if (kb < 0 || kb >= s.Tk) {
              report_error(a.status, kDevErrBounds);
              kb = 0;
            }
            if (J >= kKStages && !mbar_wait(bar_kempty(ks), ((J / kKStages) - 1) & 1, wc)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar_kfull(ks), L::kParts * L::kKVBytes);
            for (int p = 0; p < L::kPanels; ++p) {
              tma_load_4d(sbase + L::kOffK + ks * L::kKVBytes + p * 8192, &mk, bar_kfull(ks), p * 64, kb * 64, h,
                          b);
              if constexpr (SPLIT)
                tma_load_4d(sbase + L::kOffKlo + ks * L::kKVBytes + p * 8192, &mkl, bar_kfull(ks), p * 64, kb * 64,
                            h, b);
            }
            ++nk;
            if (J >= kVStages && !mbar_wait(bar_vempty(vs), ((J / kVStages) - 1) & 1, wc)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar_vfull(vs), L::kKVBytes);
            for (int p = 0; p < L::kPanels; ++p)
              tma_load_4d(sbase + L::kOffV + vs * L::kKVBytes + p * 8192, &mv, bar_vfull(vs), p * 64, kb * 64, h,
                          b);
            ++nv;
          }
        }
        x = xn;
      }
      // No copy may still be in flight when the CTA exits, whether the loop ran to its end or
      // gave up: drain the last load of each stage and of each Q / dO slot (each is its
      // barrier's latest phase).
      for (uint32_t v = nk > kKStages ? nk - kKStages : 0; v < nk; ++v)
        mbar_drain(bar_kfull(v % kKStages), (v / kKStages) & 1, abort_flag);
      for (uint32_t v = nv > kVStages ? nv - kVStages : 0; v < nv; ++v)
        mbar_drain(bar_vfull(v % kVStages), (v / kVStages) & 1, abort_flag);
      for (uint32_t v = qn > (uint32_t)L::kQBuf ? qn - L::kQBuf : 0; v < qn; ++v)
        mbar_drain(bar_q((int)(v % L::kQBuf)), (v / L::kQBuf) & 1, abort_flag);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S_j, dP_j issuer
    constexpr uint32_t idS = idesc_f16_f32(128, 64, false, false);
    bool ok = true;
    uint32_t J = 0, qn = 0;
    for (int n = 0; ok; ++n) {
      const int x = take_item(n, ok);
      if (x < 0) break;
      const int nkv = item_len(x, false);
      if (nkv == 0) continue;
      // Q, dO of the block landed in slot qs (and, for Q in TMEM, Q copied there)
      const int qs = (int)(qn % L::kQBuf);
      if (!__all_sync(0xffffffffu, mbar_wait(bar_q(qs), (qn / L::kQBuf) & 1, wc) &&
                                       (!L::kQInTmem || mbar_wait(bar_qt, qn & 1, wc)))) {
        ok = false;
        break;
      }
      ++qn;
      const uint32_t slot_base = sbase + qs * L::kQSlot;
      const uint64_t qd = smem_desc(slot_base + L::kSlotQ, 16, 1024), dod = smem_desc(slot_base + L::kSlotDO, 16, 1024);
      for (int j = 0; j < nkv; ++j, ++J) {
        const int ks = J % kKStages, vs = J % kVStages, bb = J & 1;
        // K_j and V_j present, and buffer bb (S_{j-2} / dP_{j-2}) read out by the row
        // threads, before the S_j and dP_j MMAs issue as one group
        if (!__all_sync(0xffffffffu,
                        mbar_wait(bar_kfull(ks), (J / kKStages) & 1, wc) &&
                            (J < 2 || mbar_wait(bar_sfree(bb), ((J >> 1) - 1) & 1, wc)) &&
                            mbar_wait(bar_vfull(vs), (J / kVStages) & 1, wc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t kd = smem_desc(sbase + L::kOffK + ks * L::kKVBytes, 16, 1024);
        const uint64_t vd = smem_desc(sbase + L::kOffV + vs * L::kKVBytes, 16, 1024);
        if (elect_one()) {
          if constexpr (L::kQInTmem)
            mma_ts_bkmajor<idS, 64, D / 16>(tmem + kColS + bb * 64, tmem + kColQ, kd);
          else
            mma_ss_kmajor<idS, 128, 64, D / 16>(tmem + kColS + bb * 64, qd, kd);
          if constexpr (SPLIT) {
            const uint64_t kld = smem_desc(sbase + L::kOffKlo + ks * L::kKVBytes, 16, 1024);
            const uint64_t qld = smem_desc(slot_base + L::kSlotQlo, 16, 1024);
            mma_ss_kmajor_acc<idS, 128, 64, D / 16>(tmem + kColS + bb * 64, qd, kld);
            mma_ss_kmajor_acc<idS, 128, 64, D / 16>(tmem + kColS + bb * 64, qld, kd);
          }
          mma_ss_kmajor<idS, 128, 64, D / 16>(tmem + kColDP + bb * 64, dod, vd);
          umma_commit(bar_sfull(bb));
          umma_commit(bar_vempty(vs));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) umma_commit(bar_qfree(qs));
      __syncwarp();
    }
    // no MMA of this warp may still run when TMEM is released, on the abort path too
    if (elect_one()) umma_commit(bar_sdrain);
    __syncwarp();
    mbar_drain(bar_sdrain, 0, abort_flag);
  } else if (warp == 2) {
    // ------------------------------------------------------------------ dQ issuer
    constexpr uint32_t idQ = idesc_f16_f32(128, D, false, true);
    bool ok = true;
    uint32_t J = 0;
    for (int n = 0; ok; ++n) {
      const int x = take_item(n, ok);
      if (x < 0) break;
      const int nkv = item_len(x, false);
      for (int j = 0; j < nkv; ++j, ++J) {
        const int ks = J % kKStages, bb = J & 1;
        // dS_j written.  For the first entry of a query block this also orders the
        // overwrite of the dQ accumulator after the previous block's epilogue: every row
        // thread read dQ out before it wrote this dS.
        if (!__all_sync(0xffffffffu, mbar_wait(bar_pready(bb), (J >> 1) & 1, wc) &&
                                         mbar_wait(bar_kfull(ks), (J / kKStages) & 1, wc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // K as the MN-major B operand: N = D (64-element groups 8 KB apart), K = 16 keys
        const uint64_t kmn = smem_desc(sbase + L::kOffK + ks * L::kKVBytes, 8192, 1024);
        if (elect_one()) {
          mma_ts_bmn<idQ, 4>(tmem + kColDQ, tmem + kColDS + bb * 32, kmn, j == 0);
          umma_commit(bar_kempty(ks));
          umma_commit(bar_pfree(bb));
        }
        __syncwarp();
      }
      if (!ok) break;
      // the block's S_j / dP_j MMAs all completed before its last dS was written, so this
      // commit covers every MMA of the block
      if (nkv > 0 && elect_one()) umma_commit(bar_dq);
      __syncwarp();
    }
    if (elect_one()) umma_commit(bar_gdrain);
    __syncwarp();
    mbar_drain(bar_gdrain, 0, abort_flag);
  } else {
    // -------------------------------------------------------------- query-row threads
    if (s.stall_ns && blockIdx.x == 0) stall_for(s.stall_ns);  // failure-path test hook
    const int wg = (warp - 3) >> 2;  // row warpgroup 0 or 1
    const int sub = warp & 3;
    const int r = 32 * sub + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * sub) << 16);
    const int c_begin = wg * (D / 2), c_end = c_begin + D / 2;
    bool ok = true;
    uint32_t J = 0, an = 0, qc = 0;
    // Q of the next query block with a non-empty list into TMEM: thread = row = TMEM lane,
    // group wg the 64 channels of panel wg (for d = 64 group 0 copies the one panel).  Every
    // S_j MMA reading the TMEM copy of the previous block has completed: the rows read the
    // last S_j of every earlier block before they get here.
    auto copy_q = [&]() {
      const int qs = (int)(qc % L::kQBuf);
      if (!__all_sync(0xffffffffu, mbar_wait(bar_q(qs), (qc / L::kQBuf) & 1, wc))) return false;
      ++qc;
      if (wg < L::kPanels) {
        const uint8_t* src = smem + qs * L::kQSlot + L::kSlotQ + wg * 16384 + r * 128;
        uint32_t v[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // 16-byte chunk c of the row sits at chunk c ^ (r % 8)
          const uint4 w = *reinterpret_cast<const uint4*>(src + ((c ^ (r & 7)) << 4));
          v[4 * c] = w.x;
          v[4 * c + 1] = w.y;
          v[4 * c + 2] = w.z;
          v[4 * c + 3] = w.w;
        }
        tmem_st32(trow + kColQ + 32 * wg, v);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(bar_qt);
      return true;
    };
    int x = take_item(0, ok);
    if (L::kQInTmem && ok && x >= 0 && item_len(x, false) > 0) ok = copy_q();
    for (int n = 0; ok && x >= 0; ++n) {
      const int nkv = item_len(x, false);
      const int bh = x / s.Tq, qi = x - bh * s.Tq, b = bh / s.H, h = bh - b * s.H;
      const int32_t* list = a.row_idx + (int64_t)x * s.Tk;
      const int64_t tok = (int64_t)qi * s.bq + r;
      const bool row_valid = r < s.bq && tok < s.N;
      // statistics record of this row: 64-row sub-tile (qi * bq + r) / 64 of the head
      const float* rec =
          a.stats + ((int64_t)bh * (s.Tq * (s.bq / 64)) + ((qi * s.bq + r) >> 6)) * 128 + (r & 63);
      const float lse2 = row_valid && nkv > 0 ? rec[0] : 0.f;
      const float Dr = row_valid && nkv > 0 ? rec[64] : 0.f;
      // both groups take every entry j (TMEM buffers J % 2), group wg its key columns
      // 32 wg .. 32 wg + 31
      int next_kb = nkv > 0 ? list[0] : 0;
      for (int j = 0; j < nkv; ++j, ++J) {
        const int bb = J & 1, jn = J >> 1;
        int kb = next_kb;
        if (j + 1 < nkv) next_kb = list[j + 1];
        if (!__all_sync(0xffffffffu, mbar_wait(bar_sfull(bb), jn & 1, wc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        kb = (kb < 0 || kb >= s.Tk) ? 0 : kb;
        const int kv_valid = min(64, s.N - kb * 64);
        uint32_t sv[32], dv[32], pk[16];
        tmem_ld32(trow + kColS + bb * 64 + 32 * wg, sv);
        tmem_ld32(trow + kColDP + bb * 64 + 32 * wg, dv);
        tmem_ld_wait(sv);
        tmem_ld_wait(dv);
        // S_j / dP_j are in registers: their buffer may be overwritten
        tc_fence_before();
        mbar_arrive(bar_sfree(bb));
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float ds[2];
#pragma unroll
          for (int z = 0; z < 2; ++z) {
            const bool cv = row_valid && (32 * wg + c + z) < kv_valid;
            const float p = cv ? ex2(fmaf(__uint_as_float(sv[c + z]), a.scale_log2, -lse2)) : 0.f;
            ds[z] = p * (__uint_as_float(dv[c + z]) - Dr);
          }
          pk[c / 2] = pack_f16x2(ds[0], ds[1]);
        }
        // dS buffer bb was last read by the dQ MMA of entry J - 2
        if (jn >= 1 && !__all_sync(0xffffffffu, mbar_wait(bar_pfree(bb), (jn - 1) & 1, wc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st16(trow + kColDS + bb * 32 + 16 * wg, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_pready(bb));
      }
      if (!ok) break;
      // the next query block, so that its Q is in TMEM (and its S_j can start) before this
      // block's epilogue
      const int xn = take_item(n + 1, ok);
      if (!ok) break;
      if (L::kQInTmem && xn >= 0 && item_len(xn, false) > 0 && !copy_q()) {
        ok = false;
        break;
      }
      // ---- epilogue: dQ = scale * (dS K) accumulated over the list; each group stores
      // half of the channels of every row
      OutT* dqrow = reinterpret_cast<OutT*>(a.dq) + (int64_t)b * a.g_sb + (int64_t)h * a.g_sh + tok * a.g_sn;
      if (nkv == 0) {
        if (row_valid) {
          float z[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) z[c] = 0.f;
          for (int c0 = c_begin; c0 < c_end; c0 += 32) store_chunk<OutT>(dqrow + c0, z);
        }
      } else {
        if (!__all_sync(0xffffffffu, mbar_wait(bar_dq, an & 1, wc))) {
          ok = false;
          break;
        }
        ++an;
        tc_fence_after();
#pragma unroll 1
        for (int c0 = c_begin; c0 < c_end; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(trow + kColDQ + c0, o);
          tmem_ld_wait(o);
          float v[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = __uint_as_float(o[c]) * a.scale;
          if (row_valid) store_chunk<OutT>(dqrow + c0, v);
        }
        tc_fence_before();
      }
      x = xn;
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

template <int D, typename OutT, bool SPLIT>
cudaError_t launch_t(const ShapeArgs& s, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                     const CUtensorMap& mdo, const CUtensorMap& mql, const CUtensorMap& mkl, const DqArgs& a,
                     cudaStream_t st) {
  const int smem = DqSmem<D, SPLIT>::kBytes;
  auto kern = attn_bwd_dq_kernel<D, OutT, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long items = (long long)s.B * s.H * s.Tq;
  const long long grid = items < sms ? items : sms;  // persistent: one CTA per SM
  // the work counter is zeroed by the pair-list pass of the same call
  if (!a.order_ready) e = launch_item_order(a.row_cnt, s.B * s.H, s.Tq, s.Tk, (int)grid, a.order, a.work_ctr, st);
  prof_start(st, kAttnBwdDq);
  if (e == cudaSuccess) kern<<<(unsigned)grid, kThreads, smem, st>>>(mq, mk, mv, mdo, mql, mkl, s, a);
  prof_stop(st, kAttnBwdDq);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace

cudaError_t launch_attn_bwd_dq(const ShapeArgs& s, const CUtensorMap& mq, const CUtensorMap& mk,
                               const CUtensorMap& mv, const CUtensorMap& mdo, const CUtensorMap* mql,
                               const CUtensorMap* mkl, const DqArgs& a, cudaStream_t st) {
  if ((long long)s.B * s.H * s.Tq > INT32_MAX) return cudaErrorInvalidValue;
  // fp32 calls take the split S product
  if (s.dtype != 0 && (!mql || !mkl)) return cudaErrorInvalidValue;
  if (s.d == 128)
    return s.dtype == 0 ? launch_t<128, __nv_bfloat16, false>(s, mq, mk, mv, mdo, mq, mk, a, st)
                        : launch_t<128, float, true>(s, mq, mk, mv, mdo, *mql, *mkl, a, st);
  return s.dtype == 0 ? launch_t<64, __nv_bfloat16, false>(s, mq, mk, mv, mdo, mq, mk, a, st)
                      : launch_t<64, float, true>(s, mq, mk, mv, mdo, *mql, *mkl, a, st);
}

}  // namespace sa2
