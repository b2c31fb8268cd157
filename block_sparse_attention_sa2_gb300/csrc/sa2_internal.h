// Internal declarations shared by the translation units of libsa2 (not part of the ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/sa2.h"
#include "sa2_device.cuh"

namespace sa2 {

constexpr size_t kMaxDynSmem = 227 * 1024;

// Launch profiler (profiler.cu): kernel ids and the brackets every launch wrapper calls.
enum KernelId {
  kPool = 0, kScoreSelect, kCsc, kToF16, kAttnFwd, kBwdPre, kAttnBwd, kAttnBwdDq, kBwdPairs, kVdLoss, kScoreTc,
  kItemOrder, kNumKernelIds
};
void prof_start(cudaStream_t st, int id);
void prof_stop(cudaStream_t st, int id);

// Shape of one call, with the derived block counts.  Strides are in elements.  wait_ns is
// the time limit of the attention kernels' bounded waits; stall_ns (0 in normal use) makes
// the row warps of their first CTA sleep that long before they start, so that a test of the
// failure path can make a wait expire (sa2_debug_set_wait_limit).
struct ShapeArgs {
  int B, H, N, d, bq, bk, Tq, Tk, dtype;
  int64_t sb, sh, sn;
  unsigned long long wait_ns, stall_ns;
};

// Validates a shape and fills the derived block counts and the wait settings (sa2_api.cu).
sa2_status check_shape(const sa2_shape* shape, ShapeArgs* s);
bool aligned16(const void* p);

// Selection parameters of the hybrid mask, prepared on the host.
struct SelectArgs {
  int K;                      // ceil(k * Tk) clamped to [0, Tk]
  int p_mode;                 // 0: 0 < p < 1, 1: p <= 0 (m = 0), 2: p >= 1 (m = Tk)
  unsigned long long p_fix;   // floor(p * 2^60), used when p_mode == 0
  float inv_sqrt_d;           // 1/sqrt(d) rounded to fp32
};

// Validates k and p of a mask call and prepares the selection parameters (sa2_api.cu).
sa2_status make_select_args(const ShapeArgs& s, float topk, float topp, SelectArgs* sel);

struct MaskOut {
  int32_t* row_cnt;
  int32_t* row_idx;
  int32_t* col_cnt;
  int32_t* col_idx;
  uint8_t* mask;      // may be null (not written)
  float* pooled_p;    // may be null
  unsigned* status;   // device status word
};

// Mask builder (mask_kernels.cu).
int score_rows_per_cta(int Tk, int d);
// Bytes of the builder's scratch: the pooled TF32 pairs of Q and K and the score tiles of
// one chunk of heads.  budget = 0: the default chunk; otherwise the scratch of the largest
// chunk that fits `budget` bytes (a result above budget means not even one head fits).
size_t mask_scratch_bytes(const ShapeArgs& s, size_t budget);
// scratch_bytes: the bytes behind `scratch` (0: mask_scratch_bytes(s, 0) of them).
cudaError_t launch_build_mask(const ShapeArgs& s, const void* q, const void* k, const SelectArgs& sel, void* scratch,
                              size_t scratch_bytes, const MaskOut& out, cudaStream_t st);

// Tensor maps of bf16 token tensors [B, H, N, d] (attn_common.cu).
bool make_token_map(CUtensorMap* map, const void* base, const ShapeArgs& s, int64_t sb, int64_t sh, int64_t sn,
                    int box_rows, bool f16);

// Element-wise helpers (attn_common.cu).
// fp16 copy of a token tensor into contiguous [B, H, N, d]; with dst_lo, also the residual
// fp16(x - hi) of each element (fp32 sources: hi + lo carries ~22 bits).
cudaError_t launch_to_f16(const void* src, const ShapeArgs& s, __half* dst, unsigned* status, cudaStream_t st,
                          __half* dst_lo = nullptr);

// The launch order of the B*H*Tq query blocks for kernels that take one query block per
// work item: head by head, each head's blocks by descending kept-list length (lengths clamped
// to [0, Tk]; equal lengths in no fixed order), except that lists too long to start late
// (longer than (heads - h) * W_h / slots blocks for head h with W_h its total, slots the CTAs
// resident at once) come first, all heads' together by descending length.  order holds
// item_order_ints(heads, Tq, Tk) integers: the order, then the scratch of the two passes.
// Also zeroes *work_ctr (when not null).  One CTA per head and pass.
size_t item_order_ints(int heads, int Tq, int Tk);
cudaError_t launch_item_order(const int32_t* row_cnt, int heads, int Tq, int Tk, int slots, int32_t* order,
                              int* work_ctr, cudaStream_t st);

struct FwdArgs {
  const int32_t* row_cnt;
  const int32_t* row_idx;
  int32_t* order;    // workspace: the launch order of the query blocks (launch_item_order)
  void* o;           // output, dtype of the call
  void* o_lo;        // optional bf16 residual O - bf16(O) (bf16 calls only), or null
  float* lse;        // [B, H, N]
  int64_t o_sb, o_sh, o_sn;
  float scale_log2;  // softmax scale * log2(e)
  unsigned* status;
};

// S = Q K^T reads bf16 Q and K (s_f16 = false, bf16 calls) or their fp16 copies (fp32
// calls; with the maps of their fp16 residuals mql, mkl, S is the split product
// Qhi Khi^T + Qhi Klo^T + Qlo Khi^T); P V always reads fp16 P and V.
cudaError_t launch_attn_fwd(const ShapeArgs& s, bool s_f16, const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& mv, const CUtensorMap* mql, const CUtensorMap* mkl, const FwdArgs& a,
                            cudaStream_t st);

// Per-row statistics of the backward, one record per 64-row query sub-tile:
// stats[(bh * Tsub + r) * 128 + i] = log2(e) * LSE of row 64 r + i (+inf past N), and
// stats[... + 64 + i] = D of that row (0 past N), with Tsub = Tq * bq / 64.
inline int64_t bwd_stats_floats(const ShapeArgs& s) { return (int64_t)s.B * s.H * s.Tq * (s.bq / 64) * 128; }

struct BwdArgs {
  const int32_t* col_cnt;  // mask column lists: input of the pair-union pass
  const int32_t* col_idx;
  int32_t* pair_cnt;       // [B*H, ceil(Tk/2)] union lengths (workspace)
  uint32_t* pair_idx;      // [B*H, ceil(Tk/2), Tq] union entries: q block | bit 30 kept by
                           // block 2m | bit 31 kept by block 2m+1 (workspace)
  const float* stats;      // per-row statistics, layout above
  int* work_ctr;           // [kBwdWorkCounters] item counters of the persistent kernels
                           // (workspace; zeroed by the pair-union pass)
  void* dk;
  void* dv;
  int64_t g_sb, g_sh, g_sn;  // strides of dk / dv (dtype of the call)
  float scale;
  float scale_log2;
  unsigned* status;
};

struct DqArgs {
  const int32_t* row_cnt;
  const int32_t* row_idx;
  int32_t* order;    // workspace: the launch order of the query blocks (launch_item_order)
  bool order_ready;  // order already holds a launch order (the forward's): not rebuilt
  const float* stats;
  int* work_ctr;  // item counter of the persistent kernel (workspace; zeroed by the pair-list pass)
  void* dq;
  int64_t g_sb, g_sh, g_sn;
  float scale;
  float scale_log2;
  unsigned* status;
};

// Entries of BwdArgs::pair_idx.
size_t bwd_pair_entries(const ShapeArgs& s);
constexpr int kBwdWorkCounters = 2;  // dK/dV kernel, dQ kernel

// dO -> fp16 copy, D = rowsum(dO * (O + O_lo)) and log2(e) * LSE into the per-row
// statistics, in one pass (attn_common.cu).
cudaError_t launch_do_prep(const ShapeArgs& s, const void* dO, const void* o, const void* o_lo, const float* lse,
                           __half* dO16, float* stats, unsigned* status, cudaStream_t st);
// fp32 calls (dtype 1) pass the maps of the fp16 residuals of Q and K (mql, mkl): their S
// product is split like the forward's; bf16 calls pass null.
cudaError_t launch_attn_bwd(const ShapeArgs& s, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            const CUtensorMap& mdo, const CUtensorMap* mql, const CUtensorMap* mkl, const BwdArgs& a,
                            cudaStream_t st);
cudaError_t launch_attn_bwd_dq(const ShapeArgs& s, const CUtensorMap& mq, const CUtensorMap& mk,
                               const CUtensorMap& mv, const CUtensorMap& mdo, const CUtensorMap* mql,
                               const CUtensorMap* mkl, const DqArgs& a, cudaStream_t st);

// Toy distillation loss (attn_common.cu): loss = sum (O_s - O_t)^2 into *loss (device),
// d_o = 2 (O_s - O_t); residuals optional (bf16 calls).  `partial` holds
// vd_loss_workspace_bytes() of per-CTA sums.
size_t vd_loss_workspace_bytes();
cudaError_t launch_vd_loss(const ShapeArgs& s, const void* os, const void* os_lo, const void* ot, const void* ot_lo,
                           void* d_o, double* loss, double* partial, cudaStream_t st);

}  // namespace sa2
