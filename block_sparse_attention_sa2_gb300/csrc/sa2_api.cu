// The C ABI (include/sa2.h): argument checks, workspace layout, tensor maps and launches.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>

#include "../../include/sa2.h"
#include "sa2_internal.h"

using namespace sa2;

namespace {

// Device-side error word; kernels write the first error code into it.
__device__ unsigned g_device_status;

constexpr int kMaxDevices = 64;
unsigned* g_status_ptr[kMaxDevices];
std::once_flag g_status_once[kMaxDevices];

unsigned* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::call_once(g_status_once[dev], [dev]() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) == cudaSuccess) g_status_ptr[dev] = static_cast<unsigned*>(p);
  });
  return g_status_ptr[dev];
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Limits of the attention kernels' bounded waits, set by sa2_debug_set_wait_limit (0: the
// default limit, no stall).
std::atomic<unsigned long long> g_wait_limit_ns{0}, g_stall_ns{0};

}  // namespace

namespace sa2 {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

sa2_status check_shape(const sa2_shape* shape, ShapeArgs* s) {
  if (!shape) return SA2_ERR_INVALID_ARG;
  const sa2_shape& x = *shape;
  if (x.B < 1 || x.H < 1 || x.N < 1 || x.reserved != 0) return SA2_ERR_INVALID_ARG;
  if (x.dtype != SA2_BF16 && x.dtype != SA2_FP32) return SA2_ERR_UNSUPPORTED;
  if (x.d != 64 && x.d != 128) return SA2_ERR_UNSUPPORTED;
  if ((x.bq != 64 && x.bq != 128) || x.bk != 64) return SA2_ERR_UNSUPPORTED;
  const int64_t esz = x.dtype == SA2_BF16 ? 2 : 4;
  if (x.stride_n < x.d || x.stride_h < 1 || x.stride_b < 1) return SA2_ERR_INVALID_ARG;
  if ((x.stride_n * esz) % 16 || (x.stride_h * esz) % 16 || (x.stride_b * esz) % 16) return SA2_ERR_ALIGNMENT;
  s->B = x.B;
  s->H = x.H;
  s->N = x.N;
  s->d = x.d;
  s->bq = x.bq;
  s->bk = x.bk;
  s->Tq = (x.N + x.bq - 1) / x.bq;
  s->Tk = (x.N + x.bk - 1) / x.bk;
  s->dtype = x.dtype;
  s->sb = x.stride_b;
  s->sh = x.stride_h;
  s->sn = x.stride_n;
  const unsigned long long w = g_wait_limit_ns.load(std::memory_order_relaxed);
  s->wait_ns = w ? w : kWaitLimitNs;
  s->stall_ns = g_stall_ns.load(std::memory_order_relaxed);
  if (s->Tk > 7680 || score_rows_per_cta(s->Tk, s->d) == 0) return SA2_ERR_UNSUPPORTED;
  if ((int64_t)s->B * s->H * s->Tq >= (int64_t)1 << 31) return SA2_ERR_UNSUPPORTED;
  return SA2_OK;
}

sa2_status make_select_args(const ShapeArgs& s, float topk, float topp, SelectArgs* sel) {
  if (!std::isfinite(topk) || !std::isfinite(topp) || topk < 0.f || topk > 1.f || topp < 0.f || topp > 1.f)
    return SA2_ERR_INVALID_ARG;
  const double Kd = std::ceil((double)topk * s.Tk - 1e-9);
  sel->K = (int)std::fmin(std::fmax(Kd, 0.0), (double)s.Tk);
  if (topp <= 0.f) {
    sel->p_mode = 1;
    sel->p_fix = 0;
  } else if (topp >= 1.f) {
    sel->p_mode = 2;
    sel->p_fix = 0;
  } else {
    sel->p_mode = 0;
    sel->p_fix = (unsigned long long)std::ldexp((double)topp, 60);
  }
  sel->inv_sqrt_d = (float)(1.0 / std::sqrt((double)s.d));
  return SA2_OK;
}

}  // namespace sa2

namespace {

size_t token_elems(const ShapeArgs& s) { return (size_t)s.B * s.H * s.N * s.d; }

sa2_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SA2_OK : SA2_ERR_CUDA; }

// Mask workspace: the builder's scratch (pooled pairs, the chunk buffers).
struct MaskWs {
  size_t pooled, total;
};
MaskWs mask_ws(const ShapeArgs& s) {
  MaskWs w;
  w.pooled = 0;
  w.total = align_up(mask_scratch_bytes(s, 0));
  return w;
}

// Forward workspace: the fp16 copy of V; for fp32 calls also the fp16 copies of Q and K and
// their fp16 residuals (the split S product); the launch order of the query blocks.
struct FwdWs {
  size_t v16, q16, k16, q16lo, k16lo, order, total;
};
FwdWs fwd_ws(const ShapeArgs& s) {
  const size_t t = align_up(2 * token_elems(s));
  FwdWs w{};
  w.v16 = 0;
  w.total = t;
  if (s.dtype == SA2_FP32) {
    w.q16 = t;
    w.k16 = 2 * t;
    w.q16lo = 3 * t;
    w.k16lo = 4 * t;
    w.total = 5 * t;
  }
  w.order = w.total;  // the launch order of the query blocks
  w.total += align_up(sizeof(int32_t) * item_order_ints(s.B * s.H, s.Tq, s.Tk));
  return w;
}

// Backward workspace: per-row statistics, the pair-union lists of the dK / dV kernel, and
// fp16 copies of Q, K, V, dO.
struct BwdWs {
  size_t stats, pair_cnt, pair_idx, q16, k16, v16, do16, ctr, order, q16lo, k16lo, total;
};
BwdWs bwd_ws(const ShapeArgs& s) {
  BwdWs w{};
  const size_t t = align_up(2 * token_elems(s));
  w.stats = 0;
  w.pair_cnt = align_up(sizeof(float) * (size_t)bwd_stats_floats(s));
  w.pair_idx = w.pair_cnt + align_up(sizeof(int32_t) * (size_t)s.B * s.H * ((s.Tk + 1) / 2));
  w.q16 = w.pair_idx + align_up(sizeof(uint32_t) * bwd_pair_entries(s));
  w.k16 = w.q16 + t;
  w.v16 = w.k16 + t;
  w.do16 = w.v16 + t;
  w.ctr = w.do16 + t;
  w.order = w.ctr + align_up(sizeof(int) * kBwdWorkCounters);
  w.total = w.order + align_up(sizeof(int32_t) * item_order_ints(s.B * s.H, s.Tq, s.Tk));
  if (s.dtype == SA2_FP32) {  // fp16 residuals of Q and K (the split S product)
    w.q16lo = w.total;
    w.k16lo = w.q16lo + t;
    w.total = w.k16lo + t;
  }
  return w;
}

// Tensor maps over 16-bit token tensors: the caller's bf16 tensors (strided) or the
// library's contiguous fp16 copies.
bool caller_map(const ShapeArgs& s, const void* base, CUtensorMap* map, int box_rows) {
  return make_token_map(map, base, s, s.sb, s.sh, s.sn, box_rows, false);
}
bool copy_map(const ShapeArgs& s, const void* base, CUtensorMap* map, int box_rows) {
  return make_token_map(map, base, s, (int64_t)s.H * s.N * s.d, (int64_t)s.N * s.d, s.d, box_rows, true);
}

}  // namespace

extern "C" {

int sa2_version(void) { return 100; }

const char* sa2_status_string(sa2_status st) {
  switch (st) {
    case SA2_OK: return "ok";
    case SA2_ERR_INVALID_ARG: return "invalid argument";
    case SA2_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case SA2_ERR_ALIGNMENT: return "pointer or stride not 16-byte aligned";
    case SA2_ERR_WORKSPACE: return "workspace missing or too small";
    case SA2_ERR_CUDA: return "CUDA error";
    case SA2_ERR_TIMEOUT: return "device wait timed out";
    case SA2_ERR_DEVICE_BOUNDS: return "block index out of range on the device";
    case SA2_ERR_RANGE: return "input magnitude beyond the fp16 range (saturated)";
  }
  return "unknown status";
}

size_t sa2_mask_workspace_size(const sa2_shape* shape) {
  ShapeArgs s;
  if (check_shape(shape, &s) != SA2_OK) return 0;
  return mask_ws(s).total;
}

sa2_status sa2_build_mask(const sa2_shape* shape, const void* q, const void* k, float topk, float topp,
                          const sa2_blockmask* out, void* ws, size_t ws_bytes, void* stream) {
  ShapeArgs s;
  sa2_status st = check_shape(shape, &s);
  if (st != SA2_OK) return st;
  if (!q || !k || !out || !out->row_cnt || !out->row_idx || !out->col_cnt || !out->col_idx)
    return SA2_ERR_INVALID_ARG;
  SelectArgs sel;
  st = make_select_args(s, topk, topp, &sel);
  if (st != SA2_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(out->row_cnt) || !aligned16(out->row_idx) ||
      !aligned16(out->col_cnt) || !aligned16(out->col_idx) || (out->mask && !aligned16(out->mask)) ||
      (out->pooled_p && !aligned16(out->pooled_p)) || !aligned16(ws))
    return SA2_ERR_ALIGNMENT;
  const MaskWs w = mask_ws(s);
  if (!ws || ws_bytes < w.total) return SA2_ERR_WORKSPACE;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  MaskOut mo;
  mo.row_cnt = out->row_cnt;
  mo.row_idx = out->row_idx;
  mo.col_cnt = out->col_cnt;
  mo.col_idx = out->col_idx;
  mo.mask = out->mask;  // null: not written
  mo.pooled_p = out->pooled_p;
  mo.status = status_ptr();
  return cuda_status(launch_build_mask(s, q, k, sel, wsb + w.pooled, 0, mo, static_cast<cudaStream_t>(stream)));
}

size_t sa2_fwd_workspace_size(const sa2_shape* shape) {
  ShapeArgs s;
  if (check_shape(shape, &s) != SA2_OK) return 0;
  return fwd_ws(s).total;
}

sa2_status sa2_attn_fwd(const sa2_shape* shape, const void* q, const void* k, const void* v,
                        const sa2_blockmask* mask, float softmax_scale, void* o, void* o_lo, float* lse, void* ws,
                        size_t ws_bytes, void* stream) {
  ShapeArgs s;
  sa2_status st = check_shape(shape, &s);
  if (st != SA2_OK) return st;
  if (!q || !k || !v || !o || !lse || !mask || !mask->row_cnt || !mask->row_idx) return SA2_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return SA2_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(o_lo) || !aligned16(lse) ||
      !aligned16(mask->row_cnt) || !aligned16(mask->row_idx) || !aligned16(ws))
    return SA2_ERR_ALIGNMENT;
  const FwdWs w = fwd_ws(s);
  if (!ws || ws_bytes < w.total) return SA2_ERR_WORKSPACE;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  unsigned* status = status_ptr();
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  __half* v16 = reinterpret_cast<__half*>(wsb + w.v16);
  if (launch_to_f16(v, s, v16, status, cs) != cudaSuccess) return SA2_ERR_CUDA;
  const bool f16_inputs = s.dtype == SA2_FP32;
  CUtensorMap mq, mk, mv, mql, mkl;
  if (f16_inputs) {
    __half* q16 = reinterpret_cast<__half*>(wsb + w.q16);
    __half* k16 = reinterpret_cast<__half*>(wsb + w.k16);
    __half* q16lo = reinterpret_cast<__half*>(wsb + w.q16lo);
    __half* k16lo = reinterpret_cast<__half*>(wsb + w.k16lo);
    if (launch_to_f16(q, s, q16, status, cs, q16lo) != cudaSuccess ||
        launch_to_f16(k, s, k16, status, cs, k16lo) != cudaSuccess)
      return SA2_ERR_CUDA;
    if (!copy_map(s, q16, &mq, 128) || !copy_map(s, k16, &mk, 64) || !copy_map(s, q16lo, &mql, 128) ||
        !copy_map(s, k16lo, &mkl, 64))
      return SA2_ERR_CUDA;
  } else {
    if (!caller_map(s, q, &mq, 128) || !caller_map(s, k, &mk, 64)) return SA2_ERR_CUDA;
  }
  if (!copy_map(s, v16, &mv, 64)) return SA2_ERR_CUDA;
  const float scale = softmax_scale > 0.f ? softmax_scale : (float)(1.0 / std::sqrt((double)s.d));
  FwdArgs a;
  a.row_cnt = mask->row_cnt;
  a.row_idx = mask->row_idx;
  a.order = reinterpret_cast<int32_t*>(wsb + w.order);
  a.o = o;
  a.o_lo = s.dtype == SA2_BF16 ? o_lo : nullptr;
  a.lse = lse;
  a.o_sb = s.sb;
  a.o_sh = s.sh;
  a.o_sn = s.sn;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
  return cuda_status(launch_attn_fwd(s, f16_inputs, mq, mk, mv, f16_inputs ? &mql : nullptr,
                                     f16_inputs ? &mkl : nullptr, a, cs));
}

size_t sa2_bwd_workspace_size(const sa2_shape* shape) {
  ShapeArgs s;
  if (check_shape(shape, &s) != SA2_OK) return 0;
  return bwd_ws(s).total;
}

namespace {

// The backward; fwd_workspace, when not null, is the (already validated) workspace of the
// forward call on the same q, k, v, whose fp16 copies replace the conversions here.
sa2_status attn_bwd_impl(const sa2_shape* shape, const void* q, const void* k, const void* v, const void* o,
                         const void* o_lo, const float* lse, const void* dO, const sa2_blockmask* mask,
                         float softmax_scale, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                         const void* fwd_workspace, void* stream) {
  ShapeArgs s;
  sa2_status st = check_shape(shape, &s);
  if (st != SA2_OK) return st;
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !mask || !mask->col_cnt || !mask->col_idx ||
      !mask->row_cnt || !mask->row_idx)
    return SA2_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return SA2_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(o_lo) || !aligned16(lse) ||
      !aligned16(dO) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(mask->col_cnt) ||
      !aligned16(mask->col_idx) || !aligned16(mask->row_cnt) || !aligned16(mask->row_idx) || !aligned16(ws))
    return SA2_ERR_ALIGNMENT;
  const BwdWs w = bwd_ws(s);
  if (!ws || ws_bytes < w.total) return SA2_ERR_WORKSPACE;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  unsigned* status = status_ptr();
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  float* stats = reinterpret_cast<float*>(wsb + w.stats);
  __half* c16[4] = {reinterpret_cast<__half*>(wsb + w.q16), reinterpret_cast<__half*>(wsb + w.k16),
                    reinterpret_cast<__half*>(wsb + w.v16), reinterpret_cast<__half*>(wsb + w.do16)};
  const bool split = s.dtype == SA2_FP32;  // fp32 calls: fp16 residuals of Q and K too
  __half* lo16[3] = {split ? reinterpret_cast<__half*>(wsb + w.q16lo) : nullptr,
                     split ? reinterpret_cast<__half*>(wsb + w.k16lo) : nullptr, nullptr};
  const void* src[3] = {q, k, v};
  bool copied[3] = {false, false, false};
  int32_t* fwd_order = nullptr;
  if (fwd_workspace) {
    // the forward's fp16 copies: v always, q and k (and their residuals) for fp32 inputs; and
    // its launch order of the query blocks, a permutation the dQ kernel takes as it is
    const FwdWs fw = fwd_ws(s);
    const uint8_t* fb = static_cast<const uint8_t*>(fwd_workspace);
    fwd_order = reinterpret_cast<int32_t*>(const_cast<uint8_t*>(fb + fw.order));
    c16[2] = reinterpret_cast<__half*>(const_cast<uint8_t*>(fb + fw.v16));
    copied[2] = true;
    if (split) {
      c16[0] = reinterpret_cast<__half*>(const_cast<uint8_t*>(fb + fw.q16));
      c16[1] = reinterpret_cast<__half*>(const_cast<uint8_t*>(fb + fw.k16));
      lo16[0] = reinterpret_cast<__half*>(const_cast<uint8_t*>(fb + fw.q16lo));
      lo16[1] = reinterpret_cast<__half*>(const_cast<uint8_t*>(fb + fw.k16lo));
      copied[0] = copied[1] = true;
    }
  }
  for (int i = 0; i < 3; ++i)
    if (!copied[i] && launch_to_f16(src[i], s, c16[i], status, cs, lo16[i]) != cudaSuccess) return SA2_ERR_CUDA;
  // fp16 dO, and D = rowsum(dO * O) from that same fp16 dO, in one pass
  if (launch_do_prep(s, dO, o, s.dtype == SA2_BF16 ? o_lo : nullptr, lse, c16[3], stats, status, cs) !=
      cudaSuccess)
    return SA2_ERR_CUDA;
  // the dK / dV kernel reads 64-row query sub-tiles, the dQ kernel 128-row query tiles
  CUtensorMap mq64, mdo64, mq, mk, mv, mdo, mql64, mql, mkl;
  if (!copy_map(s, c16[0], &mq64, 64) || !copy_map(s, c16[3], &mdo64, 64) || !copy_map(s, c16[0], &mq, 128) ||
      !copy_map(s, c16[1], &mk, 64) || !copy_map(s, c16[2], &mv, 64) || !copy_map(s, c16[3], &mdo, 128))
    return SA2_ERR_CUDA;
  if (split && (!copy_map(s, lo16[0], &mql64, 64) || !copy_map(s, lo16[0], &mql, 128) ||
                !copy_map(s, lo16[1], &mkl, 64)))
    return SA2_ERR_CUDA;
  const float scale = softmax_scale > 0.f ? softmax_scale : (float)(1.0 / std::sqrt((double)s.d));
  BwdArgs a;
  a.col_cnt = mask->col_cnt;
  a.col_idx = mask->col_idx;
  a.pair_cnt = reinterpret_cast<int32_t*>(wsb + w.pair_cnt);
  a.pair_idx = reinterpret_cast<uint32_t*>(wsb + w.pair_idx);
  a.work_ctr = reinterpret_cast<int*>(wsb + w.ctr);
  a.stats = stats;
  a.dk = dk;
  a.dv = dv;
  a.g_sb = s.sb;
  a.g_sh = s.sh;
  a.g_sn = s.sn;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
  if (launch_attn_bwd(s, mq64, mk, mv, mdo64, split ? &mql64 : nullptr, split ? &mkl : nullptr, a, cs) !=
      cudaSuccess)
    return SA2_ERR_CUDA;
  DqArgs g;
  g.row_cnt = mask->row_cnt;
  g.row_idx = mask->row_idx;
  g.order = fwd_order ? fwd_order : reinterpret_cast<int32_t*>(wsb + w.order);
  g.order_ready = fwd_order != nullptr;
  g.stats = stats;
  g.work_ctr = a.work_ctr + 1;
  g.dq = dq;
  g.g_sb = s.sb;
  g.g_sh = s.sh;
  g.g_sn = s.sn;
  g.scale = scale;
  g.scale_log2 = a.scale_log2;
  g.status = status;
  return cuda_status(launch_attn_bwd_dq(s, mq, mk, mv, mdo, split ? &mql : nullptr, split ? &mkl : nullptr, g, cs));
}

}  // namespace

sa2_status sa2_attn_bwd(const sa2_shape* shape, const void* q, const void* k, const void* v, const void* o,
                        const void* o_lo, const float* lse, const void* dO, const sa2_blockmask* mask,
                        float softmax_scale, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, void* stream) {
  return attn_bwd_impl(shape, q, k, v, o, o_lo, lse, dO, mask, softmax_scale, dq, dk, dv, ws, ws_bytes, nullptr,
                       stream);
}

sa2_status sa2_attn_bwd_with_fwd_ws(const sa2_shape* shape, const void* q, const void* k, const void* v,
                                    const void* o, const void* o_lo, const float* lse, const void* dO,
                                    const sa2_blockmask* mask, float softmax_scale, void* dq, void* dk, void* dv,
                                    void* ws, size_t ws_bytes, const void* fwd_workspace,
                                    size_t fwd_workspace_bytes, void* stream) {
  ShapeArgs s;
  sa2_status st = check_shape(shape, &s);
  if (st != SA2_OK) return st;
  if (!fwd_workspace) return SA2_ERR_INVALID_ARG;
  if (!aligned16(fwd_workspace)) return SA2_ERR_ALIGNMENT;
  if (fwd_workspace_bytes < fwd_ws(s).total) return SA2_ERR_WORKSPACE;
  return attn_bwd_impl(shape, q, k, v, o, o_lo, lse, dO, mask, softmax_scale, dq, dk, dv, ws, ws_bytes,
                       fwd_workspace, stream);
}

size_t sa2_vd_loss_workspace_size(const sa2_shape* shape) {
  ShapeArgs s;
  if (check_shape(shape, &s) != SA2_OK) return 0;
  return vd_loss_workspace_bytes();
}

sa2_status sa2_vd_loss(const sa2_shape* shape, const void* o_s, const void* o_s_lo, const void* o_t,
                       const void* o_t_lo, void* d_o, double* loss, void* ws, size_t ws_bytes, void* stream) {
  ShapeArgs s;
  sa2_status st = check_shape(shape, &s);
  if (st != SA2_OK) return st;
  if (!o_s || !o_t || !d_o || !loss) return SA2_ERR_INVALID_ARG;
  if (s.dtype == SA2_BF16 && ((o_s_lo == nullptr) != (o_t_lo == nullptr))) return SA2_ERR_INVALID_ARG;
  if (!aligned16(o_s) || !aligned16(o_t) || !aligned16(d_o) || !aligned16(o_s_lo) || !aligned16(o_t_lo) ||
      (reinterpret_cast<uintptr_t>(loss) & 7u) || !aligned16(ws))
    return SA2_ERR_ALIGNMENT;
  if (!ws || ws_bytes < vd_loss_workspace_bytes()) return SA2_ERR_WORKSPACE;
  const bool lo = s.dtype == SA2_BF16 && o_s_lo;
  return cuda_status(launch_vd_loss(s, o_s, lo ? o_s_lo : nullptr, o_t, lo ? o_t_lo : nullptr, d_o, loss,
                                    static_cast<double*>(ws), static_cast<cudaStream_t>(stream)));
}

void sa2_debug_set_wait_limit(unsigned long long limit_ns, unsigned long long stall_ns) {
  g_wait_limit_ns.store(limit_ns, std::memory_order_relaxed);
  g_stall_ns.store(stall_ns, std::memory_order_relaxed);
}

sa2_status sa2_get_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SA2_ERR_CUDA;
  unsigned* p = status_ptr();
  if (!p) return SA2_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return SA2_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return SA2_ERR_CUDA;
  }
  return v == 0 ? SA2_OK : static_cast<sa2_status>(v);
}

}  // extern "C"
