// sa2_build_mask_noalloc: the hybrid block mask for callers that cannot allocate device
// memory.
//
// Some callers of this library have no way to hand it a workspace: code that runs inside
// another runtime's memory pool and may not call cudaMalloc (a custom allocator that is
// not re-entrant, a framework plugin that only receives tensors), or code on a path where
// an allocation would synchronize the device.  For them this entry point keeps the
// builder's scratch -- the fp32 pooled queries and keys -- in a fixed array of device
// memory that belongs to the library itself.  The array is static: every GPU that loads
// the library holds it until the process exits.
//
// The kernels are the ones sa2_build_mask launches; only where their scratch lives differs.
#include <cmath>
#include <mutex>

#include "../../include/sa2.h"
#include "sa2_internal.h"

using namespace sa2;

namespace {

// The builder's scratch.  In host code this name is only a host-side stand-in for the
// device array: its device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SA2_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];
std::once_flag g_scratch_once[kMaxDevices];

// Device address of the scratch array on the current device (set up on first use there).
void* scratch_for_current_device(cudaError_t* err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
    return nullptr;
  }
  std::call_once(g_scratch_once[dev], [dev]() {
    void* p = nullptr;
    g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    g_scratch_ptr[dev] = g_scratch_err[dev] == cudaSuccess ? p : nullptr;
  });
  *err = g_scratch_err[dev];
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" sa2_status sa2_build_mask_noalloc(const sa2_shape* shape, const void* q, const void* k, float topk,
                                             float topp, const sa2_blockmask* out, void* stream) {
  // the same validation as sa2_build_mask, then the size check of the static scratch
  ShapeArgs s;
  sa2_status st = check_shape(shape, &s);
  if (st != SA2_OK) return st;
  if (!q || !k || !out || !out->row_cnt || !out->row_idx || !out->col_cnt || !out->col_idx)
    return SA2_ERR_INVALID_ARG;
  SelectArgs sel;
  st = make_select_args(s, topk, topp, &sel);
  if (st != SA2_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(out->row_cnt) || !aligned16(out->row_idx) ||
      !aligned16(out->col_cnt) || !aligned16(out->col_idx) || !aligned16(out->mask) || !aligned16(out->pooled_p))
    return SA2_ERR_ALIGNMENT;

  // the pooled pairs of Q and K and the score tiles of at least one head must fit
  if (mask_scratch_bytes(s, SA2_NOALLOC_SCRATCH_BYTES) > (size_t)SA2_NOALLOC_SCRATCH_BYTES) return SA2_ERR_WORKSPACE;

  cudaError_t err = cudaSuccess;
  unsigned char* scratch = static_cast<unsigned char*>(scratch_for_current_device(&err));
  if (!scratch) return SA2_ERR_CUDA;

  MaskOut mo;
  mo.row_cnt = out->row_cnt;
  mo.row_idx = out->row_idx;
  mo.col_cnt = out->col_cnt;
  mo.col_idx = out->col_idx;
  mo.mask = out->mask;
  mo.pooled_p = out->pooled_p;
  mo.status = nullptr;
  // The pooling kernel writes every pooled element the scores read (rows past Tq / Tk are
  // read as zeros by the tensor copies and never come from the scratch), and the score
  // tiles are written before they are read, so nothing in the scratch has to start at zero.
  err = launch_build_mask(s, q, k, sel, scratch, SA2_NOALLOC_SCRATCH_BYTES, mo, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? SA2_OK : SA2_ERR_CUDA;
}
