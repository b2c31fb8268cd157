/*
 * sa2.h -- C ABI of the GB300 (sm_103a) hot path of SpargeAttention2: the hybrid
 * Top-k + Top-p block mask and trainable block-sparse attention.
 *
 * Source of every operation: the pages on "SpargeAttention2: Trainable Sparse Attention
 * via Hybrid Top-k+Top-p Masking and Distillation Fine-Tuning" (arXiv 2602.13515); the
 * passage each entry point follows is cited at its declaration.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Token tensors (q, k, v, o, dO, dq, dk, dv) are [B, H, N, d] with element strides
 *   stride_b, stride_h, stride_n (the last dimension is contiguous).  All token tensors of
 *   one call share these strides.  dtype is SA2_BF16 or SA2_FP32 for all of them.
 * - Blocks: query block i covers tokens [i*bq, min(N, (i+1)*bq)); key block j covers
 *   [j*bk, min(N, (j+1)*bk)).  Tq = ceil(N/bq), Tk = ceil(N/bk).  The last block of each
 *   may be partial.
 * - Supported: d in {64, 128}; bq in {64, 128}; bk = 64; 1 <= N; Tk <= 7680.
 * - Pointers are device pointers unless stated otherwise; every device pointer must be
 *   16-byte aligned and every stride * element size a multiple of 16 bytes.
 * - The caller owns every buffer, including the workspaces (sizes from the *_workspace_size
 *   queries).  The library allocates no device memory; it keeps one device status word, a
 *   few bytes of per-device set-up state, and the static scratch array of
 *   sa2_build_mask_noalloc (SA2_NOALLOC_SCRATCH_BYTES, part of the loaded module).
 * - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *   Argument errors are returned before anything is launched.  Errors raised by a kernel
 *   on the device (a bounded wait that timed out, a block index out of range) are recorded
 *   in the status word and reported by sa2_get_device_status.
 * - Attention is non-causal.  The softmax scale of the attention is an argument
 *   (1/sqrt(d) when <= 0 is passed); the pooled scores always use 1/sqrt(d).
 */
#ifndef SA2_H_
#define SA2_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sa2_status {
  SA2_OK = 0,
  SA2_ERR_INVALID_ARG = 1, /* null pointer, negative size, k/p not finite, ... */
  SA2_ERR_UNSUPPORTED = 2, /* d, bq, bk, dtype or size outside the supported set */
  SA2_ERR_ALIGNMENT = 3,   /* a pointer or stride is not 16-byte aligned */
  SA2_ERR_WORKSPACE = 4,   /* workspace missing or smaller than the size query returns */
  SA2_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed */
  SA2_ERR_TIMEOUT = 6,     /* device: a bounded wait inside a kernel gave up */
  SA2_ERR_DEVICE_BOUNDS = 7, /* device: a block list held an index out of range */
  SA2_ERR_RANGE = 8          /* device: an attention input exceeded the fp16 range (saturated) */
} sa2_status;

typedef enum sa2_dtype { SA2_BF16 = 0, SA2_FP32 = 1 } sa2_dtype;

typedef struct sa2_shape {
  int32_t B, H, N, d;
  int32_t bq, bk;
  int32_t dtype; /* sa2_dtype */
  int32_t reserved; /* must be 0 */
  int64_t stride_b, stride_h, stride_n; /* in elements */
} sa2_shape;

/*
 * The block mask in compact form.  All arrays are device arrays owned by the caller.
 *   row_cnt [B, H, Tq]      int32: number of kept key blocks of each query block
 *   row_idx [B, H, Tq, Tk]  int32: the first row_cnt entries of each row are the kept key
 *                                  blocks in ascending order; the rest is unspecified
 *   col_cnt [B, H, Tk]      int32: number of query blocks that keep each key block
 *   col_idx [B, H, Tk, Tq]  int32: the first col_cnt entries are those query blocks,
 *                                  ascending; the rest is unspecified
 *   mask    [B, H, Tq, Tk]  uint8: 1 = kept (optional output of sa2_build_mask; NULL skips)
 *   pooled_p[B, H, Tq, Tk]  fp32 : the pooled probabilities P-bar (optional; NULL skips)
 * sa2_attn_fwd reads row_cnt/row_idx; sa2_attn_bwd reads all four lists.
 */
typedef struct sa2_blockmask {
  int32_t* row_cnt;
  int32_t* row_idx;
  int32_t* col_cnt;
  int32_t* col_idx;
  uint8_t* mask;
  float* pooled_p;
} sa2_blockmask;

/* Library version (major*10000 + minor*100 + patch). */
int sa2_version(void);

/* Human-readable name of a status code (static string). */
const char* sa2_status_string(sa2_status status);

/*
 * Bytes of device workspace sa2_build_mask needs for this shape (the pooled queries and
 * keys as fp32 TF32 pairs, and two buffers of the score rows and kept bits of a chunk of
 * heads).  Returns 0 for an invalid shape.
 */
size_t sa2_mask_workspace_size(const sa2_shape* shape);

/*
 * sa2_build_mask -- the hybrid Top-k + Top-p block mask.
 * gist.science explainer of the paper, section 2.A (hybrid Top-k + Top-p masking):
 * P-bar is the attention map of block-pooled queries and keys; block j of row i is kept
 * iff j is in Top-k(P-bar_i, k%) or in Top-p(P-bar_i, p%).  Section 1 of the same page
 * defines Top-k (the k largest entries) and Top-p (the smallest set whose cumulative
 * probability reaches p).
 *
 * Steps: q-bar_i, k-bar_j = means of Q and K over the valid tokens of each block (fp32);
 * P-bar_i = softmax_j(q-bar_i . k-bar_j / sqrt(d)) (fp32); K = ceil(topk * Tk) clamped to
 * [0, Tk]; m = length of the shortest prefix of the row sorted by P-bar descending (equal
 * values by ascending block index) whose mass reaches topp (topp <= 0: m = 0; topp >= 1:
 * m = Tk; a mass that never reaches topp: m = Tk); the row keeps the first max(K, m)
 * blocks of that order.
 *
 *   q, k      token tensors (see conventions); read only
 *   topk      k as a fraction of Tk, in [0, 1]
 *   topp      p in [0, 1]
 *   out       the lists to fill; row_cnt, row_idx, col_cnt, col_idx are required; mask and
 *             pooled_p optional
 *   ws        device workspace of at least sa2_mask_workspace_size(shape) bytes
 */
sa2_status sa2_build_mask(const sa2_shape* shape, const void* q, const void* k, float topk, float topp,
                          const sa2_blockmask* out, void* ws, size_t ws_bytes, void* stream);

/*
 * sa2_build_mask_noalloc -- sa2_build_mask for callers that cannot allocate device memory.
 * The paper has no counterpart to this entry point; it exists for callers that are not
 * allowed to call cudaMalloc or hand the library a workspace: code running under another
 * runtime's memory pool or a non-re-entrant custom allocator, plugins that only receive
 * tensors, and paths where an allocation would synchronize the device.
 *
 * Same computation and outputs as sa2_build_mask, except that the builder's scratch (the
 * pooled queries and keys as fp32 TF32 pairs, 2*B*H*d*(Tq+Tk) floats, and two buffers of the
 * score rows and kept bits of a chunk of heads, the chunk as large as the array allows)
 * lives in a static device array of SA2_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads the library
 * holds until the process exits.  Nothing is allocated: no cudaMalloc, no cudaFree.
 *   - A shape whose scratch exceeds SA2_NOALLOC_SCRATCH_BYTES is rejected with
 *     SA2_ERR_WORKSPACE before anything is launched.
 *   - The first call on a device looks up the array's device address on that device (the
 *     device must be current); make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents.  Calls whose
 *     kernels overlap on the GPU (different streams, no ordering between them) race on it:
 *     order them on one stream or with events.
 */
#define SA2_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
sa2_status sa2_build_mask_noalloc(const sa2_shape* shape, const void* q, const void* k, float topk, float topp,
                                  const sa2_blockmask* out, void* stream);

/*
 * Bytes of device workspace sa2_attn_fwd needs: an fp16 copy of v, plus for SA2_FP32
 * inputs fp16 copies of q and k and their fp16 residuals fp16(x - fp16(x)), and the launch
 * order of the query blocks with its scratch (B*H*Tq + 2*(Tk + 1) + 2*B*H int32, rebuilt by
 * every call).
 */
size_t sa2_fwd_workspace_size(const sa2_shape* shape);

/*
 * sa2_attn_fwd -- block-sparse attention forward.
 * gist.science explainer, section 2.C (efficient kernel implementation): a FlashAttention
 * style block-sparse kernel; tiles are kept or skipped whole, and the matmul and softmax of
 * skipped tiles are not computed.  Equals softmax attention with the scores of dropped
 * blocks at -inf:
 *   O_a = sum over kept key tokens c of exp(s_ac - LSE_a) v_c,  s_ac = scale * q_a . k_c,
 *   LSE_a = log sum over kept c of exp(s_ac)   (natural log).
 * A query block with no kept key block gets O = 0 and LSE = -inf.
 * Arithmetic: S = Q K^T on the tensor cores in bf16 (SA2_BF16), or for SA2_FP32 inputs as
 * the split fp16 product Qhi Khi^T + Qhi Klo^T + Qlo Khi^T of hi = fp16(x), lo = fp16(x - hi)
 * (about 22 bits of the fp32 inputs), fp32 accumulation, fp32 online softmax, then P V with
 * P and V in fp16 (P lies in [0, 1]; bf16 V converts to fp16 exactly).  Attention inputs must lie
 * within the fp16 range (|x| <= 65504); larger values are saturated and reported as
 * SA2_ERR_RANGE through sa2_get_device_status.
 *
 *   q, k, v   token tensors; o: token tensor (output, same dtype); lse: [B, H, N] fp32 output
 *   o_lo      optional (NULL skips; ignored for SA2_FP32): token tensor that receives the
 *             low-order bf16 part of O, bf16(O - bf16(O)), with the strides of o.  Handing
 *             it to sa2_attn_bwd makes its D = rowsum(dO * O) accurate to ~16 bits instead
 *             of bf16's 8, which matters where dS = P (dP - D) cancels (sink-dominated rows).
 *   mask      row_cnt / row_idx of the block mask (e.g. from sa2_build_mask)
 *   softmax_scale  scale of q.k (<= 0 means 1/sqrt(d))
 */
sa2_status sa2_attn_fwd(const sa2_shape* shape, const void* q, const void* k, const void* v,
                        const sa2_blockmask* mask, float softmax_scale, void* o, void* o_lo, float* lse,
                        void* ws, size_t ws_bytes, void* stream);

/*
 * Bytes of device workspace sa2_attn_bwd needs: per-row statistics (log2(e) * LSE and
 * D = rowsum(dO * O), padded to whole 64-row query sub-tiles), the merged column lists of
 * each pair of adjacent key blocks ([B, H, ceil(Tk/2), Tq] uint32 plus their lengths),
 * fp16 copies of q, k, v and dO (and for SA2_FP32 inputs the fp16 residuals of q and k),
 * the work counters of the two persistent backward kernels and the order of the query
 * blocks (reset and rebuilt by the call itself).
 */
size_t sa2_bwd_workspace_size(const sa2_shape* shape);

/*
 * sa2_attn_bwd -- backward of sa2_attn_fwd with the block mask held fixed.
 * The abstract of the paper (shd-paper.top, fugumt.com and thelatestinai.com pages),
 * contribution (ii), makes the sparse attention trainable; the pages do not spell the
 * backward out, so this is the gradient of the forward above:
 *   P = exp(s - LSE),  dV = P^T dO,  dP = dO V^T,  D_a = dO_a . O_a,
 *   dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q,
 * over kept tiles only.  Rows with LSE = -inf contribute nothing.
 *
 * Every product runs on the tensor cores in fp16 (q, k, v, dO converted; P and dS written
 * in fp16, which keeps 11 significant bits where the rows of dS cancel in dQ = dS K; for
 * SA2_FP32 inputs the recomputed scores are the split product of the forward) with fp32
 * accumulation in tensor memory: dK and dV per pair of key blocks across its query
 * blocks, dQ per query block across its key blocks, so no output is reduced across CTAs
 * and the result does not depend on scheduling.
 *
 *   q, k, v, o, dO  token tensors (o, o_lo and lse from sa2_attn_fwd); dq, dk, dv outputs
 *   o_lo      optional residual of O from sa2_attn_fwd (NULL: D uses O alone)
 *   mask      all four lists of the block mask; the column lists must be the transpose of
 *             the row lists the forward used
 *   ws        device workspace of at least sa2_bwd_workspace_size(shape) bytes
 */
sa2_status sa2_attn_bwd(const sa2_shape* shape, const void* q, const void* k, const void* v, const void* o,
                        const void* o_lo, const float* lse, const void* dO, const sa2_blockmask* mask,
                        float softmax_scale, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                        void* stream);

/*
 * sa2_attn_bwd_with_fwd_ws -- sa2_attn_bwd that takes the fp16 copies the forward already
 * made instead of converting again: the copy of v, and for SA2_FP32 inputs those of q and
 * k and their residuals, which sa2_attn_fwd leaves in its workspace; the dQ kernel also
 * takes the forward's launch order of the query blocks instead of building its own (any
 * order gives the same dQ: every query block is one CTA's).  The result is the same, bit for
 * bit.
 *
 *   fwd_ws, fwd_ws_bytes  the workspace of the sa2_attn_fwd call on the same shape, q, k
 *                         and v (the call that produced o, o_lo and lse), ordered before
 *                         this call on the device and not written since; at least
 *                         sa2_fwd_workspace_size(shape) bytes, 16-byte aligned.  Only read.
 *   other arguments       as for sa2_attn_bwd.
 * Errors as for sa2_attn_bwd, and: fwd_ws NULL -> SA2_ERR_INVALID_ARG, misaligned ->
 * SA2_ERR_ALIGNMENT, too small -> SA2_ERR_WORKSPACE, all before any launch.  A workspace
 * that does not hold the forward's copies of these q, k, v is not detected: the gradients
 * are then those of the tensors it holds.
 */
sa2_status sa2_attn_bwd_with_fwd_ws(const sa2_shape* shape, const void* q, const void* k, const void* v,
                                    const void* o, const void* o_lo, const float* lse, const void* dO,
                                    const sa2_blockmask* mask, float softmax_scale, void* dq, void* dk, void* dv,
                                    void* ws, size_t ws_bytes, const void* fwd_ws, size_t fwd_ws_bytes,
                                    void* stream);

/*
 * Toy distillation step (gist.science explainer, section 2.B: the fine-tuning loss is the
 * squared L2 distance between the velocity of the sparse model and that of the frozen
 * full-attention model; on a single attention block the block's output stands in for the
 * velocity).  With a teacher forward under the dense mask (k = 1) and a student forward
 * under the hybrid mask, sa2_vd_loss gives the loss and the student's output gradient,
 * which sa2_attn_bwd then carries to dQ, dK, dV:
 *   loss = sum over all elements of (O_s - O_t)^2,   d_o = 2 (O_s - O_t)   (O_t held fixed)
 *
 *   o_s, o_t        token tensors (dtype and strides of the call): student, teacher output
 *   o_s_lo, o_t_lo  optional residuals from sa2_attn_fwd (bf16 calls; both or neither; NULL
 *                   for none, ignored for SA2_FP32): O is read as O + O_lo, so the difference
 *                   of two close outputs keeps ~16 bits instead of bf16's 8
 *   d_o             token tensor (output, same layout)
 *   loss            device pointer to one double (output), 8-byte aligned
 *   ws              device workspace of at least sa2_vd_loss_workspace_size(shape) bytes
 * The sum is deterministic: per-CTA partial sums in fp64, then one ordered final sum.
 */
size_t sa2_vd_loss_workspace_size(const sa2_shape* shape);
sa2_status sa2_vd_loss(const sa2_shape* shape, const void* o_s, const void* o_s_lo, const void* o_t,
                       const void* o_t_lo, void* d_o, double* loss, void* ws, size_t ws_bytes, void* stream);

/*
 * Launch profiler (instrumentation of this library; the pages have no counterpart).
 * sa2_profiler_enable(1) makes every later kernel launch of the library record a CUDA
 * event before and after it on its stream; sa2_profiler_enable(0) stops that.
 * sa2_profiler_collect waits for the recorded events, writes up to max_entries records
 * (one per kernel of the library: name, launches, summed device milliseconds) and clears
 * them; it returns the number of records written, or -1 when an event could not be read.
 * With out == NULL it returns the number of kernels and leaves the records in place.  Not thread-safe against concurrent
 * launches from several host threads on different streams of the same kernel.
 */
typedef struct sa2_kernel_time {
  const char* name; /* static string */
  int launches;
  double total_ms;
} sa2_kernel_time;

void sa2_profiler_enable(int on);
int sa2_profiler_collect(sa2_kernel_time* out, int max_entries);

/*
 * Synchronizes `stream`, then returns and clears the device status word of the current
 * device: SA2_OK, or the first error a kernel recorded since the last call --
 * SA2_ERR_TIMEOUT (a bounded wait gave up), SA2_ERR_DEVICE_BOUNDS (a block list held an
 * index or count out of range; the kernel clamped it and went on) or SA2_ERR_RANGE (an
 * attention input beyond the fp16 range was saturated) -- or SA2_ERR_CUDA when the
 * synchronization itself fails.
 */
sa2_status sa2_get_device_status(void* stream);

/*
 * Test hook of the failure path (the pages have no counterpart).  Every wait inside the
 * attention kernels is bounded in time; when one expires, its CTA raises an abort flag,
 * every role leaves its loop, the copies and MMAs already issued are drained, tensor memory
 * is freed and sa2_get_device_status reports SA2_ERR_TIMEOUT.  This call lets a test make
 * that happen on purpose:
 *   limit_ns  limit of the waits of the attention calls made after it (0 restores the
 *             default of 2 s);
 *   stall_ns  the row warps of the first CTA of each attention kernel sleep this long before
 *             they start (0: no stall), so that waits on them expire when limit_ns is shorter.
 * Both apply to the calls made after it, from any thread; not for production use.  The
 * drains of the abort path keep their own 2 s bound.
 */
void sa2_debug_set_wait_limit(unsigned long long limit_ns, unsigned long long stall_ns);

#ifdef __cplusplus
}
#endif

#endif /* SA2_H_ */
