/*
 * csa_index.h -- C ABI of the GB300 (sm_103a) CSA indexer library.
 *
 * The library computes the DeepSeek-V4 CSA / StreamIndex indexer hot path:
 *
 *   score[b,s,t] = sum_h w[b,s,h] * ReLU(scale * <q[b,h,s,:], k[b,t,:]>)
 *
 * (the head-reduced indexer score of "Add StreamIndex Kernel for CSA
 * [Deepseek v4]", Description and BlockSpec review hunk: q [B,H,S,D],
 * compressed [B,W,D], weights [B,S,H] -> scores [B,S,W]; the activation is
 * not named there and is taken to be ReLU), masked by the future mask
 * t >= (pos+1) // compress_rate and by the packed-document segment mask of
 * "DSV4: Add indexer_save_selection and indexer_sharded_topk" (mask review
 * hunk), followed by a per-row top-k selection of entry indices (same page,
 * Description: the selection handed to sparse attention).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller (except
 *    those of csa_index_fused_host, which are host pointers), row-major
 *    (contiguous unless csa_problem gives strides for q, k or w), with
 *    16-byte aligned bases.  The library never allocates,
 *    frees or synchronises in these calls; work is enqueued on `stream`
 *    (a cudaStream_t passed as void*; NULL = the legacy default stream) on
 *    the current device.
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns CSA_ERR_INVALID_ARG, a valid but unimplemented shape
 *    returns CSA_ERR_UNSUPPORTED.  There is no fallback path.
 *  - A launch failure returns CSA_ERR_CUDA.  Every wait inside a kernel is
 *    bounded; a wait that gives up records CSA_ERR_TIMEOUT in a device status
 *    word, read (and cleared) by csa_index_device_status().
 *  - Position of query row s of batch b: pos = q_start[b] + s (q_start NULL
 *    means 0).  Entry t is visible from row s iff
 *        t < min(W, (pos + 1) / compress_rate)                (future mask)
 *    and, when segment ids are given, q_seg[b,s] == kv_seg[b,t].
 *  - Selection: among visible entries, the min(top_k, visible) largest
 *    scores; equal scores go to the lower entry index and compare by value
 *    (-0.0 == +0.0).  Each row's indices are written in ascending order and
 *    padded with -1 up to top_k.
 */
#ifndef CSA_INDEX_H
#define CSA_INDEX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned base, scale <= 0 ... */
  CSA_ERR_UNSUPPORTED = 2, /* valid problem outside the implemented (H, D, W) set   */
  CSA_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a launch failed          */
  CSA_ERR_TIMEOUT = 4,     /* a bounded in-kernel wait gave up (device status word)  */
  CSA_ERR_DEVICE = 5       /* the kernel recorded another device-side error          */
} csa_status;

typedef enum { CSA_BF16 = 0, CSA_F32 = 1 } csa_dtype;

/* Layout of q: head-major [B,H,S,D] (the pages' kernel layout) or
 * sequence-major [B,S,H,D] (the layout the pages' RoPE produces, used to
 * avoid transposes).                                                      */
typedef enum { CSA_Q_HEAD_MAJOR = 0, CSA_Q_SEQ_MAJOR = 1 } csa_q_layout;

/* Problem description (all sizes in elements).
 *   B  batch, H indexer heads, S query rows per batch, D head dim,
 *   W  compressed entries per batch (the compressed KV length),
 *   compress_rate  tokens per compressed entry (>= 1),
 *   scale  > 0, applied to q.k inside the ReLU (e.g. D^-0.5),
 *   top_k  >= 1 (may exceed the visible count or W: -1 padding),
 *   w_dtype  storage type of the weights (csa_dtype),
 *   q_layout  csa_q_layout of q (added in ABI version 101).
 * Strided inputs (added in ABI version 104): q, k and w may be views into
 * larger buffers -- e.g. q sliced out of a [B,S,H',D] projection output,
 * so no copy is needed before the call.  Their innermost dimension (D for
 * q and k, H for w) must be contiguous; the other strides are given in
 * elements, and 0 (the value a zero-initialised struct holds) means the
 * contiguous layout:
 *   q_stride_b, q_stride_h, q_stride_s  of q's batch, head and row
 *       dimensions (default: from q_layout); with the 16-byte-aligned base
 *       they must be multiples of 8 elements (16 bytes, the TMA rule);
 *   k_stride_b, k_stride_w  of k's batch and entry dimensions (default
 *       W*D and D; multiples of 8 elements);
 *   w_stride_b, w_stride_s  of w's batch and row dimensions (default S*H
 *       and H; any positive value).
 * Outputs (scores, idx, dq, dk, dw, gathered rows) are always contiguous;
 * dq follows q_layout.  A stride that breaks these rules returns
 * CSA_ERR_INVALID_ARG.
 * A decode batch with sequences of different lengths shares one k buffer
 * [B,W,D] sized for the longest; q_start[b] (the row's position) bounds
 * each sequence's visible entries, so entries past a sequence's length are
 * never selected and their tiles are never multiplied.                  */
typedef struct {
  int32_t B, H, S, D, W;
  int32_t compress_rate;
  float scale;
  int32_t top_k;
  int32_t w_dtype;
  int32_t q_layout;
  int64_t q_stride_b, q_stride_h, q_stride_s;
  int64_t k_stride_b, k_stride_w;
  int64_t w_stride_b, w_stride_s;
} csa_problem;

/* Scores.  q [B,H,S,D] (or [B,S,H,D], q_layout) bf16, k [B,W,D] bf16, w [B,S,H] (w_dtype),
 * q_seg [B,S] int32 or NULL, kv_seg [B,W] int32 or NULL (both or neither),
 * q_start [B] int64 or NULL.  Writes scores [B,S,W] fp32, -inf where masked.
 * Defined by the score formula above ("Add StreamIndex Kernel for CSA
 * [Deepseek v4]", Description; masks per "DSV4: Add indexer_save_selection
 * and indexer_sharded_topk", mask review hunk).
 * Supported: (H, D) in {(64, 128), (4, 32)}, any B, S, W >= 1.           */
csa_status csa_index_score(const csa_problem* p, const void* q, const void* k, const void* w,
                           const int32_t* q_seg, const int32_t* kv_seg, const int64_t* q_start,
                           float* scores, void* stream);

/* Selection only, from precomputed scores [B,S,W] fp32 (an entry is visible
 * iff its score > -inf).  Writes idx [B,S,top_k] int32 (selection rule
 * above; "DSV4: Add indexer_save_selection and indexer_sharded_topk",
 * Description).  workspace may be NULL when csa_index_workspace_size(p, 0)
 * returns 0 (it does for every supported W).  Supported: W <= 49152.     */
csa_status csa_index_topk(const csa_problem* p, const float* scores, int32_t* idx,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Scores and selection in one call: same inputs as csa_index_score, writes
 * idx [B,S,top_k] int32.  Needs `workspace`: csa_index_workspace_size(p, 1)
 * bytes of device memory owned by the caller (16-byte aligned).
 *  - W <= 4096 and S > 2: one persistent kernel.  Each CTA stages the score
 *    rows of its two most recent items of four rows in its slice of the
 *    workspace (2 x 4 x W fp32 per CTA, at most 256 CTAs: a few tens of MB
 *    that stay in L2), so the selection of one item overlaps the scores of
 *    the next; the [B,S,W] score tensor is never formed.  With segment
 *    ids a short pre-pass kernel first summarises each item's segment ids
 *    (64 bytes per item of four rows, after the ring in the workspace).
 *  - otherwise (decode-style single rows, long rows): the scores go to the
 *    workspace ([B,S,W] fp32) and a second kernel selects.
 * scores_dbg [B,S,W] fp32, if non-NULL, also receives the exact fp32 scores
 * the selection used (every entry, -inf where masked).                    */
csa_status csa_index_fused(const csa_problem* p, const void* q, const void* k, const void* w,
                           const int32_t* q_seg, const int32_t* kv_seg, const int64_t* q_start,
                           int32_t* idx, float* scores_dbg, void* workspace,
                           size_t workspace_bytes, void* stream);

/* csa_index_fused on HOST buffers (added in ABI version 106): q, k, w,
 * q_seg, kv_seg, q_start and idx are host pointers (page-locked memory
 * makes the copies asynchronous), contiguous and in the layouts of
 * csa_index_fused (each stride in csa_problem 0 or the contiguous one).  The call
 * enqueues on `stream`, in order: the copies of the inputs into
 * `workspace`, the computation of csa_index_fused, and the copy of idx
 * back to the host; it returns without waiting, so idx may be read, and the
 * input buffers reused, only after the stream has been synchronised.
 * q_start, when given, is also read on the host during the call.
 * Only the q rows the computation can read are copied.  A row whose
 * future-mask bound min(W, (pos + 1) / compress_rate) is at most top_k
 * keeps all its visible entries, whatever its scores; when csa_index_fused
 * runs as one kernel, the q block of an item of four such rows is never
 * loaded, so the rows before the first item holding a row with a larger
 * bound are not transferred (on prefill with q_start = 0 that is rows
 * s < ((top_k + 1) * compress_rate - 1) rounded down to a multiple of 4).
 * The other paths copy all of q.  csa_index_fused_host_bytes() gives the
 * bytes one call moves each way.
 * Needs `workspace`: csa_index_workspace_size(p, 3) bytes of device memory
 * owned by the caller, 256-byte aligned, holding the device copies of the
 * inputs and of idx and csa_index_fused's own workspace; calls that may be
 * in flight at the same time need separate workspaces.  Errors: as for
 * csa_index_fused; a stride other than the contiguous one returns
 * CSA_ERR_INVALID_ARG.                                                    */
csa_status csa_index_fused_host(const csa_problem* p, const void* q, const void* k, const void* w,
                                const int32_t* q_seg, const int32_t* kv_seg, const int64_t* q_start,
                                int32_t* idx, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes one csa_index_fused_host call copies host -> device (*h2d: the q
 * rows it transfers, k, w, the segment ids when with_segments != 0, and
 * q_start when given) and device -> host (*d2h: idx).  q_start is the host
 * array the call would get (NULL = 0).  Enqueues nothing.                 */
csa_status csa_index_fused_host_bytes(const csa_problem* p, const int64_t* q_start, int32_t with_segments,
                                      size_t* h2d, size_t* d2h);

/* Gather of the selected compressed entries, the rows sparse attention reads
 * ("DSV4: Add indexer_save_selection and indexer_sharded_topk", Description:
 * the selection is handed to sparse attention in sequence layout):
 *   out[b,s,i,:] = k[b, idx[b,s,i], :],  zeros where idx[b,s,i] == -1.
 * k [B,W,D] bf16, idx [B,S,top_k] int32 (a selection from this library or
 * any int32 indices), out [B,S,top_k,D] bf16; uses B, S, W, D, top_k of p.
 * An index outside [-1, W) writes a zero row and records CSA_ERR_DEVICE in
 * the device status word.  Supported: D in {32, 128}.                    */
csa_status csa_index_gather(const csa_problem* p, const void* k, const int32_t* idx, void* out, void* stream);

/* csa_index_fused without any caller workspace and without any allocation.
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory at the call site -- for instance a host
 * process whose memory pool already owns (and has reserved) the free device
 * memory, or a code path where the implicit device synchronisation of a
 * cudaMalloc is not allowed.  Inputs and idx are as for csa_index_fused;
 * the result equals csa_index_fused's for the same problem.
 *  - Scores go through a scratch array compiled into the library (fp32,
 *    at most 2,097,152 = 2^21 scores, i.e. 8 MiB: B*S*W must not exceed it,
 *    e.g. 64 decode rows of 32768 entries).  Larger problems return
 *    CSA_ERR_UNSUPPORTED before anything is launched.  Every GPU that loads
 *    the library holds this array until the process exits.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and keeps it; make that first call before any
 *    stream capture in the calling program.  A failed lookup returns
 *    CSA_ERR_CUDA and is tried again on the next call.  The kept address
 *    belongs to the device's primary context: do not reset the device
 *    (cudaDeviceReset) between calls.
 *  - All calls share the one array: calls whose work overlaps on the GPU
 *    (other streams, other host threads) race and corrupt each other's
 *    results.  Each call writes every score it later reads, so nothing needs
 *    clearing between calls.                                              */
csa_status csa_index_fused_noalloc(const csa_problem* p, const void* q, const void* k, const void* w,
                                   const int32_t* q_seg, const int32_t* kv_seg, const int64_t* q_start,
                                   int32_t* idx, void* stream);

/* Backward of the score step: the gradients of sum(g * score) over the
 * visible entries, for a cotangent g of the scores ("Add StreamIndex Kernel
 * for CSA [Deepseek v4]", Description: the custom_vjp whose backward is the
 * autodiff of the reference computation; its backward review asks for a
 * fused kernel).  With x = q[b,h,s,:].k[b,t,:] and gm = g on visible
 * entries, 0 on masked ones (masked scores are constants):
 *   dw[b,s,h] = sum_t gm * ReLU(scale * x)
 *   P         = gm * w[b,s,h] * scale * [x > 0]
 *   dq[b,h,s,:] = sum_t P * k[b,t,:],   dk[b,t,:] = sum_{h,s} P * q[b,h,s,:].
 * Inputs as for csa_index_score; g [B,S,W] fp32 (values at masked entries
 * are ignored); writes dq in q's layout ([B,H,S,D] or [B,S,H,D], q_layout),
 * dk [B,W,D] and dw [B,S,H], all fp32, every element; dq and dk need
 * 16-byte aligned bases.  Two tensor-core kernels recompute the logits tile
 * by tile and keep P (rounded to bf16) on the SM: one forms dw and dq per
 * pair of query rows, the other dk per tile of 128 entries and run of row
 * pairs, adding its partial sums into dk with fp32 atomics (so the last bits
 * of dk may differ from call to call); the [B,H,S,W] tensor and P never
 * reach HBM.  With segment ids, a pre-pass summarises each item of four
 * rows (the tiles holding entries visible to its rows, as for
 * csa_index_fused) and the kernels skip the tiles, and the dk kernel the
 * row pairs, that the segment mask leaves without a visible entry.  Needs
 * `workspace`: csa_index_workspace_size(p, 2) bytes (256 + 64 per item of
 * four rows, B * ceil(S/4) items; 16-byte aligned): a work counter the call
 * resets, then the summaries.  dk is zeroed and the kernels run on
 * `stream`; the call returns once they are enqueued and allocates nothing.
 * Supported: H = 64, D = 128, either q layout.  Added in ABI version 102;
 * the workspace shrank to 256 bytes in 103 and holds the segment summaries
 * since 105.                                                              */
csa_status csa_index_backward(const csa_problem* p, const void* q, const void* k, const void* w,
                              const int32_t* q_seg, const int32_t* kv_seg, const int64_t* q_start,
                              const float* g, float* dq, float* dk, float* dw, void* workspace,
                              size_t workspace_bytes, void* stream);

/* Bytes of device workspace an entry point needs: which = 0 for
 * csa_index_topk (always 0), 1 for csa_index_fused, 2 for
 * csa_index_backward, 3 for csa_index_fused_host.  Depends only on the
 * problem (no device query).  Returns 0 when the problem is invalid.      */
size_t csa_index_workspace_size(const csa_problem* p, int32_t which);

/* Synchronises `stream`, then reads and clears the device status word of
 * the current device: CSA_OK, CSA_ERR_TIMEOUT (a bounded wait gave up) or
 * CSA_ERR_DEVICE.  CSA_ERR_CUDA if the synchronisation itself failed.     */
csa_status csa_index_device_status(void* stream);

/* Runs a kernel whose single wait can never be satisfied, bounded by
 * `timeout_us` microseconds; it must give up, record CSA_ERR_TIMEOUT and
 * return.  Used to test the give-up path without faulting a GPU.          */
csa_status csa_index_selftest_timeout(uint32_t timeout_us, void* stream);

/* Static string for a status code. */
const char* csa_status_string(csa_status s);

/* ABI version (major * 100 + minor): 106 (csa_index_fused_host; 105:
 * backward workspace holds the segment summaries; 104: strides in
 * csa_problem). */
int32_t csa_index_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CSA_INDEX_H */
