// csa_api.cu -- the C ABI declared in include/csa_index.h: argument checks,
// TMA tensor maps, choice of kernel instantiation and launches.  Nothing here
// computes any part of the indexer; every step runs in the kernels.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <atomic>
#include <mutex>

#include "csa_index.h"
#include "csa_internal.h"

namespace csa {
namespace {

constexpr int kFusedMaxW = 4096;   // shared-memory score rows of the fused kernel
constexpr int kFusedLongMaxW = 16384;  // its long-row mode: one shared row, selected by a team
constexpr int kMaxGrid = 256;      // CTAs of the persistent kernel (bounds the fused staging ring)
constexpr int kTopkMaxW = 49152;   // one row staged in shared memory by the top-k kernel
constexpr int kDecodeChunkTiles = 8;
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s per wait before giving up

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Element strides of the inputs, the problem's own or the contiguous
// defaults (a zero field selects the default).
struct Strides {
  long long qb, qh, qs;  // q: batch, head, row
  long long kb, kw;      // k: batch, entry
  long long wb, ws;      // w: batch, row
};
Strides strides_of(const csa_problem* p) {
  const bool sm = p->q_layout == CSA_Q_SEQ_MAJOR;
  const long long D = p->D, H = p->H, S = p->S, W = p->W;
  Strides t;
  t.qb = p->q_stride_b ? p->q_stride_b : H * S * D;
  t.qh = p->q_stride_h ? p->q_stride_h : (sm ? D : S * D);
  t.qs = p->q_stride_s ? p->q_stride_s : (sm ? H * D : D);
  t.kb = p->k_stride_b ? p->k_stride_b : W * D;
  t.kw = p->k_stride_w ? p->k_stride_w : D;
  t.wb = p->w_stride_b ? p->w_stride_b : S * H;
  t.ws = p->w_stride_s ? p->w_stride_s : H;
  return t;
}

// q and k strides feed TMA maps: multiples of 16 bytes (8 bf16) below 2^40 bytes.
bool tma_stride_ok(long long s) { return s >= 0 && (s % 8) == 0 && s < (1ll << 38); }

csa_status check_problem(const csa_problem* p) {
  if (p == nullptr) return CSA_ERR_INVALID_ARG;
  if (p->B < 1 || p->H < 1 || p->S < 1 || p->D < 1 || p->W < 1) return CSA_ERR_INVALID_ARG;
  if (p->compress_rate < 1 || p->top_k < 1) return CSA_ERR_INVALID_ARG;
  if (!(p->scale > 0.f) || !std::isfinite(p->scale)) return CSA_ERR_INVALID_ARG;
  if (p->w_dtype != CSA_BF16 && p->w_dtype != CSA_F32) return CSA_ERR_INVALID_ARG;
  if (p->q_layout != CSA_Q_HEAD_MAJOR && p->q_layout != CSA_Q_SEQ_MAJOR) return CSA_ERR_INVALID_ARG;
  const double rows = (double)p->B * (double)p->S;
  if (rows * (double)p->W > 4.0e18 || rows * (double)p->top_k > 4.0e18) return CSA_ERR_INVALID_ARG;
  for (long long st : {p->q_stride_b, p->q_stride_h, p->q_stride_s, p->k_stride_b, p->k_stride_w})
    if (!tma_stride_ok(st)) return CSA_ERR_INVALID_ARG;
  if (p->w_stride_b < 0 || p->w_stride_s < 0 || p->w_stride_b > (1ll << 40) || p->w_stride_s > (1ll << 40))
    return CSA_ERR_INVALID_ARG;
  return CSA_OK;
}

csa_status check_inputs(const csa_problem* p, const void* q, const void* k, const void* w, const int32_t* q_seg,
                        const int32_t* kv_seg, const int64_t* q_start) {
  if (q == nullptr || k == nullptr || w == nullptr) return CSA_ERR_INVALID_ARG;
  if ((q_seg == nullptr) != (kv_seg == nullptr)) return CSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16)) return CSA_ERR_INVALID_ARG;  // TMA bases
  if (!aligned(w, p->w_dtype == CSA_F32 ? 4 : 2)) return CSA_ERR_INVALID_ARG;
  if (q_seg && (!aligned(q_seg, 4) || !aligned(kv_seg, 4))) return CSA_ERR_INVALID_ARG;
  if (q_start && !aligned(q_start, 8)) return CSA_ERR_INVALID_ARG;
  return CSA_OK;
}

bool shape_supported(const csa_problem* p) {
  return (p->H == 64 && p->D == 128) || (p->H == 4 && p->D == 32);
}

// Single-row problems use the R = 1 kernel with tile chunks, which keeps every
// SM busy streaming k; everything else uses blocks of four query rows.
bool use_row_kernel(const csa_problem* p) { return p->S <= 2 && p->H == 64 && p->D == 128; }

// Fused in one kernel (selection on the SM) unless the problem is single-row
// or its rows are too long for shared memory; those go through two passes.
// Rows of 4097..16384 entries take the kernel's long-row mode (H = 64, D = 128).
bool fused_long(const csa_problem* p) {
  return !use_row_kernel(p) && p->W > kFusedMaxW && p->W <= kFusedLongMaxW && p->H == 64 && p->D == 128;
}
bool fused_one_kernel(const csa_problem* p) {
  return !use_row_kernel(p) && (p->W <= kFusedMaxW || fused_long(p));
}

int w_pad_of(const csa_problem* p) { return ((p->W + kTileT - 1) / kTileT) * kTileT; }

// Staging ring of the one-kernel fused path: two items of four rows per CTA.
size_t fused_ring_bytes(const csa_problem* p) {
  const long long items = (long long)p->B * ((p->S + 3) / 4);
  const long long ctas = std::min<long long>(items, kMaxGrid);
  return (size_t)ctas * 2 * 4 * (size_t)w_pad_of(p) * sizeof(float);
}
// Segment summaries of the one-kernel fused path (one per item of four rows),
// after the ring in the same workspace.
size_t fused_seginfo_bytes(const csa_problem* p) {
  return (size_t)p->B * (size_t)((p->S + 3) / 4) * sizeof(SegInfo);
}
size_t fused_seginfo_offset(const csa_problem* p) { return (fused_ring_bytes(p) + 255) & ~(size_t)255; }

int num_sms() {
  static int cached[64];
  static std::once_flag flags[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::call_once(flags[dev], [dev] {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 0;
    cached[dev] = n;
  });
  return cached[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag flag;
  std::call_once(flag, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// q viewed as dims (D, H, S, B) so one box {KC, H, R, 1} lands as R*H rows
// ordered (row j, head h) -> j*H + h.  Head-major [B,H,S,D], sequence-major
// [B,S,H,D] and strided views differ only in the strides of H, S and B.
bool make_q_map(CUtensorMap* m, const csa_problem* p, const void* q, int R) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int KC = (p->D % 64 == 0) ? 64 : 32;
  cuuint64_t dims[4] = {(cuuint64_t)p->D, (cuuint64_t)p->H, (cuuint64_t)p->S, (cuuint64_t)p->B};
  const Strides st = strides_of(p);
  cuuint64_t strides[3] = {(cuuint64_t)st.qh * 2, (cuuint64_t)st.qs * 2, (cuuint64_t)st.qb * 2};
  cuuint32_t box[4] = {(cuuint32_t)KC, (cuuint32_t)p->H, (cuuint32_t)R, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw = (KC == 64) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// k [B,W,D] bf16 as dims (D, W, B); box {KC, 128, 1}.  Entries past W read as zero.
bool make_k_map(CUtensorMap* m, const csa_problem* p, const void* k) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int KC = (p->D % 64 == 0) ? 64 : 32;
  cuuint64_t dims[3] = {(cuuint64_t)p->D, (cuuint64_t)p->W, (cuuint64_t)p->B};
  const Strides st = strides_of(p);
  cuuint64_t strides[2] = {(cuuint64_t)st.kw * 2, (cuuint64_t)st.kb * 2};
  cuuint32_t box[3] = {(cuuint32_t)KC, (cuuint32_t)kTileT, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = (KC == 64) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(k), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Backward workspace: the dk kernel's item counter (256 bytes), then the
// segment summaries of the items of four rows (64 bytes each; written and
// read only when segment ids are given).
constexpr size_t kBwdWorkspace = 256;
size_t backward_workspace_bytes(const csa_problem* p) {
  if (check_problem(p) != CSA_OK) return 0;
  return kBwdWorkspace + (size_t)p->B * (size_t)((p->S + 3) / 4) * sizeof(SegInfo);
}

// Row pairs per dk item: 256, halved while the problem would give fewer than
// about eight items per SM before the causal half is skipped (down to 32).
int bwd_chunk_pairs(const csa_problem* p, int sms) {
  const long long n_pairs = (p->S + 1) / 2;
  const long long n_tiles = (p->W + kTileT - 1) / kTileT;
  int cp = 256;
  while (cp > 32 && (long long)p->B * n_tiles * ((n_pairs + cp - 1) / cp) < 8ll * sms) cp /= 2;
  return cp;
}

csa_status run_index_kernel(const csa_problem* p, bool fused, const void* q, const void* k, const void* w,
                            const int32_t* q_seg, const int32_t* kv_seg, const int64_t* q_start, float* scores,
                            int32_t* idx, float* ring, cudaStream_t stream, SegInfo* seginfo = nullptr) {
  const bool row_kernel = use_row_kernel(p);
  KernelChoice kc{p->H, p->D, row_kernel ? 1 : 4, fused};
  kc.long_rows = fused && p->W > kFusedMaxW;
  CUtensorMap tq, tk;
  if (!make_q_map(&tq, p, q, kc.R) || !make_k_map(&tk, p, k)) return CSA_ERR_CUDA;
  KParams kp;
  std::memset(&kp, 0, sizeof(kp));
  kp.B = p->B;
  kp.S = p->S;
  kp.W = p->W;
  kp.r = p->compress_rate;
  kp.r_shift = -1;
  for (int sh = 0; sh < 31; ++sh)
    if ((1 << sh) == p->compress_rate) kp.r_shift = sh;
  kp.K = p->top_k;
  kp.scale = p->scale;
  kp.w_f32 = (p->w_dtype == CSA_F32) ? 1 : 0;
  kp.w = w;
  kp.w_sb = strides_of(p).wb;
  kp.w_ss = strides_of(p).ws;
  kp.q_seg = q_seg;
  kp.kv_seg = kv_seg;
  kp.q_start = q_start;
  kp.scores = scores;
  kp.idx = idx;
  kp.ring = ring;
  kp.n_rb = (p->S + kc.R - 1) / kc.R;
  kp.n_tiles = (p->W + kTileT - 1) / kTileT;
  kp.chunk_tiles = row_kernel ? std::min(kp.n_tiles, kDecodeChunkTiles) : kp.n_tiles;
  kp.n_chunks = (kp.n_tiles + kp.chunk_tiles - 1) / kp.chunk_tiles;
  const long long items = (long long)p->B * kp.n_rb * kp.n_chunks;
  if (items > 0x7FFFFFFFll) return CSA_ERR_UNSUPPORTED;
  kp.n_items = (int)items;
  kp.w_pad = kp.n_tiles * kTileT;
  kp.wait_ns = kWaitNs;
  if (index_kernel_smem(kc, kp.w_pad) == 0) return CSA_ERR_UNSUPPORTED;
  if (index_kernel_smem(kc, kp.w_pad) > 227u * 1024u) return CSA_ERR_UNSUPPORTED;
  const int sms = num_sms();
  if (sms <= 0) return CSA_ERR_CUDA;
  const int grid = (int)std::min<long long>(items, std::min(sms, kMaxGrid));
  if (seginfo != nullptr && q_seg != nullptr && kc.R == 4 && kp.n_chunks == 1) {
    // segment ids scanned once per item across the whole GPU, ahead of the kernel
    if (launch_segscan(kp, seginfo, sms, stream) != cudaSuccess) return CSA_ERR_CUDA;
    kp.seginfo = seginfo;
    // packed documents: the kernel's document mode
    kc.docs = fused && !kc.long_rows && p->H == 64 && p->D == 128;
  }
  if (launch_index_kernel(kc, tq, tk, kp, grid, stream) != cudaSuccess) return CSA_ERR_CUDA;
  return CSA_OK;
}

size_t fused_workspace_bytes(const csa_problem* p) {
  if (check_problem(p) != CSA_OK) return 0;
  if (fused_one_kernel(p)) return fused_seginfo_offset(p) + fused_seginfo_bytes(p);
  return (size_t)p->B * p->S * p->W * sizeof(float);
}

// ----------------------------------------------------------------- host buffers
// Device workspace of csa_index_fused_host: the inputs' device copies, idx
// and csa_index_fused's own workspace, each 256-byte aligned.
struct HostPlan {
  size_t q, k, w, qseg, kvseg, qst, idx, fws;              // bytes
  size_t off_q, off_k, off_w, off_qseg, off_kvseg, off_qst, off_idx, off_fws, total;
};
size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }
HostPlan host_plan(const csa_problem* p) {
  HostPlan h{};
  const size_t B = (size_t)p->B, S = (size_t)p->S, W = (size_t)p->W;
  h.q = B * (size_t)p->H * S * (size_t)p->D * 2;
  h.k = B * W * (size_t)p->D * 2;
  h.w = B * S * (size_t)p->H * (p->w_dtype == CSA_F32 ? 4 : 2);
  h.qseg = B * S * 4;
  h.kvseg = B * W * 4;
  h.qst = B * 8;
  h.idx = B * S * (size_t)p->top_k * 4;
  h.fws = fused_workspace_bytes(p);
  size_t o = 0;
  h.off_q = o;
  o = up256(o + h.q);
  h.off_k = o;
  o = up256(o + h.k);
  h.off_w = o;
  o = up256(o + h.w);
  h.off_qseg = o;
  o = up256(o + h.qseg);
  h.off_kvseg = o;
  o = up256(o + h.kvseg);
  h.off_qst = o;
  o = up256(o + h.qst);
  h.off_idx = o;
  o = up256(o + h.idx);
  h.off_fws = o;
  h.total = up256(o + h.fws);
  return h;
}

// First query row of a sequence starting at position qs whose q the
// one-kernel fused path can read.  An item of four rows is scored only if
// one of its rows sees more than top_k entries, which needs that row's
// future-mask bound min(W, (qs + s + 1) / r) to exceed top_k, i.e. W > top_k
// and qs + s + 1 >= (top_k + 1) * r.  Bounds grow with s, so every item
// before the one holding the first such row keeps its visible sets without
// its q block ever being loaded.  The other paths read all of q.
int first_read_row(const csa_problem* p, long long qs) {
  if (!fused_one_kernel(p)) return 0;
  if (p->W <= p->top_k) return p->S;
  const long long lim = 1ll << 62;
  qs = qs < -lim ? -lim : (qs > lim ? lim : qs);
  const long long s = (long long)(p->top_k + 1) * p->compress_rate - qs - 1;
  if (s >= p->S) return p->S;
  return s <= 0 ? 0 : (int)(s / 4 * 4);
}

// Host -> device bytes of q that csa_index_fused_host copies.
size_t host_q_bytes(const csa_problem* p, const int64_t* q_start) {
  size_t n = 0;
  for (int b = 0; b < p->B; ++b)
    n += (size_t)(p->S - first_read_row(p, q_start ? q_start[b] : 0)) * (size_t)p->H * (size_t)p->D * 2;
  return n;
}

// Host buffers are contiguous: every stride is 0 or the contiguous one.
bool host_layout_ok(const csa_problem* p) {
  csa_problem dense = *p;
  dense.q_stride_b = dense.q_stride_h = dense.q_stride_s = 0;
  dense.k_stride_b = dense.k_stride_w = dense.w_stride_b = dense.w_stride_s = 0;
  const Strides a = strides_of(p), c = strides_of(&dense);
  return a.qb == c.qb && a.qh == c.qh && a.qs == c.qs && a.kb == c.kb && a.kw == c.kw && a.wb == c.wb &&
         a.ws == c.ws;
}

// ----------------------------------------------------------------- allocation-free variant
// Scratch for csa_index_fused_noalloc: the fp32 scores of one call, at most
// kNoAllocMaxScores of them (8 MiB).  Every GPU that loads the library keeps
// this array until the process exits.  Host code must not use the symbol as
// a pointer: noalloc_scratch() fetches its device address.
constexpr size_t kNoAllocMaxScores = (size_t)2 * 1024 * 1024;
static __device__ __align__(256) float g_noalloc_scores[kNoAllocMaxScores];

// Device address of g_noalloc_scores on the current device, looked up with
// that device current on the first successful call there and kept for later
// calls.  A failed lookup is not kept: the next call tries again.  The
// address stays valid for the life of the device's primary context.
float* noalloc_scratch(cudaError_t* err) {
  static std::atomic<float*> ptrs[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  float* p = ptrs[dev].load(std::memory_order_acquire);
  if (p != nullptr) {
    *err = cudaSuccess;
    return p;
  }
  void* ptr = nullptr;
  *err = cudaGetSymbolAddress(&ptr, g_noalloc_scores);
  if (*err != cudaSuccess) return nullptr;
  ptrs[dev].store(static_cast<float*>(ptr), std::memory_order_release);
  return static_cast<float*>(ptr);
}

}  // namespace
}  // namespace csa

using namespace csa;

extern "C" {

csa_status csa_index_score(const csa_problem* p, const void* q, const void* k, const void* w,
                           const int32_t* q_seg, const int32_t* kv_seg, const int64_t* q_start, float* scores,
                           void* stream) {
  csa_status st = check_problem(p);
  if (st != CSA_OK) return st;
  if ((st = check_inputs(p, q, k, w, q_seg, kv_seg, q_start)) != CSA_OK) return st;
  if (scores == nullptr || !aligned(scores, 4)) return CSA_ERR_INVALID_ARG;
  if (!shape_supported(p)) return CSA_ERR_UNSUPPORTED;
  return run_index_kernel(p, false, q, k, w, q_seg, kv_seg, q_start, scores, nullptr, nullptr,
                          static_cast<cudaStream_t>(stream));
}

csa_status csa_index_topk(const csa_problem* p, const float* scores, int32_t* idx, void* workspace,
                          size_t workspace_bytes, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  csa_status st = check_problem(p);
  if (st != CSA_OK) return st;
  if (scores == nullptr || idx == nullptr || !aligned(scores, 4) || !aligned(idx, 4)) return CSA_ERR_INVALID_ARG;
  if (p->W > kTopkMaxW) return CSA_ERR_UNSUPPORTED;
  const long long rows = (long long)p->B * p->S;
  if (launch_topk(scores, idx, rows, p->W, p->top_k, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CSA_ERR_CUDA;
  return CSA_OK;
}

csa_status csa_index_fused(const csa_problem* p, const void* q, const void* k, const void* w,
                           const int32_t* q_seg, const int32_t* kv_seg, const int64_t* q_start, int32_t* idx,
                           float* scores_dbg, void* workspace, size_t workspace_bytes, void* stream) {
  csa_status st = check_problem(p);
  if (st != CSA_OK) return st;
  if ((st = check_inputs(p, q, k, w, q_seg, kv_seg, q_start)) != CSA_OK) return st;
  if (idx == nullptr || !aligned(idx, 4)) return CSA_ERR_INVALID_ARG;
  if (scores_dbg != nullptr && !aligned(scores_dbg, 4)) return CSA_ERR_INVALID_ARG;
  if (!shape_supported(p)) return CSA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t need = fused_workspace_bytes(p);
  if (fused_one_kernel(p)) {
    if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 16)) return CSA_ERR_INVALID_ARG;
    SegInfo* seginfo =
        reinterpret_cast<SegInfo*>(static_cast<uint8_t*>(workspace) + fused_seginfo_offset(p));
    return run_index_kernel(p, true, q, k, w, q_seg, kv_seg, q_start, scores_dbg, idx,
                            static_cast<float*>(workspace), s, seginfo);
  }
  // Long rows or single-row problems: scores through the workspace (or the
  // caller's debug copy), then the selection kernel.
  if (p->W > kTopkMaxW) return CSA_ERR_UNSUPPORTED;
  float* sc = scores_dbg;
  if (sc == nullptr) {
    if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 16)) return CSA_ERR_INVALID_ARG;
    sc = static_cast<float*>(workspace);
  }
  st = run_index_kernel(p, false, q, k, w, q_seg, kv_seg, q_start, sc, nullptr, nullptr, s);
  if (st != CSA_OK) return st;
  if (launch_topk(sc, idx, (long long)p->B * p->S, p->W, p->top_k, s) != cudaSuccess) return CSA_ERR_CUDA;
  return CSA_OK;
}

csa_status csa_index_fused_host(const csa_problem* p, const void* q, const void* k, const void* w,
                                const int32_t* q_seg, const int32_t* kv_seg, const int64_t* q_start, int32_t* idx,
                                void* workspace, size_t workspace_bytes, void* stream) {
  csa_status st = check_problem(p);
  if (st != CSA_OK) return st;
  if (q == nullptr || k == nullptr || w == nullptr || idx == nullptr) return CSA_ERR_INVALID_ARG;
  if ((q_seg == nullptr) != (kv_seg == nullptr)) return CSA_ERR_INVALID_ARG;
  if (!host_layout_ok(p)) return CSA_ERR_INVALID_ARG;
  if (!shape_supported(p)) return CSA_ERR_UNSUPPORTED;
  if (!fused_one_kernel(p) && p->W > kTopkMaxW) return CSA_ERR_UNSUPPORTED;
  const HostPlan h = host_plan(p);
  if (workspace == nullptr || workspace_bytes < h.total || !aligned(workspace, 256)) return CSA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto in = [&](size_t off, const void* src, size_t n) {
    return n == 0 || cudaMemcpyAsync(ws + off, src, n, cudaMemcpyHostToDevice, s) == cudaSuccess;
  };
  // q: only the rows the computation can read (whole items of four rows)
  const size_t row = (size_t)p->D * 2;
  for (int b = 0; b < p->B; ++b) {
    const int s0 = first_read_row(p, q_start ? q_start[b] : 0);
    if (s0 >= p->S) continue;
    const size_t rows = (size_t)(p->S - s0);
    const uint8_t* hq = static_cast<const uint8_t*>(q);
    if (p->q_layout == CSA_Q_HEAD_MAJOR) {  // H slabs of S rows: one strided copy
      const size_t pitch = (size_t)p->S * row, off = ((size_t)b * p->H * p->S + (size_t)s0) * row;
      if (cudaMemcpy2DAsync(ws + h.off_q + off, pitch, hq + off, pitch, rows * row, (size_t)p->H,
                            cudaMemcpyHostToDevice, s) != cudaSuccess)
        return CSA_ERR_CUDA;
    } else {  // rows of H heads: one contiguous range
      const size_t off = ((size_t)b * p->S + (size_t)s0) * (size_t)p->H * row;
      if (!in(h.off_q + off, hq + off, rows * (size_t)p->H * row)) return CSA_ERR_CUDA;
    }
  }
  if (!in(h.off_k, k, h.k) || !in(h.off_w, w, h.w)) return CSA_ERR_CUDA;
  if (q_seg != nullptr && (!in(h.off_qseg, q_seg, h.qseg) || !in(h.off_kvseg, kv_seg, h.kvseg))) return CSA_ERR_CUDA;
  if (q_start != nullptr && !in(h.off_qst, q_start, h.qst)) return CSA_ERR_CUDA;
  st = csa_index_fused(p, ws + h.off_q, ws + h.off_k, ws + h.off_w,
                       q_seg ? reinterpret_cast<const int32_t*>(ws + h.off_qseg) : nullptr,
                       kv_seg ? reinterpret_cast<const int32_t*>(ws + h.off_kvseg) : nullptr,
                       q_start ? reinterpret_cast<const int64_t*>(ws + h.off_qst) : nullptr,
                       reinterpret_cast<int32_t*>(ws + h.off_idx), nullptr, ws + h.off_fws, h.fws, stream);
  if (st != CSA_OK) return st;
  if (cudaMemcpyAsync(idx, ws + h.off_idx, h.idx, cudaMemcpyDeviceToHost, s) != cudaSuccess) return CSA_ERR_CUDA;
  return CSA_OK;
}

csa_status csa_index_fused_host_bytes(const csa_problem* p, const int64_t* q_start, int32_t with_segments,
                                      size_t* h2d, size_t* d2h) {
  csa_status st = check_problem(p);
  if (st != CSA_OK) return st;
  if (h2d == nullptr || d2h == nullptr) return CSA_ERR_INVALID_ARG;
  const HostPlan h = host_plan(p);
  *h2d = host_q_bytes(p, q_start) + h.k + h.w + (with_segments ? h.qseg + h.kvseg : 0) + (q_start ? h.qst : 0);
  *d2h = h.idx;
  return CSA_OK;
}

csa_status csa_index_fused_noalloc(const csa_problem* p, const void* q, const void* k, const void* w,
                                   const int32_t* q_seg, const int32_t* kv_seg, const int64_t* q_start,
                                   int32_t* idx, void* stream) {
  csa_status st = check_problem(p);
  if (st != CSA_OK) return st;
  if ((st = check_inputs(p, q, k, w, q_seg, kv_seg, q_start)) != CSA_OK) return st;
  if (idx == nullptr || !aligned(idx, 4)) return CSA_ERR_INVALID_ARG;
  if (!shape_supported(p)) return CSA_ERR_UNSUPPORTED;
  if (p->W > kTopkMaxW) return CSA_ERR_UNSUPPORTED;
  const size_t n_scores = (size_t)p->B * (size_t)p->S * (size_t)p->W;
  if (n_scores > kNoAllocMaxScores) return CSA_ERR_UNSUPPORTED;  // beyond the library's static scratch
  cudaError_t err = cudaSuccess;
  float* scratch = noalloc_scratch(&err);
  if (scratch == nullptr) return CSA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the score pass writes every entry the selection pass reads, so the
  // scratch needs no clearing between calls
  st = run_index_kernel(p, false, q, k, w, q_seg, kv_seg, q_start, scratch, nullptr, nullptr, s);
  if (st != CSA_OK) return st;
  if (launch_topk(scratch, idx, (long long)p->B * p->S, p->W, p->top_k, s) != cudaSuccess) return CSA_ERR_CUDA;
  return CSA_OK;
}

size_t csa_index_workspace_size(const csa_problem* p, int32_t which) {
  if (which == 1) return fused_workspace_bytes(p);
  if (which == 2) return backward_workspace_bytes(p);
  if (which == 3) return check_problem(p) == CSA_OK ? host_plan(p).total : 0;
  return 0;
}

csa_status csa_index_backward(const csa_problem* p, const void* q, const void* k, const void* w,
                              const int32_t* q_seg, const int32_t* kv_seg, const int64_t* q_start, const float* g,
                              float* dq, float* dk, float* dw, void* workspace, size_t workspace_bytes,
                              void* stream) {
  csa_status st = check_problem(p);
  if (st != CSA_OK) return st;
  if ((st = check_inputs(p, q, k, w, q_seg, kv_seg, q_start)) != CSA_OK) return st;
  if (g == nullptr || dq == nullptr || dk == nullptr || dw == nullptr) return CSA_ERR_INVALID_ARG;
  if (!aligned(g, 4) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dw, 4)) return CSA_ERR_INVALID_ARG;
  if (p->H != 64 || p->D != 128) return CSA_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < backward_workspace_bytes(p) || !aligned(workspace, 16))
    return CSA_ERR_INVALID_ARG;
  const long long n_pairs = (p->S + 1) / 2;
  if ((long long)p->B * n_pairs > 0x7FFFFFFFll) return CSA_ERR_UNSUPPORTED;
  const int sms = num_sms();
  if (sms <= 0) return CSA_ERR_CUDA;
  CUtensorMap tq, tk;
  if (!make_q_map(&tq, p, q, 2) || !make_k_map(&tk, p, k)) return CSA_ERR_CUDA;
  BwdParams bp;
  std::memset(&bp, 0, sizeof(bp));
  bp.B = p->B;
  bp.S = p->S;
  bp.W = p->W;
  bp.r = p->compress_rate;
  bp.r_shift = -1;
  for (int sh = 0; sh < 31; ++sh)
    if ((1 << sh) == p->compress_rate) bp.r_shift = sh;
  bp.n_pairs = (int)n_pairs;
  bp.n_items = (int)((long long)p->B * n_pairs);
  bp.n_tiles = (p->W + kTileT - 1) / kTileT;
  bp.chunk_pairs = bwd_chunk_pairs(p, sms);
  bp.n_chunks = (int)((n_pairs + bp.chunk_pairs - 1) / bp.chunk_pairs);
  if ((long long)p->B * bp.n_chunks * bp.n_tiles > 0x7FFFFFFFll) return CSA_ERR_UNSUPPORTED;
  bp.w_f32 = (p->w_dtype == CSA_F32) ? 1 : 0;
  bp.scale = p->scale;
  bp.w = w;
  bp.w_sb = strides_of(p).wb;
  bp.w_ss = strides_of(p).ws;
  bp.q_seg = q_seg;
  bp.kv_seg = kv_seg;
  bp.q_start = q_start;
  bp.g = g;
  bp.dq = dq;
  bp.dq_seq_major = p->q_layout == CSA_Q_SEQ_MAJOR ? 1 : 0;
  bp.dk = dk;
  bp.dw = dw;
  bp.counter = static_cast<unsigned int*>(workspace);
  bp.n_rb = (p->S + 3) / 4;
  bp.wait_ns = kWaitNs;
  if (q_seg != nullptr) {
    // segment summaries of the items of four rows, by the forward's pre-pass
    SegInfo* si = reinterpret_cast<SegInfo*>(static_cast<uint8_t*>(workspace) + kBwdWorkspace);
    KParams kp;
    std::memset(&kp, 0, sizeof(kp));
    kp.B = p->B;
    kp.S = p->S;
    kp.W = p->W;
    kp.r = p->compress_rate;
    kp.r_shift = bp.r_shift;
    kp.q_seg = q_seg;
    kp.kv_seg = kv_seg;
    kp.q_start = q_start;
    kp.n_rb = bp.n_rb;
    kp.n_tiles = bp.n_tiles;
    kp.n_chunks = 1;
    kp.chunk_tiles = bp.n_tiles;
    if (launch_segscan(kp, si, sms, static_cast<cudaStream_t>(stream)) != cudaSuccess) return CSA_ERR_CUDA;
    bp.seginfo = si;
  }
  if (launch_backward(tq, tk, bp, sms, static_cast<cudaStream_t>(stream)) != cudaSuccess) return CSA_ERR_CUDA;
  return CSA_OK;
}

csa_status csa_index_gather(const csa_problem* p, const void* k, const int32_t* idx, void* out, void* stream) {
  csa_status st = check_problem(p);
  if (st != CSA_OK) return st;
  if (k == nullptr || idx == nullptr || out == nullptr) return CSA_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(out, 16) || !aligned(idx, 4)) return CSA_ERR_INVALID_ARG;
  if (p->D != 128 && p->D != 32) return CSA_ERR_UNSUPPORTED;
  const int sms = num_sms();
  if (sms <= 0) return CSA_ERR_CUDA;
  const long long n_rows = (long long)p->B * p->S * p->top_k;
  const Strides ks = strides_of(p);
  if (launch_gather(k, ks.kb, ks.kw, idx, out, n_rows, p->S, p->top_k, p->W, p->D, sms,
                    static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return CSA_ERR_CUDA;
  return CSA_OK;
}

csa_status csa_index_device_status(void* stream) {
  uint32_t a = 0, b = 0, c = 0, d = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (take_status_prefill(&a, s) != cudaSuccess) return CSA_ERR_CUDA;
  if (take_status_other(&b, s) != cudaSuccess) return CSA_ERR_CUDA;
  if (take_status_gather(&c, s) != cudaSuccess) return CSA_ERR_CUDA;
  if (take_status_backward(&d, s) != cudaSuccess) return CSA_ERR_CUDA;
  const uint32_t v = a | b | c | d;
  if (v & kErrTimeout) return CSA_ERR_TIMEOUT;
  if (v != 0u) return CSA_ERR_DEVICE;
  return CSA_OK;
}

csa_status csa_index_selftest_timeout(uint32_t timeout_us, void* stream) {
  if (timeout_us == 0 || timeout_us > 10000000u) return CSA_ERR_INVALID_ARG;
  if (launch_selftest_timeout((unsigned long long)timeout_us * 1000ull, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return CSA_ERR_CUDA;
  return CSA_OK;
}

const char* csa_status_string(csa_status s) {
  switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_INVALID_ARG: return "invalid argument";
    case CSA_ERR_UNSUPPORTED: return "unsupported problem shape";
    case CSA_ERR_CUDA: return "CUDA call or launch failed";
    case CSA_ERR_TIMEOUT: return "a bounded device wait gave up";
    case CSA_ERR_DEVICE: return "device-side error";
  }
  return "unknown status";
}

int32_t csa_index_abi_version(void) { return 106; }

}  // extern "C"
