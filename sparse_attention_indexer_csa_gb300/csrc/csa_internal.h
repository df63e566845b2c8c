// csa_internal.h -- host-side interface between the C ABI (csa_api.cu) and
// the translation units that instantiate and launch the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "csa_score_kernel.cuh"

namespace csa {

constexpr int kMaxDevices = 64;

// Raises the dynamic shared-memory limit of kernel `Fn` to `bytes` on the
// current device, once per device and thread-safe; a failed attempt is not
// remembered, so a later call tries again.
template <auto Fn>
cudaError_t smem_limit_once(int bytes) {
  static std::atomic<bool> done[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> guard(mu);
  if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  e = cudaFuncSetAttribute(Fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
  return e;
}

// Which instantiation of the persistent kernel to launch.
struct KernelChoice {
  int H, D, R;
  bool fused;
};

// Launch the persistent score (or fused score + selection) kernel.
cudaError_t launch_index_kernel(const KernelChoice& kc, const CUtensorMap& tq, const CUtensorMap& tk,
                                const KParams& p, int grid, cudaStream_t stream);
// Dynamic shared memory of that kernel (0 if the choice is not instantiated).
size_t index_kernel_smem(const KernelChoice& kc, int w_pad);

// Standalone per-row selection over [rows, W] fp32 scores.
cudaError_t launch_topk(const float* scores, int32_t* idx, long long rows, int W, int K,
                        cudaStream_t stream);
int topk_threads(int W);

// Gather of the selected compressed entries (D in {32, 128}).
cudaError_t launch_gather(const void* k, const int32_t* idx, void* out, long long n_rows, int S, int K, int W, int D,
                          int sms, cudaStream_t stream);
cudaError_t take_status_gather(uint32_t* out, cudaStream_t stream);

// Backward of the score step for one batch and one chunk of query rows
// (csa_backward.cu): P in bf16 into the chunk buffer and dw, then two GEMMs.
struct BwdParams {
  int B, S, W, r;
  int b;        // batch of this launch
  int s_base;   // first row of the chunk
  int rows;     // rows in the chunk
  int n_items;  // pairs of rows: (rows + 1) / 2
  int grid;     // CTAs (persistent; at most n_items are launched)
  int T_eff;    // tiles of the chunk's GEMM range: P is written for [0, T_eff*128)
  int sub_rows; // > 0: rows of a GEMM sub-block (even); a pair's P spans its sub-block's
                // range, ceil(min(W, (s_base + end of sub-block) / r) / 128) tiles
  int w_f32;
  float scale;
  const void* w;
  const int32_t* q_seg;
  const int32_t* kv_seg;
  const int64_t* q_start;
  const float* g;
  float* dw;
  const void* q_gather;  // head-major q [B,H,S,D] to copy into qc, or null
  void* qc;              // the chunk's q rows in (row, head) order [rows, H, D], or null
  unsigned long long wait_ns;
};
struct BwdGemms {
  int H, D, rows, w_eff, w_pad;  // rows and GEMM range of one sub-block of a chunk
  const void* p;       // P rows of the sub-block: [rows, H, w_pad] bf16
  const void* k;       // [W, D] bf16 of the batch
  const void* qc;      // the sub-block's q rows in the same (row, head) order: [rows, H, D] bf16
  float* dq;           // dq of the sub-block's first row, head 0
  long long dq_head_stride;  // floats between heads (S*D head-major, D sequence-major)
  int dq_row_stride;         // floats between rows (D head-major, H*D sequence-major)
  float* dk;           // dk[b] [W, D]
};
cudaError_t launch_backward_kernel(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tp,
                                   const BwdParams& bp, cudaStream_t stream);
size_t backward_kernel_smem();
bool backward_gemms(const BwdGemms& gm, cudaStream_t stream);
// qc[h][r][:] = q[b, s0 + r, h, :] for a sequence-major q (bf16, D = 128).
cudaError_t take_status_backward(uint32_t* out, cudaStream_t stream);

// Kernel that waits on a barrier nothing completes, bounded by `ns`.
cudaError_t launch_selftest_timeout(unsigned long long ns, cudaStream_t stream);

// Read and clear the status words of each translation unit (stream-ordered copy + sync).
cudaError_t take_status_prefill(uint32_t* out, cudaStream_t stream);
cudaError_t take_status_other(uint32_t* out, cudaStream_t stream);

}  // namespace csa
