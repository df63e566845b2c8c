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

// Launch of `kernel` on `stream` with programmatic stream serialization: it
// may start while the previous kernel on the stream finishes, and waits in
// griddep_wait() before reading global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Which instantiation of the persistent kernel to launch.
struct KernelChoice {
  int H, D, R;
  bool fused;
  bool long_rows = false;  // fused with rows of 4097..16384 entries
  bool docs = false;       // fused with segment summaries: the document mode (H = 64, D = 128)
};

// Launch the persistent score (or fused score + selection) kernel.
cudaError_t launch_index_kernel(const KernelChoice& kc, const CUtensorMap& tq, const CUtensorMap& tk,
                                const KParams& p, int grid, cudaStream_t stream);
// Dynamic shared memory of that kernel (0 if the choice is not instantiated).
size_t index_kernel_smem(const KernelChoice& kc, int w_pad);
// Segment pre-pass of the fused path: SegInfo of every item of four rows.
cudaError_t launch_segscan(const KParams& p, SegInfo* out, int sms, cudaStream_t stream);

// Standalone per-row selection over [rows, W] fp32 scores.
cudaError_t launch_topk(const float* scores, int32_t* idx, long long rows, int W, int K,
                        cudaStream_t stream);
int topk_threads(int W);

// Gather of the selected compressed entries (D in {32, 128}).
// k_sb, k_sw: element strides of k's batch and entry dimensions.
cudaError_t launch_gather(const void* k, long long k_sb, long long k_sw, const int32_t* idx, void* out,
                          long long n_rows, int S, int K, int W, int D, int sms, cudaStream_t stream);
cudaError_t take_status_gather(uint32_t* out, cudaStream_t stream);

// Backward of the score step (csa_backward.cu): the dq / dw kernel over
// pairs of query rows, then the dk kernel over (k tile, run of row pairs)
// items handed out through `counter`.
struct BwdParams {
  int B, S, W, r;
  int r_shift;      // log2(r) when r is a power of two, else -1
  int n_pairs;      // pairs of query rows per batch: (S + 1) / 2
  int n_items;      // dq kernel items: B * n_pairs
  int n_tiles;      // k tiles of 128 entries: ceil(W / 128)
  int chunk_pairs;  // dk kernel: row pairs per item at most
  int n_chunks;     // dk kernel: ceil(n_pairs / chunk_pairs)
  int w_f32;
  float scale;
  const void* w;
  long long w_sb, w_ss;   // element strides of w's batch and row dimensions
  const int32_t* q_seg;
  const int32_t* kv_seg;
  const int64_t* q_start;
  const float* g;
  float* dq;          // fp32 in q's layout
  int dq_seq_major;   // dq [B,S,H,D] (1) or [B,H,S,D] (0)
  float* dk;          // [B,W,D] fp32 (zeroed, then accumulated)
  float* dw;          // [B,S,H] fp32
  unsigned int* counter;  // dk item counter (device memory, zeroed before the launch)
  const SegInfo* seginfo;  // with segment ids: [B][n_rb] summaries of items of four rows, else null
  int n_rb;                // items of four rows per batch: ceil(S / 4)
  unsigned long long wait_ns;
};
// Enqueues the whole backward on `stream` (two memsets, two kernels).
cudaError_t launch_backward(const CUtensorMap& tq, const CUtensorMap& tk, const BwdParams& bp, int sms,
                            cudaStream_t stream);
size_t backward_kernel_smem();
cudaError_t take_status_backward(uint32_t* out, cudaStream_t stream);

// Kernel that waits on a barrier nothing completes, bounded by `ns`.
cudaError_t launch_selftest_timeout(unsigned long long ns, cudaStream_t stream);

// Read and clear the status words of each translation unit (stream-ordered copy + sync).
cudaError_t take_status_prefill(uint32_t* out, cudaStream_t stream);
cudaError_t take_status_other(uint32_t* out, cudaStream_t stream);

}  // namespace csa
