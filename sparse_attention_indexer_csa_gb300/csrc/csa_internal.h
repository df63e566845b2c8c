// csa_internal.h -- host-side interface between the C ABI (csa_api.cu) and
// the translation units that instantiate and launch the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "csa_score_kernel.cuh"

namespace csa {

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

// Kernel that waits on a barrier nothing completes, bounded by `ns`.
cudaError_t launch_selftest_timeout(unsigned long long ns, cudaStream_t stream);

// Read and clear the status words of each translation unit (stream-ordered copy + sync).
cudaError_t take_status_prefill(uint32_t* out, cudaStream_t stream);
cudaError_t take_status_other(uint32_t* out, cudaStream_t stream);

}  // namespace csa
