// csa_topk.cu -- standalone per-row selection over precomputed scores, and
// the bounded-wait self-test kernel.
#include "csa_internal.h"
#include "csa_select.cuh"

namespace csa {

namespace {

constexpr uint32_t kTopkSmemHeader = (sizeof(SelectScratch) + 15u) & ~15u;

// One CTA per row (grid-strided): the row is staged in shared memory, then
// the whole CTA runs the radix selection and the ordered write.
template <int NT>
__global__ void __launch_bounds__(NT) csa_topk_kernel(const float* __restrict__ scores, int32_t* __restrict__ idx,
                                                      long long rows, int W, int K) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelectScratch* sc = reinterpret_cast<SelectScratch*>(smem_raw);
  float* row = reinterpret_cast<float*>(smem_raw + kTopkSmemHeader);
  const Team<NT> team{1u, threadIdx.x};
  const bool vec = (W % 4) == 0 && (reinterpret_cast<uintptr_t>(scores) % 16) == 0;
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    const float* src = scores + (size_t)r * W;
    if (vec) {
      const float4* s4 = reinterpret_cast<const float4*>(src);
      float4* d4 = reinterpret_cast<float4*>(row);
      for (int i = threadIdx.x; i < W / 4; i += NT) d4[i] = __ldcs(s4 + i);
    } else {
      for (int i = threadIdx.x; i < W; i += NT) row[i] = __ldcs(src + i);
    }
    team.sync();
    team_topk_row<NT>(row, 0, W, (uint32_t)K, idx + (size_t)r * K, sc, team);
    team.sync();
  }
}

__global__ void csa_selftest_timeout_kernel(unsigned long long ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl ctl{&abort_flag, ns};
  // phase 0 of `bar` never completes: nothing arrives on it
  mbar_wait(&bar, 0, ctl);
  __syncthreads();
}

template <int NT>
cudaError_t launch_topk_nt(const float* scores, int32_t* idx, long long rows, int W, int K, cudaStream_t stream) {
  const size_t smem = topk_smem(W);
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(csa_topk_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const long long grid = rows < 1048576 ? rows : 1048576;
  csa_topk_kernel<NT><<<(unsigned)grid, NT, smem, stream>>>(scores, idx, rows, W, K);
  return cudaGetLastError();
}

}  // namespace

int topk_threads(int W) {
  if (W <= 2048) return 128;
  if (W <= 8192) return 256;
  if (W <= 16384) return 512;
  return 1024;
}

size_t topk_smem(int W) { return kTopkSmemHeader + (size_t)W * sizeof(float); }

cudaError_t launch_topk(const float* scores, int32_t* idx, long long rows, int W, int K, cudaStream_t stream) {
  switch (topk_threads(W)) {
    case 128: return launch_topk_nt<128>(scores, idx, rows, W, K, stream);
    case 256: return launch_topk_nt<256>(scores, idx, rows, W, K, stream);
    case 512: return launch_topk_nt<512>(scores, idx, rows, W, K, stream);
    default: return launch_topk_nt<1024>(scores, idx, rows, W, K, stream);
  }
}

cudaError_t launch_selftest_timeout(unsigned long long ns, cudaStream_t stream) {
  csa_selftest_timeout_kernel<<<1, 32, 0, stream>>>(ns);
  return cudaGetLastError();
}

cudaError_t take_status_other(uint32_t* out, cudaStream_t stream) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_status, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e;
}

}  // namespace csa
