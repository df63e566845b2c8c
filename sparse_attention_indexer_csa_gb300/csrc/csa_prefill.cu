// csa_prefill.cu -- instantiations of the persistent indexer kernel and their
// launcher: R = 4 query rows per item (prefill score and fused score +
// selection) and R = 1 with tile chunks (single-row decode scores).
#include "csa_internal.h"

namespace csa {

namespace {

template <class C>
cudaError_t launch_cfg(const CUtensorMap& tq, const CUtensorMap& tk, const KParams& p, int grid,
                       cudaStream_t stream) {
  const size_t smem = C::smem_bytes(p.w_pad);
  cudaError_t e = smem_limit_once<csa_index_kernel<C>>(227 * 1024);
  if (e != cudaSuccess) return e;
  csa_index_kernel<C><<<grid, C::NTHREADS, smem, stream>>>(tq, tk, p);
  return cudaGetLastError();
}

template <class C>
size_t smem_cfg(int w_pad) {
  return C::smem_bytes(w_pad);
}

}  // namespace

#define CSA_DISPATCH(H_, D_, R_, F_, CALL)                  \
  if (kc.H == H_ && kc.D == D_ && kc.R == R_ && kc.fused == F_) { \
    using C = Cfg<H_, D_, R_, F_>;                          \
    CALL;                                                   \
  }

cudaError_t launch_index_kernel(const KernelChoice& kc, const CUtensorMap& tq, const CUtensorMap& tk,
                                const KParams& p, int grid, cudaStream_t stream) {
  CSA_DISPATCH(64, 128, 4, false, return launch_cfg<C>(tq, tk, p, grid, stream))
  CSA_DISPATCH(64, 128, 4, true, return launch_cfg<C>(tq, tk, p, grid, stream))
  CSA_DISPATCH(64, 128, 1, false, return launch_cfg<C>(tq, tk, p, grid, stream))
  CSA_DISPATCH(4, 32, 4, false, return launch_cfg<C>(tq, tk, p, grid, stream))
  CSA_DISPATCH(4, 32, 4, true, return launch_cfg<C>(tq, tk, p, grid, stream))
  return cudaErrorInvalidConfiguration;
}

size_t index_kernel_smem(const KernelChoice& kc, int w_pad) {
  CSA_DISPATCH(64, 128, 4, false, return smem_cfg<C>(w_pad))
  CSA_DISPATCH(64, 128, 4, true, return smem_cfg<C>(w_pad))
  CSA_DISPATCH(64, 128, 1, false, return smem_cfg<C>(w_pad))
  CSA_DISPATCH(4, 32, 4, false, return smem_cfg<C>(w_pad))
  CSA_DISPATCH(4, 32, 4, true, return smem_cfg<C>(w_pad))
  return 0;
}

cudaError_t take_status_prefill(uint32_t* out, cudaStream_t stream) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_status, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e;
}

}  // namespace csa
