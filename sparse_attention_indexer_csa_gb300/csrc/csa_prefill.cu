// csa_prefill.cu -- instantiations of the persistent indexer kernel and their
// launcher: R = 4 query rows per item (prefill score, fused score +
// selection, its long-row mode for rows of up to 16384 entries and its
// document mode for packed documents) and R = 1 with tile chunks
// (single-row decode scores).
#include "csa_internal.h"

namespace csa {

namespace {

// Segment pre-pass of the one-kernel fused path: one warp per item of four
// whole rows scans the item's segment ids and writes its SegInfo, so the
// persistent kernel's scheduler warps read a summary instead of scanning
// up to W ids per item themselves.
__global__ void __launch_bounds__(256) csa_segscan_kernel(const KParams p, SegInfo* out) {
  griddep_wait();
  const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int n_warps = (int)((gridDim.x * blockDim.x) >> 5);
  const long long n = (long long)p.B * p.n_rb;
  for (long long i = warp; i < n; i += n_warps) {
    const int b = (int)(i / p.n_rb), rb = (int)(i % p.n_rb);
    int thr[4], seg[4], nvis[4], tfirst[4], contig[4];
    const int thr_max = item_rows<4>(p, b, rb * 4, thr, seg);
    int t_lo, t_hi;
    scan_segments<4>(p, b, 0, min(p.n_tiles * kTileT, thr_max), thr, seg, nvis, tfirst, contig, t_lo, t_hi);
    if (lane_id() == 0) {
      SegInfo si;
      si.t_lo = t_lo;
      si.t_hi = t_hi;
      si.pad0 = si.pad1 = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        si.nvis[j] = nvis[j];
        si.tfirst[j] = tfirst[j];
        si.contig[j] = contig[j];
      }
      out[i] = si;
    }
  }
}

template <class C>
cudaError_t launch_cfg(const CUtensorMap& tq, const CUtensorMap& tk, const KParams& p, int grid,
                       cudaStream_t stream) {
  const size_t smem = C::smem_bytes(p.w_pad);
  cudaError_t e = smem_limit_once<csa_index_kernel<C>>(227 * 1024);
  if (e != cudaSuccess) return e;
  // the document mode as a dependent launch after the segment pre-pass: its
  // set-up overlaps the pre-pass's end (packed_8k seed 0: -4 %)
  if constexpr (C::DOCS) return launch_pdl(csa_index_kernel<C>, dim3(grid), dim3(C::NTHREADS), smem, stream, tq, tk, p);
  csa_index_kernel<C><<<grid, C::NTHREADS, smem, stream>>>(tq, tk, p);
  return cudaGetLastError();
}

template <class C>
size_t smem_cfg(int w_pad) {
  return C::smem_bytes(w_pad);
}

}  // namespace

#define CSA_DISPATCH(H_, D_, R_, F_, CALL)                                                     \
  if (kc.H == H_ && kc.D == D_ && kc.R == R_ && kc.fused == F_ && !kc.long_rows && !kc.docs) { \
    using C = Cfg<H_, D_, R_, F_>;                                                             \
    CALL;                                                                                      \
  }
#define CSA_DISPATCH_DOCS(H_, D_, CALL)                                             \
  if (kc.H == H_ && kc.D == D_ && kc.R == 4 && kc.fused && !kc.long_rows && kc.docs) { \
    using C = Cfg<H_, D_, 4, true, false, true>;                                    \
    CALL;                                                                           \
  }
#define CSA_DISPATCH_LONG(H_, D_, CALL)                                        \
  if (kc.H == H_ && kc.D == D_ && kc.R == 4 && kc.fused && kc.long_rows) {     \
    using C = Cfg<H_, D_, 4, true, true>;                                      \
    CALL;                                                                      \
  }

cudaError_t launch_index_kernel(const KernelChoice& kc, const CUtensorMap& tq, const CUtensorMap& tk,
                                const KParams& p, int grid, cudaStream_t stream) {
  CSA_DISPATCH(64, 128, 4, false, return launch_cfg<C>(tq, tk, p, grid, stream))
  CSA_DISPATCH(64, 128, 4, true, return launch_cfg<C>(tq, tk, p, grid, stream))
  CSA_DISPATCH_LONG(64, 128, return launch_cfg<C>(tq, tk, p, grid, stream))
  CSA_DISPATCH_DOCS(64, 128, return launch_cfg<C>(tq, tk, p, grid, stream))
  CSA_DISPATCH(64, 128, 1, false, return launch_cfg<C>(tq, tk, p, grid, stream))
  CSA_DISPATCH(4, 32, 4, false, return launch_cfg<C>(tq, tk, p, grid, stream))
  CSA_DISPATCH(4, 32, 4, true, return launch_cfg<C>(tq, tk, p, grid, stream))
  return cudaErrorInvalidConfiguration;
}

size_t index_kernel_smem(const KernelChoice& kc, int w_pad) {
  CSA_DISPATCH(64, 128, 4, false, return smem_cfg<C>(w_pad))
  CSA_DISPATCH(64, 128, 4, true, return smem_cfg<C>(w_pad))
  CSA_DISPATCH_LONG(64, 128, return smem_cfg<C>(w_pad))
  CSA_DISPATCH_DOCS(64, 128, return smem_cfg<C>(w_pad))
  CSA_DISPATCH(64, 128, 1, false, return smem_cfg<C>(w_pad))
  CSA_DISPATCH(4, 32, 4, false, return smem_cfg<C>(w_pad))
  CSA_DISPATCH(4, 32, 4, true, return smem_cfg<C>(w_pad))
  return 0;
}

cudaError_t launch_segscan(const KParams& p, SegInfo* out, int sms, cudaStream_t stream) {
  const long long items = (long long)p.B * p.n_rb;
  const long long blocks = (items + 7) / 8;  // eight warps per block, one item each
  const int grid = (int)std::min<long long>(std::max<long long>(blocks, 1), (long long)sms * 16);
  return launch_pdl(csa_segscan_kernel, dim3(grid), dim3(256), 0, stream, p, out);
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
