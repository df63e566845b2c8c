// csa_gather.cu -- gather of the selected compressed entries:
//   out[b,s,i,:] = k[b, idx[b,s,i], :]   (zeros where idx == -1)
// the rows the sparse attention consumes after the selection ("DSV4: Add
// indexer_save_selection and indexer_sharded_topk", Description: selected
// indices go back to the sequence layout before sparse attention).
// Memory-bound: each output row is D bf16 (D*2 bytes) read from k and
// written once with streaming stores.
#include "csa_internal.h"

namespace csa {

namespace {

// One group of G = D*2/16 lanes per output row; each lane moves 16 bytes.
template <int G>
// k_sb, k_sw: strides of k's batch and entry dimensions in 16-byte units.
__global__ void __launch_bounds__(256) csa_gather_kernel(const uint4* __restrict__ k, long long k_sb, long long k_sw,
                                                         const int32_t* __restrict__ idx, uint4* __restrict__ out,
                                                         long long n_rows, int S, int K, int W) {
  constexpr int ROWS_PER_BLOCK = 256 / G;
  const int g = threadIdx.x / G, l = threadIdx.x % G;
  for (long long r = (long long)blockIdx.x * ROWS_PER_BLOCK + g; r < n_rows; r += (long long)gridDim.x * ROWS_PER_BLOCK) {
    const long long bs = r / K;  // (b, s) row of the selection
    const long long b = bs / S;
    const int t = __ldcs(idx + r);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (t >= 0 && t < W) {
      v = __ldg(k + (size_t)b * k_sb + (size_t)t * k_sw + l);
    } else if (t != -1 && l == 0) {
      record_error(kErrDevice);  // index outside [-1, W): the row is written as zeros
    }
    __stcs(out + (size_t)r * G + l, v);
  }
}

}  // namespace

cudaError_t launch_gather(const void* k, long long k_sb, long long k_sw, const int32_t* idx, void* out,
                          long long n_rows, int S, int K, int W, int D, int sms, cudaStream_t stream) {
  // strides in 16-byte units (8 bf16 elements; the caller checked divisibility)
  const long long sb = k_sb / 8, sw = k_sw / 8;
  const long long blocks_needed = (n_rows * (D * 2 / 16) + 255) / 256;
  const int grid = (int)std::min<long long>(std::max<long long>(blocks_needed, 1), (long long)sms * 8);
  if (D == 128) {
    csa_gather_kernel<16><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(k), sb, sw, idx,
                                                   static_cast<uint4*>(out), n_rows, S, K, W);
  } else if (D == 32) {
    csa_gather_kernel<4><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(k), sb, sw, idx,
                                                  static_cast<uint4*>(out), n_rows, S, K, W);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t take_status_gather(uint32_t* out, cudaStream_t stream) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_status, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e;
}

}  // namespace csa
