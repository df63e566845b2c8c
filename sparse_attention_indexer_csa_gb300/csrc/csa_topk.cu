// csa_topk.cu -- standalone per-row selection over precomputed scores, and
// the bounded-wait self-test kernel.
#include "csa_internal.h"
#include "csa_select.cuh"

namespace csa {

namespace {

constexpr int kTopkMaxRow = 49152;  // longest row the kernel stages in shared memory

template <int NT>
struct TopkCfg {
  static constexpr int NB = (NT >= 512) ? 2048 : (NT >= 256 ? 1024 : 512);
  static constexpr int CAP = (NT >= 512) ? 1024 : 256;
  struct Scratch {
    SelectScratch sc;
    BinScratch<NB, CAP, 4 * (kTopkMaxRow / 128 + 1)> bs;
    RowStats st;
  };
  static constexpr uint32_t HEADER = (sizeof(Scratch) + 15u) & ~15u;
  static size_t smem(int W) { return HEADER + (size_t)((W + 127) & ~127) * sizeof(float); }
};

// One CTA per row (grid-strided): the row is staged in shared memory while its
// visible count and value range are reduced, then the whole CTA runs the
// selection and the ordered write.
template <int NT>
__global__ void __launch_bounds__(NT) csa_topk_kernel(const float* __restrict__ scores, int32_t* __restrict__ idx,
                                                      long long rows, int W, int K) {
  using TC = TopkCfg<NT>;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  typename TC::Scratch* scr = reinterpret_cast<typename TC::Scratch*>(smem_raw);
  float* row = reinterpret_cast<float*>(smem_raw + TC::HEADER);
  const Team<NT> team{1u, threadIdx.x};
  const bool vec = (W % 4) == 0 && (reinterpret_cast<uintptr_t>(scores) % 16) == 0;
  const int wpad = (W + 127) & ~127;
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    if (threadIdx.x == 0) {
      scr->st.nvis = 0u;
      scr->st.min_key = 0xFFFFFFFFu;
      scr->st.max_key = 0u;
    }
    team.sync();
    const float* src = scores + (size_t)r * W;
    uint32_t cnt = 0, kmin = 0xFFFFFFFFu, kmax = 0u;
    auto note = [&](float x) {
      const uint32_t k = score_key(x);
      if (k != 0u) {
        ++cnt;
        kmin = min(kmin, k);
        kmax = max(kmax, k);
      }
    };
    if (vec) {  // four 16-byte loads in flight per thread
      const float4* s4 = reinterpret_cast<const float4*>(src);
      float4* d4 = reinterpret_cast<float4*>(row);
      const int w4 = W / 4;
#pragma unroll 1
      for (int i0 = threadIdx.x; i0 < w4; i0 += 4 * NT) {
        float4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          v[q] = (i0 + q * NT < w4) ? __ldcs(s4 + i0 + q * NT)
                                    : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (i0 + q * NT < w4) d4[i0 + q * NT] = v[q];
          note(v[q].x);
          note(v[q].y);
          note(v[q].z);
          note(v[q].w);
        }
      }
    } else {
      for (int i = threadIdx.x; i < W; i += NT) {
        const float v = __ldcs(src + i);
        row[i] = v;
        note(v);
      }
    }
    for (int i = W + threadIdx.x; i < wpad; i += NT) row[i] = -INFINITY;
    cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
    kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
    kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
    if ((threadIdx.x & 31u) == 0 && cnt > 0u) {
      atomicAdd(&scr->st.nvis, cnt);
      atomicMin(&scr->st.min_key, kmin);
      atomicMax(&scr->st.max_key, kmax);
    }
    team.sync();
    const RowStats st = scr->st;
    team_topk_row(row, 0, wpad, (uint32_t)K, st, idx + (size_t)r * K, &scr->bs, &scr->sc, team);
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
  // sized from the very layout the kernel instantiation uses
  const size_t smem = TopkCfg<NT>::smem(W);
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

cudaError_t launch_topk(const float* scores, int32_t* idx, long long rows, int W, int K, cudaStream_t stream) {
  if (W > kTopkMaxRow) return cudaErrorInvalidValue;
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
