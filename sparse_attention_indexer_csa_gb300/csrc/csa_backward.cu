// csa_backward.cu -- backward of the score step for one chunk of query rows,
// and the two library GEMMs that finish it.
//
// The score of "Add StreamIndex Kernel for CSA [Deepseek v4]" (Description) is
//   score[b,s,t] = sum_h w[b,s,h] * ReLU(scale * x),  x = q[b,h,s,:] . k[b,t,:];
// the page's custom_vjp takes the cotangent g[b,s,t] of the scores back to
//   dw[b,s,h] = sum_t gm * ReLU(scale * x)
//   P[b,h,s,t] = gm * w[b,s,h] * scale * [scale * x > 0]
//   dq[b,h,s,:] = sum_t P * k[b,t,:]         dk[b,t,:] = sum_{h,s} P * q[b,h,s,:]
// with gm = g on visible entries and 0 on masked ones (masked scores are
// constants).  For a chunk of rows this kernel recomputes x on the tensor
// cores, forms P in bf16 for the chunk only ([H, rows, W_pad] in the caller's
// workspace -- never the whole [B,H,S,W]) and dw in registers; dq and dk are
// then two plain GEMMs over that chunk (cuBLAS).
//
// Kernel layout (one CTA per pair of query rows, 192 threads):
//   warp 0  TMA: the q block (2 rows x 64 heads x 128, as the UMMA A operand:
//           M = 128 rows (row j, head h) -> 64 j + h) once, then k tiles
//           (128 entries, the B operand, N = 128) into three stages;
//   warp 1  TMEM owner and UMMA issuer: per k tile one 128x128x128 product
//           into one of two 128-column accumulators;
//   warps 2-5  epilogue: warp w reads TMEM lanes 32*(w%4) .. (rows (j, h)),
//           so each thread owns one (row, head) and walks the tile's 128
//           entries: dw in a register, P converted to bf16 into a
//           128-byte-swizzled staging tile that one thread writes out with
//           3-D TMA stores (box {64 entries, 2 rows, 64 heads}).
// Tiles past the pair's visible range but inside the chunk's GEMM range are
// written as zeros without any product.
#include <cublas_v2.h>
#include <cuda_bf16.h>

#include <mutex>

#include "csa_internal.h"

namespace csa {

namespace {

constexpr int kBH = 64, kBD = 128, kBR = 2;
constexpr int kBM = kBR * kBH;                      // 128 (row, head) pairs: UMMA M
constexpr int kBNKC = kBD / 64;                     // K chunks of 64 (128-byte swizzled rows)
constexpr uint32_t kBQChunk = kBM * 128;            // 16 KB
constexpr uint32_t kBQBytes = kBQChunk * kBNKC;     // 32 KB
constexpr uint32_t kBKChunk = kTileT * 128;         // 16 KB
constexpr uint32_t kBKBytes = kBKChunk * kBNKC;     // 32 KB
constexpr int kBStages = 3;
constexpr uint32_t kBPHalf = kBM * 128;             // 16 KB: 128 rows x 64 entries of bf16
constexpr uint32_t kBPTile = 2 * kBPHalf;           // 32 KB
constexpr uint32_t kBIdesc = idesc_bf16_f32(kBM, kTileT);
constexpr int kBThreads = 192;
constexpr uint32_t kBTmemCols = 256;                // two 128-column accumulators
constexpr uint32_t kBEpiBar = 2;                    // named barrier of the epilogue warps

constexpr uint32_t OFF_BQ = 0;
constexpr uint32_t OFF_BK = OFF_BQ + kBQBytes;
constexpr uint32_t OFF_BP = OFF_BK + kBStages * kBKBytes;
constexpr uint32_t OFF_BG = OFF_BP + 2 * kBPTile;          // 4 warps x 128 fp32 cotangents
constexpr uint32_t OFF_BBAR = OFF_BG + 4 * kTileT * 4;     // 1 + 2*stages + 4 barriers
constexpr uint32_t OFF_BMISC = OFF_BBAR + 16 * 8;
constexpr uint32_t kBSmem = OFF_BMISC + 64 + 1024;         // + alignment slack

struct BSm {
  uint8_t* base;
  __device__ uint8_t* q() const { return base + OFF_BQ; }
  __device__ uint8_t* k(int i) const { return base + OFF_BK + i * kBKBytes; }
  __device__ uint8_t* ptile(int i) const { return base + OFF_BP + i * kBPTile; }
  __device__ float* g(int e) const { return reinterpret_cast<float*>(base + OFF_BG) + e * kTileT; }
  __device__ uint64_t* bar(int i) const { return reinterpret_cast<uint64_t*>(base + OFF_BBAR) + i; }
  __device__ uint64_t* q_full() const { return bar(0); }
  __device__ uint64_t* k_full(int i) const { return bar(1 + i); }
  __device__ uint64_t* k_empty(int i) const { return bar(1 + kBStages + i); }
  __device__ uint64_t* acc_full(int i) const { return bar(1 + 2 * kBStages + i); }
  __device__ uint64_t* acc_empty(int i) const { return bar(3 + 2 * kBStages + i); }
  __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(base + OFF_BMISC); }
  __device__ volatile uint32_t* abort_flag() const {
    return reinterpret_cast<volatile uint32_t*>(base + OFF_BMISC + 4);
  }
};

// Visible-entry threshold of absolute row s (future mask): entries t < thr.
__device__ __forceinline__ int row_threshold(const BwdParams& p, int s) {
  if (s >= p.S) return 0;
  const long long qs0 = p.q_start ? (long long)p.q_start[p.b] : 0ll;
  long long tv = (qs0 + s + 1) / p.r;
  tv = tv < 0 ? 0 : (tv > p.W ? p.W : tv);
  return (int)tv;
}

__global__ void __launch_bounds__(kBThreads, 1)
    csa_backward_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_p, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const BSm sm{base};
  const int warp = threadIdx.x / 32;
  const uint32_t lane = lane_id();
  // pairs in reverse order: the longest rows (most tiles) start first
  const int pair = p.n_items - 1 - (int)blockIdx.x;
  const int sl0 = 2 * pair;         // first row of the pair, relative to the chunk
  const int s0 = p.s_base + sl0;    // absolute row
  const int thr0 = row_threshold(p, s0);
  const int thr1 = (sl0 + 1 < p.rows) ? row_threshold(p, s0 + 1) : 0;
  const int t_hi = min(p.T_eff, (max(thr0, thr1) + kTileT - 1) / kTileT);  // tiles with products

  if (threadIdx.x == 0) {
    mbar_init(sm.q_full(), 1);
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(sm.k_full(i), 1);
      mbar_init(sm.k_empty(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sm.acc_full(i), 1);
      mbar_init(sm.acc_empty(i), 4);
    }
    *sm.abort_flag() = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_p);
  }
  if (warp == 1) {
    tmem_alloc(sm.tmem_slot(), kBTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot();
  const WaitCtl ctl{sm.abort_flag(), p.wait_ns};

  if (warp == 0) {
    if (lane == 0 && t_hi > 0) {
      const uint64_t q_pol = l2_policy_evict_first(), k_pol = l2_policy_evict_last();
      mbar_arrive_expect_tx(sm.q_full(), kBQBytes);
#pragma unroll
      for (int c = 0; c < kBNKC; ++c)
        tma_load_4d_hint(sm.q() + c * kBQChunk, &tmap_q, sm.q_full(), c * 64, 0, s0, p.b, q_pol);
      for (int tile = 0; tile < t_hi; ++tile) {
        const int st = tile % kBStages;
        if (!mbar_wait(sm.k_empty(st), ((tile / kBStages) & 1) ^ 1, ctl)) break;
        mbar_arrive_expect_tx(sm.k_full(st), kBKBytes);
#pragma unroll
        for (int c = 0; c < kBNKC; ++c)
          tma_load_3d_hint(sm.k(st) + c * kBKChunk, &tmap_k, sm.k_full(st), c * 64, tile * kTileT, p.b, k_pol);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && t_hi > 0) {
      const bool q_ok = mbar_wait(sm.q_full(), 0, ctl);
      tc_fence_after();
      const uint32_t q_addr = smem_u32(sm.q());
      for (int tile = 0; tile < t_hi; ++tile) {
        const int st = tile % kBStages, a = tile & 1;
        const bool k_ok = mbar_wait(sm.k_full(st), (tile / kBStages) & 1, ctl);
        const bool a_ok = mbar_wait(sm.acc_empty(a), ((tile >> 1) & 1) ^ 1, ctl);
        tc_fence_after();
        if (q_ok && k_ok && a_ok) {
          const uint32_t k_addr = smem_u32(sm.k(st));
          const uint32_t d_tmem = tmem_base + (uint32_t)(a * kTileT);
#pragma unroll
          for (int c = 0; c < kBNKC; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t adesc = smem_desc_kmajor(q_addr + c * kBQChunk + kk * 32, 128);
              const uint64_t bdesc = smem_desc_kmajor(k_addr + c * kBKChunk + kk * 32, 128);
              umma_bf16(d_tmem, adesc, bdesc, kBIdesc, (c | kk) != 0 ? 1u : 0u);
            }
          }
        }
        umma_commit(sm.k_empty(st));
        umma_commit(sm.acc_full(a));
        if (!(q_ok && k_ok && a_ok)) break;
      }
    }
  } else {
    // epilogue: thread = TMEM lane m = 32*quarter + lane = (row j, head h)
    const int e = warp - 2;
    const int quarter = warp & 3;
    const int m = quarter * 32 + (int)lane;
    const int j = m >> 6, h = m & 63;  // row of the pair (warp-uniform), head
    const int s = s0 + j;
    const bool row_ok = (sl0 + j < p.rows) && s < p.S;
    const int thr = j ? thr1 : thr0;
    const bool segs = p.q_seg != nullptr;
    const int seg = (segs && row_ok) ? p.q_seg[(size_t)p.b * p.S + s] : 0;
    float wc = 0.f;
    if (row_ok) {
      const size_t off = ((size_t)p.b * p.S + s) * kBH + h;
      wc = (p.w_f32 ? reinterpret_cast<const float*>(p.w)[off]
                    : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.w)[off])) *
           p.scale;
    }
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
    float* gb = sm.g(e);
    // staging row of this thread in the TMA box order {entry, row, head}
    const uint32_t srow = (uint32_t)(h * 2 + j);
    float dw_acc = 0.f;
    for (int tile = 0; tile < p.T_eff; ++tile) {
      // masked cotangents of this warp's row for the tile
      {
        const int t0 = tile * kTileT + 4 * (int)lane;
        float gv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int t = t0 + u;
          bool vis = row_ok && t < thr;
          if (vis && segs) vis = p.kv_seg[(size_t)p.b * p.W + t] == seg;
          gv[u] = vis ? p.g[((size_t)p.b * p.S + s) * p.W + t] : 0.f;
        }
        *reinterpret_cast<float4*>(gb + 4 * lane) = make_float4(gv[0], gv[1], gv[2], gv[3]);
      }
      __syncwarp();
      // the staging tile of two tiles ago has been read by its TMA store
      if (e == 0 && lane == 0) bulk_wait_group_read<1>();
      named_bar_sync(kBEpiBar, 128);
      uint8_t* pt = sm.ptile(tile & 1);
      const bool computed = tile < t_hi;
      const int a = tile & 1;
      bool ok = true;
      if (computed) {
        ok = mbar_wait(sm.acc_full(a), (tile >> 1) & 1, ctl);
        tc_fence_after();
      }
      float va[32], vb[32];
      if (computed && ok) {
        tmem_ld32_start(t_lane + (uint32_t)(a * kTileT), va);
        tmem_wait32(va);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 32 entries per chunk
        float(&cur)[32] = (c & 1) ? vb : va;
        float(&nxt)[32] = (c & 1) ? va : vb;
        if (computed && ok && c + 1 < 4) tmem_ld32_start(t_lane + (uint32_t)(a * kTileT + (c + 1) * 32), nxt);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float pr[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int col = c * 32 + 2 * i + u;
            const float x = (computed && ok) ? cur[2 * i + u] * p.scale : 0.f;
            const float gm = gb[col];
            dw_acc = fmaf(gm, fmaxf(x, 0.f), dw_acc);
            pr[u] = (x > 0.f) ? gm * wc : 0.f;
          }
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(pr[0], pr[1]);
          pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        // 32 entries = 64 bytes: 16-byte chunks 4*(c&1) .. 4*(c&1)+3 of half c>>1
        uint8_t* half = pt + (c >> 1) * kBPHalf + srow * 128u;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const uint32_t chunk = (uint32_t)(4 * (c & 1) + q4);
          const uint32_t pos = chunk ^ (srow & 7u);  // 128-byte swizzle
          *reinterpret_cast<uint4*>(half + pos * 16u) =
              make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
        }
        if (computed && ok && c + 1 < 4) tmem_wait32(nxt);
      }
      if (computed) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.acc_empty(a));
      }
      fence_proxy_async_shared();
      named_bar_sync(kBEpiBar, 128);
      if (e == 0 && lane == 0) {
        tma_store_3d(&tmap_p, pt, tile * kTileT, sl0, 0);
        tma_store_3d(&tmap_p, pt + kBPHalf, tile * kTileT + 64, sl0, 0);
        bulk_commit_group();
      }
      __syncwarp();
    }
    if (row_ok) p.dw[((size_t)p.b * p.S + s) * kBH + h] = dw_acc;
    if (e == 0 && lane == 0) bulk_wait_group_all();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kBTmemCols);
}

cublasHandle_t blas_handle() {
  static cublasHandle_t handles[64];
  static std::once_flag flags[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::call_once(flags[dev], [dev] {
    cublasHandle_t h = nullptr;
    if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) h = nullptr;
    handles[dev] = h;
  });
  return handles[dev];
}

}  // namespace

size_t backward_kernel_smem() { return kBSmem; }

cudaError_t launch_backward_kernel(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tp,
                                   const BwdParams& bp, cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(csa_backward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBSmem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  if (bp.n_items <= 0) return cudaSuccess;
  csa_backward_kernel<<<bp.n_items, kBThreads, kBSmem, stream>>>(tq, tk, tp, bp);
  return cudaGetLastError();
}

// dq rows of the chunk (one GEMM per head, batched) and the chunk's share of
// dk (one GEMM over all heads and rows), fp32 accumulation of bf16 operands.
// Row-major operands are passed to the column-major library transposed.
bool backward_gemms(const BwdGemms& gm, cudaStream_t stream) {
  cublasHandle_t h = blas_handle();
  if (h == nullptr || cublasSetStream(h, stream) != CUBLAS_STATUS_SUCCESS) return false;
  const float one = 1.f, zero = 0.f;
  // dq[h][rows x D] = P[h][rows x W_eff] . k[W_eff x D]   (column-major: D x rows = k^T . P^T)
  if (cublasGemmStridedBatchedEx(h, CUBLAS_OP_N, CUBLAS_OP_N, gm.D, gm.rows, gm.w_eff, &one, gm.k, CUDA_R_16BF,
                                 gm.D, 0, gm.p, CUDA_R_16BF, gm.w_pad, (long long)gm.rows * gm.w_pad, &zero, gm.dq,
                                 CUDA_R_32F, gm.D, gm.dq_head_stride, gm.H, CUBLAS_COMPUTE_32F,
                                 CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
    return false;
  // dk[W_eff x D] += P_all^T[W_eff x (H rows)] . Q[(H rows) x D]   (column-major: D x W_eff = Q^T . P_all)
  if (cublasGemmEx(h, CUBLAS_OP_N, CUBLAS_OP_T, gm.D, gm.w_eff, gm.H * gm.rows, &one, gm.qc, CUDA_R_16BF, gm.D,
                   gm.p, CUDA_R_16BF, gm.w_pad, &one, gm.dk, CUDA_R_32F, gm.D, CUBLAS_COMPUTE_32F,
                   CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
    return false;
  return true;
}

cudaError_t take_status_backward(uint32_t* out, cudaStream_t stream) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_status, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e;
}

}  // namespace csa
