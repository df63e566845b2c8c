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
// cores, forms P in bf16 for the chunk only ([rows, H, W_pad] in the caller's
// workspace -- never the whole [B,H,S,W]) and dw in registers; dq and dk are
// then two plain GEMMs per sub-block of the chunk's rows (cuBLAS), each over
// the entries the sub-block's last row sees -- the range of P a pair of rows
// writes here.
//
// Kernel layout (persistent: each CTA takes pairs of query rows in turn, 352
// threads):
//   warp 0  TMA: per pair the q block (2 rows x 64 heads x 128, as the UMMA A
//           operand: M = 128 rows (row j, head h) -> 64 j + h), then its k
//           tiles (128 entries, the B operand, N = 128) into three stages;
//   warp 1  TMEM owner and UMMA issuer: per k tile one 128x128x128 product
//           into one of two 128-column accumulators;
//   warps 2-9  epilogue: warp w reads TMEM lanes 32*(w%4) .. (rows (j, h))
//           and one half of the tile's 128 entries (warps 2-5 the first,
//           6-9 the second), so each thread owns one (row, head) and walks
//           64 entries per tile: dw in a register (the halves added once per
//           pair), P converted to bf16 into the warp's own 128-byte-swizzled
//           staging tile (32 heads x 64 entries), which lane 0 writes out
//           with a 3-D TMA store (box {64 entries, 32 heads, 1 row}); each
//           warp double-buffers its staging, so the warps never wait for
//           one another inside a tile.
//   warp 10  for head-major q, copies the chunk's q rows into P's (row, head)
//           order (the dk GEMMs' operand) while the other warps form P.
// Tiles past the pair's visible range but inside its sub-block's GEMM range
// are written as zeros without any product.
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
constexpr uint32_t kBPWarp = 32 * 128;              // 4 KB: one warp's 32 heads x 64 entries of bf16
constexpr uint32_t kBIdesc = idesc_bf16_f32(kBM, kTileT);
constexpr int kBEpiWarps = 8;
constexpr int kBGatherWarp = 2 + kBEpiWarps;       // copies the chunk's head-major q rows
constexpr int kBThreads = 64 + 32 * kBEpiWarps + 32;
constexpr uint32_t kBTmemCols = 256;                // two 128-column accumulators
constexpr uint32_t kBEpiBar = 2;                    // named barrier of the epilogue warps

constexpr uint32_t OFF_BQ = 0;
constexpr uint32_t OFF_BK = OFF_BQ + kBQBytes;
constexpr uint32_t OFF_BP = OFF_BK + kBStages * kBKBytes;
constexpr uint32_t OFF_BG = OFF_BP + kBEpiWarps * 2 * kBPWarp;  // 8 warps x 64 fp32 cotangents
constexpr uint32_t OFF_BDW = OFF_BG + kBEpiWarps * 64 * 4;       // 2 x 128 partial dw of the second half
constexpr uint32_t OFF_BBAR = OFF_BDW + 2 * kBM * 4;             // 2 + 2*stages + 4 barriers
constexpr uint32_t OFF_BMISC = OFF_BBAR + 16 * 8;
constexpr uint32_t kBSmem = OFF_BMISC + 64 + 1024;         // + alignment slack

struct BSm {
  uint8_t* base;
  __device__ uint8_t* q() const { return base + OFF_BQ; }
  __device__ uint8_t* k(int i) const { return base + OFF_BK + i * kBKBytes; }
  __device__ uint8_t* pstage(int e, int i) const { return base + OFF_BP + (e * 2 + i) * kBPWarp; }
  __device__ float* g(int e) const { return reinterpret_cast<float*>(base + OFF_BG) + e * 64; }
  __device__ float* dwp(int i) const { return reinterpret_cast<float*>(base + OFF_BDW) + i * kBM; }
  __device__ uint64_t* bar(int i) const { return reinterpret_cast<uint64_t*>(base + OFF_BBAR) + i; }
  __device__ uint64_t* q_full() const { return bar(0); }
  __device__ uint64_t* q_empty() const { return bar(1); }
  __device__ uint64_t* k_full(int i) const { return bar(2 + i); }
  __device__ uint64_t* k_empty(int i) const { return bar(2 + kBStages + i); }
  __device__ uint64_t* acc_full(int i) const { return bar(2 + 2 * kBStages + i); }
  __device__ uint64_t* acc_empty(int i) const { return bar(4 + 2 * kBStages + i); }
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

// Tiles of P written for the pair whose first row is sl0 (relative): the GEMM
// range of its sub-block of rows, the same expression the host uses for that
// sub-block's GEMMs; the chunk's range without sub-blocks.
__device__ __forceinline__ int pair_tiles(const BwdParams& p, int sl0) {
  if (p.sub_rows <= 0) return p.T_eff;
  const int end = min(p.rows, (sl0 / p.sub_rows + 1) * p.sub_rows);
  long long tv = ((long long)p.s_base + end) / p.r;
  tv = tv > p.W ? p.W : tv;
  return (int)((tv + kTileT - 1) / kTileT);
}

// Pair number `pair` of the chunk: its first row (relative and absolute), the
// visible thresholds of its two rows, the tiles of P it writes and the tiles
// that need products.
struct PairInfo {
  int sl0, s0, thr0, thr1, T, t_hi;
};
__device__ __forceinline__ PairInfo pair_info(const BwdParams& p, int pair) {
  PairInfo pi;
  pi.sl0 = 2 * pair;
  pi.s0 = p.s_base + pi.sl0;
  pi.thr0 = row_threshold(p, pi.s0);
  pi.thr1 = (pi.sl0 + 1 < p.rows) ? row_threshold(p, pi.s0 + 1) : 0;
  pi.T = pair_tiles(p, pi.sl0);
  pi.t_hi = min(pi.T, (max(pi.thr0, pi.thr1) + kTileT - 1) / kTileT);
  return pi;
}

__global__ void __launch_bounds__(kBThreads, 1)
    csa_backward_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_p, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const BSm sm{base};
  const int warp = threadIdx.x / 32;
  const uint32_t lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(sm.q_full(), 1);
    mbar_init(sm.q_empty(), 1);
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(sm.k_full(i), 1);
      mbar_init(sm.k_empty(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sm.acc_full(i), 1);
      mbar_init(sm.acc_empty(i), kBEpiWarps);
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
  // pairs in reverse order (the longest rows, most tiles, first), strided over the CTAs

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t q_pol = l2_policy_evict_first(), k_pol = l2_policy_evict_last();
      uint32_t qcount = 0, kcount = 0;
      for (int it = blockIdx.x; it < p.n_items; it += gridDim.x) {
        const PairInfo pi = pair_info(p, p.n_items - 1 - it);
        if (pi.t_hi == 0) continue;
        if (!mbar_wait(sm.q_empty(), (qcount & 1u) ^ 1u, ctl)) break;
        mbar_arrive_expect_tx(sm.q_full(), kBQBytes);
#pragma unroll
        for (int c = 0; c < kBNKC; ++c)
          tma_load_4d_hint(sm.q() + c * kBQChunk, &tmap_q, sm.q_full(), c * 64, 0, pi.s0, p.b, q_pol);
        ++qcount;
        bool ok = true;
        for (int tile = 0; tile < pi.t_hi; ++tile, ++kcount) {
          const int st = kcount % kBStages;
          if (!(ok = mbar_wait(sm.k_empty(st), ((kcount / kBStages) & 1u) ^ 1u, ctl))) break;
          mbar_arrive_expect_tx(sm.k_full(st), kBKBytes);
#pragma unroll
          for (int c = 0; c < kBNKC; ++c)
            tma_load_3d_hint(sm.k(st) + c * kBKChunk, &tmap_k, sm.k_full(st), c * 64, tile * kTileT, p.b, k_pol);
        }
        if (!ok) break;
      }
      // no copy may still be landing in shared memory when the CTA exits
      volatile uint32_t dummy = 0;
      const WaitCtl drain_ctl{&dummy, ctl.limit_ns};
      for (uint32_t i = 0; i < (uint32_t)kBStages && i < kcount; ++i) {
        const uint32_t last = kcount - 1 - i;
        mbar_wait(sm.k_full(last % kBStages), (last / kBStages) & 1u, drain_ctl);
      }
      if (qcount > 0) mbar_wait(sm.q_full(), (qcount - 1) & 1u, drain_ctl);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t qcount = 0, kcount = 0, acount = 0;
      const uint32_t q_addr = smem_u32(sm.q());
      for (int it = blockIdx.x; it < p.n_items; it += gridDim.x) {
        const PairInfo pi = pair_info(p, p.n_items - 1 - it);
        if (pi.t_hi == 0) continue;
        const bool q_ok = mbar_wait(sm.q_full(), qcount & 1u, ctl);
        tc_fence_after();
        bool ok = q_ok;
        for (int tile = 0; tile < pi.t_hi; ++tile, ++kcount, ++acount) {
          const int st = kcount % kBStages, a = acount & 1;
          const bool k_ok = ok && mbar_wait(sm.k_full(st), (kcount / kBStages) & 1u, ctl);
          const bool a_ok = k_ok && mbar_wait(sm.acc_empty(a), ((acount >> 1) & 1u) ^ 1u, ctl);
          tc_fence_after();
          ok = q_ok && k_ok && a_ok;
          if (ok) {
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
          if (!ok) break;
        }
        umma_commit(sm.q_empty());  // the q block may be replaced once these products are done
        ++qcount;
        if (!ok) break;
      }
    }
  } else if (warp < kBGatherWarp) {
    // epilogue: thread = TMEM lane m = 32*quarter + lane = (row j, head h);
    // warp half hf takes entries hf*64 .. hf*64+63 of every tile
    const int e = warp - 2;
    const int hf = e >> 2;
    const int quarter = warp & 3;
    const int m = quarter * 32 + (int)lane;
    const int j = m >> 6, h = m & 63;  // row of the pair (warp-uniform), head
    const int h0 = 32 * (quarter & 1);  // first head of this warp
    const bool segs = p.q_seg != nullptr;
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
    float* gb = sm.g(e);
    const uint64_t p_pol = l2_policy_evict_last();
    uint32_t acount = 0, scount = 0, icount = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < p.n_items; it += gridDim.x, ++icount) {
      const PairInfo pi = pair_info(p, p.n_items - 1 - it);
      const int s = pi.s0 + j;
      const bool row_ok = (pi.sl0 + j < p.rows) && s < p.S;
      const int thr = j ? pi.thr1 : pi.thr0;
      const int seg = (segs && row_ok) ? p.q_seg[(size_t)p.b * p.S + s] : 0;
      float wc = 0.f;
      if (row_ok) {
        const size_t off = ((size_t)p.b * p.S + s) * kBH + h;
        wc = (p.w_f32 ? reinterpret_cast<const float*>(p.w)[off]
                      : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.w)[off])) *
             p.scale;
      }
      // dw / scale in four independent packed partial sums (eight floats)
      float2 dwa[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      const float2 wc2 = make_float2(wc, wc);
      // masked cotangents of this warp's row and half for one tile (two per
      // lane); the next tile's are loaded while the current tile is processed
      auto load_g = [&](int tile) -> float2 {
        const int t0 = tile * kTileT + hf * 64 + 2 * (int)lane;
        float gv[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int t = t0 + u;
          bool vis = row_ok && t < thr;
          if (vis && segs) vis = p.kv_seg[(size_t)p.b * p.W + t] == seg;
          gv[u] = vis ? p.g[((size_t)p.b * p.S + s) * p.W + t] : 0.f;
        }
        return make_float2(gv[0], gv[1]);
      };
      float2 g_next = (pi.T > 0) ? load_g(0) : make_float2(0.f, 0.f);
      for (int tile = 0; tile < pi.T; ++tile, ++scount) {
        *reinterpret_cast<float2*>(gb + 2 * lane) = g_next;
        if (tile + 1 < pi.T) g_next = load_g(tile + 1);
        // this warp's staging buffer of two stores ago has been read
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        uint8_t* stg = sm.pstage(e, (int)(scount & 1u)) + lane * 128u;
        const bool computed = tile < pi.t_hi;
        const int a = acount & 1;
        if (computed && ok) {
          ok = mbar_wait(sm.acc_full(a), (acount >> 1) & 1u, ctl);
          tc_fence_after();
        }
        const bool live = computed && ok;
        float va[32], vb[32];
        const uint32_t col0 = (uint32_t)(a * kTileT + hf * 64);
        if (live) {
          tmem_ld32_start(t_lane + col0, va);
          tmem_wait32(va);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {  // 32 entries per chunk
          float(&cur)[32] = (c & 1) ? vb : va;
          float(&nxt)[32] = (c & 1) ? va : vb;
          uint32_t pk[16];
          if (live) {
            if (c == 0) tmem_ld32_start(t_lane + col0 + 32u, nxt);
            // scale > 0: [scale*x > 0] = [x > 0].  gm = g * [x > 0] gives both
            // P = gm * w * scale and the dw term gm * x = g * ReLU(x) (the
            // scale of dw is applied once per pair)
            const float4* g4 = reinterpret_cast<const float4*>(gb + c * 32);
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
              const float4 gq = g4[i4];
#pragma unroll
              for (int i2 = 0; i2 < 2; ++i2) {
                const int i = 2 * i4 + i2;
                const float2 x = make_float2(cur[2 * i], cur[2 * i + 1]);
                const float2 gg = i2 ? make_float2(gq.z, gq.w) : make_float2(gq.x, gq.y);
                const float2 gm = fmul2(gg, make_float2(step_pos(x.x), step_pos(x.y)));
                dwa[i & 3] = ffma2(gm, x, dwa[i & 3]);
                const float2 pv = fmul2(gm, wc2);
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(pv.x, pv.y);
                pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
              }
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = 0u;  // tile without products: P = 0
          }
          // 32 entries = 64 bytes: 16-byte chunks 4c .. 4c+3 of the row
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const uint32_t chunk = (uint32_t)(4 * c + q4);
            const uint32_t pos = chunk ^ (lane & 7u);  // 128-byte swizzle (row = lane)
            *reinterpret_cast<uint4*>(stg + pos * 16u) =
                make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
          }
          if (live && c == 0) tmem_wait32(nxt);
        }
        if (computed) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(sm.acc_empty(a));
          ++acount;
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0 && pi.sl0 + j < p.rows) {
          // evict_last: the dq and dk GEMMs that follow read P back, and the
          // part of the chunk that stays in L2 is not read from DRAM again
          tma_store_3d_hint(&tmap_p, sm.pstage(e, (int)(scount & 1u)), tile * kTileT + hf * 64, h0, pi.sl0 + j,
                            p_pol);
          bulk_commit_group();
        }
        __syncwarp();
      }
      // dw: the second half's partial sums join the first half's (buffers
      // alternate by pair, so one barrier per pair suffices)
      const float dw_acc =
          (((dwa[0].x + dwa[0].y) + (dwa[1].x + dwa[1].y)) + ((dwa[2].x + dwa[2].y) + (dwa[3].x + dwa[3].y))) *
          p.scale;
      float* dwp = sm.dwp((int)(icount & 1u));
      if (hf == 1) dwp[m] = dw_acc;
      named_bar_sync(kBEpiBar, 32 * kBEpiWarps);
      if (hf == 0 && row_ok) p.dw[((size_t)p.b * p.S + s) * kBH + h] = dw_acc + dwp[m];
    }
    if (lane == 0) bulk_wait_group_all();
  } else if (p.qc != nullptr) {
    // head-major q: the chunk's q rows in P's (row, head) order for the dk
    // GEMMs, as plain 16-byte copies spread over the CTAs while the other
    // warps form P (eight loads in flight per lane)
    const uint4* src = static_cast<const uint4*>(p.q_gather);
    uint4* dst = static_cast<uint4*>(p.qc);
    const long long n = (long long)p.rows * kBH * 16;  // 16 x 16 bytes per row of 128 bf16
    const long long stride = (long long)gridDim.x * 32;
    constexpr int U = 8;
    for (long long i0 = (long long)blockIdx.x * 32 + lane; i0 < n; i0 += stride * U) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const long long i = i0 + u * stride;
        if (i < n) {
          const long long rh = i >> 4;
          const int r = (int)(rh / kBH), hh = (int)(rh % kBH);
          v[u] = src[(((size_t)p.b * kBH + hh) * p.S + p.s_base + r) * 16 + (i & 15)];
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const long long i = i0 + u * stride;
        if (i < n) dst[i] = v[u];
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kBTmemCols);
}

// One cuBLAS handle per device, created on first use.  Setting its stream
// and enqueueing the GEMMs happen under the device's mutex, so calls from
// several host threads on one device do not race on the handle's stream.
struct BlasSlot {
  cublasHandle_t handle = nullptr;
  std::mutex lock;
};
BlasSlot* blas_slot() {
  static BlasSlot slots[64];
  static std::once_flag flags[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::call_once(flags[dev], [dev] {
    cublasHandle_t h = nullptr;
    if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) h = nullptr;
    slots[dev].handle = h;
  });
  return slots[dev].handle ? &slots[dev] : nullptr;
}

}  // namespace

size_t backward_kernel_smem() { return kBSmem; }

cudaError_t launch_backward_kernel(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tp,
                                   const BwdParams& bp, cudaStream_t stream) {
  cudaError_t e = smem_limit_once<csa_backward_kernel>((int)kBSmem);
  if (e != cudaSuccess) return e;
  if (bp.n_items <= 0) return cudaSuccess;
  const int grid = bp.grid < bp.n_items ? bp.grid : bp.n_items;
  csa_backward_kernel<<<grid, kBThreads, kBSmem, stream>>>(tq, tk, tp, bp);
  return cudaGetLastError();
}

// dq rows of the chunk (one GEMM per head, batched) and the chunk's share of
// dk (one GEMM over all heads and rows), fp32 accumulation of bf16 operands.
// Row-major operands are passed to the column-major library transposed.
bool backward_gemms(const BwdGemms& gm, cudaStream_t stream) {
  BlasSlot* slot = blas_slot();
  if (slot == nullptr) return false;
  std::lock_guard<std::mutex> guard(slot->lock);
  cublasHandle_t h = slot->handle;
  if (cublasSetStream(h, stream) != CUBLAS_STATUS_SUCCESS) return false;
  const float one = 1.f, zero = 0.f;
  // dq[h][rows x D] = P[:, h][rows x W_eff] . k[W_eff x D]   (column-major: D x rows = k^T . P^T);
  // the rows of head h are H * w_pad apart in P, the heads w_pad apart
  if (cublasGemmStridedBatchedEx(h, CUBLAS_OP_N, CUBLAS_OP_N, gm.D, gm.rows, gm.w_eff, &one, gm.k, CUDA_R_16BF,
                                 gm.D, 0, gm.p, CUDA_R_16BF, gm.H * gm.w_pad, (long long)gm.w_pad, &zero, gm.dq,
                                 CUDA_R_32F, gm.dq_row_stride, gm.dq_head_stride, gm.H, CUBLAS_COMPUTE_32F,
                                 CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
    return false;
  // dk[W_eff x D] += P_all^T[W_eff x (rows H)] . Q[(rows H) x D]   (column-major: D x W_eff = Q^T . P_all),
  // P_all and Q with their rows in the same (row, head) order
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
