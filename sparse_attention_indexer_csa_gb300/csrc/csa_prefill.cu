// csa_prefill.cu -- instantiations of the persistent indexer kernel and their
// launcher: R = 4 query rows per item (prefill score, fused score +
// selection, its long-row mode for rows of up to 16384 entries and its
// document mode for packed documents) and R = 1 with tile chunks
// (single-row decode scores).
#include "csa_internal.h"

namespace csa {

namespace {

// Segment pre-pass of the one-kernel fused path (and of the backward): the
// SegInfo of every item of four whole rows, so the persistent kernels'
// scheduler warps read a summary instead of scanning up to W ids per item.
//
// A block takes kScanRows consecutive query rows of one batch.  Their
// future-mask bounds lie in [lo, hi] with hi - lo < kScanRows (a row's bound
// exceeds the previous row's by at most one), and every entry below lo is
// below every row's bound.  One coalesced pass over the ids [0, hi) gives,
// for each of the block's first kScanIds distinct row ids, the count, first
// and last of its entries below lo and which entries of the window [lo, hi)
// carry it; a row with one of these ids reads its visible count and first /
// last visible entry from prefix tables of the window.  Rows with another id
// (more than kScanIds documents among the block's rows, or scattered ids)
// are scanned one by one by a warp.
constexpr int kScanRows = 128;
constexpr int kScanThreads = 256;
constexpr int kScanWarps = kScanThreads / 32;
constexpr int kScanIds = 4;
constexpr int kBig = 0x7FFFFFFF;

struct ScanShared {
  int rid[kScanRows], rthr[kScanRows];                            // row id and bound
  int row_n[kScanRows], row_first[kScanRows], row_last[kScanRows];  // row results
  int other[kScanRows];                                           // rows scanned one by one
  int ids[kScanIds];
  int n_ids, lo, hi, n_other;
  unsigned char win[kScanIds][kScanRows];  // entry lo + j carries ids[k]
  int wcnt[kScanIds][kScanRows + 1];       // window entries j' < j carrying ids[k]
  int wlast[kScanIds][kScanRows + 1];      // the last of them, or -1
  int part_cnt[kScanIds][kScanWarps], part_min[kScanIds][kScanWarps], part_max[kScanIds][kScanWarps];
  int c0[kScanIds], first[kScanIds], last0[kScanIds];  // below lo: count, last; first over [0, hi)
};

__global__ void __launch_bounds__(kScanThreads) csa_segscan_kernel(const KParams p, SegInfo* out) {
  __shared__ ScanShared sh;
  griddep_wait();
  const int tid = (int)threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nblk = (p.S + kScanRows - 1) / kScanRows;
  const int b = (int)blockIdx.x / nblk;
  const int s0 = ((int)blockIdx.x - b * nblk) * kScanRows;
  const long long qs0 = p.q_start ? (long long)p.q_start[b] : 0ll;
  const int32_t* kv = p.kv_seg + (size_t)b * p.W;

  // 1. the rows' ids and bounds (bound 0 past S); window flags cleared
  if (tid < kScanRows) {
    const int s = s0 + tid;
    int thr[1];
    row_bounds<1>(p, qs0, s, thr);
    sh.rid[tid] = s < p.S ? p.q_seg[(size_t)b * p.S + s] : 0;
    sh.rthr[tid] = thr[0];
  }
  for (int i = tid; i < kScanIds * kScanRows; i += kScanThreads) (&sh.win[0][0])[i] = 0;
  __syncthreads();

  // 2. warp 0: smallest and largest bound of the rows before S, and the
  //    first kScanIds distinct ids in row order
  if (warp == 0) {
    int lo = kBig, hi = 0;
    for (int r = lane; r < kScanRows && s0 + r < p.S; r += 32) {
      lo = min(lo, sh.rthr[r]);
      hi = max(hi, sh.rthr[r]);
    }
    lo = __reduce_min_sync(0xFFFFFFFFu, lo);
    hi = __reduce_max_sync(0xFFFFFFFFu, hi);
    int n = 0;
    for (int k = 0; k < kScanIds; ++k) {
      int cand = kBig;  // this lane's first row whose id is not yet listed
      for (int r = lane; r < kScanRows && s0 + r < p.S; r += 32) {
        const int id = sh.rid[r];
        bool seen = false;
        for (int j = 0; j < k; ++j) seen = seen || sh.ids[j] == id;
        if (!seen) {
          cand = r;
          break;
        }
      }
      cand = __reduce_min_sync(0xFFFFFFFFu, cand);
      if (cand == kBig) break;
      if (lane == 0) sh.ids[k] = sh.rid[cand];
      __syncwarp();
      n = k + 1;
    }
    if (lane == 0) {
      sh.lo = lo == kBig ? 0 : lo;
      sh.hi = hi;
      sh.n_ids = n;
      sh.n_other = 0;
    }
  }
  __syncthreads();
  const int n_ids = sh.n_ids, lo = sh.lo, hi = sh.hi;

  // 3. one pass over the ids [0, hi): per listed id its entries below lo
  //    (count, last), its first entry, and its entries in the window
  {
    int idv[kScanIds], cnt[kScanIds], mn[kScanIds], mx[kScanIds];
#pragma unroll
    for (int k = 0; k < kScanIds; ++k) {
      idv[k] = k < n_ids ? sh.ids[k] : 0;
      cnt[k] = 0;
      mn[k] = kBig;
      mx[k] = -1;
    }
#pragma unroll 4
    for (int t = tid; t < hi; t += kScanThreads) {
      const int v = kv[t];
#pragma unroll
      for (int k = 0; k < kScanIds; ++k) {
        if (k < n_ids && v == idv[k]) {
          mn[k] = min(mn[k], t);
          if (t < lo) {
            ++cnt[k];
            mx[k] = t;  // entries ascend within a thread: the last match wins
          } else if (t - lo < kScanRows) {
            sh.win[k][t - lo] = 1;
          }
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kScanIds; ++k) {
      const int c = (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)cnt[k]);
      const int a = __reduce_min_sync(0xFFFFFFFFu, mn[k]);
      const int z = __reduce_max_sync(0xFFFFFFFFu, mx[k]);
      if (lane == 0) {
        sh.part_cnt[k][warp] = c;
        sh.part_min[k][warp] = a;
        sh.part_max[k][warp] = z;
      }
    }
  }
  __syncthreads();
  if (tid < n_ids) {
    int c = 0, a = kBig, z = -1;
    for (int w = 0; w < kScanWarps; ++w) {
      c += sh.part_cnt[tid][w];
      a = min(a, sh.part_min[tid][w]);
      z = max(z, sh.part_max[tid][w]);
    }
    sh.c0[tid] = c;
    sh.first[tid] = a;
    sh.last0[tid] = z;
  }
  // 4. warp k: prefix tables of the window for id k (positions 0 .. 128)
  if (warp < n_ids) {
    const int k = warp;
    int base = 0, lastp = -1;
    for (int c = 0; c < kScanRows / 32; ++c) {
      const int j = c * 32 + lane;
      const bool m = j < hi - lo && sh.win[k][j];
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, m);
      const uint32_t below = bal & ((1u << lane) - 1u);
      sh.wcnt[k][j] = base + __popc(below);
      sh.wlast[k][j] = below ? c * 32 + 31 - __clz(below) : lastp;
      base += __popc(bal);
      if (bal) lastp = c * 32 + 31 - __clz(bal);
    }
    if (lane == 0) {
      sh.wcnt[k][kScanRows] = base;
      sh.wlast[k][kScanRows] = lastp;
    }
  }
  __syncthreads();

  // 5. rows with a listed id: count and first / last visible entry from
  //    the tables; the others are queued for a scan
  if (tid < kScanRows) {
    int n = 0, f = -1, l = -1;
    if (s0 + tid < p.S) {
      const int thr = sh.rthr[tid], id = sh.rid[tid];
      int k = -1;
      for (int j = 0; j < n_ids; ++j)
        if (sh.ids[j] == id) k = j;
      if (k >= 0) {
        const int j = thr - lo;  // 0 .. hi - lo
        n = sh.c0[k] + sh.wcnt[k][j];
        const int wl = sh.wlast[k][j];
        l = wl >= 0 ? lo + wl : sh.last0[k];
        f = sh.first[k] < thr ? sh.first[k] : -1;
      } else {
        sh.other[atomicAdd(&sh.n_other, 1)] = tid;
      }
    }
    sh.row_n[tid] = n;
    sh.row_first[tid] = f;
    sh.row_last[tid] = l;
  }
  __syncthreads();
  // 6. queued rows: one warp per row over the ids below its bound
  const int n_other = sh.n_other;
  for (int i = warp; i < n_other; i += kScanWarps) {
    const int r = sh.other[i], thr = sh.rthr[r], id = sh.rid[r];
    int c = 0, f = kBig, l = -1;
    for (int t = lane; t < thr; t += 32) {
      if (kv[t] == id) {
        ++c;
        f = min(f, t);
        l = t;
      }
    }
    c = (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)c);
    f = __reduce_min_sync(0xFFFFFFFFu, f);
    l = __reduce_max_sync(0xFFFFFFFFu, l);
    if (lane == 0) {
      sh.row_n[r] = c;
      sh.row_first[r] = c > 0 ? f : -1;
      sh.row_last[r] = l;
    }
  }
  __syncthreads();

  // 7. the items of four rows
  if (tid < kScanRows / 4) {
    const int rb = s0 / 4 + tid;
    if (rb < p.n_rb) {
      SegInfo si;
      int tmin = kBig, tmax = -1;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = 4 * tid + j, n = sh.row_n[r], f = sh.row_first[r], l = sh.row_last[r];
        si.nvis[j] = n;
        si.tfirst[j] = n > 0 ? f : 0;
        si.contig[j] = (n == 0) || (l - f + 1 == n);
        if (n > 0) {
          tmin = min(tmin, f);
          tmax = max(tmax, l);
        }
      }
      si.t_lo = tmax >= 0 ? tmin / kTileT : 0;
      si.t_hi = tmax >= 0 ? tmax / kTileT + 1 : 0;
      si.pad0 = si.pad1 = 0;
      out[(size_t)b * p.n_rb + rb] = si;
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
  (void)sms;
  const long long blocks = (long long)p.B * ((p.S + kScanRows - 1) / kScanRows);  // kScanRows rows each
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
  return launch_pdl(csa_segscan_kernel, dim3((unsigned)blocks), dim3(kScanThreads), 0, stream, p, out);
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
