// csa_topk.cu -- standalone per-row selection over precomputed scores, and
// the bounded-wait self-test kernel.
#include <cooperative_groups.h>

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

// ----------------------------------------------------------------------------
// Long rows (W > 16384): one row per cluster of kCl CTAs.  CTA c of a cluster
// stages entries [c*seg, (c+1)*seg) of the row and every step that needs the
// whole row is a merge over the cluster's shared memory (distributed shared
// memory reads after a cluster barrier):
//   row statistics (visible count, value range)        -> identical in all CTAs
//   binned path: bin histogram -> threshold bin b*, then the members of b*
//     of every CTA -> exact rank of the local members, then each CTA's kept
//     count -> its offset in the output row;
//   radix path (rows that keep all visible entries, equal values, ranges that
//     overflow, b* over capacity): per-digit histograms -> the K-th largest
//     key T and the number of keys equal to T kept; per-CTA counts above / at
//     T -> offsets and each CTA's share of the ties (lowest index first).
// Every decision is taken on cluster-wide values, so all CTAs follow the same
// path through the same sequence of cluster barriers.
namespace cg = cooperative_groups;

constexpr int kCl = 4;                           // CTAs per row
constexpr int kClSegMax = kTopkMaxRow / kCl;     // entries staged per CTA (multiple of 128)
constexpr int kClNT = 512;                       // threads per CTA
constexpr int kClNB = 2048, kClCAP = 1024;

struct ClusterScratch {
  uint32_t hist[kClNB];  // local counts: bins (binned path) or two 256-digit buffers (radix path)
  uint32_t ghist[kClNB];  // cluster-wide counts
  uint32_t cand[kClCAP], cand_t[kClCAP];    // local members of b*: key, entry number in the row
  uint32_t acand[kClCAP], acand_t[kClCAP];  // members of every CTA
  uint32_t keep[4 * (kClSegMax / 128)];     // word 4*c+u, bit l: entry c*128 + 4*l + u of the segment
  uint32_t seg_gt[32], seg_sel[32], warp_sum[32], warp_a[32], warp_b[32];
  uint32_t bcast[8];
  RowStats gst;  // the row's statistics over the cluster
  // read by the other CTAs of the cluster
  uint32_t super[kClNB / 32];  // bin totals of 32 consecutive bins
  RowStats st;
  uint32_t ncand, kept, n_gt, n_eq;
};
constexpr uint32_t kClHeader = (sizeof(ClusterScratch) + 127u) & ~127u;

__global__ void __cluster_dims__(kCl, 1, 1) __launch_bounds__(kClNT)
    csa_topk_cluster_kernel(const float* __restrict__ scores, int32_t* __restrict__ idx, int W, int K) {
  constexpr int NT = kClNT, NW = NT / 32, NB = kClNB, CAP = kClCAP, PER = NB / NT;
  cg::cluster_group cluster = cg::this_cluster();
  const uint32_t cr = cluster.block_rank();
  const long long r = blockIdx.x / kCl;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ClusterScratch* cs = reinterpret_cast<ClusterScratch*>(smem_raw);
  float* row = reinterpret_cast<float*>(smem_raw + kClHeader);
  const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
  const Team<NT> team{1u, tid};
  ClusterScratch* peer[kCl];
#pragma unroll
  for (int c = 0; c < kCl; ++c) peer[c] = cluster.map_shared_rank(cs, c);

  const int seg = (((W + kCl - 1) / kCl) + 127) & ~127;
  const int e_lo = min(W, (int)cr * seg), e_hi = min(W, e_lo + seg);
  const int n = e_hi - e_lo, npad = (n + 127) & ~127, chunks = npad >> 7;
  int32_t* out = idx + (size_t)r * K;

  // 1. stage the segment, local statistics
  if (tid == 0) {
    cs->st.nvis = 0u;
    cs->st.min_key = 0xFFFFFFFFu;
    cs->st.max_key = 0u;
  }
  team.sync();
  {
    const float* src = scores + (size_t)r * W + e_lo;
    uint32_t cnt = 0, kmin = 0xFFFFFFFFu, kmax = 0u;
    auto note = [&](float x) {
      const uint32_t k = score_key(x);
      if (k != 0u) {
        ++cnt;
        kmin = min(kmin, k);
        kmax = max(kmax, k);
      }
    };
    if ((W % 4) == 0 && (reinterpret_cast<uintptr_t>(scores) % 16) == 0) {  // e_lo, n multiples of 4
      const float4* s4 = reinterpret_cast<const float4*>(src);
      float4* d4 = reinterpret_cast<float4*>(row);
      const int n4 = n / 4;
#pragma unroll 1
      for (int i0 = (int)tid; i0 < n4; i0 += 4 * NT) {
        float4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          v[q] = (i0 + q * NT < n4) ? __ldcs(s4 + i0 + q * NT) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (i0 + q * NT < n4) d4[i0 + q * NT] = v[q];
          note(v[q].x);
          note(v[q].y);
          note(v[q].z);
          note(v[q].w);
        }
      }
    } else {
      for (int i = (int)tid; i < n; i += NT) {
        const float v = __ldcs(src + i);
        row[i] = v;
        note(v);
      }
    }
    for (int i = n + (int)tid; i < npad; i += NT) row[i] = -INFINITY;
    cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
    kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
    kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
    if (lane == 0 && cnt > 0u) {
      atomicAdd(&cs->st.nvis, cnt);
      atomicMin(&cs->st.min_key, kmin);
      atomicMax(&cs->st.max_key, kmax);
    }
  }
  cluster.sync();
  // 2. row statistics over the cluster (lane c of warp 0 reads CTA c)
  if (warp == 0) {
    RowStats s{0u, 0xFFFFFFFFu, 0u};
    if (lane < (uint32_t)kCl) s = cluster.map_shared_rank(cs, lane)->st;
    const uint32_t nv = __reduce_add_sync(0xFFFFFFFFu, s.nvis);
    const uint32_t mn = __reduce_min_sync(0xFFFFFFFFu, s.min_key);
    const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, s.max_key);
    if (lane == 0) cs->gst = RowStats{nv, mn, mx};
  }
  team.sync();
  const RowStats g = cs->gst;
  const uint32_t UK = (uint32_t)K;
  const float lo = key_score(g.min_key), hi = key_score(g.max_key);
  const float span = hi - lo;
  const float scale = (float)(NB - 1) / span;
  const float bias = -lo * scale;
  bool binned = g.nvis > UK && hi > lo && span < INFINITY && scale < INFINITY && fabsf(bias) < 2097152.0f;
  const uint32_t lt_mask = (1u << lane) - 1u;
  const uint32_t row_s = smem_u32(row);
  if (binned) {
    const BinMap bin_of(lo, span, NB);
    const uint32_t hist_s = smem_u32(cs->hist);
#pragma unroll
    for (int j = 0; j < PER; ++j) cs->hist[tid * PER + j] = 0u;
    if (tid < 32) {
      cs->seg_gt[tid] = 0u;
      cs->seg_sel[tid] = 0u;
    }
    if (tid == 0) cs->ncand = 0u;
    team.sync();
    // 3. local histogram
    const int n4 = npad >> 2;
#pragma unroll 1
    for (int i0 = (int)tid; i0 < n4; i0 += 4 * NT) {
      float4 a[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        a[q] = (i0 + q * NT < n4) ? lds_f4(row_s + 16u * (uint32_t)(i0 + q * NT))
                                  : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float xs[4] = {a[q].x, a[q].y, a[q].z, a[q].w};
#pragma unroll
        for (int u = 0; u < 4; ++u) red_add_shared_if(hist_s + 4u * bin_of(xs[u]), 1u, xs[u] > -INFINITY);
      }
    }
    team.sync();
    for (uint32_t sb = tid; sb < (uint32_t)(NB / 32); sb += NT) {  // super-bin totals
      uint32_t v = 0;
#pragma unroll 8
      for (int j = 0; j < 32; ++j) v += cs->hist[sb * 32 + j];
      cs->super[sb] = v;
    }
    cluster.sync();
    // 4. b* over the cluster: the super-bin holding the K-th largest entry from
    //    the CTAs' super-bin totals, then that super-bin's 32 bins (warp 0)
    if (warp == 0) {
      constexpr int NS = NB / 32, SPL = NS / 32;  // super-bins, super-bins per lane
      uint32_t sv[SPL], sum = 0;
#pragma unroll
      for (int j = 0; j < SPL; ++j) {
        uint32_t v = 0;
#pragma unroll
        for (int c = 0; c < kCl; ++c) v += peer[c]->super[lane * SPL + j];
        sv[j] = v;
        sum += v;
      }
      uint32_t incl = sum;  // entries in the super-bins of lanes >= this one
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t x = __shfl_down_sync(0xFFFFFFFFu, incl, off);
        if (lane + off < 32) incl += x;
      }
      const uint32_t excl = incl - sum;
      uint32_t sb_star = 0, sb_above = 0;
      bool here = excl < UK && UK <= incl;
      if (here) {
        uint32_t acc = excl;
        bool found = false;
#pragma unroll
        for (int j = SPL - 1; j >= 0; --j) {
          if (!found && acc + sv[j] >= UK) {
            found = true;
            sb_star = lane * SPL + (uint32_t)j;
            sb_above = acc;
          }
          if (!found) acc += sv[j];
        }
      }
      const uint32_t src = __ffs(__ballot_sync(0xFFFFFFFFu, here)) - 1u;
      sb_star = __shfl_sync(0xFFFFFFFFu, sb_star, src);
      sb_above = __shfl_sync(0xFFFFFFFFu, sb_above, src);
      // lane l: bin sb_star*32 + l over the cluster; suffix sums over lanes
      uint32_t bv = 0;
#pragma unroll
      for (int c = 0; c < kCl; ++c) bv += peer[c]->hist[sb_star * 32 + lane];
      uint32_t bincl = bv;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t x = __shfl_down_sync(0xFFFFFFFFu, bincl, off);
        if (lane + off < 32) bincl += x;
      }
      const uint32_t bexcl = sb_above + bincl - bv;
      if (bexcl < UK && UK <= sb_above + bincl) {
        cs->bcast[0] = sb_star * 32 + lane;
        cs->bcast[1] = bexcl;
        cs->bcast[2] = bv;
      }
    }
    team.sync();
    const uint32_t bstar = cs->bcast[0], above = cs->bcast[1], m = cs->bcast[2];
    binned = m <= (uint32_t)CAP;  // identical in every CTA
    if (!binned) cluster.sync();  // the radix path reuses `hist`, which the other CTAs may still be reading
    if (binned) {
      const uint32_t need = UK - above;
      const uint32_t keep_s = smem_u32(cs->keep), cand_s = smem_u32(cs->cand), cand_t_s = smem_u32(cs->cand_t);
      const uint32_t ncand_s = smem_u32(&cs->ncand), seg_sel_s = smem_u32(cs->seg_sel);
      // 5. local bitmap of sure entries, members of b*
      const int seg_chunks = (chunks + NW - 1) / NW;
      const int c_lo = min(chunks, (int)warp * seg_chunks);
      const int c_hi = min(chunks, c_lo + seg_chunks);
      uint32_t gt = 0;
#pragma unroll 1
      for (int c0 = c_lo; c0 < c_hi; ++c0) {
        const float4 v = lds_f4(row_s + 16u * (uint32_t)(c0 * 32 + (int)lane));
        const float xs[4] = {v.x, v.y, v.z, v.w};
        uint32_t sure[4], memb[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const bool vis = xs[u] > -INFINITY;
          const uint32_t bb = bin_of(xs[u]);
          sure[u] = __ballot_sync(0xFFFFFFFFu, vis && bb > bstar);
          memb[u] = __ballot_sync(0xFFFFFFFFu, vis && bb == bstar);
        }
        sts_u4_if(keep_s + 16u * (uint32_t)c0, make_uint4(sure[0], sure[1], sure[2], sure[3]), lane == 0);
        gt += (__popc(sure[0]) + __popc(sure[1])) + (__popc(sure[2]) + __popc(sure[3]));
        const uint32_t p1 = __popc(memb[0]), p2 = p1 + __popc(memb[1]), p3 = p2 + __popc(memb[2]);
        const uint32_t nm = p3 + __popc(memb[3]);
        if (nm != 0u) {
          uint32_t slot = 0;
          if (lane == 0) slot = atom_add_shared(ncand_s, nm);
          slot = __shfl_sync(0xFFFFFFFFu, slot, 0);
          const uint32_t pre[4] = {0u, p1, p2, p3};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t o = slot + pre[u] + __popc(memb[u] & lt_mask);
            sts_u32x2_if(cand_s + 4u * o, score_key(xs[u]), cand_t_s + 4u * o,
                         (uint32_t)(e_lo + c0 * 128 + 4 * (int)lane + u),  // entry number in the row
                         ((memb[u] >> lane) & 1u) && o < (uint32_t)CAP);
          }
        }
      }
      if (lane == 0) cs->seg_gt[warp] = gt;
      cluster.sync();
      // 6. members of every CTA, exact rank of the local ones
      {
        uint32_t ncs[kCl], pre[kCl + 1];
#pragma unroll
        for (int c = 0; c < kCl; ++c) ncs[c] = min(peer[c]->ncand, (uint32_t)CAP);
        pre[0] = 0u;
#pragma unroll
        for (int c = 0; c < kCl; ++c) pre[c + 1] = pre[c] + ncs[c];
        const uint32_t off = pre[kCl];
        // one round of remote reads: member j comes from the CTA whose range holds it
        for (uint32_t j = tid; j < min(off, (uint32_t)CAP); j += NT) {
          int c = 0;
          uint32_t base = 0u;
#pragma unroll
          for (int q = 1; q < kCl; ++q) {
            if (j >= pre[q]) {
              c = q;
              base = pre[q];
            }
          }
          const ClusterScratch* pc = cluster.map_shared_rank(cs, c);
          cs->acand[j] = pc->cand[j - base];
          cs->acand_t[j] = pc->cand_t[j - base];
        }
        team.sync();
        const uint32_t mall = min(off, (uint32_t)CAP), mine = min(cs->ncand, (uint32_t)CAP);
#pragma unroll 1
        for (uint32_t i = tid; i < mine; i += NT) {
          const uint32_t ki = cs->cand[i], ti = cs->cand_t[i];
          uint32_t rank = 0;
#pragma unroll 4
          for (uint32_t j = 0; j < mall; ++j) {
            const uint32_t kj = cs->acand[j], tj = cs->acand_t[j];
            rank += (kj > ki) || (kj == ki && tj < ti);
          }
          if (rank < need) {
            const uint32_t lt = ti - (uint32_t)e_lo;
            const uint32_t c = lt >> 7, l = (lt >> 2) & 31u, u = lt & 3u;
            red_or_shared(keep_s + 4u * (4u * c + u), 1u << l);
            red_add_shared_if(seg_sel_s + 4u * (c / (uint32_t)max(seg_chunks, 1)), 1u, true);
          }
        }
      }
      team.sync();
      // 7. offsets: kept entries of the earlier CTAs
      uint32_t mine_kept = 0, wbase = 0;
      for (int w = 0; w < NW; ++w) {
        const uint32_t cnt = cs->seg_gt[w] + cs->seg_sel[w];
        wbase += (w < (int)warp) ? cnt : 0u;
        mine_kept += cnt;
      }
      if (tid == 0) cs->kept = mine_kept;
      cluster.sync();
      uint32_t before = 0, total = 0;
#pragma unroll
      for (int c = 0; c < kCl; ++c) {
        const uint32_t kc = peer[c]->kept;
        before += (c < (int)cr) ? kc : 0u;
        total += kc;
      }
      // 8. ordered write of the local kept entries
      uint32_t base = before + wbase;
#pragma unroll 4
      for (int c = c_lo; c < c_hi; ++c) {
        const uint4 mw = lds_u4(keep_s + 16u * (uint32_t)c);
        const uint32_t b0 = (mw.x >> lane) & 1u, b1 = (mw.y >> lane) & 1u, b2 = (mw.z >> lane) & 1u;
        const uint32_t b3 = (mw.w >> lane) & 1u;
        const uint32_t p0 = base + __popc(mw.x & lt_mask) + __popc(mw.y & lt_mask) + __popc(mw.z & lt_mask) +
                            __popc(mw.w & lt_mask);
        const uint32_t q1 = p0 + b0, q2 = q1 + b1, q3 = q2 + b2;
        const int tb = e_lo + c * 128 + 4 * (int)lane;
        if (b0 && p0 < UK) out[p0] = tb;
        if (b1 && q1 < UK) out[q1] = tb + 1;
        if (b2 && q2 < UK) out[q2] = tb + 2;
        if (b3 && q3 < UK) out[q3] = tb + 3;
        base += __popc(mw.x) + __popc(mw.y) + __popc(mw.z) + __popc(mw.w);
      }
      if (cr == kCl - 1)
        for (uint32_t i = min(total, UK) + tid; i < UK; i += NT) out[i] = -1;
    }
  }
  if (!binned) {
    // radix search for the K-th largest key over the cluster (two digit
    // buffers alternate, so a buffer is only cleared after every CTA has read it)
    uint32_t prefix = 0, rem = UK, T = 0u, take_eq = 0u;
    bool done = false;
    for (int pass = 0; pass < 4 && !done; ++pass) {
      const int shift = 24 - 8 * pass;
      uint32_t* h = cs->hist + (pass & 1) * 256;
      for (uint32_t i = tid; i < 256; i += NT) h[i] = 0u;
      team.sync();
      const uint32_t hi_mask = (pass == 0) ? 0u : (0xFFFFFFFFu << (shift + 8));
      for (int t = (int)tid; t < n; t += NT) {
        const uint32_t key = score_key(row[t]);
        if (key != 0u && (key & hi_mask) == prefix) atomicAdd(&h[(key >> shift) & 255u], 1u);
      }
      cluster.sync();
      if (warp == 0) {
        uint32_t c8[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t v = 0;
#pragma unroll
          for (int c = 0; c < kCl; ++c) v += (peer[c]->hist + (pass & 1) * 256)[lane * 8 + j];
          c8[j] = v;
          sum += v;
        }
        uint32_t incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, incl, off);
          if (lane + off < 32) incl += v;
        }
        const uint32_t totalk = __shfl_sync(0xFFFFFFFFu, incl, 0);
        const uint32_t rr = (pass == 0 && totalk <= UK) ? 0u : rem;
        const uint32_t excl = incl - sum;
        if (lane == 0) {
          cs->bcast[0] = 0xFFFFFFFFu;
          cs->bcast[1] = 0u;
          cs->bcast[2] = 0u;
        }
        __syncwarp();
        if (rr > 0u && excl < rr && rr <= incl) {
          uint32_t acc = excl, d = 0, cd = 0;
          bool found = false;
#pragma unroll
          for (int j = 7; j >= 0; --j) {
            if (!found && acc + c8[j] >= rr) {
              found = true;
              d = (uint32_t)j;
              cd = c8[j];
            }
            if (!found) acc += c8[j];
          }
          cs->bcast[0] = lane * 8 + d;
          cs->bcast[1] = acc;
          cs->bcast[2] = cd;
        }
      }
      team.sync();
      const uint32_t digit = cs->bcast[0], abv = cs->bcast[1], inbin = cs->bcast[2];
      team.sync();  // bcast is rewritten by the next pass
      if (digit == 0xFFFFFFFFu) {  // at most K visible: keep every visible entry
        T = 0u;
        take_eq = 0u;
        done = true;
      } else {
        prefix |= digit << shift;
        rem -= abv;
        if (inbin == rem) {  // the whole bin is kept
          T = (prefix == 0u) ? 0u : prefix - 1u;
          take_eq = 0u;
          done = true;
        } else if (pass == 3) {
          T = prefix;
          take_eq = rem;
          done = true;
        }
      }
    }
    // local counts above / at T, then offsets and this CTA's share of the ties
    auto pred = [&](int t) -> int {
      const uint32_t key = score_key(row[t]);
      if (key == 0u) return 0;
      if (key > T) return 1;
      return (key == T) ? 2 : 0;
    };
    const int sg = ((n + NW - 1) / NW + 31) & ~31;
    const int s_lo = min(n, (int)warp * sg), s_hi = min(n, s_lo + sg);
    uint32_t ngt = 0, neq = 0;
    for (int t = s_lo + (int)lane; t < s_hi; t += 32) {
      const int pv = pred(t);
      ngt += (pv == 1);
      neq += (pv == 2);
    }
    ngt = __reduce_add_sync(0xFFFFFFFFu, ngt);
    neq = __reduce_add_sync(0xFFFFFFFFu, neq);
    if (lane == 0) {
      cs->warp_a[warp] = ngt;
      cs->warp_b[warp] = neq;
    }
    team.sync();
    if (tid == 0) {
      uint32_t a = 0, b = 0;
      for (int w = 0; w < NW; ++w) {
        a += cs->warp_a[w];
        b += cs->warp_b[w];
      }
      cs->n_gt = a;
      cs->n_eq = b;
    }
    cluster.sync();
    // ties are taken lowest index first: in CTA order, then warp order
    uint32_t eqb = 0, eqb_cta = 0, sel_before = 0, total = 0;
#pragma unroll
    for (int c = 0; c < kCl; ++c) {
      const uint32_t g_c = peer[c]->n_gt, e_c = peer[c]->n_eq;
      const uint32_t tk = (take_eq > eqb) ? min(e_c, take_eq - eqb) : 0u;
      if (c < (int)cr) {
        sel_before += g_c + tk;
        eqb_cta += e_c;
      }
      total += g_c + tk;
      eqb += e_c;
    }
    uint32_t w_eq_before = eqb_cta, w_sel_before = sel_before;
    for (int w = 0; w < (int)warp; ++w) {
      const uint32_t gw = cs->warp_a[w], ew = cs->warp_b[w];
      const uint32_t tk = (take_eq > w_eq_before) ? min(ew, take_eq - w_eq_before) : 0u;
      w_sel_before += gw + tk;
      w_eq_before += ew;
    }
    uint32_t pos = w_sel_before, eq_seen = w_eq_before;
    for (int t0 = s_lo; t0 < s_hi; t0 += 32) {
      const int t = t0 + (int)lane;
      const int pv = (t < s_hi) ? pred(t) : 0;
      const uint32_t eqm = __ballot_sync(0xFFFFFFFFu, pv == 2);
      const uint32_t my_eq_rank = eq_seen + __popc(eqm & lt_mask);
      const bool keep = (pv == 1) || (pv == 2 && my_eq_rank < take_eq);
      const uint32_t km = __ballot_sync(0xFFFFFFFFu, keep);
      if (keep) {
        const uint32_t o = pos + __popc(km & lt_mask);
        if (o < UK) out[o] = e_lo + t;
      }
      pos += __popc(km);
      eq_seen += __popc(eqm);
    }
    if (cr == kCl - 1)
      for (uint32_t i = min(total, UK) + tid; i < UK; i += NT) out[i] = -1;
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
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
  cudaError_t e = smem_limit_once<csa_topk_kernel<NT>>(227 * 1024);
  if (e != cudaSuccess) return e;
  const long long grid = rows < 1048576 ? rows : 1048576;
  csa_topk_kernel<NT><<<(unsigned)grid, NT, smem, stream>>>(scores, idx, rows, W, K);
  return cudaGetLastError();
}

cudaError_t launch_topk_cluster(const float* scores, int32_t* idx, long long rows, int W, int K,
                                cudaStream_t stream) {
  const int seg = (((W + kCl - 1) / kCl) + 127) & ~127;
  const size_t smem = kClHeader + (size_t)seg * sizeof(float);
  cudaError_t e = smem_limit_once<csa_topk_cluster_kernel>(227 * 1024);
  if (e != cudaSuccess) return e;
  // one cluster per row; rows beyond one launch's grid go to further launches
  const long long per_launch = 65536;
  for (long long r0 = 0; r0 < rows; r0 += per_launch) {
    const long long nr = (rows - r0) < per_launch ? (rows - r0) : per_launch;
    csa_topk_cluster_kernel<<<(unsigned)(nr * kCl), kClNT, smem, stream>>>(scores + (size_t)r0 * W, idx + (size_t)r0 * K,
                                                                           W, K);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
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
  if (W > 16384 && rows > 0) return launch_topk_cluster(scores, idx, rows, W, K, stream);
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
