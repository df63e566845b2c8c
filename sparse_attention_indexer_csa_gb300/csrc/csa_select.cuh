// csa_select.cuh -- per-row top-k selection by a team of warps over one row
// of fp32 scores held in shared memory.
//
// Selection rule (the per-row selection of "DSV4: Add indexer_save_selection
// and indexer_sharded_topk", Description; tie and order rule as documented in
// csa_index.h): among visible entries (score > -inf) keep the min(K, visible)
// largest, equal scores going to the lower entry index and comparing by value
// (-0.0 == +0.0); write the kept indices ascending and pad with -1.
//
// Method (team_topk_row): scores map to order-preserving 32-bit keys (0 =
// invisible).  With the row's visible count and value range known,
//   1. a histogram of NB bins spaced linearly between the row's smallest and
//      largest visible score (a monotone map, so bins are ordered value
//      intervals and a row's scores spread over many bins);
//   2. the bin b* holding the K-th largest score (team-wide suffix scan);
//   3. one pass per warp over a contiguous segment: a ballot bitmap of the
//      entries in bins above b* (kept for sure), per-segment counts, and the
//      members of b* gathered with their entry numbers;
//   4. an exact rank of the gathered members by (value desc, index asc);
//   5. an ordered write from the bitmap (popcounts only).
// Rows that keep all their visible entries, rows of equal scores, rows whose
// value range overflows fp32 and rows whose b* holds more than CAP members
// take the general path: a most-significant-digit-first radix search over
// the keys (four 8-bit digits) for the K-th largest key T and the number of
// keys equal to T that are kept, then an ordered compaction.
#pragma once

#include "csa_ptx.cuh"

namespace csa {

// Order-preserving key of a score; 0 marks an invisible entry (-inf or NaN).
__device__ __forceinline__ uint32_t score_key(float f) {
  if (!(f > -INFINITY)) return 0u;
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0u) u = 0u;  // -0.0 and +0.0 share one key
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inverse of score_key for a visible key.
__device__ __forceinline__ float key_score(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

struct SelectScratch {
  uint32_t hist[256];
  uint32_t warp_a[32];
  uint32_t warp_b[32];
  uint32_t bcast[4];
};

// Scratch of the binned search: NB histogram bins, up to CAP gathered
// (key, entry) pairs of the threshold bin, and a keep-bitmap of up to MAXW
// words (word 4*c+u holds bit `lane` for entry c*128 + 4*lane + u).
template <int NB, int CAP, int MAXW>
struct BinScratch {
  uint32_t hist[NB];
  uint32_t cand[CAP];
  uint32_t cand_t[CAP];
  uint32_t seg_gt[32];   // per warp segment: entries in bins above the threshold bin
  uint32_t seg_sel[32];  // per warp segment: kept entries of the threshold bin
  uint32_t warp_sum[32];
  uint32_t bcast[4];
  uint32_t keep[MAXW];
};

// Bin of a score in a row whose visible scores span [lo, hi] (lo < hi): a
// monotone map onto 0 .. NB-1.  A saturating fma takes x onto [0, 1]; a
// second fma scales that to [0, NB-1] and adds 2^23, which rounds it to an
// integer read from the mantissa.  Each step is a monotone function of its
// input, so bins are ordered value intervals (not exactly equal in width),
// and every finite x lands in range.
struct BinMap {
  float s, b, nb1;
  __device__ BinMap(float lo, float span, int nb) : s(1.0f / span), b(-lo / span), nb1((float)(nb - 1)) {}
  __device__ __forceinline__ uint32_t operator()(float x) const {
    float y;
    asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(x), "f"(s), "f"(b));
    return __float_as_uint(fmaf(y, nb1, 8388608.0f)) - 0x4B000000u;
  }
};

// Visible count and value range of one row.
struct RowStats {
  uint32_t nvis;
  uint32_t min_key;  // score_key of the smallest visible score
  uint32_t max_key;  // score_key of the largest visible score
};

// A team: NT threads (a multiple of 32) synchronised by named barrier `bar_id`.
template <int NT>
struct Team {
  static_assert(NT % 32 == 0, "team size must be whole warps");
  static constexpr int kThreads = NT;
  uint32_t bar_id;
  uint32_t tid;  // 0 .. NT-1
  __device__ __forceinline__ void sync() const {
    if (NT == 32)
      __syncwarp();
    else
      named_bar_sync(bar_id, NT);
  }
  __device__ __forceinline__ uint32_t warp() const { return tid >> 5; }
};

struct SelectResult {
  uint32_t T;        // keys > T are kept
  uint32_t take_eq;  // plus this many keys == T, lowest index first
  uint32_t nvis;     // visible entries in the row
};

// Radix search for the K-th largest key among row[t_begin, t_end).
template <int NT>
__device__ SelectResult team_select_threshold(const float* row, int t_begin, int t_end, uint32_t K,
                                              SelectScratch* sc, const Team<NT>& team) {
  const uint32_t lane = team.tid & 31u;
  uint32_t prefix = 0, rem = K, nvis = 0;
  SelectResult res;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (uint32_t i = team.tid; i < 256; i += NT) sc->hist[i] = 0u;
    team.sync();
    const uint32_t hi_mask = (pass == 0) ? 0u : (0xFFFFFFFFu << (shift + 8));
    for (int t = t_begin + (int)team.tid; t < t_end; t += NT) {
      const uint32_t key = score_key(row[t]);
      if (key != 0u && (key & hi_mask) == prefix) atomicAdd(&sc->hist[(key >> shift) & 255u], 1u);
    }
    team.sync();
    if (team.warp() == 0) {
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = sc->hist[lane * 8 + j];
        sum += c[j];
      }
      // inclusive suffix sum over lanes: keys in bins >= lane*8
      uint32_t incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, incl, off);
        if (lane + off < 32) incl += v;
      }
      const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 0);
      const uint32_t r = (pass == 0 && total <= K) ? 0u : rem;
      const uint32_t excl = incl - sum;  // keys in bins above this lane's bins
      const bool here = (r > 0) && (excl < r) && (r <= incl);
      if (lane == 0) {
        sc->bcast[0] = 0xFFFFFFFFu;  // stays: keep every visible entry
        sc->bcast[1] = 0u;
        sc->bcast[2] = 0u;
        sc->bcast[3] = total;
      }
      __syncwarp();
      if (here) {
        uint32_t acc = excl, d = 0, cd = 0;
        bool found = false;
#pragma unroll
        for (int j = 7; j >= 0; --j) {
          if (!found && acc + c[j] >= r) {
            found = true;
            d = (uint32_t)j;
            cd = c[j];
          }
          if (!found) acc += c[j];
        }
        sc->bcast[0] = lane * 8 + d;  // digit
        sc->bcast[1] = acc;           // keys strictly above the digit's bin
        sc->bcast[2] = cd;            // keys inside the digit's bin
      }
    }
    team.sync();
    const uint32_t digit = sc->bcast[0], above = sc->bcast[1], inbin = sc->bcast[2];
    if (pass == 0) nvis = sc->bcast[3];
    if (digit == 0xFFFFFFFFu) {  // nvis <= K: keep all visible (key > 0)
      res.T = 0u;
      res.take_eq = 0u;
      res.nvis = nvis;
      return res;
    }
    prefix |= digit << shift;
    rem -= above;
    if (inbin == rem) {  // the whole bin is kept: keys >= prefix (low bits zero)
      res.T = (prefix == 0u) ? 0u : prefix - 1u;
      res.take_eq = 0u;
      res.nvis = nvis;
      return res;
    }
  }
  res.T = prefix;  // exact K-th largest key
  res.take_eq = rem;
  res.nvis = nvis;
  return res;
}

// Ordered compaction: writes, in ascending t, every t in [t_begin, t_end)
// with pred(t) == 1 (kept) -- pred(t) == 2 marks a tie candidate that is kept
// only while fewer than `take_eq` earlier tie candidates were kept -- to
// out[0..), then pads out[count..K) with -1.  Each warp owns one contiguous
// segment of the range; a team-wide scan orders the segments.
template <int NT, typename Pred>
__device__ void team_write_ordered(int t_begin, int t_end, uint32_t take_eq, uint32_t K, int32_t* out,
                                   SelectScratch* sc, const Team<NT>& team, Pred pred) {
  constexpr int NW = NT / 32;
  const uint32_t lane = team.tid & 31u, warp = team.warp();
  const int n = t_end > t_begin ? t_end - t_begin : 0;
  const int seg = ((n + NW - 1) / NW + 31) & ~31;
  const int s_lo = t_begin + (int)warp * seg;
  const int s_hi = min(t_end, s_lo + seg);
  uint32_t n_gt = 0, n_eq = 0;
  for (int t = s_lo + (int)lane; t < s_hi; t += 32) {
    const int p = pred(t);
    n_gt += (p == 1);
    n_eq += (p == 2);
  }
  n_gt = __reduce_add_sync(0xFFFFFFFFu, n_gt);
  n_eq = __reduce_add_sync(0xFFFFFFFFu, n_eq);
  if (lane == 0) {
    sc->warp_a[warp] = n_gt;
    sc->warp_b[warp] = n_eq;
  }
  team.sync();
  // exclusive prefix over warps (NW <= 32, done redundantly by every thread)
  uint32_t eq_before = 0, sel_before = 0;
  for (uint32_t w = 0; w < warp; ++w) {
    const uint32_t g = sc->warp_a[w], e = sc->warp_b[w];
    const uint32_t e_take = (take_eq > eq_before) ? min(e, take_eq - eq_before) : 0u;
    sel_before += g + e_take;
    eq_before += e;
  }
  uint32_t total = 0;
  {
    uint32_t eb = 0;
    for (uint32_t w = 0; w < (uint32_t)NW; ++w) {
      const uint32_t g = sc->warp_a[w], e = sc->warp_b[w];
      const uint32_t e_take = (take_eq > eb) ? min(e, take_eq - eb) : 0u;
      total += g + e_take;
      eb += e;
    }
  }
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint32_t pos = sel_before, eq_seen = eq_before;
  for (int t0 = s_lo; t0 < s_hi; t0 += 32) {
    const int t = t0 + (int)lane;
    const int p = (t < s_hi) ? pred(t) : 0;
    const uint32_t eqm = __ballot_sync(0xFFFFFFFFu, p == 2);
    const uint32_t my_eq_rank = eq_seen + __popc(eqm & lt_mask);
    const bool keep = (p == 1) || (p == 2 && my_eq_rank < take_eq);
    const uint32_t km = __ballot_sync(0xFFFFFFFFu, keep);
    if (keep) {
      const uint32_t o = pos + __popc(km & lt_mask);
      if (o < K) out[o] = t;
    }
    pos += __popc(km);
    eq_seen += __popc(eqm);
  }
  for (uint32_t i = min(total, K) + team.tid; i < K; i += NT) out[i] = -1;
  team.sync();  // scratch reuse by the caller
}

// Cold paths kept out of line so the hot selection stays small in the
// instruction cache: the radix search and the general ordered write.
template <int NT>
__device__ __noinline__ void select_general(const float* row, int t0, int n, uint32_t K, uint32_t T,
                                            uint32_t take_eq, bool search, int32_t* out, SelectScratch* sc,
                                            uint32_t bar_id, uint32_t tid) {
  const Team<NT> team{bar_id, tid};
  if (search) {
    const SelectResult r = team_select_threshold<NT>(row, t0, t0 + n, K, sc, team);
    T = r.T;
    take_eq = r.take_eq;
  }
  team_write_ordered<NT>(t0, t0 + n, take_eq, K, out, sc, team, [&](int t) -> int {
    const uint32_t key = score_key(row[t]);
    if (key == 0u) return 0;
    if (key > T) return 1;
    return (key == T) ? 2 : 0;
  });
}

// Selection of one row whose scores live in shared memory at row[t0, t0+n):
// t0 and n multiples of 128, row 16-byte aligned, entries past the row's end
// hold -inf; the indices written are absolute entry numbers.  `st` holds the
// row's visible count and value range.  The bin of x is BinMap: a monotone
// map of x, identical in every pass.
template <int NT, int NB, int CAP, int MAXW>
__device__ void team_topk_row(float* row, int t0, int n, uint32_t K, const RowStats& st, int32_t* out,
                              BinScratch<NB, CAP, MAXW>* bs, SelectScratch* sc, const Team<NT>& team) {
  constexpr int NW = NT / 32;
  constexpr int PER = NB / NT;  // bins per thread in the scan
  static_assert(NB % NT == 0 && PER >= 1, "bins must be a multiple of the team size");
  const uint32_t lane = team.tid & 31u, warp = team.warp();
  const float lo = key_score(st.min_key), hi = key_score(st.max_key);
  const float span = hi - lo;
  const float scale = (float)(NB - 1) / span;
  const int chunks = n >> 7;
  if (st.nvis <= K) {
    select_general<NT>(row, t0, n, K, 0u, 0u, false, out, sc, team.bar_id, team.tid);
    return;
  }
  if (!(hi > lo)) {
    select_general<NT>(row, t0, n, K, st.min_key, K, false, out, sc, team.bar_id, team.tid);
    return;
  }
  const float bias = -lo * scale;
  // |bias| < 2^21 keeps the rounding of x*scale + bias within a quarter bin,
  // so the bin map below stays monotone and in range
  if (!(span < INFINITY) || !(scale < INFINITY) || !(fabsf(bias) < 2097152.0f) || chunks * 4 > MAXW) {
    select_general<NT>(row, t0, n, K, 0u, 0u, true, out, sc, team.bar_id, team.tid);
    return;
  }
  const BinMap bin_of(lo, span, NB);  // in [0, NB-1] for any finite x
  // shared-space addresses: entry e of the row's range at row_s + 4*e
  const uint32_t row_s = smem_u32(row + t0);
  const uint32_t hist_s = smem_u32(bs->hist), keep_s = smem_u32(bs->keep);
  const uint32_t cand_s = smem_u32(bs->cand), cand_t_s = smem_u32(bs->cand_t);
  const uint32_t ncand_s = smem_u32(&bs->bcast[3]), seg_sel_s = smem_u32(bs->seg_sel);
  const int n4 = n >> 2;
#pragma unroll
  for (int j = 0; j < PER; ++j) bs->hist[team.tid * PER + j] = 0u;
  if (team.tid < 32) {
    bs->seg_gt[team.tid] = 0u;
    bs->seg_sel[team.tid] = 0u;
  }
  team.sync();
  // 1. histogram: four float4 loads in flight per thread, then sixteen
  //    predicated shared-memory adds with no returned value
#pragma unroll 1
  for (int i0 = (int)team.tid; i0 < n4; i0 += 4 * NT) {
    float4 a[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      a[q] = (i0 + q * NT < n4) ? lds_f4(row_s + 16u * (uint32_t)(i0 + q * NT))
                                : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    uint32_t addr[16];
    bool vis[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float xs[4] = {a[q].x, a[q].y, a[q].z, a[q].w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        vis[4 * q + u] = xs[u] > -INFINITY;
        addr[4 * q + u] = hist_s + 4u * bin_of(xs[u]);
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) red_add_shared_if(addr[i], 1u, vis[i]);
  }
  team.sync();
  // 2. b*: thread t owns bins [t*PER, (t+1)*PER); suffix sums over threads
  {
    uint32_t c[PER], sum = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      c[j] = bs->hist[team.tid * PER + j];
      sum += c[j];
    }
    uint32_t incl = sum;  // suffix sum within the warp (lanes >= this one)
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t x = __shfl_down_sync(0xFFFFFFFFu, incl, off);
      if (lane + off < 32) incl += x;
    }
    if (lane == 0) bs->warp_sum[warp] = incl;
    team.sync();
    uint32_t higher = 0;  // entries in the bins of later warps
    for (int w = (int)warp + 1; w < NW; ++w) higher += bs->warp_sum[w];
    incl += higher;
    const uint32_t excl = incl - sum;
    if (excl < K && K <= incl) {
      uint32_t acc = excl;
#pragma unroll
      for (int j = PER - 1; j >= 0; --j) {
        if (acc < K && acc + c[j] >= K) {
          bs->bcast[0] = team.tid * PER + (uint32_t)j;
          bs->bcast[1] = acc;
          bs->bcast[2] = c[j];
          bs->bcast[3] = 0u;
        }
        acc += c[j];
      }
    }
  }
  team.sync();
  const uint32_t bstar = bs->bcast[0], above = bs->bcast[1], m = bs->bcast[2];
  if (m > (uint32_t)CAP) {
    select_general<NT>(row, t0, n, K, 0u, 0u, true, out, sc, team.bar_id, team.tid);
    return;
  }
  const uint32_t need = K - above;
  const uint32_t lt_mask = (1u << lane) - 1u;
  // 3. bitmap of sure entries and per-segment counts from ballots; members
  //    of b* gathered by a ballot compaction (slots from a register count in
  //    one-warp teams, else one reservation per warp and pair of chunks);
  //    two chunks in flight, stores predicated rather than branched
  const int seg_chunks = (chunks + NW - 1) / NW;
  const int c_lo = min(chunks, (int)warp * seg_chunks);
  const int c_hi = min(chunks, c_lo + seg_chunks);
  uint32_t gt = 0;      // warp-uniform
  uint32_t ncand = 0u;  // one-warp teams: members gathered so far
#pragma unroll 1
  for (int c0 = c_lo; c0 < c_hi; c0 += 2) {
    float4 v[2];
#pragma unroll
    for (int q = 0; q < 2; ++q)
      v[q] = (c0 + q < c_hi) ? lds_f4(row_s + 16u * (uint32_t)((c0 + q) * 32 + (int)lane))
                             : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    uint32_t sure[8], memb[8];
    float xk[8];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float xs[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool vis = xs[u] > -INFINITY;
        const uint32_t bb = bin_of(xs[u]);
        xk[4 * q + u] = xs[u];
        sure[4 * q + u] = __ballot_sync(0xFFFFFFFFu, vis && bb > bstar);
        memb[4 * q + u] = __ballot_sync(0xFFFFFFFFu, vis && bb == bstar);
      }
    }
    sts_u4_if(keep_s + 16u * (uint32_t)c0, make_uint4(sure[0], sure[1], sure[2], sure[3]), lane == 0);
    sts_u4_if(keep_s + 16u * (uint32_t)(c0 + 1), make_uint4(sure[4], sure[5], sure[6], sure[7]),
              lane == 0 && c0 + 1 < c_hi);
    // counts as balanced sums (short dependency chains)
    uint32_t pm[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) pm[i] = __popc(memb[i]);
    gt += ((__popc(sure[0]) + __popc(sure[1])) + (__popc(sure[2]) + __popc(sure[3]))) +
          ((__popc(sure[4]) + __popc(sure[5])) + (__popc(sure[6]) + __popc(sure[7])));
    // exclusive prefix of the member counts over the eight ballots
    uint32_t pre[8];
    pre[0] = 0u;
    pre[1] = pm[0];
    pre[2] = pm[0] + pm[1];
    pre[3] = pre[2] + pm[2];
    const uint32_t h4 = pre[2] + (pm[2] + pm[3]);
    pre[4] = h4;
    pre[5] = h4 + pm[4];
    pre[6] = h4 + (pm[4] + pm[5]);
    pre[7] = pre[6] + pm[6];
    const uint32_t nm = pre[7] + pm[7];
    if (nm != 0u) {  // warp-uniform: most pairs of chunks hold no member
      uint32_t slot;
      if constexpr (NT == 32) {  // one warp: the running member count lives in a register
        slot = ncand;
        ncand += nm;
      } else {
        slot = 0;
        if (lane == 0) slot = atom_add_shared(ncand_s, nm);
        slot = __shfl_sync(0xFFFFFFFFu, slot, 0);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t o = slot + pre[i] + __popc(memb[i] & lt_mask);
        sts_u32x2_if(cand_s + 4u * o, score_key(xk[i]), cand_t_s + 4u * o,
                     (uint32_t)((c0 + i / 4) * 128 + 4 * (int)lane + (i & 3)),  // entry relative to t0
                     ((memb[i] >> lane) & 1u) && o < (uint32_t)CAP);
      }
    }
  }
  if (lane == 0) bs->seg_gt[warp] = gt;
  team.sync();
  // 4. exact rank inside b*
#pragma unroll 1
  for (uint32_t i = team.tid; i < m; i += NT) {
    const uint32_t ki = bs->cand[i], ti = bs->cand_t[i];
    uint32_t rank = 0;
#pragma unroll 4
    for (uint32_t j = 0; j < m; ++j) {
      const uint32_t kj = bs->cand[j], tj = bs->cand_t[j];
      rank += (kj > ki) || (kj == ki && tj < ti);
    }
    if (rank < need) {
      const uint32_t c = ti >> 7, l = (ti >> 2) & 31u, u = ti & 3u;
      red_or_shared(keep_s + 4u * (4u * c + u), 1u << l);
      red_add_shared_if(seg_sel_s + 4u * (c / (uint32_t)seg_chunks), 1u, true);
    }
  }
  team.sync();
  // 5. ordered write from the bitmap: positions from popcounts, predicated stores
  uint32_t base = 0, total = 0;
  for (int w = 0; w < NW; ++w) {
    const uint32_t cnt = bs->seg_gt[w] + bs->seg_sel[w];
    base += (w < (int)warp) ? cnt : 0u;
    total += cnt;
  }
#pragma unroll 4
  for (int c = c_lo; c < c_hi; ++c) {
    const uint4 mw = lds_u4(keep_s + 16u * (uint32_t)c);
    const uint32_t b0 = (mw.x >> lane) & 1u, b1 = (mw.y >> lane) & 1u, b2 = (mw.z >> lane) & 1u;
    const uint32_t b3 = (mw.w >> lane) & 1u;
    const uint32_t p0 = base + __popc(mw.x & lt_mask) + __popc(mw.y & lt_mask) + __popc(mw.z & lt_mask) +
                        __popc(mw.w & lt_mask);
    const uint32_t p1 = p0 + b0, p2 = p1 + b1, p3 = p2 + b2;
    const int tb = t0 + c * 128 + 4 * (int)lane;
    if (b0 && p0 < K) out[p0] = tb;
    if (b1 && p1 < K) out[p1] = tb + 1;
    if (b2 && p2 < K) out[p2] = tb + 2;
    if (b3 && p3 < K) out[p3] = tb + 3;
    base += __popc(mw.x) + __popc(mw.y) + __popc(mw.z) + __popc(mw.w);
  }
  for (uint32_t i = min(total, K) + team.tid; i < K; i += NT) out[i] = -1;
  team.sync();
}

}  // namespace csa
