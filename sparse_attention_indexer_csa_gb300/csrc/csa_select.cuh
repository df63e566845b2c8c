// csa_select.cuh -- per-row top-k selection by a team of warps over one row
// of fp32 scores held in shared memory.
//
// Selection rule (the per-row selection of "DSV4: Add indexer_save_selection
// and indexer_sharded_topk", Description; tie and order rule as documented in
// csa_index.h): among visible entries (score > -inf) keep the min(K, visible)
// largest, equal scores going to the lower entry index and comparing by value
// (-0.0 == +0.0); write the kept indices ascending and pad with -1.
//
// Method: scores map to order-preserving 32-bit keys (0 = invisible).  A
// most-significant-digit-first radix search (four 8-bit digits) finds the
// K-th largest key T and how many keys equal to T are kept (the lowest
// indices first).  One ordered compaction pass then writes, per row, every
// index whose key is above T plus the first `take_eq` indices whose key
// equals T, in ascending order.
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

struct SelectScratch {
  uint32_t hist[256];
  uint32_t warp_a[32];
  uint32_t warp_b[32];
  uint32_t bcast[4];
};

// A team: NT threads (a multiple of 32) synchronised by named barrier `bar_id`.
template <int NT>
struct Team {
  static_assert(NT % 32 == 0, "team size must be whole warps");
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
        uint32_t acc = excl;
        int d = 0;
#pragma unroll
        for (int j = 7; j >= 0; --j) {
          if (acc + c[j] >= r) {
            d = j;
            break;
          }
          acc += c[j];
        }
        sc->bcast[0] = lane * 8 + (uint32_t)d;  // digit
        sc->bcast[1] = acc;                      // keys strictly above the digit's bin
        sc->bcast[2] = c[d];                     // keys inside the digit's bin
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

// Full selection of one row held in shared memory.
template <int NT>
__device__ void team_topk_row(const float* row, int t_begin, int t_end, uint32_t K, int32_t* out,
                              SelectScratch* sc, const Team<NT>& team) {
  const SelectResult r = team_select_threshold<NT>(row, t_begin, t_end, K, sc, team);
  const uint32_t T = r.T;
  team_write_ordered<NT>(t_begin, t_end, r.take_eq, K, out, sc, team, [&](int t) -> int {
    const uint32_t key = score_key(row[t]);
    if (key == 0u) return 0;
    if (key > T) return 1;
    return (key == T) ? 2 : 0;
  });
}

}  // namespace csa
