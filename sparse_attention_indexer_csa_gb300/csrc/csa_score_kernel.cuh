// csa_score_kernel.cuh -- the persistent, warp-specialised indexer kernel.
//
// One CTA per SM walks a static list of work items.  An item is R query rows
// of one batch (all H heads) and a range of compressed-entry tiles of 128.
// Per item the tensor cores compute, for every tile,
//     acc[t, (j,h)] = sum_d k[b,t,d] * q[b,h,s0+j,d]        (tcgen05 UMMA)
// with the k tile as operand A (M = 128 entries) and the item's q block as
// operand B (N = R*H columns ordered j*H + h), accumulating in TMEM.  The
// epilogue warps read their lane's row of the accumulator, so each thread
// owns one entry t and reduces over heads in registers:
//     score[s0+j, t] = scale * sum_h w[s0+j,h] * max(acc[t,(j,h)], 0)
// (ReLU(scale*x) = scale*ReLU(x) because scale > 0), then apply the future
// and segment masks.  This is the head-reduced score of "Add StreamIndex
// Kernel for CSA [Deepseek v4]" (Description; head-chunked on-chip
// accumulation instead of the [B,H,S,W] tensor) with the masks of "DSV4: Add
// indexer_save_selection and indexer_sharded_topk" (mask review hunk).
//
// Warp roles (block = 4 control warps + EW epilogue warps [+ R select warps]):
//   warp 0  TMA producer: q block per item, k tiles into a ring of stages
//   warp 1  TMEM owner and UMMA issuer (one elected thread)
//   warps 2, 3  schedulers (alternate items): per item compute the visible
//           tile range, per-row thresholds / segment ids / visible counts and
//           stage the weights into a ring of item slots
//   warps 4..4+EW-1  epilogue (warp w reads TMEM lanes 32*(w%4) ..)
//   FUSED: warps 4+EW .. 4+EW+R-1  select warps, one query row each.
// FUSED: the epilogue writes each item's R score rows into one of two
// per-CTA staging slots in the caller's workspace (2 x R x W fp32 per CTA,
// small enough to stay in L2) and folds per-row min / max / visible counts
// into shared memory; the select warps pull the item's rows into shared
// memory with one bulk copy, free the slot and select, so the selection of
// item i runs while the tensor cores and the epilogue work on item i+1.
//
// Tiles wholly past the rows' future-mask bound, or (with segment ids)
// outside the range of entries sharing a segment with the item's rows, are
// never loaded or multiplied.  Every mbarrier wait is bounded.
#pragma once

#include "csa_ptx.cuh"
#include "csa_select.cuh"

namespace csa {

constexpr int kTileT = 128;  // compressed entries per tile (UMMA M)

// Per-item segment summary written by csa_segscan_kernel for whole-row items
// of four rows (64 bytes): tiles holding visible entries, and per row the
// visible count, first visible entry and contiguity.
struct SegInfo {
  int t_lo, t_hi, pad0, pad1;
  int nvis[4], tfirst[4], contig[4];
};

struct KParams {
  int B, S, W, r, K;
  int r_shift;  // log2(r) when r is a power of two, else -1
  float scale;
  int w_f32;
  const void* w;
  long long w_sb, w_ss;  // element strides of w's batch and row dimensions
  const int32_t* q_seg;
  const int32_t* kv_seg;
  const int64_t* q_start;
  float* scores;  // score mode: output; fused: optional debug copy
  int32_t* idx;   // fused: selection output
  float* ring;    // fused: per-CTA staging of two items' score rows [grid][2][R][w_pad]
  const SegInfo* seginfo;  // with segment ids and whole-row items: [B][n_rb] summaries, or null
  int n_rb, n_tiles, n_chunks, chunk_tiles, n_items;
  int w_pad;  // fused: row pitch (floats) of the shared score rows
  unsigned long long wait_ns;
};

template <int R>
struct ItemDesc {
  int b, s0;
  int t_lo, t_hi;  // tiles computed: [t_lo, t_hi)
  int c_lo, c_hi;  // tiles owned by the item: [c_lo, c_hi)
  int trivial;     // fused: every row keeps all its visible entries, no scores needed
  int thr[R];      // rows' visible bound min(W, (pos+1)/r); 0 for rows past S
  int seg[R];
  int nvis[R];     // visible entries of the row inside [c_lo, c_hi) tiles
  int tfirst[R];   // first visible entry of the row
  int contig[R];   // the row's visible entries are tfirst .. tfirst + nvis - 1
};

// Selection scratch of one select warp of the fused kernel.
struct FusedRowScratch {
  SelectScratch sc;
  BinScratch<512, 256, 128> bs;  // rows of up to 4096 entries
};

// Long-row mode (rows of up to 16384 entries): the select warps select as one
// team of 128 threads, one row at a time, from a single shared row buffer.
constexpr int kLongMaxW = 16384;
struct LongRowScratch {
  SelectScratch sc[4];                          // per warp (visible-set writes); sc[0] for the team
  BinScratch<1024, 1024, kLongMaxW / 32> bs;    // the team's binned search
};

constexpr uint32_t pow2_cols(uint32_t n) {
  uint32_t c = 32;
  while (c < n) c <<= 1;
  return c;
}

template <int H_, int D_, int R_, bool FUSED_, bool LONG_ = false, bool DOCS_ = false>
struct Cfg {
  static constexpr int H = H_, D = D_, R = R_;
  static constexpr bool FUSED = FUSED_;
  static constexpr bool LONG = LONG_;  // fused, rows of 4097..16384 entries
  // fused with segment summaries (packed documents): the scheduler posts only
  // the items that need scores to the item ring, which ends with a marker
  static constexpr bool DOCS = DOCS_;
  static_assert(!DOCS || (FUSED && !LONG), "the document mode is the fused kernel's");
  static_assert(!LONG || (FUSED && R_ == 4), "long-row mode is the fused four-row kernel");
  static constexpr int N = R * H;
  static_assert(N % 16 == 0 && N >= 16 && N <= 256, "UMMA N must be 16..256 in steps of 16");
  static constexpr int KC = (D % 64 == 0) ? 64 : 32;  // K elements per swizzled row
  static constexpr int ROWB = KC * 2;                  // 128 B (SW128) or 64 B (SW64)
  static constexpr int NKC = D / KC;
  static_assert(D % 32 == 0, "head dim must be a multiple of 32");
  static constexpr int KSTAGES = (R == 1) ? 5 : 2;
  static constexpr int QBUF = FUSED ? 1 : 2;
  static constexpr int SLOTS = FUSED ? 6 : 4;      // item ring depth
  // fused: the select warps' own ring of item descriptors, deeper than the
  // item ring, so a selection that waits for its scores holds no item slot
  static constexpr int SSLOTS = FUSED ? 16 : 0;
  static constexpr int EW = (R >= 2) ? 8 : 4;      // epilogue warps
  static constexpr int SW = FUSED ? R : 0;         // select warps (one row each)
  static constexpr int RW = (R >= 2) ? R / 2 : 1;  // rows per epilogue warp
  static_assert(R == 1 || R % 2 == 0, "R must be 1 or even");
  static constexpr int NTHREADS = 128 + (EW + SW) * 32;
  static constexpr uint32_t QCHUNK = N * ROWB;       // bytes of one K-chunk of the q block
  static constexpr uint32_t KCHUNK = kTileT * ROWB;  // bytes of one K-chunk of a k tile
  static constexpr uint32_t QBYTES = QCHUNK * NKC;
  static constexpr uint32_t KBYTES = KCHUNK * NKC;
  static constexpr uint32_t TMEM_COLS = pow2_cols(2 * N);
  static constexpr uint32_t IDESC = idesc_bf16_f32(kTileT, N);
  // shared memory layout (offsets from a 1024-aligned base)
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = (OFF_Q + QBUF * QBYTES + 1023) & ~1023u;
  static constexpr uint32_t OFF_W = (OFF_K + KSTAGES * KBYTES + 1023) & ~1023u;
  static constexpr uint32_t OFF_DESC = OFF_W + SLOTS * R * H * 4;
  static constexpr uint32_t OFF_SDESC = OFF_DESC + SLOTS * sizeof(ItemDesc<R>);
  static constexpr uint32_t OFF_BAR = (OFF_SDESC + SSLOTS * sizeof(ItemDesc<R>) + 15) & ~15u;
  // barriers: item_full[SLOTS], item_empty[SLOTS], q_full[QB], q_empty[QB], k_full[KS], k_empty[KS],
  //           acc_full[2], acc_empty[2], drain, ring_full[2], ring_empty[2], copy_full,
  //           sel_full[SSLOTS], sel_empty[SSLOTS]
  static constexpr int NBAR = 2 * SLOTS + 2 * QBUF + 2 * KSTAGES + 4 + 1 + 5 + 2 * SSLOTS;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;  // tmem base, abort flag
  static constexpr uint32_t OFF_STATS = (OFF_MISC + 16 + 15) & ~15u;  // RowStats[2][R]
  static constexpr uint32_t OFF_SCR = (OFF_STATS + 2 * R * sizeof(RowStats) + 15) & ~15u;
  static constexpr uint32_t SCR_BYTES = LONG ? (uint32_t)sizeof(LongRowScratch) : SW * (uint32_t)sizeof(FusedRowScratch);
  static constexpr uint32_t OFF_SROW = (OFF_SCR + SCR_BYTES + 127) & ~127u;
  static constexpr uint32_t SROWS = FUSED ? (LONG ? 1u : (uint32_t)R) : 0u;  // shared score rows
  // dynamic shared memory for a given fused row pitch (+1 KB alignment slack)
  static constexpr uint32_t smem_bytes(int w_pad) { return OFF_SROW + SROWS * (uint32_t)w_pad * 4u + 1024u; }
};

template <class C>
struct Smem {
  uint8_t* base;
  static constexpr int B0 = 2 * C::SLOTS;         // first q barrier
  static constexpr int B1 = B0 + 2 * C::QBUF;     // first k barrier
  static constexpr int B2 = B1 + 2 * C::KSTAGES;  // first accumulator barrier
  __device__ uint8_t* q(int i) const { return base + C::OFF_Q + i * C::QBYTES; }
  __device__ uint8_t* k(int i) const { return base + C::OFF_K + i * C::KBYTES; }
  __device__ float* w(int slot) const { return reinterpret_cast<float*>(base + C::OFF_W) + slot * C::R * C::H; }
  __device__ ItemDesc<C::R>* desc(int slot) const {
    return reinterpret_cast<ItemDesc<C::R>*>(base + C::OFF_DESC) + slot;
  }
  __device__ ItemDesc<C::R>* sdesc(int slot) const {
    return reinterpret_cast<ItemDesc<C::R>*>(base + C::OFF_SDESC) + slot;
  }
  __device__ uint64_t* bar(int i) const { return reinterpret_cast<uint64_t*>(base + C::OFF_BAR) + i; }
  __device__ uint64_t* item_full(int s) const { return bar(s); }
  __device__ uint64_t* item_empty(int s) const { return bar(C::SLOTS + s); }
  __device__ uint64_t* q_full(int i) const { return bar(B0 + i); }
  __device__ uint64_t* q_empty(int i) const { return bar(B0 + C::QBUF + i); }
  __device__ uint64_t* k_full(int i) const { return bar(B1 + i); }
  __device__ uint64_t* k_empty(int i) const { return bar(B1 + C::KSTAGES + i); }
  __device__ uint64_t* acc_full(int i) const { return bar(B2 + i); }
  __device__ uint64_t* acc_empty(int i) const { return bar(B2 + 2 + i); }
  __device__ uint64_t* drain() const { return bar(B2 + 4); }
  __device__ uint64_t* ring_full(int i) const { return bar(B2 + 5 + i); }
  __device__ uint64_t* ring_empty(int i) const { return bar(B2 + 7 + i); }
  __device__ uint64_t* copy_full() const { return bar(B2 + 9); }
  __device__ uint64_t* sel_full(int s) const { return bar(B2 + 10 + s); }
  __device__ uint64_t* sel_empty(int s) const { return bar(B2 + 10 + C::SSLOTS + s); }
  __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(base + C::OFF_MISC); }
  __device__ volatile uint32_t* abort_flag() const {
    return reinterpret_cast<volatile uint32_t*>(base + C::OFF_MISC + 4);
  }
  __device__ RowStats* stats(int slot, int j) const {
    return reinterpret_cast<RowStats*>(base + C::OFF_STATS) + slot * C::R + j;
  }
  __device__ FusedRowScratch* scratch(int j) const {
    return reinterpret_cast<FusedRowScratch*>(base + C::OFF_SCR) + j;
  }
  __device__ LongRowScratch* long_scratch() const { return reinterpret_cast<LongRowScratch*>(base + C::OFF_SCR); }
  __device__ float* srow(int j, int w_pad) const {
    return reinterpret_cast<float*>(base + C::OFF_SROW) + (size_t)j * w_pad;
  }
};

// Item index -> (b, row block, chunk).  Row blocks run from the last (most
// visible entries, most work) to the first, the batch index fastest.
__device__ __forceinline__ void item_coords(const KParams& p, int item, int& b, int& rb, int& c) {
  c = item % p.n_chunks;
  const int rest = item / p.n_chunks;
  b = rest % p.B;
  rb = p.n_rb - 1 - rest / p.B;
}

// The items are dealt to the CTAs in rounds of gridDim.x.  Items of several
// rows (ROT): in round k, CTA x takes item k * gridDim.x + (x + k) %
// gridDim.x.  Each CTA's list keeps the longest-first order, and the
// rotation moves a CTA to another batch every round; a plain round-robin
// would give CTA x only batch x % B whenever B divides the grid, and batches
// that differ (segments, offsets) would load the CTAs unevenly.  Single-row
// items (decode chunks) carry equal work and take the plain round-robin.
template <bool ROT>
__device__ __forceinline__ int cta_item_count(const KParams& p) {
  const int g = (int)gridDim.x, x = (int)blockIdx.x;
  if constexpr (ROT) {
    const int rounds = p.n_items / g, rem = p.n_items - rounds * g;
    return rounds + (((x + rounds) % g) < rem ? 1 : 0);
  } else {
    return x < p.n_items ? (p.n_items - x + g - 1) / g : 0;
  }
}
template <bool ROT>
__device__ __forceinline__ int cta_item(int k) {
  const int g = (int)gridDim.x;
  return ROT ? k * g + ((int)blockIdx.x + k) % g : k * g + (int)blockIdx.x;
}

// Visible bound min(W, (pos+1)/r) of rows s0 .. s0+R-1 of a sequence that
// starts at position qs0 (0 for rows past S); returns the largest.
template <int R>
__device__ __forceinline__ int row_bounds(const KParams& p, long long qs0, int s0, int (&thr)[R]) {
  int thr_max = 0;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    const int s = s0 + j;
    long long tv = 0;
    if (s < p.S) {
      const long long pos1 = qs0 + s + 1;
      tv = pos1 <= 0 ? 0 : (p.r_shift >= 0 ? (pos1 >> p.r_shift) : pos1 / p.r);
      tv = tv > p.W ? p.W : tv;
    }
    thr[j] = (int)tv;
    thr_max = max(thr_max, thr[j]);
  }
  return thr_max;
}

// Rows s0 .. s0+R-1 of batch b: each row's visible bound under the future
// mask and its segment id (0 without segments); returns the largest bound.
template <int R>
__device__ __forceinline__ int item_rows(const KParams& p, int b, int s0, int (&thr)[R], int (&seg)[R]) {
  const long long qs0 = p.q_start ? (long long)p.q_start[b] : 0ll;
#pragma unroll
  for (int j = 0; j < R; ++j) seg[j] = (p.q_seg != nullptr && s0 + j < p.S) ? p.q_seg[(size_t)b * p.S + s0 + j] : 0;
  return row_bounds<R>(p, qs0, s0, thr);
}

// Segment scan of one item (a warp): over entries [e_lo, e_hi) of batch b,
// per row j the entries visible under both masks -- count, first entry and
// whether they form one contiguous run -- and the tiles [t_lo, t_hi) that
// hold any of them (t_lo = t_hi when none does).  Segment ids are read with
// 16-byte loads, four in flight per lane, when they are aligned.
//
// When the item's rows share one segment id (the usual case: four
// consecutive rows of one document), entries below the smallest row bound
// are visible to every row or to none, so that prefix takes one comparison
// per entry; only the few entries between the rows' bounds are checked per
// row.
template <int R>
__device__ void scan_segments(const KParams& p, int b, int e_lo, int e_hi, const int (&thr)[R], const int (&seg)[R],
                              int (&nvis)[R], int (&tfirst)[R], int (&contig)[R], int& t_lo, int& t_hi) {
  const uint32_t lane = lane_id();
  t_lo = t_hi = e_lo / kTileT;
  int cnt[R], tmn[R], tmx[R];
#pragma unroll
  for (int j = 0; j < R; ++j) {
    cnt[j] = 0;
    tmn[j] = 0x7FFFFFFF;
    tmx[j] = -1;
  }
  const int32_t* kv = p.kv_seg + (size_t)b * p.W;
  auto visit = [&](int t, int ks) {
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const bool m = (t < thr[j]) && (ks == seg[j]);
      cnt[j] += m;
      if (m) {
        tmn[j] = min(tmn[j], t);
        tmx[j] = max(tmx[j], t);
      }
    }
  };
  // calls f(t, kv[t]) for every entry of [lo, hi) this lane owns
  auto scan = [&](int lo, int hi, auto&& f) {
    const bool vec = ((reinterpret_cast<uintptr_t>(kv) & 15u) == 0) && (lo % 4 == 0);
    if (vec) {
      // four 16-byte loads in flight per lane per round (512 entries per warp)
      for (int t0 = lo + 4 * (int)lane; t0 < hi; t0 += 512) {
        int4 v4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int t = t0 + 128 * u;
          v4[u] = (t + 3 < hi) ? *reinterpret_cast<const int4*>(kv + t) : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int t = t0 + 128 * u;
          if (t + 3 < hi) {
            f(t, v4[u].x);
            f(t + 1, v4[u].y);
            f(t + 2, v4[u].z);
            f(t + 3, v4[u].w);
          } else {
            for (int x = t; x < hi; ++x) f(x, kv[x]);
          }
        }
      }
    } else {
      for (int t = lo + (int)lane; t < hi; t += 32) f(t, kv[t]);
    }
  };
  bool uni = true;
  int ta = e_hi;  // smallest row bound (rows past S have bound 0 and id 0)
#pragma unroll
  for (int j = 0; j < R; ++j) {
    uni = uni && seg[j] == seg[0];
    ta = min(ta, thr[j]);
  }
  ta = max(ta, e_lo);
  if (uni && ta > e_lo) {
    // [e_lo, ta): every row's bound is at or above ta
    const int sg = seg[0];
    int c = 0, mn = 0x7FFFFFFF, mx = -1;
    scan(e_lo, ta, [&](int t, int ks) {
      const bool m = ks == sg;
      c += m;
      if (m) {
        mn = min(mn, t);
        mx = max(mx, t);
      }
    });
#pragma unroll
    for (int j = 0; j < R; ++j) {
      cnt[j] = c;
      tmn[j] = mn;
      tmx[j] = mx;
    }
    for (int t = ta + (int)lane; t < e_hi; t += 32) visit(t, kv[t]);
  } else {
    scan(e_lo, e_hi, visit);
  }
  int tmin = 0x7FFFFFFF, tmax = -1;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    nvis[j] = (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)cnt[j]);
    tfirst[j] = __reduce_min_sync(0xFFFFFFFFu, tmn[j]);
    const int last = __reduce_max_sync(0xFFFFFFFFu, tmx[j]);
    contig[j] = (nvis[j] == 0) || (last - tfirst[j] + 1 == nvis[j]);
    if (nvis[j] > 0) {
      tmin = min(tmin, tfirst[j]);
      tmax = max(tmax, last);
    } else {
      tfirst[j] = 0;
    }
  }
  if (tmax >= 0) {
    t_lo = tmin / kTileT;
    t_hi = tmax / kTileT + 1;
  }
}

// Item `it` of this CTA's list.  Fused: the items alternate from both ends of
// the list (longest rows first, shortest last), so the cheap trivial items
// are interleaved with scored ones instead of leaving the tensor cores idle
// at the end.
template <class C>
__device__ __forceinline__ void sched_coords(const KParams& p, int it, int n_mine, int& b, int& rb, int& c) {
  if constexpr (C::FUSED) {
    const int jj = (it & 1) ? (n_mine - 1 - (it >> 1)) : (it >> 1);
    item_coords(p, cta_item<(C::R > 1)>(jj), b, rb, c);
  } else {
    item_coords(p, cta_item<(C::R > 1)>(it), b, rb, c);
  }
}

template <int R>
__device__ __forceinline__ void write_desc(ItemDesc<R>* d, int b, int s0, int t_lo, int t_hi, int c_lo, int c_hi,
                                           int trivial, const int (&thr)[R], const int (&seg)[R],
                                           const int (&nvis)[R], const int (&tfirst)[R], const int (&contig)[R]) {
  d->b = b;
  d->s0 = s0;
  d->t_lo = t_lo;
  d->t_hi = t_hi;
  d->c_lo = c_lo;
  d->c_hi = c_hi;
  d->trivial = trivial;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    d->thr[j] = thr[j];
    d->seg[j] = seg[j];
    d->nvis[j] = nvis[j];
    d->tfirst[j] = tfirst[j];
    d->contig[j] = contig[j];
  }
}

// Scheduler warp `sw` (0 or 1) prepares the items it = sw, sw + 2, ...: per
// item the visible tile range, per-row thresholds / segment ids / visible
// counts, the trivial flag, and the weights of scored items.  The global
// reads of 32 items at a time are made at once, one item per lane (the
// items' latencies overlap instead of adding up), and handed to the item
// loop through shuffles.
template <class C>
__device__ void run_scheduler(const KParams& p, const Smem<C>& sm, const WaitCtl& ctl, int sw) {
  constexpr int R = C::R, H = C::H;
  constexpr int NWL = (R * H + 31) / 32;  // weights per lane
  static_assert(R <= 4, "a segment summary covers four rows");
  const uint32_t lane = lane_id();
  const bool segs = p.q_seg != nullptr;
  const bool pre = p.seginfo != nullptr;  // scanned ahead by csa_segscan_kernel (whole-row items)
  const int n_mine = cta_item_count<(C::R > 1)>(p);
  for (int it0 = sw; it0 < n_mine; it0 += 64) {
    // lane l fetches item it0 + 2l
    const int my_it = it0 + 2 * (int)lane;
    int b_l = 0, rb_l = 0, c_l = 0;
    long long qs_l = 0;
    int seg_l[R];
    SegInfo si_l{};
#pragma unroll
    for (int j = 0; j < R; ++j) seg_l[j] = 0;
    if (my_it < n_mine) {
      sched_coords<C>(p, my_it, n_mine, b_l, rb_l, c_l);
      if (p.q_start != nullptr) qs_l = p.q_start[b_l];
      if (segs) {
#pragma unroll
        for (int j = 0; j < R; ++j)
          if (rb_l * R + j < p.S) seg_l[j] = p.q_seg[(size_t)b_l * p.S + rb_l * R + j];
      }
      if (pre) si_l = p.seginfo[(size_t)b_l * p.n_rb + rb_l];
      // the weight rows of the item into L2: the item loop reads them from
      // there if the item needs scores (a few hundred bytes per item)
      const size_t esz = p.w_f32 ? 4 : 2;
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int s = rb_l * R + j;
        if (s < p.S) {
          const char* a = static_cast<const char*>(p.w) + ((size_t)b_l * p.w_sb + (size_t)s * p.w_ss) * esz;
          prefetch_l2(a);
          prefetch_l2(a + H * esz - 1);
        }
      }
    }
    const int cnt = min(32, (n_mine - it0 + 1) / 2);
    for (int k = 0; k < cnt; ++k) {
      const int it = it0 + 2 * k;
      const int b = __shfl_sync(0xFFFFFFFFu, b_l, k);
      const int rb = __shfl_sync(0xFFFFFFFFu, rb_l, k);
      const int c = __shfl_sync(0xFFFFFFFFu, c_l, k);
      const long long qs0 = __shfl_sync(0xFFFFFFFFu, qs_l, k);
      const int s0 = rb * R;
      int thr[R], seg[R], nvis[R], tfirst[R], contig[R];
#pragma unroll
      for (int j = 0; j < R; ++j) seg[j] = __shfl_sync(0xFFFFFFFFu, seg_l[j], k);
      const int thr_max = row_bounds<R>(p, qs0, s0, thr);
      const int c_lo = c * p.chunk_tiles;
      const int c_hi = min(p.n_tiles, c_lo + p.chunk_tiles);
      int t_lo = c_lo, t_hi = c_lo;
      if (!segs) {
#pragma unroll
        for (int j = 0; j < R; ++j) {
          nvis[j] = max(0, min(thr[j], c_hi * kTileT) - c_lo * kTileT);
          tfirst[j] = c_lo * kTileT;
          contig[j] = 1;
        }
        t_hi = max(c_lo, min(c_hi, (thr_max + kTileT - 1) / kTileT));
      } else if (pre) {
#pragma unroll
        for (int j = 0; j < R; ++j) {
          nvis[j] = __shfl_sync(0xFFFFFFFFu, si_l.nvis[j], k);
          tfirst[j] = __shfl_sync(0xFFFFFFFFu, si_l.tfirst[j], k);
          contig[j] = __shfl_sync(0xFFFFFFFFu, si_l.contig[j], k);
        }
        t_lo = __shfl_sync(0xFFFFFFFFu, si_l.t_lo, k);
        t_hi = __shfl_sync(0xFFFFFFFFu, si_l.t_hi, k);
      } else {
        scan_segments<R>(p, b, c_lo * kTileT, min(c_hi * kTileT, thr_max), thr, seg, nvis, tfirst, contig, t_lo,
                         t_hi);
      }
      int trivial = 0;
      if (C::FUSED && p.scores == nullptr) {
        trivial = 1;
#pragma unroll
        for (int j = 0; j < R; ++j) trivial &= (nvis[j] <= p.K) ? 1 : 0;
        if (trivial) t_hi = t_lo;
      }
      // the weights (fp32) of a scored item's rows, every load in flight
      // before the first store; rows past S get 0 (an item whose rows keep
      // every visible entry computes no score and needs none)
      float wv[NWL];
#pragma unroll
      for (int u = 0; u < NWL; ++u) {
        const int i = (int)lane + 32 * u;
        const int j = i / H, h = i % H;
        const int s = s0 + j;
        float v = 0.f;
        if (!trivial && i < R * H && s < p.S) {
          const size_t off = (size_t)b * p.w_sb + (size_t)s * p.w_ss + h;
          v = p.w_f32 ? reinterpret_cast<const float*>(p.w)[off]
                      : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.w)[off]);
        }
        wv[u] = v;
      }
      const int slot = it % C::SLOTS;
      mbar_wait(sm.item_empty(slot), ((it / C::SLOTS) & 1) ^ 1, ctl);
      if (!trivial) {
        float* ws = sm.w(slot);
#pragma unroll
        for (int u = 0; u < NWL; ++u) {
          const int i = (int)lane + 32 * u;
          if (i < R * H) ws[i] = wv[u];
        }
      }
      if (lane == 0) write_desc<R>(sm.desc(slot), b, s0, t_lo, t_hi, c_lo, c_hi, trivial, thr, seg, nvis, tfirst, contig);
      if constexpr (C::FUSED) {
        const int ss = it % C::SSLOTS;
        mbar_wait(sm.sel_empty(ss), ((it / C::SSLOTS) & 1) ^ 1, ctl);
        if (lane == 1)
          write_desc<R>(sm.sdesc(ss), b, s0, t_lo, t_hi, c_lo, c_hi, trivial, thr, seg, nvis, tfirst, contig);
        __syncwarp();
        if (lane == 1) mbar_arrive(sm.sel_full(ss));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.item_full(slot));
    }
  }
}

// Write the selection of a row that keeps all its visible entries.
template <int NT>
__device__ void write_visible_set(int32_t* out, int K, int nvis, int tfirst, int contig, int thr, int seg,
                                  const int32_t* kv, SelectScratch* sc, const Team<NT>& team) {
  if (contig) {  // visible entries are tfirst .. tfirst + nvis - 1
    if ((K & 3) == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0) {
      int4* o4 = reinterpret_cast<int4*>(out);
      for (int i = (int)team.tid; i < K / 4; i += NT) {
        const int i0 = 4 * i;
        int4 v;
        v.x = (i0 + 0 < nvis) ? tfirst + i0 + 0 : -1;
        v.y = (i0 + 1 < nvis) ? tfirst + i0 + 1 : -1;
        v.z = (i0 + 2 < nvis) ? tfirst + i0 + 2 : -1;
        v.w = (i0 + 3 < nvis) ? tfirst + i0 + 3 : -1;
        o4[i] = v;
      }
    } else {
      for (int i = (int)team.tid; i < K; i += NT) out[i] = (i < nvis) ? tfirst + i : -1;
    }
  } else {
    team_write_ordered<NT>(0, thr, 0u, (uint32_t)K, out, sc, team,
                           [&](int tt) -> int { return (kv[tt] == seg) ? 1 : 0; });
  }
}

// Scheduler of the document mode (C::DOCS, segment summaries present).
// The items are taken in rounds of 32: their global reads are made at once,
// one item per lane, and handed to the item loop through shuffles; from the
// lanes' flags both warps know, for every item of the round, where it goes.
//  * Items that need scores go to the item ring (producer, MMA issuer,
//    epilogue), all posted by warp 0 in order, which then ends the ring with
//    a marker: trivial items never hold a slot the tensor-core roles wait
//    behind.
//  * In a round that also holds scored items, the trivial items whose rows
//    each keep one contiguous run of visible entries -- the usual case with
//    documents -- are written by the scheduler warps themselves, so the
//    select warps spend their time on the selections: the even-ranked ones
//    of the round by warp 1 (after it has posted the round's select
//    entries), the odd-ranked ones by warp 0 in a second pass over its
//    rounds once it has posted every item (its posts keep the tensor cores
//    fed; a single warp writing them all finished last on packed inputs).
//  * Every other item is an entry of the select warps' ring; entry e is
//    posted by warp e % 2 (the slot's parity is the entry's, so every slot
//    has one writer, written in order), and the ring ends with a marker.
//    In a round of trivial items only that is every item, spread over both
//    warps and written by the four select warps.
template <class C>
__device__ void run_scheduler_docs(const KParams& p, const Smem<C>& sm, const WaitCtl& ctl, int sw) {
  constexpr int R = C::R, H = C::H;
  constexpr int NWL = (R * H + 31) / 32;  // weights per lane
  static_assert(C::DOCS && R == 4, "the document mode's scheduler");
  static_assert(C::SSLOTS % 2 == 0, "select slots alternate between the two scheduler warps");
  const uint32_t lane = lane_id();
  const Team<32> team{0u, lane};
  const bool can_trivial = p.scores == nullptr;  // no debug copy of the scores
  const int n_mine = cta_item_count<true>(p);
  int posted = 0;   // item-ring entries written (warp 0)
  int sposted = 0;  // select-ring entries of the rounds before (both warps)
  for (int it0 = 0; it0 < n_mine; it0 += 32) {
    // lane l fetches item it0 + l
    const int my_it = it0 + (int)lane;
    int b_l = 0, rb_l = 0, c_l = 0;
    long long qs_l = 0;
    int seg_l[R];
    SegInfo si_l{};
    bool scored_l = false, ctriv_l = false;
#pragma unroll
    for (int j = 0; j < R; ++j) seg_l[j] = 0;
    if (my_it < n_mine) {
      sched_coords<C>(p, my_it, n_mine, b_l, rb_l, c_l);
      if (p.q_start != nullptr) qs_l = p.q_start[b_l];
#pragma unroll
      for (int j = 0; j < R; ++j)
        if (rb_l * R + j < p.S) seg_l[j] = p.q_seg[(size_t)b_l * p.S + rb_l * R + j];
      si_l = p.seginfo[(size_t)b_l * p.n_rb + rb_l];
      bool triv = can_trivial, contig = true;
#pragma unroll
      for (int j = 0; j < R; ++j) {
        triv = triv && si_l.nvis[j] <= p.K;
        contig = contig && si_l.contig[j] != 0;
      }
      scored_l = !triv;
      ctriv_l = triv && contig;
      if (sw == 0 && scored_l) {
        // the weight rows of the item into L2: the item loop reads them
        // from there (a few hundred bytes per item)
        const size_t esz = p.w_f32 ? 4 : 2;
#pragma unroll
        for (int j = 0; j < R; ++j) {
          const int s = rb_l * R + j;
          if (s < p.S) {
            const char* a = static_cast<const char*>(p.w) + ((size_t)b_l * p.w_sb + (size_t)s * p.w_ss) * esz;
            prefetch_l2(a);
            prefetch_l2(a + H * esz - 1);
          }
        }
      }
    }
    const bool mixed = __ballot_sync(0xFFFFFFFFu, scored_l) != 0u;
    const bool w1_l = mixed && ctriv_l;  // written by the scheduler warps
    const uint32_t sel_mask = __ballot_sync(0xFFFFFFFFu, my_it < n_mine && !w1_l);
    const int cnt = min(32, n_mine - it0);
    for (int k = 0; k < cnt; ++k) {
      const bool w1 = __shfl_sync(0xFFFFFFFFu, w1_l, k);
      const bool scored = __shfl_sync(0xFFFFFFFFu, scored_l, k);
      const int e = sposted + __popc(sel_mask & ((1u << k) - 1u));  // select entry (if not w1)
      if (w1) continue;  // written by warp 1 after the round's posts
      const bool my_entry = (e & 1) == sw;
      if (!my_entry && !(sw == 0 && scored)) continue;
      const int b = __shfl_sync(0xFFFFFFFFu, b_l, k);
      const int rb = __shfl_sync(0xFFFFFFFFu, rb_l, k);
      const int c = __shfl_sync(0xFFFFFFFFu, c_l, k);
      const long long qs0 = __shfl_sync(0xFFFFFFFFu, qs_l, k);
      const int s0 = rb * R;
      int thr[R], seg[R], nvis[R], tfirst[R], contig[R];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        seg[j] = __shfl_sync(0xFFFFFFFFu, seg_l[j], k);
        nvis[j] = __shfl_sync(0xFFFFFFFFu, si_l.nvis[j], k);
        tfirst[j] = __shfl_sync(0xFFFFFFFFu, si_l.tfirst[j], k);
        contig[j] = __shfl_sync(0xFFFFFFFFu, si_l.contig[j], k);
      }
      row_bounds<R>(p, qs0, s0, thr);
      const int c_lo = c * p.chunk_tiles;
      const int c_hi = min(p.n_tiles, c_lo + p.chunk_tiles);
      const int t_lo = __shfl_sync(0xFFFFFFFFu, si_l.t_lo, k);
      const int t_hi = scored ? __shfl_sync(0xFFFFFFFFu, si_l.t_hi, k) : t_lo;
      const int trivial = scored ? 0 : 1;
      if (my_entry) {  // the select ring
        const int ss = e % C::SSLOTS;
        mbar_wait(sm.sel_empty(ss), ((e / C::SSLOTS) & 1) ^ 1, ctl);
        if (lane == 0)
          write_desc<R>(sm.sdesc(ss), b, s0, t_lo, t_hi, c_lo, c_hi, trivial, thr, seg, nvis, tfirst, contig);
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.sel_full(ss));
      }
      if (sw != 0 || !scored) continue;
      // the item ring, with the weights (fp32) of the item's rows: every
      // load in flight before the first store; rows past S get 0
      float wv[NWL];
#pragma unroll
      for (int u = 0; u < NWL; ++u) {
        const int i = (int)lane + 32 * u;
        const int j = i / H, h = i % H;
        const int s = s0 + j;
        float v = 0.f;
        if (i < R * H && s < p.S) {
          const size_t off = (size_t)b * p.w_sb + (size_t)s * p.w_ss + h;
          v = p.w_f32 ? reinterpret_cast<const float*>(p.w)[off]
                      : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.w)[off]);
        }
        wv[u] = v;
      }
      const int slot = posted % C::SLOTS;
      mbar_wait(sm.item_empty(slot), ((posted / C::SLOTS) & 1) ^ 1, ctl);
      float* ws = sm.w(slot);
#pragma unroll
      for (int u = 0; u < NWL; ++u) {
        const int i = (int)lane + 32 * u;
        if (i < R * H) ws[i] = wv[u];
      }
      if (lane == 0) write_desc<R>(sm.desc(slot), b, s0, t_lo, t_hi, c_lo, c_hi, trivial, thr, seg, nvis, tfirst, contig);
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.item_full(slot));
      ++posted;
    }
    if (sw == 1 && mixed) {
      // the round's even-ranked contiguous trivial items: each row's visible
      // entries tfirst .. tfirst + nvis - 1, -1 padded
      const uint32_t w1_mask = __ballot_sync(0xFFFFFFFFu, w1_l);
      for (int k = 0; k < cnt; ++k) {
        if (!((w1_mask >> k) & 1u) || (__popc(w1_mask & ((1u << k) - 1u)) & 1)) continue;
        const int b = __shfl_sync(0xFFFFFFFFu, b_l, k);
        const int rb = __shfl_sync(0xFFFFFFFFu, rb_l, k);
#pragma unroll
        for (int j = 0; j < R; ++j) {
          const int nv = __shfl_sync(0xFFFFFFFFu, si_l.nvis[j], k);
          const int tf = __shfl_sync(0xFFFFFFFFu, si_l.tfirst[j], k);
          const int s = rb * R + j;
          if (s < p.S)
            write_visible_set<32>(p.idx + ((size_t)b * p.S + s) * p.K, p.K, nv, tf, 1, 0, 0, nullptr, nullptr, team);
        }
      }
    }
    sposted += __popc(sel_mask);
  }
  // the end markers (b < 0): the select ring's from the warp of its
  // entry's parity, the item ring's from warp 0
  if ((sposted & 1) == sw) {
    const int ss = sposted % C::SSLOTS;
    mbar_wait(sm.sel_empty(ss), ((sposted / C::SSLOTS) & 1) ^ 1, ctl);
    if (lane == 0) sm.sdesc(ss)->b = -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.sel_full(ss));
  }
  if (sw == 0) {
    const int slot = posted % C::SLOTS;
    mbar_wait(sm.item_empty(slot), ((posted / C::SLOTS) & 1) ^ 1, ctl);
    if (lane == 0) sm.desc(slot)->b = -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.item_full(slot));
    // second pass: the odd-ranked contiguous trivial items of the rounds
    // that also hold scored items (the same classification as above)
    for (int it0 = 0; it0 < n_mine; it0 += 32) {
      const int my_it = it0 + (int)lane;
      int b_l = 0, rb_l = 0, c_l = 0;
      SegInfo si_l{};
      bool scored_l = false, ctriv_l = false;
      if (my_it < n_mine) {
        sched_coords<C>(p, my_it, n_mine, b_l, rb_l, c_l);
        si_l = p.seginfo[(size_t)b_l * p.n_rb + rb_l];
        bool triv = can_trivial, contig = true;
#pragma unroll
        for (int j = 0; j < R; ++j) {
          triv = triv && si_l.nvis[j] <= p.K;
          contig = contig && si_l.contig[j] != 0;
        }
        scored_l = !triv;
        ctriv_l = triv && contig;
      }
      if (__ballot_sync(0xFFFFFFFFu, scored_l) == 0u) continue;
      const uint32_t w1_mask = __ballot_sync(0xFFFFFFFFu, ctriv_l);
      const int cnt = min(32, n_mine - it0);
      for (int k = 0; k < cnt; ++k) {
        if (!((w1_mask >> k) & 1u) || !(__popc(w1_mask & ((1u << k) - 1u)) & 1)) continue;
        const int b = __shfl_sync(0xFFFFFFFFu, b_l, k);
        const int rb = __shfl_sync(0xFFFFFFFFu, rb_l, k);
#pragma unroll
        for (int j = 0; j < R; ++j) {
          const int nv = __shfl_sync(0xFFFFFFFFu, si_l.nvis[j], k);
          const int tf = __shfl_sync(0xFFFFFFFFu, si_l.tfirst[j], k);
          const int s = rb * R + j;
          if (s < p.S)
            write_visible_set<32>(p.idx + ((size_t)b * p.S + s) * p.K, p.K, nv, tf, 1, 0, 0, nullptr, nullptr, team);
        }
      }
    }
  }
}

template <class C>
__device__ void run_producer(const KParams& p, const Smem<C>& sm, const WaitCtl& ctl, const CUtensorMap* tq,
                             const CUtensorMap* tk) {
  uint32_t kcount = 0, qcount = 0;
  // q blocks are read once; k tiles are re-read by every row block of the
  // batch, except with single-row items (decode), where k streams once and
  // should not push the scores of the selection pass out of L2
  const uint64_t q_pol = l2_policy_evict_first();
  const uint64_t k_pol = (C::R == 1) ? l2_policy_evict_first() : l2_policy_evict_last();
  // document mode: the item ring until its end marker
  const int n_mine = C::DOCS ? 0x7FFFFFFF : cta_item_count<(C::R > 1)>(p);
  // Row-block items already posted to the item ring are looked at ahead of
  // their turn, and the q block of each one that needs scores is prefetched
  // into L2, so its load into the q buffer (which waits for the previous
  // item's products) comes from L2.  `look` is the next item to look at.
  int look = 1;
  auto look_ahead = [&](int it) {
    if constexpr (C::R > 1) {
      look = max(look, it + 1);
      const int lim = min(n_mine, it + C::SLOTS);
      for (; look < lim; ++look) {
        const int sl = look % C::SLOTS;
        if (!mbar_test_wait(sm.item_full(sl), (look / C::SLOTS) & 1)) break;
        const ItemDesc<C::R>* da = sm.desc(sl);
        if (C::DOCS && da->b < 0) break;  // the end marker
        if (da->t_hi > da->t_lo) {
#pragma unroll
          for (int c = 0; c < C::NKC; ++c) tma_prefetch_4d(tq, c * C::KC, 0, da->s0, da->b);
        }
      }
    }
  };
  for (int it = 0; it < n_mine; ++it) {
    const int slot = it % C::SLOTS;
    const bool ok_item = mbar_wait(sm.item_full(slot), (it / C::SLOTS) & 1, ctl);
    const ItemDesc<C::R>* d = sm.desc(slot);
    const int b = d->b, s0 = d->s0, t_lo = d->t_lo, t_hi = d->t_hi;
    mbar_arrive(sm.item_empty(slot));
    if (C::DOCS && (!ok_item || b < 0)) break;
    if (!ok_item || t_hi <= t_lo) {
      if (ok_item) look_ahead(it);
      continue;
    }
    const int qb = qcount % C::QBUF;
    if (mbar_wait(sm.q_empty(qb), ((qcount / C::QBUF) & 1) ^ 1, ctl)) {
      mbar_arrive_expect_tx(sm.q_full(qb), C::QBYTES);
#pragma unroll
      for (int c = 0; c < C::NKC; ++c)
        tma_load_4d_hint(sm.q(qb) + c * C::QCHUNK, tq, sm.q_full(qb), c * C::KC, 0, s0, b, q_pol);
    }
    ++qcount;
    look_ahead(it);
    for (int tile = t_lo; tile < t_hi; ++tile) {
      const int st = kcount % C::KSTAGES;
      if (mbar_wait(sm.k_empty(st), ((kcount / C::KSTAGES) & 1) ^ 1, ctl)) {
        mbar_arrive_expect_tx(sm.k_full(st), C::KBYTES);
#pragma unroll
        for (int c = 0; c < C::NKC; ++c)
          tma_load_3d_hint(sm.k(st) + c * C::KCHUNK, tk, sm.k_full(st), c * C::KC, tile * kTileT, b, k_pol);
      }
      ++kcount;
      look_ahead(it);
    }
  }
  // make sure no copy is still landing in shared memory when the CTA exits
  volatile uint32_t dummy = 0;
  const WaitCtl drain_ctl{&dummy, ctl.limit_ns};
  for (uint32_t i = 0; i < C::KSTAGES && i < kcount; ++i) {
    const uint32_t last = kcount - 1 - i;  // most recent use of stage last % KSTAGES
    mbar_wait(sm.k_full(last % C::KSTAGES), (last / C::KSTAGES) & 1, drain_ctl);
  }
  for (uint32_t i = 0; i < C::QBUF && i < qcount; ++i) {
    const uint32_t last = qcount - 1 - i;
    mbar_wait(sm.q_full(last % C::QBUF), (last / C::QBUF) & 1, drain_ctl);
  }
}

template <class C>
__device__ void run_mma(const KParams& p, const Smem<C>& sm, const WaitCtl& ctl, uint32_t tmem_base) {
  uint32_t kcount = 0, qcount = 0, acount = 0;
  // document mode: the item ring until its end marker
  const int n_mine = C::DOCS ? 0x7FFFFFFF : cta_item_count<(C::R > 1)>(p);
  for (int it = 0; it < n_mine; ++it) {
    const int slot = it % C::SLOTS;
    const bool ok_item = mbar_wait(sm.item_full(slot), (it / C::SLOTS) & 1, ctl);
    const ItemDesc<C::R>* d = sm.desc(slot);
    const int t_lo = d->t_lo, t_hi = d->t_hi;
    const int b_mark = d->b;
    mbar_arrive(sm.item_empty(slot));
    if (C::DOCS && (!ok_item || b_mark < 0)) break;
    if (!ok_item || t_hi <= t_lo) continue;
    const int qb = qcount % C::QBUF;
    const bool q_ok = mbar_wait(sm.q_full(qb), (qcount / C::QBUF) & 1, ctl);
    tc_fence_after();
    const uint32_t q_addr = smem_u32(sm.q(qb));
    for (int tile = t_lo; tile < t_hi; ++tile) {
      const int st = kcount % C::KSTAGES;
      const int a = acount & 1;
      const bool k_ok = mbar_wait(sm.k_full(st), (kcount / C::KSTAGES) & 1, ctl);
      const bool a_ok = mbar_wait(sm.acc_empty(a), ((acount >> 1) & 1) ^ 1, ctl);
      tc_fence_after();
      if (q_ok && k_ok && a_ok) {
        const uint32_t k_addr = smem_u32(sm.k(st));
        const uint32_t d_tmem = tmem_base + (uint32_t)(a * C::N);
#pragma unroll
        for (int c = 0; c < C::NKC; ++c) {
#pragma unroll
          for (int kk = 0; kk < C::KC / 16; ++kk) {
            const uint64_t adesc = smem_desc_kmajor(k_addr + c * C::KCHUNK + kk * 32, C::ROWB);
            const uint64_t bdesc = smem_desc_kmajor(q_addr + c * C::QCHUNK + kk * 32, C::ROWB);
            umma_bf16(d_tmem, adesc, bdesc, C::IDESC, (c | kk) != 0 ? 1u : 0u);
          }
        }
      }
      umma_commit(sm.k_empty(st));
      umma_commit(sm.acc_full(a));
      ++kcount;
      ++acount;
    }
    umma_commit(sm.q_empty(qb));
    ++qcount;
  }
  // every MMA issued above has completed once this barrier fires
  umma_commit(sm.drain());
  volatile uint32_t dummy = 0;
  const WaitCtl drain_ctl{&dummy, ctl.limit_ns};
  mbar_wait(sm.drain(), 0, drain_ctl);
}

// Accumulate this warp's rows over heads from one TMEM accumulator buffer.
// `loaded()` runs once every TMEM load of the buffer has completed, before
// the arithmetic on the last chunk, so the buffer can go back to the MMA
// issuer early.
template <class C, class F>
__device__ __forceinline__ void epilogue_accumulate(uint32_t t_row, const float* ws, int hf,
                                                    float (&acc)[C::RW], F&& loaded) {
  constexpr int H = C::H, RW = C::RW;
#pragma unroll
  for (int jj = 0; jj < RW; ++jj) acc[jj] = 0.f;
  if constexpr (H == 64) {
    // 2*RW chunks of 32 columns (row jj, heads hh*32 .. hh*32+31); the load
    // of the next chunk is in flight while the current one is reduced with
    // four independent packed-FMA chains
    float va[32], vb[32];
    float2 a[4];
    tmem_ld32_start(t_row + (uint32_t)(hf * RW * H), va);
    tmem_wait32(va);
#pragma unroll
    for (int c = 0; c < 2 * RW; ++c) {
      float(&cur)[32] = (c & 1) ? vb : va;
      float(&nxt)[32] = (c & 1) ? va : vb;
      if (c + 1 < 2 * RW) tmem_ld32_start(t_row + (uint32_t)(hf * RW * H + (c + 1) * 32), nxt);
      const int jj = c >> 1, hh = c & 1;
      const float4* w4 = reinterpret_cast<const float4*>(ws + (hf * RW + jj) * H + hh * 32);
      if (hh == 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) a[q] = make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 wq = w4[i];
        const float2 r0 = make_float2(fmaxf(cur[4 * i], 0.f), fmaxf(cur[4 * i + 1], 0.f));
        const float2 r1 = make_float2(fmaxf(cur[4 * i + 2], 0.f), fmaxf(cur[4 * i + 3], 0.f));
        a[(2 * i) & 3] = ffma2(make_float2(wq.x, wq.y), r0, a[(2 * i) & 3]);
        a[(2 * i + 1) & 3] = ffma2(make_float2(wq.z, wq.w), r1, a[(2 * i + 1) & 3]);
      }
      if (hh == 1)
        acc[jj] = ((a[0].x + a[0].y) + (a[1].x + a[1].y)) + ((a[2].x + a[2].y) + (a[3].x + a[3].y));
      if (c + 1 < 2 * RW) tmem_wait32(nxt);
      if (c + 2 == 2 * RW) loaded();  // the last chunk is in registers
    }
  } else {
    static_assert((C::RW * H) % 8 == 0, "small-head path loads 8 columns at a time");
#pragma unroll
    for (int c0 = 0; c0 < RW * H; c0 += 8) {
      float v[8];
      tmem_ld8(t_row + (uint32_t)(hf * RW * H + c0), v);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int col = c0 + i;
        const int jj = col / H, h = col % H;
        acc[jj] = fmaf(ws[(hf * RW + jj) * H + h], fmaxf(v[i], 0.f), acc[jj]);
      }
    }
    loaded();
  }
}

template <class C>
__device__ void run_epilogue(const KParams& p, const Smem<C>& sm, const WaitCtl& ctl, uint32_t tmem_base,
                             int e /* epilogue warp 0..EW-1 */) {
  constexpr int R = C::R, RW = C::RW;
  const uint32_t lane = lane_id();
  const int quarter = (4 + e) % 4;  // warp id % 4 selects the TMEM lane quarter
  const int hf = (C::EW == 8) ? (e / 4) : 0;
  const bool segs = p.q_seg != nullptr;
  const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
  uint32_t acount = 0, nt = 0;
  const uint64_t sc_pol = l2_policy_evict_last();
  // document mode: the item ring until its end marker
  const int n_mine = C::DOCS ? 0x7FFFFFFF : cta_item_count<(C::R > 1)>(p);
  for (int it = 0; it < n_mine; ++it) {
    const int slot = it % C::SLOTS;
    const bool ok_it = mbar_wait(sm.item_full(slot), (it / C::SLOTS) & 1, ctl);
    const ItemDesc<R>* d = sm.desc(slot);
    if (C::DOCS && (!ok_it || d->b < 0)) break;
    const int b = d->b, s0 = d->s0, t_lo = d->t_lo, t_hi = d->t_hi, c_lo = d->c_lo, c_hi = d->c_hi;
    if (C::FUSED && d->trivial) {  // the select warps write the visible sets
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.item_empty(slot));
      continue;
    }
    int thr[RW], seg[RW];
    float smin[RW], smax[RW];
    uint32_t scnt[RW];
#pragma unroll
    for (int jj = 0; jj < RW; ++jj) {
      thr[jj] = d->thr[hf * RW + jj];
      seg[jj] = d->seg[hf * RW + jj];
      smin[jj] = INFINITY;
      smax[jj] = -INFINITY;
      scnt[jj] = 0u;
    }
    const float* ws = sm.w(slot);
    float* ring_rows = nullptr;  // this item's staging slot (fused)
    const int rs = (int)(nt & 1u);
    if constexpr (C::FUSED) {
      mbar_wait(sm.ring_empty(rs), ((nt >> 1) & 1u) ^ 1u, ctl);
      ring_rows = p.ring + ((size_t)blockIdx.x * 2 + rs) * R * p.w_pad;
    }
    const bool write_all = !C::FUSED || p.scores != nullptr;
    const int tile_begin = write_all ? c_lo : t_lo;
    const int tile_end = write_all ? c_hi : t_hi;
    for (int tile = tile_begin; tile < tile_end; ++tile) {
      const bool computed = tile >= t_lo && tile < t_hi;
      const int t = tile * kTileT + quarter * 32 + (int)lane;
      float acc[RW];
#pragma unroll
      for (int jj = 0; jj < RW; ++jj) acc[jj] = 0.f;
      if (computed) {
        const int a = acount & 1;
        const bool ok = mbar_wait(sm.acc_full(a), (acount >> 1) & 1, ctl);
        tc_fence_after();
        bool released = false;
        auto release = [&]() {  // every TMEM read of accumulator a has completed
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(sm.acc_empty(a));
          released = true;
        };
        if (ok) epilogue_accumulate<C>(t_lane + (uint32_t)(a * C::N), ws, hf, acc, release);
        if (!released) release();
        ++acount;
      }
      int kvs = 0;
      if (segs && computed && t < p.W) kvs = p.kv_seg[(size_t)b * p.W + t];
#pragma unroll
      for (int jj = 0; jj < RW; ++jj) {
        const int j = hf * RW + jj;
        const int s = s0 + j;
        const bool vis = computed && t < thr[jj] && (!segs || kvs == seg[jj]);
        const float val = vis ? p.scale * acc[jj] : -INFINITY;
        if constexpr (C::FUSED) {
          if (computed) ring_rows[(size_t)j * p.w_pad + t] = val;
          if (vis) {
            smin[jj] = fminf(smin[jj], val);
            smax[jj] = fmaxf(smax[jj], val);
            scnt[jj] += 1u;
          }
        }
        if (p.scores != nullptr && s < p.S && t < p.W) {
          float* dst = p.scores + ((size_t)b * p.S + s) * p.W + t;
          if constexpr (C::R == 1)  // single-row items (decode): the selection pass re-reads them from L2
            st_global_hint(dst, val, sc_pol);
          else
            *dst = val;
        }
      }
    }
    if constexpr (C::FUSED) {  // row statistics, then hand the slot to the select warps
#pragma unroll
      for (int jj = 0; jj < RW; ++jj) {
        const uint32_t cnt = __reduce_add_sync(0xFFFFFFFFu, scnt[jj]);
        const uint32_t kmin = __reduce_min_sync(0xFFFFFFFFu, score_key(smin[jj]));
        const uint32_t kmax = __reduce_max_sync(0xFFFFFFFFu, score_key(smax[jj]));
        if (lane == 0 && cnt > 0u) {
          RowStats* st = sm.stats(rs, hf * RW + jj);
          atomicAdd(&st->nvis, cnt);
          atomicMin(&st->min_key, kmin);
          atomicMax(&st->max_key, kmax);
        }
      }
      fence_proxy_async_global();  // the staged rows are read back by a bulk copy
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.ring_full(rs));
      ++nt;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.item_empty(slot));
  }
}

// Select warp `j` (fused): selection of row j of every item.  Trivial items
// keep every visible entry; the others wait for their staged score rows,
// which one thread copies into shared memory for all R rows at once.
template <class C>
__device__ void run_selector(const KParams& p, const Smem<C>& sm, const WaitCtl& ctl, int j) {
  constexpr int R = C::R;
  constexpr uint32_t kSelBar = 6;  // named barrier of the select warps
  const uint32_t lane = lane_id();
  const Team<32> team{0u, lane};
  FusedRowScratch* fs = sm.scratch(j);
  uint32_t nt = 0;
  // document mode: the select ring until its end marker
  const int n_mine = C::DOCS ? 0x7FFFFFFF : cta_item_count<(C::R > 1)>(p);
  for (int it = 0; it < n_mine; ++it) {
    const int ss = it % C::SSLOTS;
    const bool ok_s = mbar_wait(sm.sel_full(ss), (it / C::SSLOTS) & 1, ctl);
    const ItemDesc<R>* d = sm.sdesc(ss);
    const int b = d->b, s0 = d->s0, s = s0 + j;
    const int trivial = d->trivial, t_lo = d->t_lo, t_hi = d->t_hi;
    const int nvis = d->nvis[j], tfirst = d->tfirst[j], contig = d->contig[j], thr = d->thr[j], seg = d->seg[j];
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.sel_empty(ss));
    if (C::DOCS && (!ok_s || b < 0)) break;
    int32_t* out = p.idx + ((size_t)b * p.S + s) * p.K;
    if (trivial) {
      if (s < p.S)
        write_visible_set<32>(out, p.K, nvis, tfirst, contig, thr, seg, p.kv_seg + (size_t)b * p.W, &fs->sc, team);
    } else {
      const int rs = (int)(nt & 1u);
      const int e0 = t_lo * kTileT;
      const uint32_t row_bytes = (uint32_t)(t_hi - t_lo) * kTileT * 4u;
      mbar_wait(sm.ring_full(rs), (nt >> 1) & 1u, ctl);
      if (j == 0 && lane == 0) {
        fence_proxy_async_global();
        const float* src = p.ring + ((size_t)blockIdx.x * 2 + rs) * R * p.w_pad;
        mbar_arrive_expect_tx(sm.copy_full(), row_bytes * R);
        if (row_bytes > 0u)
          for (int r = 0; r < R; ++r)
            bulk_copy_g2s(sm.srow(r, p.w_pad) + e0, src + (size_t)r * p.w_pad + e0, row_bytes, sm.copy_full());
      }
      mbar_wait(sm.copy_full(), nt & 1u, ctl);
      RowStats* stp = sm.stats(rs, j);
      const RowStats st = *stp;
      __syncwarp();
      if (lane == 0) {
        stp->nvis = 0u;
        stp->min_key = 0xFFFFFFFFu;
        stp->max_key = 0u;
      }
      named_bar_sync(kSelBar, 32 * R);  // every select warp holds its statistics
      if (j == 0 && lane == 0) mbar_arrive(sm.ring_empty(rs));
      if (s < p.S)
        team_topk_row(sm.srow(j, p.w_pad), e0, (t_hi - t_lo) * kTileT, (uint32_t)p.K, st, out, &fs->bs, &fs->sc,
                      team);
      named_bar_sync(kSelBar, 32 * R);  // the shared rows may be refilled
      ++nt;
    }
  }
}

// Long-row mode: the R select warps form one team.  Trivial items: each warp
// writes its own row's visible set.  Scored items: the team copies the
// item's staged rows into the single shared row buffer one at a time and
// selects each; the staging slot goes back to the epilogue once its last
// row has been copied.
template <class C>
__device__ void run_selector_long(const KParams& p, const Smem<C>& sm, const WaitCtl& ctl, int j) {
  constexpr int R = C::R;
  constexpr uint32_t kSelBar = 6;  // named barrier of the select team
  const uint32_t lane = lane_id();
  const Team<32> wteam{0u, lane};
  const Team<32 * R> team{kSelBar, (uint32_t)j * 32u + lane};
  LongRowScratch* ls = sm.long_scratch();
  float* srow = sm.srow(0, p.w_pad);
  uint32_t nt = 0, nc = 0;  // scored items, row copies
  const int n_mine = cta_item_count<(C::R > 1)>(p);
  for (int it = 0; it < n_mine; ++it) {
    const int ss = it % C::SSLOTS;
    mbar_wait(sm.sel_full(ss), (it / C::SSLOTS) & 1, ctl);
    const ItemDesc<R>* d = sm.sdesc(ss);
    const int b = d->b, s0 = d->s0;
    const int trivial = d->trivial, t_lo = d->t_lo, t_hi = d->t_hi;
    const int nvis = d->nvis[j], tfirst = d->tfirst[j], contig = d->contig[j], thr = d->thr[j], seg = d->seg[j];
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.sel_empty(ss));
    if (trivial) {
      const int s = s0 + j;
      if (s < p.S)
        write_visible_set<32>(p.idx + ((size_t)b * p.S + s) * p.K, p.K, nvis, tfirst, contig, thr, seg,
                              p.kv_seg + (size_t)b * p.W, &ls->sc[j], wteam);
    } else {
      const int rs = (int)(nt & 1u);
      const int e0 = t_lo * kTileT, n = (t_hi - t_lo) * kTileT;
      const uint32_t row_bytes = (uint32_t)n * 4u;
      mbar_wait(sm.ring_full(rs), (nt >> 1) & 1u, ctl);
      RowStats st[R];
#pragma unroll
      for (int r = 0; r < R; ++r) st[r] = *sm.stats(rs, r);
      team.sync();  // every thread holds the statistics
      if (team.tid == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          RowStats* stp = sm.stats(rs, r);
          stp->nvis = 0u;
          stp->min_key = 0xFFFFFFFFu;
          stp->max_key = 0u;
        }
        fence_proxy_async_global();
      }
      const float* src = p.ring + ((size_t)blockIdx.x * 2 + rs) * R * p.w_pad;
      for (int r = 0; r < R; ++r) {
        if (team.tid == 0) {
          mbar_arrive_expect_tx(sm.copy_full(), row_bytes);
          if (row_bytes > 0u) bulk_copy_g2s(srow + e0, src + (size_t)r * p.w_pad + e0, row_bytes, sm.copy_full());
        }
        mbar_wait(sm.copy_full(), nc & 1u, ctl);
        ++nc;
        if (r == R - 1 && team.tid == 0) mbar_arrive(sm.ring_empty(rs));  // every row of the slot is copied
        if (s0 + r < p.S)
          team_topk_row(srow, e0, n, (uint32_t)p.K, st[r], p.idx + ((size_t)b * p.S + s0 + r) * p.K, &ls->bs,
                        &ls->sc[0], team);
        team.sync();  // the row buffer may be refilled
      }
      ++nt;
    }
  }
}

template <class C>
__global__ void __launch_bounds__(C::NTHREADS, 1)
    csa_index_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Smem<C> sm{base};
  const int warp = threadIdx.x / 32;
  const uint32_t lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::SLOTS; ++s) {
      mbar_init(sm.item_full(s), 1);
      mbar_init(sm.item_empty(s), 2 + C::EW);  // producer, MMA issuer, epilogue warps
    }
    for (int s = 0; s < C::SSLOTS; ++s) {
      mbar_init(sm.sel_full(s), 1);
      mbar_init(sm.sel_empty(s), C::SW);
    }
    for (int i = 0; i < C::QBUF; ++i) {
      mbar_init(sm.q_full(i), 1);
      mbar_init(sm.q_empty(i), 1);
    }
    for (int i = 0; i < C::KSTAGES; ++i) {
      mbar_init(sm.k_full(i), 1);
      mbar_init(sm.k_empty(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sm.acc_full(i), 1);
      mbar_init(sm.acc_empty(i), C::EW);
    }
    mbar_init(sm.drain(), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(sm.ring_full(i), C::EW);
      mbar_init(sm.ring_empty(i), 1);
    }
    mbar_init(sm.copy_full(), 1);
    *sm.abort_flag() = 0u;
    for (int i = 0; i < 2 * C::R; ++i) {
      RowStats* st = sm.stats(i / C::R, i % C::R);
      st->nvis = 0u;
      st->min_key = 0xFFFFFFFFu;
      st->max_key = 0u;
    }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
  }
  if (warp == 1) {
    tmem_alloc(sm.tmem_slot(), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot();
  const WaitCtl ctl{sm.abort_flag(), p.wait_ns};
  // launched as a dependent (document mode, after the segment pre-pass): the
  // previous kernel's results (our inputs) are visible past this point;
  // every CTA of this single-wave grid is resident, so the next kernel may
  // start its own set-up on the SMs this one leaves
  if constexpr (C::DOCS) {
    griddep_wait();
    griddep_launch_dependents();
  }

  if (warp == 0) {
    if (lane == 0) run_producer<C>(p, sm, ctl, &tmap_q, &tmap_k);
  } else if (warp == 1) {
    if (lane == 0) run_mma<C>(p, sm, ctl, tmem_base);
  } else if (warp == 2 || warp == 3) {
    if constexpr (C::DOCS)
      run_scheduler_docs<C>(p, sm, ctl, warp - 2);
    else
      run_scheduler<C>(p, sm, ctl, warp - 2);
  } else if (warp < 4 + C::EW) {
    run_epilogue<C>(p, sm, ctl, tmem_base, warp - 4);
  } else {
    if constexpr (C::LONG)
      run_selector_long<C>(p, sm, ctl, warp - 4 - C::EW);
    else if constexpr (C::FUSED)
      run_selector<C>(p, sm, ctl, warp - 4 - C::EW);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

}  // namespace csa
