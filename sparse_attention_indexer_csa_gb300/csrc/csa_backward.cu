// csa_backward.cu -- backward of the score step on the tensor cores: two
// persistent kernels, no intermediate tensor in HBM.
//
// The score of "Add StreamIndex Kernel for CSA [Deepseek v4]" (Description) is
//   score[b,s,t] = sum_h w[b,s,h] * ReLU(scale * x),  x = q[b,h,s,:] . k[b,t,:];
// the page's custom_vjp takes the cotangent g[b,s,t] of the scores back to
//   dw[b,s,h] = sum_t gm * ReLU(scale * x)
//   P[b,h,s,t] = gm * w[b,s,h] * scale * [x > 0]
//   dq[b,h,s,:] = sum_t P * k[b,t,:]         dk[b,t,:] = sum_{h,s} P * q[b,h,s,:]
// with gm = g on visible entries and 0 on masked ones (masked scores are
// constants), and a fused kernel is asked for in that page's backward review
// (the reference vjp forms the [B,H,S,W] tensor).  Both kernels here
// recompute the logits x tile by tile and keep P on the SM:
//
//   csa_bwd_dq_kernel   item = a pair of query rows (2 rows x 64 heads = the
//                       128 TMEM lanes), walking the k tiles the pair sees:
//                         X  = Q . K^T                 (A = q block, B = k tile, smem)
//                         P  = gm * w * scale * [X > 0] in bf16, written back
//                              over X in tensor memory; dw += gm * X
//                         dQ += P . K                  (A = P in TMEM, B = k tile read MN-major)
//                       dQ stays in TMEM until the pair's last tile, then goes
//                       to dq once (fp32, q's layout).
//   csa_bwd_dk_kernel   item = one k tile (the 128 TMEM lanes are its entries)
//                       and a run of row pairs that see it:
//                         X^T = K . Q^T                (A = k tile, B = q block)
//                         P^T in bf16 over X^T in tensor memory
//                         dK += P^T . Q                (A = P^T in TMEM, B = q block read MN-major)
//                       each item's dK is added into dk with vector atomics;
//                       items are handed out through a counter in the
//                       caller's workspace.
//
// Tensor memory (512 columns): three 128-column logit buffers (X / P), so the
// products of tile n+1 run while the epilogue forms P of tile n and the
// product with P of tile n-1 is still queued, and one 128-column accumulator
// (dQ or dK).  P overwrites the first 32 columns of each 64-column half of
// its logit buffer (64 bf16 in 32 columns), which that half's warp has
// already read, so no warp writes columns another warp still reads.
//
// Warp roles (15 warps, both kernels):
//   warp 0      TMA producer (dk: also takes items from the counter and
//               publishes them to the other roles through a ring of slots)
//   warp 1      TMEM owner and issuer of the logit products (one thread)
//   warp 14     issuer of the accumulate products (one thread): the two
//               issuers own different accumulators, so the waits and
//               commits of one overlap the other's products on the pipe
//   warps 2-9   epilogue: warp w reads TMEM lanes 32*(w%4).., half w/6 of
//               each logit buffer (dq: entries 64*half.., dk: row `half` of
//               the pair)
//   warps 10-13 drain of the accumulator (lanes 32*(w%4)..)
// Every mbarrier wait is bounded; a wait that gives up raises the CTA's
// abort flag and records CSA_ERR_TIMEOUT, and the other roles stop waiting.
#include <cuda_bf16.h>

#include "csa_internal.h"

namespace csa {
namespace {

constexpr int kBH = 64, kBD = 128;
constexpr uint32_t kChunk = 128 * 128;             // 16 KB: 128 rows x 64 bf16 (one half of D)
constexpr uint32_t kBlk = 2 * kChunk;              // 32 KB: q block (2 rows x 64 heads) or k tile
constexpr int kQBufDq = 2, kKStDq = 4;             // dq kernel: q blocks, k tile stages
constexpr int kKtBufDk = 2, kQStDk = 4;            // dk kernel: k tiles, q block stages
constexpr int kXBuf = 3;                           // logit / P buffers in TMEM
constexpr uint32_t kAccCol = 384;                  // accumulator columns [384, 512)
constexpr uint32_t kTmemCols = 512;
constexpr int kThreads = 15 * 32;
constexpr int kAccWarp = 14;  // issuer of the accumulate products
constexpr int kEpiWarps = 8, kDrainWarps = 4;
constexpr int kItemSlots = 4;
constexpr uint32_t kIdescX = idesc_bf16_f32(128, 128);       // both operands K-major (K = D)
constexpr uint32_t kIdescAcc = idesc_bf16_f32_bmn(128, 128);  // B read MN-major (N = D)

// ----------------------------------------------------------------- shared layouts
// dq kernel: q blocks | k stages | g staging (8 warps x 2 x 64 fp32) |
//            dw exchange (2 x 128 fp32) | barriers | misc
constexpr uint32_t DQ_OFF_Q = 0;
constexpr uint32_t DQ_OFF_K = DQ_OFF_Q + kQBufDq * kBlk;
constexpr uint32_t DQ_OFF_G = DQ_OFF_K + kKStDq * kBlk;
constexpr uint32_t DQ_OFF_DW = DQ_OFF_G + kEpiWarps * 2 * 64 * 4;
constexpr uint32_t DQ_OFF_BAR = DQ_OFF_DW + 2 * 128 * 4;
constexpr int DQ_NBAR = 2 * kQBufDq + 2 * kKStDq + 3 * kXBuf + 3;
constexpr uint32_t DQ_OFF_MISC = DQ_OFF_BAR + DQ_NBAR * 8;
constexpr uint32_t kDqSmem = DQ_OFF_MISC + 16 + 1024;  // + alignment slack

// dk kernel: k tiles | q stages | w staging (8 warps x 2 x 64 fp32) |
//            item slots | barriers | misc
struct DkItem {
  int b, tile, p_lo, p_hi;  // b < 0: no more items
};
constexpr uint32_t DK_OFF_KT = 0;
constexpr uint32_t DK_OFF_Q = DK_OFF_KT + kKtBufDk * kBlk;
constexpr uint32_t DK_OFF_W = DK_OFF_Q + kQStDk * kBlk;
constexpr uint32_t DK_OFF_ITEM = DK_OFF_W + kEpiWarps * 2 * 64 * 4;
constexpr uint32_t DK_OFF_BAR = DK_OFF_ITEM + kItemSlots * sizeof(DkItem);
constexpr int DK_NBAR = 2 * kItemSlots + 2 * kKtBufDk + 2 * kQStDk + 3 * kXBuf + 3;
constexpr uint32_t DK_OFF_MISC = DK_OFF_BAR + DK_NBAR * 8;
constexpr uint32_t kDkSmem = DK_OFF_MISC + 16 + 1024;
static_assert(kDqSmem <= 227u * 1024u && kDkSmem <= 227u * 1024u, "shared memory budget");

// Barrier indices.
struct DqBars {
  static constexpr int q_full = 0, q_empty = q_full + kQBufDq, k_full = q_empty + kQBufDq,
                       k_empty = k_full + kKStDq, x_full = k_empty + kKStDq, p_full = x_full + kXBuf,
                       x_free = p_full + kXBuf, acc_full = x_free + kXBuf, acc_empty = acc_full + 1,
                       done = acc_empty + 1;
};
struct DkBars {
  static constexpr int item_full = 0, item_empty = item_full + kItemSlots, kt_full = item_empty + kItemSlots,
                       kt_empty = kt_full + kKtBufDk, q_full = kt_empty + kKtBufDk, q_empty = q_full + kQStDk,
                       x_full = q_empty + kQStDk, p_full = x_full + kXBuf, x_free = p_full + kXBuf,
                       acc_full = x_free + kXBuf, acc_empty = acc_full + 1, done = acc_empty + 1;
};

// ----------------------------------------------------------------- shared helpers
// Visible-entry bound of row s of batch b (future mask): entries t < thr.
// A shift replaces the division when the compress rate is a power of two;
// without offsets the position fits 32 bits.
__device__ __forceinline__ int row_thr(const BwdParams& p, int b, int s) {
  if (s >= p.S) return 0;
  if (p.q_start == nullptr) {
    const int tv = p.r_shift >= 0 ? ((s + 1) >> p.r_shift) : (s + 1) / p.r;
    return tv > p.W ? p.W : tv;
  }
  const long long pos1 = (long long)p.q_start[b] + s + 1;
  if (pos1 <= 0) return 0;
  const long long tv = p.r_shift >= 0 ? (pos1 >> p.r_shift) : pos1 / p.r;
  return tv > p.W ? p.W : (int)tv;
}

// Operand forms of the two products (M = 128, N = 128, eight K-steps of 16):
//  * logits: A and B are 128-row blocks in shared memory, K-major over D in
//    two 64-wide chunks of 128-byte swizzled rows (kChunk apart); K-step ks
//    starts 32 bytes further into each row (chunk ks / 4).
//  * accumulate: A is P in tensor memory as the epilogue leaves it -- K
//    indices 0..63 in columns x_col + 0..31, 64..127 in columns x_col + 64..95,
//    eight columns per K-step -- and B the 128-row block of the other operand
//    read MN-major: K index k is row k of the block, D contiguous within a
//    128-byte row (the two 64-wide chunks kChunk apart, 8-row groups 1024 B
//    apart), K-step ks starting 2048 bytes further.
// Descriptors are built once per buffer and advanced by the start-field
// increment (bytes / 16) of these offsets.

// Two fp32 to packed bf16 (lower index in the low half).
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void drain_waits(uint64_t* full_bars, int nbuf, uint32_t count, const WaitCtl& ctl) {
  // the most recent use of each buffer has landed: no copy still writes
  // shared memory when the CTA exits
  volatile uint32_t dummy = 0;
  const WaitCtl dctl{&dummy, ctl.limit_ns};
  for (uint32_t i = 0; i < (uint32_t)nbuf && i < count; ++i) {
    const uint32_t last = count - 1 - i;
    mbar_wait(full_bars + (last % nbuf), (last / nbuf) & 1u, dctl);
  }
}

// ======================================================================= dq
// Items of the dq kernel: item it is batch it % B and pair n_pairs-1 - it / B,
// the longest pairs (latest rows) first so the static round-robin over the
// CTAs stays balanced.  A CTA walks items it = blockIdx.x + k * gridDim.x
// with the quotient and remainder kept as running counters (no division per
// item in the issuing threads).
struct DqItem {
  int b, s0, thr0, thr1;
  int t0, T;  // the pair's k tiles: t0 .. t0 + T - 1
};
struct DqWalk {
  int it, b, q, gq, gr;
  __device__ explicit DqWalk(const BwdParams& p) : it((int)blockIdx.x) {
    gq = (int)gridDim.x / p.B;
    gr = (int)gridDim.x - gq * p.B;
    q = it / p.B;
    b = it - q * p.B;
  }
  __device__ bool more(const BwdParams& p) const { return it < p.n_items; }
  __device__ void next(const BwdParams& p) {
    it += (int)gridDim.x;
    q += gq;
    b += gr;
    if (b >= p.B) {
      b -= p.B;
      ++q;
    }
  }
  __device__ DqItem item(const BwdParams& p) const {
    DqItem d;
    d.b = b;
    d.s0 = 2 * (p.n_pairs - 1 - q);
    d.thr0 = row_thr(p, b, d.s0);
    d.thr1 = row_thr(p, b, d.s0 + 1);
    d.T = (max(d.thr0, d.thr1) + kTileT - 1) / kTileT;
    d.t0 = 0;
    if (p.seginfo != nullptr) {
      // with segment ids: only the tiles holding an entry visible to a row
      // of the pair's item of four rows (its segment summary)
      const SegInfo& si = p.seginfo[(size_t)b * p.n_rb + (d.s0 >> 2)];
      const int hi = min(d.T, si.t_hi);
      d.t0 = si.t_lo;
      d.T = hi > si.t_lo ? hi - si.t_lo : 0;
    }
    return d;
  }
};

__global__ void __launch_bounds__(kThreads, 1)
    csa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                      const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + DQ_OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + DQ_OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(base + DQ_OFF_MISC + 4);
  const int warp = threadIdx.x / 32;
  const uint32_t lane = lane_id();
  using Bq = DqBars;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQBufDq; ++i) {
      mbar_init(bars + Bq::q_full + i, 1);
      mbar_init(bars + Bq::q_empty + i, 1);
    }
    for (int i = 0; i < kKStDq; ++i) {
      mbar_init(bars + Bq::k_full + i, 1);
      // released by the accumulate product alone: it starts only after the
      // epilogue has read the tile's logits, so the logit product is done
      mbar_init(bars + Bq::k_empty + i, 1);
    }
    for (int i = 0; i < kXBuf; ++i) {
      mbar_init(bars + Bq::x_full + i, 1);
      mbar_init(bars + Bq::p_full + i, kEpiWarps);
      mbar_init(bars + Bq::x_free + i, 1);
    }
    mbar_init(bars + Bq::acc_full, 1);
    mbar_init(bars + Bq::acc_empty, kDrainWarps);
    mbar_init(bars + Bq::done, 2);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, p.wait_ns};

  if (warp == 0) {
    if (lane == 0) {  // ---------------------------------------------- TMA producer
      // The q block of the next pair is requested right after the first k
      // tile of the current one (its buffer was freed by the pair before),
      // so its load overlaps the current pair's tiles.
      const uint64_t q_pol = l2_policy_evict_first(), k_pol = l2_policy_evict_last();
      uint32_t qc = 0, kc = 0;
      auto load_q = [&](const DqItem& d) {
        const int qb = qc % kQBufDq;
        if (mbar_wait(bars + Bq::q_empty + qb, ((qc / kQBufDq) & 1u) ^ 1u, ctl)) {
          uint8_t* dst = base + DQ_OFF_Q + qb * kBlk;
          mbar_arrive_expect_tx(bars + Bq::q_full + qb, kBlk);
          for (int c = 0; c < 2; ++c)
            tma_load_4d_hint(dst + c * kChunk, &tmap_q, bars + Bq::q_full + qb, c * 64, 0, d.s0, d.b, q_pol);
        }
        ++qc;
      };
      // the next item that sees any tile
      auto skip_empty = [&](DqWalk& w) {
        while (w.more(p) && w.item(p).T == 0) w.next(p);
      };
      DqWalk wk(p);
      skip_empty(wk);
      if (wk.more(p)) load_q(wk.item(p));
      while (wk.more(p)) {
        const DqItem d = wk.item(p);
        DqWalk nx = wk;
        nx.next(p);
        skip_empty(nx);
        for (int tile = 0; tile < d.T; ++tile, ++kc) {
          const int st = kc % kKStDq;
          if (mbar_wait(bars + Bq::k_empty + st, ((kc / kKStDq) & 1u) ^ 1u, ctl)) {
            uint8_t* dst = base + DQ_OFF_K + st * kBlk;
            mbar_arrive_expect_tx(bars + Bq::k_full + st, kBlk);
            for (int c = 0; c < 2; ++c)
              tma_load_3d_hint(dst + c * kChunk, &tmap_k, bars + Bq::k_full + st, c * 64, (d.t0 + tile) * kTileT,
                               d.b, k_pol);
          }
          if (tile == 0 && nx.more(p)) load_q(nx.item(p));
        }
        wk = nx;
      }
      drain_waits(bars + Bq::k_full, kKStDq, kc, ctl);
      drain_waits(bars + Bq::q_full, kQBufDq, qc, ctl);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------- logits issuer
      // Two threads issue the products: this one X = Q . K^T, warp kAccWarp
      // the accumulate products.  Each keeps its loop short -- descriptors
      // built once and advanced by constants, ring indices wrapping with
      // explicit phase bits, barriers addressed directly -- and its waits
      // and commits overlap the other's products on the tensor pipe.
      const uint32_t bar0 = smem_u32(bars);
      const uint64_t qd0 = smem_desc_kmajor(smem_u32(base + DQ_OFF_Q), 128);
      const uint64_t kd0 = smem_desc_kmajor(smem_u32(base + DQ_OFF_K), 128);
      uint32_t qb = 0, qph = 0, kst = 0, kph = 0, xb = 0, xph = 0, n = 0;
      bool alive = true;
      for (DqWalk wk(p); wk.more(p); wk.next(p)) {
        const DqItem d = wk.item(p);
        if (d.T == 0) continue;
        alive = alive && mbar_wait_u32(bar0 + 8u * (Bq::q_full + qb), qph, ctl);
        const uint64_t qd = qd0 + (uint64_t)(qb * (kBlk >> 4));
        for (int tile = 0; tile < d.T; ++tile) {
          alive = alive && mbar_wait_u32(bar0 + 8u * (Bq::k_full + kst), kph, ctl);
          if (n >= (uint32_t)kXBuf) alive = alive && mbar_wait_u32(bar0 + 8u * (Bq::x_free + xb), xph ^ 1u, ctl);
          tc_fence_after();
          if (alive) {  // X = Q . K^T into logit buffer xb
            const uint64_t kd = kd0 + (uint64_t)(kst * (kBlk >> 4));
            const uint32_t xt = tmem + xb * 128u;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint64_t o = (uint64_t)(((ks >> 2) * kChunk + (ks & 3) * 32) >> 4);
              umma_bf16(xt, qd + o, kd + o, kIdescX, ks != 0 ? 1u : 0u);
            }
          }
          umma_commit_u32(bar0 + 8u * (Bq::x_full + xb));
          if (tile == d.T - 1) umma_commit_u32(bar0 + 8u * (Bq::q_empty + qb));
          ++n;
          if (++kst == (uint32_t)kKStDq) {
            kst = 0;
            kph ^= 1u;
          }
          if (++xb == (uint32_t)kXBuf) {
            xb = 0;
            xph ^= 1u;
          }
        }
        if (++qb == (uint32_t)kQBufDq) {
          qb = 0;
          qph ^= 1u;
        }
      }
      // both issuers' products have completed before TMEM is released
      umma_commit_u32(bar0 + 8u * Bq::done);
      volatile uint32_t dummy = 0;
      const WaitCtl dctl{&dummy, ctl.limit_ns};
      mbar_wait(bars + Bq::done, 0u, dctl);
    }
  } else if (warp < 2 + kEpiWarps) {  // ------------------------------ epilogue
    const int e = warp - 2;
    const int quarter = warp & 3;
    const int hf = e >> 2;                      // half of the tile's entries
    const int m = quarter * 32 + (int)lane;     // TMEM lane: (row j, head h)
    const int j = m >> 6, h = m & 63;
    const bool segs = p.q_seg != nullptr;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    float* gbuf = reinterpret_cast<float*>(base + DQ_OFF_G) + e * 128;
    float* dwx = reinterpret_cast<float*>(base + DQ_OFF_DW);
    uint32_t n = 0, ic = 0;
    for (DqWalk wk(p); wk.more(p); wk.next(p), ++ic) {
      const DqItem d = wk.item(p);
      const int s = d.s0 + j;
      const bool row_ok = s < p.S;
      const int thr = j ? d.thr1 : d.thr0;
      const int seg = (segs && row_ok) ? p.q_seg[(size_t)d.b * p.S + s] : 0;
      float wc = 0.f;
      if (row_ok) {
        const size_t off = (size_t)d.b * p.w_sb + (size_t)s * p.w_ss + h;
        wc = (p.w_f32 ? reinterpret_cast<const float*>(p.w)[off]
                      : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.w)[off])) *
             p.scale;
      }
      const float2 wc2 = make_float2(wc, wc);
      float2 dwa[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      // masked cotangents of row s for this warp's 64 entries of a tile (two per lane)
      auto load_g = [&](int tile) -> float2 {
        float gv[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int t = (d.t0 + tile) * kTileT + hf * 64 + 2 * (int)lane + u;
          bool vis = row_ok && t < thr;
          if (vis && segs) vis = p.kv_seg[(size_t)d.b * p.W + t] == seg;
          gv[u] = vis ? p.g[((size_t)d.b * p.S + s) * p.W + t] : 0.f;
        }
        return make_float2(gv[0], gv[1]);
      };
      float2 g_next = (d.T > 0) ? load_g(0) : make_float2(0.f, 0.f);
      for (int tile = 0; tile < d.T; ++tile, ++n) {
        const int xb = n % kXBuf;
        float* gb = gbuf + (n & 1u) * 64;
        *reinterpret_cast<float2*>(gb + 2 * lane) = g_next;
        __syncwarp();
        if (tile + 1 < d.T) g_next = load_g(tile + 1);
        const bool ok = mbar_wait(bars + Bq::x_full + xb, (n / kXBuf) & 1u, ctl);
        tc_fence_after();
        const uint32_t ta = t_lane + (uint32_t)xb * 128u + (uint32_t)hf * 64u;
        if (ok) {
          float va[32], vb[32];
          tmem_ld32_start(ta, va);
          tmem_wait32(va);
          tmem_ld32_start(ta + 32u, vb);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float(&cur)[32] = c ? vb : va;
            if (c) tmem_wait32(vb);
            uint32_t pk[16];
            const float4* g4 = reinterpret_cast<const float4*>(gb + c * 32);
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
              const float4 gq = g4[i4];
#pragma unroll
              for (int i2 = 0; i2 < 2; ++i2) {
                const int i = 2 * i4 + i2;
                const float2 x = make_float2(cur[2 * i], cur[2 * i + 1]);
                const float2 gg = i2 ? make_float2(gq.z, gq.w) : make_float2(gq.x, gq.y);
                // scale > 0: [scale*x > 0] = [x > 0]; gm * x = g * ReLU(x)
                const float2 gm = fmul2(gg, make_float2(step_pos(x.x), step_pos(x.y)));
                dwa[i & 3] = ffma2(gm, x, dwa[i & 3]);
                const float2 pv = fmul2(gm, wc2);
                pk[i] = pack_bf16(pv.x, pv.y);
              }
            }
            // entries 32c .. 32c+31 of this half -> columns 16c .. 16c+15
            // (already read: columns 0..31 hold va)
            tmem_st16(ta + 16u * (uint32_t)c, pk);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + Bq::p_full + xb);
      }
      // dw: this half's sum joins the other half's (buffers alternate by item)
      const float dw_acc =
          (((dwa[0].x + dwa[0].y) + (dwa[1].x + dwa[1].y)) + ((dwa[2].x + dwa[2].y) + (dwa[3].x + dwa[3].y))) *
          p.scale;
      float* slot = dwx + (ic & 1u) * 128;
      if (hf == 1) slot[m] = dw_acc;
      named_bar_sync(1 + quarter, 64);
      if (hf == 0 && row_ok) p.dw[((size_t)d.b * p.S + s) * kBH + h] = dw_acc + slot[m];
    }
  } else if (warp == kAccWarp) {
    if (lane == 0) {  // --------------------------------- accumulate issuer
      // dQ (+)= P . K per tile: P in the tile's logit buffer, K read MN-major
      const uint32_t bar0 = smem_u32(bars);
      const uint64_t km0 = smem_desc_mn_sw128(smem_u32(base + DQ_OFF_K), kChunk, 1024u);
      uint32_t kst = 0, xb = 0, xph = 0, ac = 0;
      bool alive = true;
      for (DqWalk wk(p); wk.more(p); wk.next(p)) {
        const DqItem d = wk.item(p);
        if (d.T == 0) continue;
        for (int tile = 0; tile < d.T; ++tile) {
          if (tile == 0) alive = alive && mbar_wait_u32(bar0 + 8u * Bq::acc_empty, (ac & 1u) ^ 1u, ctl);
          alive = alive && mbar_wait_u32(bar0 + 8u * (Bq::p_full + xb), xph, ctl);
          tc_fence_after();
          if (alive) {
            const uint32_t xa = tmem + xb * 128u;
            const uint64_t bd = km0 + (uint64_t)(kst * (kBlk >> 4));
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              umma_bf16_tmem_a(tmem + kAccCol, xa + 64u * (uint32_t)(ks >> 2) + 8u * (uint32_t)(ks & 3),
                               bd + (uint64_t)(128 * ks), kIdescAcc, (tile != 0 || ks != 0) ? 1u : 0u);
            }
          }
          umma_commit_u32(bar0 + 8u * (Bq::k_empty + kst));
          umma_commit_u32(bar0 + 8u * (Bq::x_free + xb));
          if (tile == d.T - 1) {
            umma_commit_u32(bar0 + 8u * Bq::acc_full);
            ++ac;
          }
          if (++kst == (uint32_t)kKStDq) kst = 0;
          if (++xb == (uint32_t)kXBuf) {
            xb = 0;
            xph ^= 1u;
          }
        }
      }
      umma_commit_u32(bar0 + 8u * Bq::done);
    }
  } else {  // ---------------------------------------------------------- dQ drain
    const int quarter = warp & 3;
    const int m = quarter * 32 + (int)lane;
    const int j = m >> 6, h = m & 63;
    const uint32_t t_acc = tmem + ((uint32_t)(quarter * 32) << 16) + kAccCol;
    uint32_t ac = 0;
    for (DqWalk wk(p); wk.more(p); wk.next(p)) {
      const DqItem d = wk.item(p);
      const int s = d.s0 + j;
      const bool row_ok = s < p.S;
      float* dst = p.dq + (p.dq_seq_major ? (((size_t)d.b * p.S + s) * kBH + h) * kBD
                                          : (((size_t)d.b * kBH + h) * p.S + s) * kBD);
      float4* d4 = reinterpret_cast<float4*>(dst);
      if (d.T == 0) {  // no visible entry: dq rows are zero
        if (row_ok)
          for (int i = 0; i < kBD / 4; ++i) d4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        continue;
      }
      const bool ok = mbar_wait(bars + Bq::acc_full, ac & 1u, ctl);
      tc_fence_after();
      ++ac;
      // the whole row in registers first: the accumulator goes back to the
      // accumulate issuer before any store (the stores of 32 different rows
      // per instruction throttle, and the next pair's first product waits)
      float v[4][32];
      if (ok) {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32_start(t_acc + 32u * c, v[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_wait32(v[c]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + Bq::acc_empty);
      if (ok && row_ok) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 8; ++i)
            d4[8 * c + i] = make_float4(v[c][4 * i], v[c][4 * i + 1], v[c][4 * i + 2], v[c][4 * i + 3]);
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ======================================================================= dk
// First pair of batch b that sees tile `tile`: the pair holding the first row
// s with (q_start + s + 1) / r > 128 * tile; n_pairs if none.
__device__ __forceinline__ int dk_first_pair(const BwdParams& p, int b, int tile) {
  const long long qs0 = p.q_start ? (long long)p.q_start[b] : 0ll;
  long long s_first = (long long)p.r * ((long long)tile * kTileT + 1) - qs0 - 1;
  if (s_first < 0) s_first = 0;
  if (s_first >= p.S) return p.n_pairs;
  return (int)(s_first / 2);
}

// With segment ids (a warp): narrows the pairs [lo, hi) of a dk item to the
// span from the first to the last pair whose item of four rows holds a
// visible entry in `tile` (its segment summary); lo = hi when none does.
// Pairs inside the span that see nothing form P = 0.
__device__ __forceinline__ void dk_trim(const BwdParams& p, int b, int tile, int& lo, int& hi) {
  const uint32_t lane = lane_id();
  int first = hi, last = lo - 1;
  for (int base = lo; base < hi; base += 32) {
    const int pr = base + (int)lane;
    bool in = false;
    if (pr < hi) {
      const SegInfo& si = p.seginfo[(size_t)b * p.n_rb + (pr >> 1)];
      in = tile >= si.t_lo && tile < si.t_hi;
    }
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, in);
    if (m != 0u) {
      first = min(first, base + __ffs((int)m) - 1);
      last = max(last, base + 31 - __clz((int)m));
    }
  }
  if (last < first) {
    hi = lo;
  } else {
    lo = first;
    hi = last + 1;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    csa_bwd_dk_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                      const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + DK_OFF_BAR);
  DkItem* slots = reinterpret_cast<DkItem*>(base + DK_OFF_ITEM);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + DK_OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(base + DK_OFF_MISC + 4);
  const int warp = threadIdx.x / 32;
  const uint32_t lane = lane_id();
  using Bk = DkBars;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(bars + Bk::item_full + i, 1);
      mbar_init(bars + Bk::item_empty + i, 2 + kEpiWarps + kDrainWarps);
    }
    for (int i = 0; i < kKtBufDk; ++i) {
      mbar_init(bars + Bk::kt_full + i, 1);
      mbar_init(bars + Bk::kt_empty + i, 1);
    }
    for (int i = 0; i < kQStDk; ++i) {
      mbar_init(bars + Bk::q_full + i, 1);
      // released by the accumulate product alone (see the dq kernel)
      mbar_init(bars + Bk::q_empty + i, 1);
    }
    for (int i = 0; i < kXBuf; ++i) {
      mbar_init(bars + Bk::x_full + i, 1);
      mbar_init(bars + Bk::p_full + i, kEpiWarps);
      mbar_init(bars + Bk::x_free + i, 1);
    }
    mbar_init(bars + Bk::acc_full, 1);
    mbar_init(bars + Bk::acc_empty, kDrainWarps);
    mbar_init(bars + Bk::done, 2);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, p.wait_ns};

  // Consumers read the item descriptors in order; false once there are no more.
  auto next_item = [&](uint32_t ic, DkItem& out) -> bool {
    const int slot = ic % kItemSlots;
    const bool ok = mbar_wait(bars + Bk::item_full + slot, (ic / kItemSlots) & 1u, ctl);
    out = slots[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + Bk::item_empty + slot);
    return ok && out.b >= 0;
  };

  if (warp == 0) {  // ------------------------------- scheduler + TMA producer
    // Lane 0 takes items from the counter, publishes them and issues the
    // copies; with segment ids the whole warp first trims each item's pairs.
    const uint64_t q_pol = l2_policy_evict_last(), k_pol = l2_policy_evict_last();
    const long long n_raw = (long long)p.B * p.n_chunks * p.n_tiles;
    uint32_t ic = 0, qc = 0;
    // raw item x -> (b, chunk, tile), tile fastest: the items of one chunk
    // of rows (the same q blocks) are taken one after another
    unsigned int x = 0;
    if (lane == 0) x = atomicAdd(p.counter, 1u);
    x = __shfl_sync(0xFFFFFFFFu, x, 0);
    while (__shfl_sync(0xFFFFFFFFu, *abort_flag, 0) == 0u) {  // lane 0's reading, for the whole warp
      DkItem d{-1, 0, 0, 0};
      while ((long long)x < n_raw) {
        const int tile = (int)(x % (unsigned)p.n_tiles);
        const int rest = (int)(x / (unsigned)p.n_tiles);
        const int chunk = rest % p.n_chunks, b = rest / p.n_chunks;
        unsigned int xn = 0;
        if (lane == 0) xn = atomicAdd(p.counter, 1u);  // the next one, while this one is set up
        int lo = max(chunk * p.chunk_pairs, dk_first_pair(p, b, tile));
        int hi = min((chunk + 1) * p.chunk_pairs, p.n_pairs);
        if (lo < hi && p.seginfo != nullptr) dk_trim(p, b, tile, lo, hi);
        x = __shfl_sync(0xFFFFFFFFu, xn, 0);
        if (lo < hi) {
          d = DkItem{b, tile, lo, hi};
          break;
        }
      }
      uint32_t go = 0u;
      if (lane == 0) {
        const int slot = ic % kItemSlots;
        if (mbar_wait(bars + Bk::item_empty + slot, ((ic / kItemSlots) & 1u) ^ 1u, ctl)) {
          slots[slot] = d;
          mbar_arrive(bars + Bk::item_full + slot);
          go = d.b >= 0 ? 1u : 0u;
        }
        if (go) {
          const int kb = ic % kKtBufDk;
          if (mbar_wait(bars + Bk::kt_empty + kb, ((ic / kKtBufDk) & 1u) ^ 1u, ctl)) {
            uint8_t* dst = base + DK_OFF_KT + kb * kBlk;
            mbar_arrive_expect_tx(bars + Bk::kt_full + kb, kBlk);
            for (int c = 0; c < 2; ++c)
              tma_load_3d_hint(dst + c * kChunk, &tmap_k, bars + Bk::kt_full + kb, c * 64, d.tile * kTileT, d.b,
                               k_pol);
          }
          ++ic;
          for (int pr = d.p_lo; pr < d.p_hi; ++pr, ++qc) {
            const int st = qc % kQStDk;
            if (mbar_wait(bars + Bk::q_empty + st, ((qc / kQStDk) & 1u) ^ 1u, ctl)) {
              uint8_t* dst = base + DK_OFF_Q + st * kBlk;
              mbar_arrive_expect_tx(bars + Bk::q_full + st, kBlk);
              for (int c = 0; c < 2; ++c)
                tma_load_4d_hint(dst + c * kChunk, &tmap_q, bars + Bk::q_full + st, c * 64, 0, 2 * pr, d.b, q_pol);
            }
          }
        }
      }
      if (__shfl_sync(0xFFFFFFFFu, go, 0) == 0u) break;
    }
    if (lane == 0) {
      drain_waits(bars + Bk::q_full, kQStDk, qc, ctl);
      drain_waits(bars + Bk::kt_full, kKtBufDk, ic, ctl);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------- logits issuer
      const uint32_t bar0 = smem_u32(bars);
      const uint64_t td0 = smem_desc_kmajor(smem_u32(base + DK_OFF_KT), 128);
      const uint64_t qd0 = smem_desc_kmajor(smem_u32(base + DK_OFF_Q), 128);
      uint32_t slot = 0, sph = 0, kb = 0, kbph = 0, qst = 0, qph = 0, xb = 0, xph = 0, n = 0;
      bool alive = true;
      while (true) {
        const bool have = mbar_wait_u32(bar0 + 8u * (Bk::item_full + slot), sph, ctl);
        const DkItem d = slots[slot];
        mbar_arrive(bars + Bk::item_empty + slot);
        if (++slot == (uint32_t)kItemSlots) {
          slot = 0;
          sph ^= 1u;
        }
        if (!have || d.b < 0) break;
        alive = alive && mbar_wait_u32(bar0 + 8u * (Bk::kt_full + kb), kbph, ctl);
        const uint64_t ad = td0 + (uint64_t)(kb * (kBlk >> 4));
        for (int pr = d.p_lo; pr < d.p_hi; ++pr) {
          alive = alive && mbar_wait_u32(bar0 + 8u * (Bk::q_full + qst), qph, ctl);
          if (n >= (uint32_t)kXBuf) alive = alive && mbar_wait_u32(bar0 + 8u * (Bk::x_free + xb), xph ^ 1u, ctl);
          tc_fence_after();
          if (alive) {  // X^T = K . Q^T into logit buffer xb
            const uint64_t bd = qd0 + (uint64_t)(qst * (kBlk >> 4));
            const uint32_t xt = tmem + xb * 128u;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint64_t o = (uint64_t)(((ks >> 2) * kChunk + (ks & 3) * 32) >> 4);
              umma_bf16(xt, ad + o, bd + o, kIdescX, ks != 0 ? 1u : 0u);
            }
          }
          umma_commit_u32(bar0 + 8u * (Bk::x_full + xb));
          if (pr == d.p_hi - 1) umma_commit_u32(bar0 + 8u * (Bk::kt_empty + kb));
          ++n;
          if (++qst == (uint32_t)kQStDk) {
            qst = 0;
            qph ^= 1u;
          }
          if (++xb == (uint32_t)kXBuf) {
            xb = 0;
            xph ^= 1u;
          }
        }
        if (++kb == (uint32_t)kKtBufDk) {
          kb = 0;
          kbph ^= 1u;
        }
      }
      umma_commit_u32(bar0 + 8u * Bk::done);
      volatile uint32_t dummy = 0;
      const WaitCtl dctl{&dummy, ctl.limit_ns};
      mbar_wait(bars + Bk::done, 0u, dctl);
    }
  } else if (warp < 2 + kEpiWarps) {  // ------------------------------ epilogue
    const int e = warp - 2;
    const int quarter = warp & 3;
    const int jr = e >> 2;  // row of the pair whose 64 heads this warp takes
    const bool segs = p.q_seg != nullptr;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    float* wbuf = reinterpret_cast<float*>(base + DK_OFF_W) + e * 128;
    uint32_t ic = 0, n = 0;
    DkItem d;
    while (next_item(ic, d)) {
      ++ic;
      const int t = d.tile * kTileT + quarter * 32 + (int)lane;  // this thread's entry
      const bool t_ok = t < p.W;
      const int kvs = (segs && t_ok) ? p.kv_seg[(size_t)d.b * p.W + t] : 0;
      // masked cotangent of (row, t) and the row's weights times scale (two per lane)
      auto load_row = [&](int pr, float& gm, float2& w2) {
        const int s = 2 * pr + jr;
        gm = 0.f;
        w2 = make_float2(0.f, 0.f);
        if (s < p.S) {
          bool vis = t < row_thr(p, d.b, s);
          if (vis && segs) vis = p.q_seg[(size_t)d.b * p.S + s] == kvs;
          if (vis) gm = p.g[((size_t)d.b * p.S + s) * p.W + t];
          const size_t off = (size_t)d.b * p.w_sb + (size_t)s * p.w_ss + 2 * lane;
          float w0, w1;
          if (p.w_f32) {
            w0 = reinterpret_cast<const float*>(p.w)[off];
            w1 = reinterpret_cast<const float*>(p.w)[off + 1];
          } else {
            w0 = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.w)[off]);
            w1 = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.w)[off + 1]);
          }
          w2 = make_float2(w0 * p.scale, w1 * p.scale);
        }
      };
      float gm_next;
      float2 w_next;
      load_row(d.p_lo, gm_next, w_next);
      for (int pr = d.p_lo; pr < d.p_hi; ++pr, ++n) {
        const int xb = n % kXBuf;
        const float gm = gm_next;
        float* wb = wbuf + (n & 1u) * 64;
        *reinterpret_cast<float2*>(wb + 2 * lane) = w_next;
        __syncwarp();
        if (pr + 1 < d.p_hi) load_row(pr + 1, gm_next, w_next);
        const bool ok = mbar_wait(bars + Bk::x_full + xb, (n / kXBuf) & 1u, ctl);
        tc_fence_after();
        const uint32_t ta = t_lane + (uint32_t)xb * 128u + (uint32_t)jr * 64u;
        if (ok) {
          if (__any_sync(0xFFFFFFFFu, gm != 0.f)) {
            float va[32], vb[32];
            tmem_ld32_start(ta, va);
            tmem_wait32(va);
            tmem_ld32_start(ta + 32u, vb);
            const float2 gm2 = make_float2(gm, gm);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              float(&cur)[32] = c ? vb : va;
              if (c) tmem_wait32(vb);
              uint32_t pk[16];
              const float4* w4 = reinterpret_cast<const float4*>(wb + c * 32);
#pragma unroll
              for (int i4 = 0; i4 < 8; ++i4) {
                const float4 wq = w4[i4];
#pragma unroll
                for (int i2 = 0; i2 < 2; ++i2) {
                  const int i = 2 * i4 + i2;
                  const float2 ww = i2 ? make_float2(wq.z, wq.w) : make_float2(wq.x, wq.y);
                  const float2 st2 = make_float2(step_pos(cur[2 * i]), step_pos(cur[2 * i + 1]));
                  const float2 pv = fmul2(fmul2(gm2, ww), st2);
                  pk[i] = pack_bf16(pv.x, pv.y);
                }
              }
              tmem_st16(ta + 16u * (uint32_t)c, pk);
            }
          } else {  // no visible entry in this warp's 32 x 64 block: P = 0
            uint32_t zk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) zk[i] = 0u;
            tmem_st16(ta, zk);
            tmem_st16(ta + 16u, zk);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + Bk::p_full + xb);
      }
    }
  } else if (warp == kAccWarp) {
    if (lane == 0) {  // --------------------------------- accumulate issuer
      // dK (+)= P^T . Q per pair: P^T in the pair's logit buffer, Q read MN-major
      const uint32_t bar0 = smem_u32(bars);
      const uint64_t qm0 = smem_desc_mn_sw128(smem_u32(base + DK_OFF_Q), kChunk, 1024u);
      uint32_t slot = 0, sph = 0, qst = 0, xb = 0, xph = 0, ac = 0;
      bool alive = true;
      while (true) {
        const bool have = mbar_wait_u32(bar0 + 8u * (Bk::item_full + slot), sph, ctl);
        const DkItem d = slots[slot];
        mbar_arrive(bars + Bk::item_empty + slot);
        if (++slot == (uint32_t)kItemSlots) {
          slot = 0;
          sph ^= 1u;
        }
        if (!have || d.b < 0) break;
        for (int pr = d.p_lo; pr < d.p_hi; ++pr) {
          if (pr == d.p_lo) alive = alive && mbar_wait_u32(bar0 + 8u * Bk::acc_empty, (ac & 1u) ^ 1u, ctl);
          alive = alive && mbar_wait_u32(bar0 + 8u * (Bk::p_full + xb), xph, ctl);
          tc_fence_after();
          if (alive) {
            const uint32_t xa = tmem + xb * 128u;
            const uint64_t bd = qm0 + (uint64_t)(qst * (kBlk >> 4));
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              umma_bf16_tmem_a(tmem + kAccCol, xa + 64u * (uint32_t)(ks >> 2) + 8u * (uint32_t)(ks & 3),
                               bd + (uint64_t)(128 * ks), kIdescAcc, (pr != d.p_lo || ks != 0) ? 1u : 0u);
          }
          umma_commit_u32(bar0 + 8u * (Bk::q_empty + qst));
          umma_commit_u32(bar0 + 8u * (Bk::x_free + xb));
          if (pr == d.p_hi - 1) {
            umma_commit_u32(bar0 + 8u * Bk::acc_full);
            ++ac;
          }
          if (++qst == (uint32_t)kQStDk) qst = 0;
          if (++xb == (uint32_t)kXBuf) {
            xb = 0;
            xph ^= 1u;
          }
        }
      }
      umma_commit_u32(bar0 + 8u * Bk::done);
    }
  } else {  // ---------------------------------------------------------- dK drain
    const int quarter = warp & 3;
    const uint32_t t_acc = tmem + ((uint32_t)(quarter * 32) << 16) + kAccCol;
    uint32_t ic = 0, ac = 0;
    DkItem d;
    while (next_item(ic, d)) {
      ++ic;
      const int t = d.tile * kTileT + quarter * 32 + (int)lane;
      const bool ok = mbar_wait(bars + Bk::acc_full, ac & 1u, ctl);
      tc_fence_after();
      ++ac;
      float* dst = p.dk + ((size_t)d.b * p.W + t) * kBD;
      // the whole row in registers, the accumulator released, then the adds
      float v[4][32];
      if (ok) {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32_start(t_acc + 32u * c, v[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_wait32(v[c]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + Bk::acc_empty);
      if (ok && t < p.W) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 8; ++i)
            red_add_f32x4(dst + 32 * c + 4 * i, v[c][4 * i], v[c][4 * i + 1], v[c][4 * i + 2], v[c][4 * i + 3]);
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

size_t backward_kernel_smem() { return kDqSmem > kDkSmem ? kDqSmem : kDkSmem; }

cudaError_t launch_backward(const CUtensorMap& tq, const CUtensorMap& tk, const BwdParams& bp, int sms,
                            cudaStream_t stream) {
  cudaError_t e = smem_limit_once<csa_bwd_dq_kernel>((int)kDqSmem);
  if (e != cudaSuccess) return e;
  e = smem_limit_once<csa_bwd_dk_kernel>((int)kDkSmem);
  if (e != cudaSuccess) return e;
  // dk accumulates the items' partial sums; the item counter starts at 0
  e = cudaMemsetAsync(bp.dk, 0, (size_t)bp.B * bp.W * kBD * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(bp.counter, 0, sizeof(unsigned int), stream);
  if (e != cudaSuccess) return e;
  const int grid_dq = bp.n_items < sms ? bp.n_items : sms;
  csa_bwd_dq_kernel<<<grid_dq, kThreads, kDqSmem, stream>>>(tq, tk, bp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  csa_bwd_dk_kernel<<<sms, kThreads, kDkSmem, stream>>>(tq, tk, bp);
  return cudaGetLastError();
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
