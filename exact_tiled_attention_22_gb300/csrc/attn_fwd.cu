// attn_fwd.cu -- forward attention kernel for sm_103a.
//
// Computes O = softmax(s Q K^T [causal mask]) V and LSE per query row, one
// CTA per (pair of 128-row query tiles, batch, head).  The K/V loop follows
// the blockwise softmax of page "突破单卡显存极限：FlashAttention-2技术解析与实战
// 指南", section 2.1 (running max m, running sum l, rescale by
// exp(m_old - m_new)), with normalisation by l deferred to the end (page
// "FlashAttention-2：GPU利用率从50%干到90%", improvement 2: reorganise the
// normalisation so most work stays in matrix products).  Query tiles are spread
// over CTAs as well as batch x head (same page, improvement 1: parallelise over
// the sequence length), and each query row is owned by one thread from start
// to end (improvement 3: independent rows, little synchronisation).
//
// sm_103a mapping (our design, not the pages'):
//   warp 8     TMA producer: Q0, Q1 once; K_j, V_j through a ring of slots.
//   warp 9     MMA issuer:   S_t = Q_t K_j^T and O_t += P_t V_j with tcgen05,
//                            fp32 accumulators in tensor memory (TMEM).
//   warp 10    waiter:       every mbarrier wait the issuer depends on,
//                            handed over at a named barrier, so the issuer
//                            never stalls the tensor pipe on one.
//   warps 0-3  softmax for query tile 0, warps 4-7 for tile 1: one thread per
//              row (= TMEM lane), exp2 with the scale folded into one FMA,
//              P written back to TMEM over S as 16-bit, O rescaled in TMEM.
//   The two tiles ping-pong: while one warpgroup does its softmax the tensor
//   core works on the other tile.
//
// The running max used as the exponent reference is only moved when a new
// tile's max exceeds it by more than kTau (log2 units).  Until then P values
// are at most 2^kTau, fine in fp32 and in the 16-bit P; O and l always share
// the same reference, so the result is the same exact attention.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dropout.cuh"
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

// Warp roles: softmax warps first, then the producer, the MMA issuer and the
// waiter.  One softmax warpgroup per query tile (8 softmax warps; query tile
// t = warp / 4), except in the dropout variant: two per tile, one per half
// of the score columns (16 softmax warps; t = warp / 8, column half
// hc = (warp / 4) % 2), which spreads the generator's integer work over
// twice the warps.  The TMEM lane quadrant of a softmax warp is warp % 4.
template <bool SPLIT>
struct FwdRoles {
  static constexpr int kSoft = SPLIT ? 16 : 8;
  static constexpr int kProducer = kSoft, kMma = kSoft + 1, kWaiter = kSoft + 2;
  static constexpr int kThreads = (kSoft + 3) * 32;
};
constexpr uint32_t kHandoffBar = 1;  // named barrier: waiter -> MMA issuer
constexpr uint32_t kTileBar0 = 2;    // named barriers 2, 3: the two column halves of tile 0, 1
constexpr float kTau = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

template <int D>
struct FwdLayout {
  static constexpr int kSub = 128 * 128;    // one 64-column box: 128 rows x 128 B
  static constexpr int kNSub = D / 64;
  static constexpr int kTile = 128 * D * 2;  // a 128-row Q, K or V tile
  static constexpr int kSlots = D == 128 ? 4 : 6;
  static constexpr int kQ0 = 0;
  static constexpr int kSlot0 = 2 * kTile;
  static constexpr int kBar = kSlot0 + kSlots * kTile;
  // barriers
  static constexpr int kBarQ = 0;
  static constexpr int kBarKVFull = 1;
  static constexpr int kBarKVEmpty = kBarKVFull + kSlots;
  static constexpr int kBarSFull = kBarKVEmpty + kSlots;  // [2]
  static constexpr int kBarPFull = kBarSFull + 2;         // [tile][half]: 2 x 2
  static constexpr int kBarOFull = kBarPFull + 4;         // [2]
  static constexpr int kBarDrain = kBarOFull + 2;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  // block-sparse variant: the K/V tiles the pair visits (int16) and, per
  // tile, which of the two query tiles keeps it (bit t); then len, count0
  static constexpr int kListTile = kTmemSlot + 16;
  static constexpr int kListFlag = kListTile + 2 * kMaxSparseTiles;
  static constexpr int kListLen = kListFlag + kMaxSparseTiles;
  // partial row maxima and sums exchanged by the two column halves of a
  // query tile: [2 parities][2 tiles][2 halves][128 rows] fp32
  static constexpr int kXch = kListLen + 16;
  static constexpr int kBytes = kXch + 2 * 2 * 2 * 128 * 4;
  static constexpr int kSmem = kBytes + 1024;  // slack to align the base to 1 KiB
  // TMEM columns (512 allocated)
  static constexpr int kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
};

// ALIBI: add the linear bias -m_h |i - j| (m_h = p.alibi[h]) to the scaled
// scores, the ALiBi of page "FlashAttention技术解析：如何让GPT训练速度提升5-9倍",
// section 4.1.
//
// SPARSE: block-sparse mask (page "FlashAttention技术解析：如何让GPT训练速度提升
// 5-9倍", section 5.2): p.bmask[h][qb][kb] = 0 removes the 128 x 128 block of
// query block qb and key block kb.  The pair visits only the K/V tiles that
// either of its query tiles keeps ("positions"); a tile kept by one query
// tile only is fully masked for the other.
//
// DROPOUT: each probability is kept or dropped by the Philox decision of
// dropout.cuh (p.drop); the row sum l takes every probability (LSE is that
// of the scores), O takes the kept ones and is scaled by 256 / t at the end.
//
// ACC (with none of the above): the epilogue merges this call's (O, LSE) into
// the running fp32 accumulators p.o_acc, p.lse instead of storing O: with
// L_old the accumulated LSE and L_new this call's, the merged LSE is
// log(e^L_old + e^L_new) and the merged output the weighted mean
// (e^L_old O_old + e^L_new O_new) / (e^L_old + e^L_new), exact because each
// O is a softmax-weighted mean over its own keys (the block recurrence of
// page "突破单卡显存极限", section 2.1, applied to whole key ranges).  On the
// last partial the merged O is written as 16-bit to p.o.
template <int D, bool BF16, bool ALIBI, bool SPARSE, bool DROPOUT, bool ACC = false>
__global__ void __launch_bounds__(FwdRoles<DROPOUT>::kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ FwdArgs p) {
  static_assert(!ACC || !(ALIBI || SPARSE || DROPOUT), "the accumulating variant is plain only");
  constexpr int kWarpProducer = FwdRoles<DROPOUT>::kProducer;
  constexpr int kWarpMma = FwdRoles<DROPOUT>::kMma;
  constexpr int kWarpWaiter = FwdRoles<DROPOUT>::kWaiter;
  using L = FwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // (launched with programmatic serialization: nothing touches global
  // memory before the previous kernel on the stream has completed)
  griddep_wait();
  const int BH = p.B * p.H;
  const int n_pairs = (p.N + 255) / 256;
  const int pair = p.causal ? (n_pairs - 1 - (int)(blockIdx.x / BH)) : (int)(blockIdx.x / BH);
  const int bh = blockIdx.x % BH;
  const int b = bh / p.H, h = bh % p.H;
  const int q0 = pair * 256;
  const int n_kv_all = (p.N + 127) / 128;
  const int n0 = p.causal ? min(2 * pair + 1, n_kv_all) : n_kv_all;
  const int n1 = p.causal ? min(2 * pair + 2, n_kv_all) : n_kv_all;
  const WaitCtl wc{p.wait.status, p.wait.limit_ns};

  auto bar = [&](int i) -> uint32_t { return base + L::kBar + 8u * i; };
  auto slot_addr = [&](int s) -> uint32_t { return base + L::kSlot0 + s * L::kTile; };

  int16_t* list_tile = reinterpret_cast<int16_t*>(sbase + L::kListTile);
  uint8_t* list_flag = sbase + L::kListFlag;
  int* list_len = reinterpret_cast<int*>(sbase + L::kListLen);
  // With ALiBi the pair visits its K/V tiles nearest first: the bias is
  // largest (0) at the diagonal, so the first tile sets each row's running
  // max and the later ones rarely move it (no O rescale per tile).  Causal:
  // descending j.  Otherwise outward from the pair's diagonal tiles c0, c1,
  // alternating sides while both have tiles.  Order k -> tile:
  auto alibi_tile = [&](int k) -> int {
    if (p.causal) return n1 - 1 - k;
    const int c0 = min(2 * pair, n_kv_all - 1), c1 = c0 + 1;
    const int left = c0 + 1, right = n_kv_all - c1, m = min(left, right);
    if (k < 2 * m) return (k & 1) ? c1 + (k >> 1) : c0 - (k >> 1);
    return left > right ? c0 - (k - m) : c1 + (k - m);
  };
  // K/V tile index of position j (the pair's j-th visited tile)
  auto kv_tile = [&](int j) -> int {
    return SPARSE ? (int)list_tile[j] : (ALIBI ? alibi_tile(j) : j);
  };
  // whether query tile t keeps the tile at position j (else it is fully
  // masked for that query tile)
  auto tile_kept = [&](int j, int t) -> bool {
    if constexpr (SPARSE) return ((list_flag[j] >> t) & 1) != 0;
    if constexpr (ALIBI) return t == 1 || alibi_tile(j) < n0;
    return true;
  };

  // The producer's lane initialises the barriers and issues the Q tiles and
  // the first ring's worth of K/V loads before the block-wide barrier, so
  // that their latency overlaps the TMEM allocation and the barrier.
  if (SPARSE && warp == kWarpProducer) {
    // Positions: tiles j < n1 kept by query tile 0 (j < n0) or 1.  In
    // order of j (without ALiBi) tile 0's tiles (j < n0) come first and it
    // takes the first count0 positions; in ALiBi's nearest-first order
    // (alibi_tile) tile 0 takes every position, those it does not keep fully
    // masked.  The producer warp reads both mask rows (all loads in flight
    // at once) and compacts them with ballots.
    constexpr int kW = kMaxSparseTiles / 32;
    const uint8_t* mk = p.bmask + (size_t)h * n_kv_all * n_kv_all;
    const int qb0 = 2 * pair, qb1 = 2 * pair + 1;
    uint8_t v0[kW], v1[kW];
    int jt[kW];
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const int k = w * 32 + lane;
      const int j = k < n1 ? (ALIBI ? alibi_tile(k) : k) : 0;
      jt[w] = j;
      v0[w] = (k < n1 && j < n0) ? mk[(size_t)qb0 * n_kv_all + j] : 0;
      v1[w] = (k < n1 && qb1 < n_kv_all) ? mk[(size_t)qb1 * n_kv_all + j] : 0;
    }
    int len = 0, cnt0 = 0;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const bool a0 = v0[w] != 0, a1 = v1[w] != 0;
      const uint32_t bal = __ballot_sync(0xffffffffu, a0 || a1);
      if (a0 || a1) {
        const int pos = len + __popc(bal & ((1u << lane) - 1u));
        list_tile[pos] = (int16_t)jt[w];
        list_flag[pos] = (uint8_t)((a0 ? 1 : 0) | (a1 ? 2 : 0));
      }
      cnt0 += __popc(__ballot_sync(0xffffffffu, (a0 || a1) && jt[w] < n0));
      len += __popc(bal);
    }
    if (lane == 0) {
      list_len[0] = len;
      list_len[1] = ALIBI ? len : cnt0;
    }
    __syncwarp();
  }
  if (warp == kWarpProducer && lane == 0) {
    const int n_early = min(L::kSlots, 2 * (SPARSE ? list_len[0] : n1));
    mbar_init(bar(L::kBarQ), 1);
    for (int s = 0; s < L::kSlots; ++s) {
      mbar_init(bar(L::kBarKVFull + s), 1);
      mbar_init(bar(L::kBarKVEmpty + s), 256);  // released by one warpgroup of each tile
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(L::kBarSFull + t), 1);
      // P half 0 ready: 128 arrivals of the tile's warpgroup; with two
      // warpgroups per tile (dropout) also column half 1 done rescaling its
      // O columns (O += P V writes all of O).  P half 1: 128.
      mbar_init(bar(L::kBarPFull + 2 * t + 0), DROPOUT ? 256 : 128);
      mbar_init(bar(L::kBarPFull + 2 * t + 1), 128);
      mbar_init(bar(L::kBarOFull + t), 1);
    }
    mbar_init(bar(L::kBarDrain), 1);
    fence_mbar_init();
    // (a pair with no position loads nothing: no copy may be left in flight)
    if (!(p.debug_flags & 1) && n_early > 0) {
      tma_prefetch(&p.tm_q);
      tma_prefetch(&p.tm_k);
      tma_prefetch(&p.tm_v);
      mbar_expect_tx(bar(L::kBarQ), 2 * L::kTile);
      for (int t = 0; t < 2; ++t)
        for (int s = 0; s < L::kNSub; ++s)
          tma_load_4d(base + L::kQ0 + t * L::kTile + s * L::kSub, &p.tm_q, bar(L::kBarQ),
                      s * 64, h, q0 + t * 128, b);
      for (int i = 0; i < n_early; ++i) {  // every slot starts empty
        mbar_expect_tx(bar(L::kBarKVFull + i), L::kTile);
        for (int s = 0; s < L::kNSub; ++s)
          tma_load_4d(slot_addr(i) + s * L::kSub, (i & 1) ? &p.tm_v : &p.tm_k,
                      bar(L::kBarKVFull + i), s * 64, h, kv_tile(i >> 1) * 128, b);
      }
    }
  }
  if (warp == kWarpProducer) {
    __syncwarp();
    tmem_alloc(base + L::kTmemSlot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sbase + L::kTmemSlot);
  // positions visited by the pair, and by query tile 0 (a prefix of them)
  const int len = SPARSE ? list_len[0] : n1;
  const int cnt0 = SPARSE ? list_len[1] : (ALIBI ? n1 : n0);
  const int n_early = min(L::kSlots, 2 * len);  // loads the producer issued before the barrier

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !(p.debug_flags & 1)) {
      int issued = n_early;
      bool ok = true;
      for (int j = n_early / 2; j < len && ok; ++j) {
        for (int kind = 0; kind < 2; ++kind) {
          const int slot = issued % L::kSlots;
          const uint32_t ph = (issued / L::kSlots) & 1;
          if (!mbar_wait(bar(L::kBarKVEmpty + slot), ph ^ 1, wc)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar(L::kBarKVFull + slot), L::kTile);
          const CUtensorMap* m = kind ? &p.tm_v : &p.tm_k;
          for (int s = 0; s < L::kNSub; ++s)
            tma_load_4d(slot_addr(slot) + s * L::kSub, m, bar(L::kBarKVFull + slot), s * 64, h,
                        kv_tile(j) * 128, b);
          ++issued;
        }
      }
      if (!ok) {
        // Let every copy already issued land before shared memory goes away.
        mbar_wait_drain(bar(L::kBarQ), 0, wc.limit_ns);
        for (int i = max(0, issued - L::kSlots); i < issued; ++i)
          mbar_wait_drain(bar(L::kBarKVFull + i % L::kSlots), (i / L::kSlots) & 1, wc.limit_ns);
      }
    }
  } else if (warp == kWarpWaiter) {
    // ------------------------------------------------------------ waiter
    // Performs every mbarrier wait the MMA issuer depends on, in the issuer's
    // order, and hands each one over at a named barrier (see named_bar_and).
    auto w = [&](int i, uint32_t parity) { return mbar_wait(bar(i), parity, wc); };
    // (no position at all: nothing is loaded and the MMA warp skips too)
    bool ok = len > 0 && named_bar_and(kHandoffBar, 64,
                                       __all_sync(0xffffffffu, w(L::kBarQ, 0) && w(L::kBarKVFull + 0, 0)));
    for (int j = 0; ok && j < len; ++j) {
      const int vi = 2 * j + 1, ki = 2 * j + 2;
      const bool more = j + 1 < len;
      auto kv = [&](int i) { return w(L::kBarKVFull + i % L::kSlots, (i / L::kSlots) & 1); };
      // A_lo: V_j, first half of P_0(j)
      bool r = kv(vi);
      if (j < cnt0) r = r && w(L::kBarPFull + 0, j & 1);
      ok = named_bar_and(kHandoffBar, 64, __all_sync(0xffffffffu, r));
      if (!ok) break;
      // A_hi: second half of P_0(j), K_{j+1} for S_0(j+1)
      r = true;
      if (j < cnt0) r = w(L::kBarPFull + 1, j & 1);
      if (j + 1 < cnt0) r = r && kv(ki);
      ok = named_bar_and(kHandoffBar, 64, __all_sync(0xffffffffu, r));
      if (!ok) break;
      // B_lo: first half of P_1(j)
      ok = named_bar_and(kHandoffBar, 64, __all_sync(0xffffffffu, w(L::kBarPFull + 2, j & 1)));
      if (!ok) break;
      // B_hi: second half of P_1(j), K_{j+1} for S_1(j+1)
      r = w(L::kBarPFull + 3, j & 1);
      if (more) r = r && kv(ki);
      ok = named_bar_and(kHandoffBar, 64, __all_sync(0xffffffffu, r));
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the schedule, converged; one elected lane
    // issues (MMAs and commits inside elect.sync, no branch around them).  This warp touches no
    // mbarrier before its last MMA: it learns that operands are ready at the
    // named-barrier hand-offs with the waiter warp.
    constexpr uint32_t idesc_s = make_idesc(BF16, 128, 128, false, false);
    constexpr uint32_t idesc_o = make_idesc(BF16, 128, D, false, true);
    // S_t = Q_t K^T : A = Q (K-major), B = K (K-major), K dimension = d.
    auto issue_s = [&](int t, uint32_t kaddr) {
      const uint32_t qaddr = base + L::kQ0 + t * L::kTile;
      const uint32_t dS = tmem + (t ? L::kColS1 : L::kColS0);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t off = (ks >> 2) * L::kSub + (ks & 3) * 32;
        mma_ss(dS, make_sdesc(qaddr + off, 16, 1024), make_sdesc(kaddr + off, 16, 1024), idesc_s,
               ks > 0);
      }
    };
    // O_t += P_t V : A = P (TMEM, 16-bit over S), B = V (MN-major, N = d).
    // Keys [64 * half, 64 * half + 64) of the tile: K steps 4 * half .. + 3.
    // Their P lies over S columns 32 * half .. + 31 (one warpgroup per
    // tile), or 64 * half .. + 31 (dropout: each column half's P over that
    // half's own S).
    auto issue_pv = [&](int t, uint32_t vaddr, bool acc, int half) {
      const uint32_t dO = tmem + (t ? L::kColO1 : L::kColO0);
      const uint32_t aP = tmem + (t ? L::kColS1 : L::kColS0) + (DROPOUT ? 64 : 32) * half;
#pragma unroll
      for (int ks = 4 * half; ks < 4 * half + 4; ++ks)
        mma_ts(dO, aP + (ks & 3) * 8, make_sdesc(vaddr + ks * 2048, L::kSub, 1024), idesc_o,
               (acc || ks > 0) ? 1u : 0u);
    };
    bool ok = len > 0 && named_bar_and(kHandoffBar, 64, true);
    if (ok) {
      tc_fence_after();
      if (cnt0 > 0) {
        issue_s(0, slot_addr(0));
        tc_commit(bar(L::kBarSFull + 0));
      }
      issue_s(1, slot_addr(0));
      tc_commit(bar(L::kBarSFull + 1));
    }
    for (int j = 0; ok && j < len; ++j) {
      const int vi = 2 * j + 1, ki = 2 * j + 2;
      const int vslot = vi % L::kSlots, kslot = ki % L::kSlots;
      const bool more = j + 1 < len;
      // Each tile's P arrives in two halves (keys 0-63, 64-127), so the first
      // half of O_t += P_t V_j overlaps the softmax of the second half.
      // A_lo: V_j loaded, first half of P_0(j) written
      ok = named_bar_and(kHandoffBar, 64, true);
      if (!ok) break;
      if (j < cnt0) {
        tc_fence_after();
        issue_pv(0, slot_addr(vslot), j > 0, 0);
      }
      // A_hi: second half of P_0(j) written (and K_{j+1} loaded)
      ok = named_bar_and(kHandoffBar, 64, true);
      if (!ok) break;
      if (j < cnt0) {
        tc_fence_after();
        issue_pv(0, slot_addr(vslot), true, 1);
        if (j + 1 < cnt0) {
          issue_s(0, slot_addr(kslot));
          tc_commit(bar(L::kBarSFull + 0));
        } else {
          tc_commit(bar(L::kBarOFull + 0));
        }
      }
      // B_lo: first half of P_1(j) written
      ok = named_bar_and(kHandoffBar, 64, true);
      if (!ok) break;
      tc_fence_after();
      issue_pv(1, slot_addr(vslot), j > 0, 0);
      // B_hi: second half of P_1(j) written (and K_{j+1} loaded)
      ok = named_bar_and(kHandoffBar, 64, true);
      if (!ok) break;
      tc_fence_after();
      issue_pv(1, slot_addr(vslot), true, 1);
      if (more) {
        issue_s(1, slot_addr(kslot));
        tc_commit(bar(L::kBarSFull + 1));
      } else {
        tc_commit(bar(L::kBarOFull + 1));
      }
    }
    // Every MMA issued above completes before tensor memory is released.
    tc_commit(bar(L::kBarDrain));
    mbar_wait_drain(bar(L::kBarDrain), 0, wc.limit_ns);
  } else if constexpr (DROPOUT) {
    // ------------------------------------------------------------ softmax
    // Two warpgroups per query tile, on the same 128 rows (TMEM lanes): hc = 0
    // takes score columns 0-63 of each K/V tile, hc = 1 columns 64-127.  Per
    // tile they exchange their partial row maxima through shared memory at a
    // named barrier (which also ANDs their give-up flags, so that a wait
    // that gives up in one cannot strand the other).  Each warpgroup reads
    // its S columns twice from TMEM (for the max, then 32 columns at a time
    // for the exponentials, which keeps the registers low enough for 19
    // warps) and writes its P over its own first 32 S columns.  Each keeps
    // a partial row sum; the two are added at the end.  O rescales and
    // stores are split by O columns.
    const int t = warp >> 3, hc = (warp >> 2) & 1, qd = warp & 3;
    const int c0 = hc * 64;  // first score column of this warpgroup
    const int row_lo = q0 + t * 128;
    const int rl = qd * 32 + lane;  // row within the tile (TMEM lane)
    const int row = row_lo + rl;
    const int n_t = t ? len : cnt0;  // positions this query tile takes
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const uint32_t tS = tmem + lane_off + (t ? L::kColS1 : L::kColS0) + c0;
    const uint32_t tO = tmem + lane_off + (t ? L::kColO1 : L::kColO0) + hc * (D / 2);
    const uint32_t tile_bar = kTileBar0 + t;
    float* xch = reinterpret_cast<float*>(sbase + L::kXch);  // [par][t][hc][row]
    auto xch_at = [&](int par, int half) -> float* { return xch + ((par * 2 + t) * 2 + half) * 128 + rl; };
    const float c = p.scale * kLog2e;
    const int lim = p.causal ? min(row + 1, p.N) : p.N;  // keys < lim are visible
    const float slope2 = ALIBI ? p.alibi[h] * kLog2e : 0.f;  // ALiBi slope, log2 units
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    // K/V ring slots are handed back to the producer by column half 0 of
    // both tiles (256 arrivals): S_t of tile j complete means K_j has been
    // read and the PV_t of tile j-1, issued before it, has read V_{j-1}.
    // Query tile 0 takes only the first cnt0 positions; tile 1 takes all of
    // them and arrives for tile 0 too on the rest, so that every
    // warpgroup's arrivals on a slot stay in the order of the slot's phases.
    auto release = [&](int pos, int load_index) {
      if (hc == 0)
        mbar_arrive_n(bar(L::kBarKVEmpty + load_index % L::kSlots), (t == 1 && pos >= cnt0) ? 2u : 1u);
    };
    // Scores of columns c0 + 32 k .. + 31 (loaded into v), masked and, with
    // ALiBi, scaled and biased (s * scale * log2 e - m |row - key|, log2
    // units; linear in the column unless the 32 keys straddle the row).
    auto fix_chunk = [&](int k, int kv0, bool kept, uint32_t* v) {
      const int kc = kv0 + c0 + 32 * k;  // key of the chunk's first column
      if ((SPARSE || ALIBI) && !kept) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(-INFINITY);  // block removed
      }
      if ((kc + 32 > p.N) || (p.causal && kc + 31 > row_lo)) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (kc + i >= lim) v[i] = __float_as_uint(-INFINITY);
      }
      if constexpr (ALIBI) {
        const int r0 = row - kc;
        const bool left = __all_sync(0xffffffffu, r0 >= 31), right = __all_sync(0xffffffffu, r0 <= 0);
        if (left || right) {
          // bias of columns (i, i + 1) = (i, i + 1) k1 + k0, in four
          // independent paired chains that step by 8 columns
          const float k1 = left ? slope2 : -slope2, k0 = -k1 * (float)r0;
          const float2 c2v = make_float2(c, c), step = make_float2(8.f * k1, 8.f * k1);
          float2 bias[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            bias[q] = make_float2(fmaf((float)(2 * q), k1, k0), fmaf((float)(2 * q + 1), k1, k0));
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const int q = (i >> 1) & 3;
            const float2 r =
                fma2(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), c2v, bias[q]);
            v[i] = __float_as_uint(r.x);
            v[i + 1] = __float_as_uint(r.y);
            bias[q] = add2(bias[q], step);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            v[i] = __float_as_uint(fmaf(__uint_as_float(v[i]), c, -slope2 * fabsf((float)(r0 - i))));
        }
      }
    };
    for (int j = 0; j < n_t; ++j) {
      // dropout: bit i of keep[k] keeps column c0 + 32 k + i of this tile
      // (drawn before the wait for S, off its critical path)
      uint32_t keep[2];
      if constexpr (DROPOUT) {
        const uint32_t g0 = (uint32_t)kv_tile(j) * 8 + (uint32_t)(c0 >> 4);  // 16-key groups
#pragma unroll
        for (int w = 0; w < 2; ++w)
          keep[w] = keep_bits16(p.drop, bh, row, g0 + 2 * w) |
                    (keep_bits16(p.drop, bh, row, g0 + 2 * w + 1) << 16);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarSFull + t), j & 1, wc));
      const int kv0 = kv_tile(j) * 128;
      const bool kept = tile_kept(j, t);
      float mx = -INFINITY;
      if (ok) {
        release(j, 2 * j);                       // K_j
        if (j > 0) release(j - 1, 2 * j - 1);    // V_{j-1}
        tc_fence_after();
        uint32_t v[64];
        tmem_ld32(tS, v);
        tmem_ld32(tS + 32, v + 32);
        tmem_ld_wait();
        reg_fence<64>(v);
        fix_chunk(0, kv0, kept, v);
        fix_chunk(1, kv0, kept, v + 32);
        // partial row max: eight independent accumulators, two values a step
        float mk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mk[k] = max3(__uint_as_float(v[k]), __uint_as_float(v[8 + k]), __uint_as_float(v[16 + k]));
#pragma unroll
        for (int i = 24; i < 56; i += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mk[k] = max3(mk[k], __uint_as_float(v[i + k]), __uint_as_float(v[i + 8 + k]));
#pragma unroll
        for (int k = 0; k < 8; ++k) mk[k] = fmaxf(mk[k], __uint_as_float(v[56 + k]));
        mx = max3(max3(mk[0], mk[1], mk[2]), max3(mk[3], mk[4], mk[5]), fmaxf(mk[6], mk[7]));
        *xch_at(j & 1, hc) = mx;
      }
      // Both halves of the tile meet: the partial maxima are visible.
      ok = named_bar_and(tile_bar, 256, ok);
      if (!ok) break;
      mx = fmaxf(mx, *xch_at(j & 1, hc ^ 1));
      const float m_tile = ALIBI ? mx : mx * c;  // with ALiBi the scale is already applied
      float alpha = 1.f;
      if (m_tile > m_ref + kTau) {
        alpha = ex2(m_ref - m_tile);  // 0 on the first tile (m_ref = -inf)
        m_ref = m_tile;
      }
      const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // this half's O columns <- alpha O; the PV of tile j-1 has completed
        // (it was issued before the S of tile j whose completion we waited for)
#pragma unroll 1
        for (int cc = 0; cc < D / 2; cc += 32) {
          uint32_t o[32];
          tmem_ld32(tO + cc, o);
          tmem_ld_wait();
          reg_fence<32>(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tO + cc, o);
        }
        tmem_st_wait();
      }
      if (hc == 1) {  // O += P V (issued on P half 0) may now write this half's O columns
        tc_fence_before();
        mbar_arrive(bar(L::kBarPFull + 2 * t + 0));
      }
      // Exponents and the partial row sum on column pairs (paired fp32
      // instructions), 32 columns at a time; their P goes over the S columns
      // already read (chunk k's 16 packed columns at 16 k).
      const float2 c2 = make_float2(c, c), neg2 = make_float2(neg, neg);
      float2 sk[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};  // independent partial sums
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        uint32_t v[32];
        tmem_ld32(tS + 32 * k, v);
        tmem_ld_wait();
        reg_fence<32>(v);
        fix_chunk(k, kv0, kept, v);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 sv = make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          const float2 x = ALIBI ? add2(sv, neg2) : fma2(sv, c2, neg2);
          const float2 e = make_float2(ex2(x.x), ex2(x.y));
          sk[i & 3] = add2(sk[i & 3], e);
          if constexpr (DROPOUT) {
            const uint32_t kw = keep[k];
            pk[i] = pack2<BF16>(((kw >> (2 * i)) & 1u) ? e.x : 0.f, ((kw >> (2 * i + 1)) & 1u) ? e.y : 0.f);
          } else {
            pk[i] = pack2<BF16>(e.x, e.y);
          }
        }
        tmem_st16(tS + 16 * k, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(L::kBarPFull + 2 * t + hc));
      const float2 s01 = add2(add2(sk[0], sk[1]), add2(sk[2], sk[3]));
      l = l * alpha + (s01.x + s01.y);
    }
    // (a query tile with no position has no O_t to wait for: it writes O = 0)
    if (ok && n_t > 0) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarOFull + t), 0, wc));
    if (ok) *xch_at(n_t & 1, hc) = l;  // this half's row sum (parity slot unused by the last tile)
    ok = named_bar_and(tile_bar, 256, ok);
    if (ok) {
      l += *xch_at(n_t & 1, hc ^ 1);
      // the last PV of this tile has read V_{n_t-1}
      if (n_t > 0) release(n_t - 1, 2 * n_t - 1);
      tc_fence_after();
      // a row that saw no key (possible only under a block-sparse mask) has
      // O = 0 and LSE = -inf
      const float inv_l = l > 0.f ? (DROPOUT ? p.drop.scale : 1.f) / l : 0.f;
      const bool valid = row < p.N;
      uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                      ((((size_t)b * p.N + (valid ? row : 0)) * p.H + h) * D + hc * (D / 2)) * 2;
#pragma unroll 1
      for (int cc = 0; cc < D / 2; cc += 32) {
        uint32_t o[32];
        if (n_t > 0) {
          tmem_ld32(tO + cc, o);
          tmem_ld_wait();
          reg_fence<32>(o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l,
                             __uint_as_float(o[2 * i + 1]) * inv_l);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 2);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (valid && hc == 0)
        p.lse[(size_t)bh * p.N + row] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
    }
  
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2, qd = warp & 3;
    const int row_lo = q0 + t * 128;
    const int row = row_lo + qd * 32 + lane;
    const int n_t = t ? len : cnt0;  // positions this query tile takes
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const uint32_t tS = tmem + lane_off + (t ? L::kColS1 : L::kColS0);
    const uint32_t tO = tmem + lane_off + (t ? L::kColO1 : L::kColO0);
    const float c = p.scale * kLog2e;
    const int lim = p.causal ? min(row + 1, p.N) : p.N;  // keys < lim are visible
    const float slope2 = ALIBI ? p.alibi[h] * kLog2e : 0.f;  // ALiBi slope, log2 units
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    // K/V ring slots are handed back to the producer by both warpgroups
    // (256 arrivals): S_t of tile j complete means K_j has been read and the
    // PV_t of tile j-1, issued before it, has read V_{j-1}.  Query tile 0
    // takes only the first cnt0 positions; tile 1 takes all of them and
    // arrives for tile 0 too on the rest, so that every warpgroup's arrivals
    // on a slot stay in the order of the slot's phases.
    auto release = [&](int pos, int load_index) {
      mbar_arrive_n(bar(L::kBarKVEmpty + load_index % L::kSlots), (t == 1 && pos >= cnt0) ? 2u : 1u);
    };
    for (int j = 0; j < n_t; ++j) {
      // dropout: bit c of keep[c / 32] keeps column c of this tile (drawn
      // before the wait for S, off its critical path)
      uint32_t keep[4];
      if constexpr (DROPOUT) {
        const uint32_t g0 = (uint32_t)kv_tile(j) * 8;  // the tile's 16-key groups
#pragma unroll
        for (int w = 0; w < 4; ++w)
          keep[w] = keep_bits16(p.drop, bh, row, g0 + 2 * w) |
                    (keep_bits16(p.drop, bh, row, g0 + 2 * w + 1) << 16);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarSFull + t), j & 1, wc));
      if (!ok) break;
      release(j, 2 * j);                       // K_j
      if (j > 0) release(j - 1, 2 * j - 1);    // V_{j-1}
      tc_fence_after();
      uint32_t s[128];
      tmem_ld32(tS + 0, s);
      tmem_ld32(tS + 32, s + 32);
      tmem_ld32(tS + 64, s + 64);
      tmem_ld32(tS + 96, s + 96);
      tmem_ld_wait();
      reg_fence<128>(s);
      const int kv0 = kv_tile(j) * 128;
      if ((SPARSE || ALIBI) && !tile_kept(j, t)) {
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] = __float_as_uint(-INFINITY);  // block removed
      }
      const bool need_mask = (kv0 + 128 > p.N) || (p.causal && kv0 + 127 > row_lo);
      if (need_mask) {
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (kv0 + i >= lim) s[i] = __float_as_uint(-INFINITY);
      }
      if constexpr (ALIBI) {
        // s <- s * scale * log2(e) - m |row - key| (log2 units).  On a tile
        // wholly left (or right) of the diagonal the bias is linear in the
        // column; only the diagonal tile needs |.| per element.
        const int r0 = row - kv0;
        const bool left = __all_sync(0xffffffffu, r0 >= 127), right = __all_sync(0xffffffffu, r0 <= 0);
        if (left || right) {
          // bias of columns (i, i + 1) = (i, i + 1) k1 + k0, carried in four
          // independent paired chains that step by 8 columns
          const float k1 = left ? slope2 : -slope2, k0 = -k1 * (float)r0;
          const float2 c2v = make_float2(c, c), step = make_float2(8.f * k1, 8.f * k1);
          float2 bias[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            bias[q] = make_float2(fmaf((float)(2 * q), k1, k0), fmaf((float)(2 * q + 1), k1, k0));
#pragma unroll
          for (int i = 0; i < 128; i += 2) {
            const int q = (i >> 1) & 3;
            const float2 r = fma2(make_float2(__uint_as_float(s[i]), __uint_as_float(s[i + 1])), c2v, bias[q]);
            s[i] = __float_as_uint(r.x);
            s[i + 1] = __float_as_uint(r.y);
            bias[q] = add2(bias[q], step);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            s[i] = __float_as_uint(
                fmaf(__uint_as_float(s[i]), c, -slope2 * fabsf((float)(r0 - i))));
        }
      }
      // Row max with eight independent accumulators (a single running max
      // would be a 128-long dependency chain), two new values per step.
      float mk[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mk[k] = max3(__uint_as_float(s[k]), __uint_as_float(s[8 + k]), __uint_as_float(s[16 + k]));
#pragma unroll
      for (int i = 24; i < 120; i += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mk[k] = max3(mk[k], __uint_as_float(s[i + k]), __uint_as_float(s[i + 8 + k]));
#pragma unroll
      for (int k = 0; k < 8; ++k) mk[k] = fmaxf(mk[k], __uint_as_float(s[120 + k]));
      const float mx = max3(max3(mk[0], mk[1], mk[2]), max3(mk[3], mk[4], mk[5]), fmaxf(mk[6], mk[7]));
      const float m_tile = ALIBI ? mx : mx * c;  // with ALiBi the scale is already applied
      float alpha = 1.f;
      if (m_tile > m_ref + kTau) {
        alpha = ex2(m_ref - m_tile);  // 0 on the first tile (m_ref = -inf)
        m_ref = m_tile;
      }
      const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O_t <- alpha O_t; the PV of tile j-1 has completed (it was issued
        // before the S of tile j whose completion we waited for).
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t o[32];
          tmem_ld32(tO + cc, o);
          tmem_ld_wait();
          reg_fence<32>(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tO + cc, o);
        }
      }
      // Exponents and row sums on column pairs (paired fp32 instructions);
      // P goes back over S as 16-bit in two halves, each handed to the MMA
      // warp as soon as it is in TMEM (after the O rescale above).
      const float2 c2 = make_float2(c, c), neg2 = make_float2(neg, neg);
      float2 sk[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};  // independent partial sums
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int cp = 32 * half + i;  // column pair
          const float2 sv = make_float2(__uint_as_float(s[2 * cp]), __uint_as_float(s[2 * cp + 1]));
          const float2 x = ALIBI ? add2(sv, neg2) : fma2(sv, c2, neg2);
          const float2 e = make_float2(ex2(x.x), ex2(x.y));
          sk[i & 3] = add2(sk[i & 3], e);
          if constexpr (DROPOUT) {
            const uint32_t kw = keep[cp >> 4];
            const int b0 = (2 * cp) & 31;
            pk[i] = pack2<BF16>(((kw >> b0) & 1u) ? e.x : 0.f, ((kw >> (b0 + 1)) & 1u) ? e.y : 0.f);
          } else {
            pk[i] = pack2<BF16>(e.x, e.y);
          }
        }
        tmem_st32(tS + 32 * half, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(L::kBarPFull + 2 * t + half));
      }
      const float2 s01 = add2(add2(sk[0], sk[1]), add2(sk[2], sk[3]));
      l = l * alpha + (s01.x + s01.y);
    }
    // (a query tile with no position has no O_t to wait for: it writes O = 0)
    if (ok && n_t > 0) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarOFull + t), 0, wc));
    if (ok) {
      // the last PV of this tile has read V_{n_t-1}
      if (n_t > 0) release(n_t - 1, 2 * n_t - 1);
      tc_fence_after();
      // a row that saw no key (possible only under a block-sparse mask) has
      // O = 0 and LSE = -inf
      const float inv_l = l > 0.f ? (DROPOUT ? p.drop.scale : 1.f) / l : 0.f;
      const bool valid = row < p.N;
      uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                      ((((size_t)b * p.N + (valid ? row : 0)) * p.H + h) * D) * 2;
      if constexpr (ACC) {
        // Merge with the accumulated (O, LSE) of earlier calls, in log2 units.
        const bool first = (p.acc_flags & kAccFirst) != 0, last = (p.acc_flags & kAccLast) != 0;
        const size_t lrow = (size_t)bh * p.N + (valid ? row : 0);
        const float l2_new = l > 0.f ? m_ref + __log2f(l) : -INFINITY;
        const float l2_old = (first || !valid) ? -INFINITY : p.lse[lrow] * kLog2e;
        const float mm = fmaxf(l2_old, l2_new);
        float w_old = 0.f, w_new = 0.f, lse_out = -INFINITY;
        if (mm != -INFINITY) {
          const float e_old = ex2(l2_old - mm), e_new = ex2(l2_new - mm);  // ex2(-inf) = 0
          const float inv_s = 1.f / (e_old + e_new);
          w_old = e_old * inv_s;
          w_new = e_new * inv_s * inv_l;
          lse_out = (mm + __log2f(e_old + e_new)) * kLn2;
        }
        float* arow = p.o_acc + (((size_t)b * p.N + (valid ? row : 0)) * p.H + h) * D;
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t o[32];
          tmem_ld32(tO + cc, o);
          tmem_ld_wait();
          reg_fence<32>(o);
          float x[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(o[i]) * w_new;
          if (!first && valid) {
            const float4* a4 = reinterpret_cast<const float4*>(arow + cc);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 a = a4[i];
              x[4 * i] = fmaf(a.x, w_old, x[4 * i]);
              x[4 * i + 1] = fmaf(a.y, w_old, x[4 * i + 1]);
              x[4 * i + 2] = fmaf(a.z, w_old, x[4 * i + 2]);
              x[4 * i + 3] = fmaf(a.w, w_old, x[4 * i + 3]);
            }
          }
          if (valid && last) {
            uint4* dst = reinterpret_cast<uint4*>(orow + cc * 2);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pack2<BF16>(x[8 * i], x[8 * i + 1]), pack2<BF16>(x[8 * i + 2], x[8 * i + 3]),
                                  pack2<BF16>(x[8 * i + 4], x[8 * i + 5]),
                                  pack2<BF16>(x[8 * i + 6], x[8 * i + 7]));
          } else if (valid) {
            float4* a4 = reinterpret_cast<float4*>(arow + cc);
#pragma unroll
            for (int i = 0; i < 8; ++i) a4[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
          }
        }
        if (valid) p.lse[lrow] = lse_out;
      } else {
      // O/l rounded to 16-bit into this tile's Q buffer (no S of the tile
      // reads Q any more: its last S completed before its last P), laid out
      // as the TMA store reads it (64-column boxes of 128 rows x 128 bytes,
      // 128-byte swizzle), then one TMA store per box; rows past N are
      // clipped by the store.
      uint8_t* stage = sbase + L::kQ0 + t * L::kTile;
      const int rl = qd * 32 + lane;
#pragma unroll 1
      for (int cc = 0; cc < D; cc += 32) {
        uint32_t o[32];
        if (n_t > 0) {
          tmem_ld32(tO + cc, o);
          tmem_ld_wait();
          reg_fence<32>(o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int col = cc + 8 * i, chunk = (col & 63) >> 3;
          uint4* dst = reinterpret_cast<uint4*>(stage + (col >> 6) * L::kSub + rl * 128 + ((chunk ^ (rl & 7)) * 16));
          *dst = make_uint4(pack2<BF16>(__uint_as_float(o[8 * i]) * inv_l, __uint_as_float(o[8 * i + 1]) * inv_l),
                            pack2<BF16>(__uint_as_float(o[8 * i + 2]) * inv_l, __uint_as_float(o[8 * i + 3]) * inv_l),
                            pack2<BF16>(__uint_as_float(o[8 * i + 4]) * inv_l, __uint_as_float(o[8 * i + 5]) * inv_l),
                            pack2<BF16>(__uint_as_float(o[8 * i + 6]) * inv_l, __uint_as_float(o[8 * i + 7]) * inv_l));
        }
      }
      if (valid) p.lse[(size_t)bh * p.N + row] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
      fence_proxy_async_smem();
      }
    }
    if constexpr (!ACC) {
      // The tile's four warps meet (agreeing on whether all of them got
      // here without giving up), then one thread stores the staged O.
      if (named_bar_and(kTileBar0 + t, 128, ok) && qd == 0 && lane == 0) {
        for (int bx = 0; bx < L::kNSub; ++bx)
          tma_store_4d(&p.tm_o, base + L::kQ0 + t * L::kTile + bx * L::kSub, bx * 64, h, row_lo, b);
        bulk_commit();
        bulk_wait_all();  // shared memory stays until the store has read it
      }
    }
  
  }
  if (threadIdx.x == 0) griddep_launch_dependents();  // (see launch_pdl)
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpProducer) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool BF16, bool ALIBI, bool SPARSE, bool DROPOUT, bool ACC = false>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t stream) {
  using L = FwdLayout<D>;
  auto* k = attn_fwd_kernel<D, BF16, ALIBI, SPARSE, DROPOUT, ACC>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(((a.N + 255) / 256) * a.B * a.H);
  e = launch_pdl(k, grid, FwdRoles<DROPOUT>::kThreads, L::kSmem, stream, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int fwd_smem_bytes(int d) {
  return d == 128 ? FwdLayout<128>::kSmem : FwdLayout<64>::kSmem;
}

template <bool ALIBI, bool SPARSE, bool DROPOUT>
cudaError_t launch_fwd_v(const FwdArgs& a, cudaStream_t stream) {
  if (a.d == 128)
    return a.bf16 ? launch_fwd_t<128, true, ALIBI, SPARSE, DROPOUT>(a, stream)
                  : launch_fwd_t<128, false, ALIBI, SPARSE, DROPOUT>(a, stream);
  return a.bf16 ? launch_fwd_t<64, true, ALIBI, SPARSE, DROPOUT>(a, stream)
                : launch_fwd_t<64, false, ALIBI, SPARSE, DROPOUT>(a, stream);
}

template <bool DROPOUT>
cudaError_t launch_fwd_d(const FwdArgs& a, cudaStream_t stream) {
  if (a.bmask)
    return a.alibi ? launch_fwd_v<true, true, DROPOUT>(a, stream) : launch_fwd_v<false, true, DROPOUT>(a, stream);
  return a.alibi ? launch_fwd_v<true, false, DROPOUT>(a, stream) : launch_fwd_v<false, false, DROPOUT>(a, stream);
}

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  return a.drop.t < 256 ? launch_fwd_d<true>(a, stream) : launch_fwd_d<false>(a, stream);
}

cudaError_t launch_fwd_acc(const FwdArgs& a, cudaStream_t stream) {
  if (a.d == 128)
    return a.bf16 ? launch_fwd_t<128, true, false, false, false, true>(a, stream)
                  : launch_fwd_t<128, false, false, false, false, true>(a, stream);
  return a.bf16 ? launch_fwd_t<64, true, false, false, false, true>(a, stream)
                : launch_fwd_t<64, false, false, false, false, true>(a, stream);
}

}  // namespace attn
