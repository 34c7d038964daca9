// attn_bwd.cu -- backward attention kernels for sm_103a.
//
// The pages describe the backward only as "recompute instead of store": the
// score and probability blocks are regenerated from Q, K and the stored
// softmax statistic (page "Flash Attention V2大模型时代的算力救星", section 3.2;
// page "突破单卡显存极限：FlashAttention-2技术解析与实战指南", sections 1 and
// 2.2).  The gradient formulas are the calculus of O = softmax(s Q K^T) V for
// L = sum(O * dO):
//   P = exp(s Q K^T - LSE),  dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),
//   dS = P * (dP - D),       dK = s dS^T Q,  dQ = s dS K.
//
// Three kernels, all on the caller's stream:
//   attn_bwd_pre   D = rowsum(dO * O) and -LSE * log2(e) per row into the
//                  workspace (padded rows get D = 0 and -inf, so their P is
//                  0), and zero the fp32 dQ accumulator.  HBM-bound.
//   attn_bwd_main  one CTA per (128-key block, b, h), parallel over key blocks;
//                  K_j and V_j stay in shared memory while the CTA walks the
//                  64-row query blocks i (causal: only i whose rows reach the
//                  key block).  Per query block, five tcgen05 contractions:
//                    S^T  = K Q_i^T  (A = K in TMEM),  dP^T = V dO_i^T
//                    dV  += P^T dO_i,  dK  += dS^T Q_i      (A from TMEM)
//                    dQ_i^T = K^T dS^T                      (smem x smem)
//                  dQ_i is added into the fp32 accumulator by bulk
//                  reduce-adds; dK, dV are stored once at the end.
//   attn_dq_post   dQ = s * accumulator, rounded to the input type.
//
// Roles in attn_bwd_main (15 warps): warp 12 TMA producer; warp 13 MMA
// issuer; warp 14 waiter (every mbarrier wait the issuer depends on, handed
// over at a named barrier so the issuer never stalls on one); warps 0-3 and
// 4-7 two warpgroups on the same 128 key rows (TMEM lanes), each computing
// P^T and dS^T for half of the query columns; warps 8-11 draining dQ from
// TMEM into the accumulator (and storing dK at the end).
//
// Template variants of attn_bwd_main (the plain kernel is unchanged by
// them): ALIBI folds a per-head linear bias into the per-query LSE term;
// SPARSE visits only the query blocks a block mask keeps; DROPOUT redraws
// the forward's Philox decisions (dropout.cuh) for P in dV and for dP, with
// four P/dS warpgroups of a quarter of the query columns each (23 warps:
// P/dS 0-15, drain 16-19, producer 20, issuer 21, waiter 22).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dropout.cuh"
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.44269504088896340736f;
// Warp roles of attn_bwd_main_kernel with NWG P/dS warpgroups: warps
// 0 .. 4 NWG - 1 compute P^T and dS^T, the next four drain dQ (and store dK),
// then the producer, the MMA issuer and the waiter.
template <int NWG>
struct BwdRoles {
  static constexpr int kPds = 4 * NWG;
  static constexpr int kDrain0 = kPds;
  static constexpr int kProducer = kPds + 4, kMma = kPds + 5, kWaiter = kPds + 6;
  static constexpr int kThreads = (kPds + 7) * 32;
};
// P/dS warpgroups per variant: the dropout variant spreads its Philox work
// over four (16 query columns each), the others use two (32 columns each).
template <bool DROPOUT>
struct BwdNwg {
  static constexpr int value = DROPOUT ? 4 : 2;
};
constexpr uint32_t kHandoffBar = 1;  // named barrier: waiter -> MMA issuer
constexpr uint32_t kDrainBar = 2;    // named barrier of the four dQ drain warps
constexpr uint32_t kPdsBar = 3;      // named barrier of the P/dS warps (dV store)

template <int D, int NWG = 2>
struct BwdLayout {
  static constexpr int BQ = 64;                   // query rows per step
  static constexpr int CW = BQ / NWG;             // query columns per P/dS warpgroup
  static constexpr int NSB = 1;                   // S^T buffers in TMEM
  static constexpr int kStages = D == 128 ? 3 : 4;
  static constexpr int kNSub = D / 64;
  static constexpr int kSubKV = 128 * 128;  // 64-column box of a 128-row tile
  static constexpr int kSubQ = BQ * 128;    // 64-column box of a BQ-row tile
  static constexpr int kKV = 128 * D * 2;
  static constexpr int kQT = BQ * D * 2;
  static constexpr int kDSsub = 128 * 128;  // dS^T: 128 key rows x 64 queries
  static constexpr int kK = 0;
  static constexpr int kV = kKV;
  static constexpr int kStage0 = 2 * kKV;  // stage s: Q at +0, dO at +kQT
  static constexpr int kDS = kStage0 + kStages * 2 * kQT;  // 2 buffers of kDSBytes
  static constexpr int kDSBytes = 128 * BQ * 2;
  static constexpr int kDQ = kDS + 2 * kDSBytes;   // dQ tile staged for the bulk reduce
  static constexpr int kDQBytes = BQ * D * 4;        // fp32, row-major like the accumulator
  static constexpr int kLse = kDQ + kDQBytes;        // [kStages][BQ] fp32
  static constexpr int kDv = kLse + kStages * BQ * 4;
  static constexpr int kBar = kDv + kStages * BQ * 4;
  static constexpr int kBarKV = 0;
  static constexpr int kBarQFull = 1;
  static constexpr int kBarQEmpty = kBarQFull + kStages;
  static constexpr int kBarSFull = kBarQEmpty + kStages;  // [2]
  static constexpr int kBarPFull = kBarSFull + 2;         // [2]
  static constexpr int kBarDPFull = kBarPFull + 2;
  static constexpr int kBarDSFull = kBarDPFull + 1;   // dS^T written to TMEM
  static constexpr int kBarDSSmem = kBarDSFull + 1;   // [2] dS^T written to shared memory
  static constexpr int kBarDQFull = kBarDSSmem + 2;
  static constexpr int kBarDQEmpty = kBarDQFull + 1;
  static constexpr int kBarDKV = kBarDQEmpty + 1;
  static constexpr int kBarKTmem = kBarDKV + 1;  // K copied into TMEM
  static constexpr int kBarItemFull = kBarKTmem + 1;    // [2] an item published in its slot
  static constexpr int kBarItemEmpty = kBarItemFull + 2;  // [2] every role has read the slot
  static constexpr int kBarDVEmpty = kBarItemEmpty + 2;   // an item's dV stored (TMEM columns free)
  static constexpr int kBarDKEmpty = kBarDVEmpty + 1;     // an item's dK stored
  static constexpr int kBarDrain = kBarDKEmpty + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kItemSlot = kTmemSlot + 8;  // int[2]: the items of the two slots
  // block-sparse variant: bit qb = this key block keeps query block qb;
  // then the number of kept steps
  static constexpr int kQBits = kItemSlot + 8;
  static constexpr int kNPos = kQBits + kMaxSparseTiles / 8;
  static constexpr int kBytes = kNPos + 16;
  static constexpr int kSmem = kBytes + 1024;
  // TMEM columns
  static constexpr int kColDV = 0;
  static constexpr int kColDK = D;
  static constexpr int kColS = 2 * D;               // NSB buffers of BQ
  static constexpr int kColDP = 2 * D + NSB * BQ;   // BQ
  static constexpr int kColDQ = kColDP + BQ;        // dQ^T: 128 lanes (d; d=64: twice) x BQ
  static constexpr int kColK = kColDQ + BQ;         // K as 16-bit MMA A operand: D/2 cols
  static_assert(kColK + D / 2 <= 512, "TMEM budget");
  static_assert(kDS % 1024 == 0 && kStage0 % 1024 == 0, "swizzle alignment");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  // Column (within an S^T or dP^T buffer) of the packed 16-bit pair for
  // queries q, q+1 of the step: each P/dS warpgroup packs its own CW columns
  // into the first half of its own column range.
  __host__ __device__ static constexpr int packed_col(int q) {
    return (q / CW) * CW + (q % CW) / 2;
  }
};

// Stores columns [c0, c0 + NC) of a row of fp32 values from TMEM as 16-bit,
// multiplied by `mul`, to dst (the row's first element), if `valid`.
template <int NC, bool BF16>
__device__ __forceinline__ void store_row_from_tmem(uint32_t taddr, int c0, float mul, bool valid,
                                                    uint8_t* dst) {
  constexpr int W = NC < 32 ? NC : 32;  // columns per TMEM load
  static_assert(NC % W == 0 && (W == 32 || W == 16), "row width");
#pragma unroll 1
  for (int cc = c0; cc < c0 + NC; cc += W) {
    uint32_t r[W];
    tmem_ld_w<W>(taddr + cc, r);
    tmem_ld_wait();
    reg_fence<W>(r);
    uint32_t w[W / 2];
#pragma unroll
    for (int i = 0; i < W / 2; ++i)
      w[i] = pack2<BF16>(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
    if (valid) {
      uint4* o = reinterpret_cast<uint4*>(dst + cc * 2);
#pragma unroll
      for (int i = 0; i < W / 8; ++i) o[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
  }
}

// Adds columns [c0, c0 + NC) of a row of fp32 values from TMEM, multiplied
// by `mul`, into the fp32 accumulator row `acc` (the row's first element);
// with `first` the accumulator is overwritten instead.  Only if `valid`.
template <int NC>
__device__ __forceinline__ void acc_row_from_tmem(uint32_t taddr, int c0, float mul, bool valid, bool first,
                                                  float* acc) {
  constexpr int W = NC < 32 ? NC : 32;  // columns per TMEM load
  static_assert(NC % W == 0 && (W == 32 || W == 16), "row width");
#pragma unroll 1
  for (int cc = c0; cc < c0 + NC; cc += W) {
    uint32_t r[W];
    tmem_ld_w<W>(taddr + cc, r);
    tmem_ld_wait();
    reg_fence<W>(r);
    if (valid) {
      float4* a4 = reinterpret_cast<float4*>(acc + cc);
#pragma unroll
      for (int i = 0; i < W / 4; ++i) {
        float4 x = make_float4(__uint_as_float(r[4 * i]) * mul, __uint_as_float(r[4 * i + 1]) * mul,
                               __uint_as_float(r[4 * i + 2]) * mul, __uint_as_float(r[4 * i + 3]) * mul);
        if (!first) {
          const float4 a = a4[i];
          x.x += a.x; x.y += a.y; x.z += a.z; x.w += a.w;
        }
        a4[i] = x;
      }
    }
  }
}

// Columns [c0, c0 + NC) of this thread's TMEM row (= tile row `row`),
// multiplied by `mul` and rounded to 16-bit, into a shared-memory tile laid
// out as a TMA store reads it: 64-column boxes of 128 rows x 128 bytes, 16 KB
// apart, 128-byte swizzle (16-byte chunk j of a row at chunk j ^ (row % 8)).
template <int NC, bool BF16>
__device__ __forceinline__ void stage_row_from_tmem(uint32_t taddr, int c0, float mul, int row, uint8_t* tile) {
  constexpr int W = NC < 32 ? NC : 32;  // columns per TMEM load
  static_assert(NC % W == 0 && (W == 32 || W == 16), "row width");
#pragma unroll 1
  for (int cc = c0; cc < c0 + NC; cc += W) {
    uint32_t r[W];
    tmem_ld_w<W>(taddr + cc, r);
    tmem_ld_wait();
    reg_fence<W>(r);
#pragma unroll
    for (int i = 0; i < W / 8; ++i) {
      const int col = cc + 8 * i;
      const int chunk = (col & 63) >> 3;
      uint4* dst = reinterpret_cast<uint4*>(tile + (col >> 6) * 16384 + row * 128 + ((chunk ^ (row & 7)) * 16));
      *dst = make_uint4(pack2<BF16>(__uint_as_float(r[8 * i]) * mul, __uint_as_float(r[8 * i + 1]) * mul),
                        pack2<BF16>(__uint_as_float(r[8 * i + 2]) * mul, __uint_as_float(r[8 * i + 3]) * mul),
                        pack2<BF16>(__uint_as_float(r[8 * i + 4]) * mul, __uint_as_float(r[8 * i + 5]) * mul),
                        pack2<BF16>(__uint_as_float(r[8 * i + 6]) * mul, __uint_as_float(r[8 * i + 7]) * mul));
    }
  }
}

// NC 16-bit zeros to dst (16-byte aligned).
template <int NC>
__device__ __forceinline__ void store_zero_row(uint8_t* dst) {
  uint4* o = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < NC / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
}

// Heads per scheduling group of the main kernel.  Every block of a head
// sweeps that head's fp32 dQ accumulator (and reads its Q and dO), so the
// blocks in flight touch about G heads' worth of N x d x (4 + 2 + 2) bytes;
// G is chosen to keep that near half of the 126 MB L2, where the bulk
// reduce-adds then hit.  Fewer heads per group would lengthen the tail (each
// head's blocks range from 1 to N/64 steps), more would spill the L2.
__host__ __device__ inline int bwd_head_group(int N, int d, int BH) {
  const long long per_head = (long long)((N + 127) / 128) * 128 * d * 8;
  const long long g = (64ll << 20) / per_head;
  return (int)(g < 1 ? 1 : (g > BH ? BH : g));
}

// ALIBI: the scores carry the linear bias -m_h |i - j| (m_h = p.alibi[h]), as
// in the forward; it is folded into the per-query -LSE*log2(e) term.
// SPARSE: block-sparse mask p.bmask[h][qb][kb] as in the forward; the CTA
// visits only the query steps whose 128-row block its key block keeps
// ("positions"); a key block that keeps none stores dK = dV = 0.
// DROPOUT: the forward's Philox decisions (dropout.cuh) are redrawn: the P
// of dV += P^T dO keeps the kept scores only, dP is multiplied by 256 / t
// where kept and 0 where dropped (dS = P (dP - D) with the undropped P), and
// dV is scaled by 256 / t at the end.  This variant runs four P/dS
// warpgroups of 16 query columns: a lane draws the 16 decisions of one query
// for one of the warp's two 16-key groups, and a bit transpose gives each
// lane its key's decisions for the warpgroup's 16 queries.
// ACC (with none of the above): dK and dV are added into the fp32
// accumulators p.dk_acc, p.dv_acc (overwritten when p.kv_flags has
// kAccFirst) instead of being stored as 16-bit, so that the gradients of a
// key block can be summed over several calls, each with another range of
// query rows (and the forward's final O and LSE for them).
//
// Work items.  An item is one (128-key block, b, h); items are numbered in
// groups of G heads (bwd_head_group), key block the slow index inside a
// group, so the longest blocks (small key index, causal) go first.  Except
// in the SPARSE variant (one item per CTA), the grid is persistent: one CTA
// per SM, each taking its first item from its block index and the next ones
// from a counter in the workspace (p.sched[0], zeroed by the preprocess
// kernel; the last CTA out zeroes it again).  The producer claims the next
// item as soon as it has issued the current one's loads and publishes it in
// one of two shared-memory slots; every role walks the same item sequence,
// and every barrier phase runs on per-CTA step and item counters, so the
// next item's loads, its K copy into TMEM and its first MMAs overlap the
// current item's dQ drain and dK, dV stores.  Only three things wait at an
// item boundary: the next K/V load waits until every MMA of the item has
// completed (they read K and V in shared memory), and the next item's first
// dV and dK MMAs (which start their accumulators) wait until the dV and dK
// stores of the item have read those TMEM columns.
template <int D, bool BF16, bool ALIBI, bool SPARSE, bool DROPOUT, bool ACC = false>
__global__ void __launch_bounds__(BwdRoles<BwdNwg<DROPOUT>::value>::kThreads, 1)
    attn_bwd_main_kernel(const __grid_constant__ BwdArgs p) {
  static_assert(!ACC || !(ALIBI || SPARSE || DROPOUT), "the accumulating variant is plain only");
  constexpr int NWG = BwdNwg<DROPOUT>::value;
  using R = BwdRoles<NWG>;
  constexpr int kWarpDrain0 = R::kDrain0, kWarpProducer = R::kProducer;
  constexpr int kWarpMma = R::kMma, kWarpWaiter = R::kWaiter;
  constexpr uint32_t kPdsThreads = 32 * R::kPds;  // arrivals of the P/dS warps on a barrier
  using L = BwdLayout<D, NWG>;
  constexpr int BQ = L::BQ, CW = L::CW;
  constexpr int CH = CW < 32 ? CW : 32;  // query columns per TMEM load
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();  // (programmatic serialization: see griddep_wait)
  const int BH = p.B * p.H;
  const int nkb = (p.N + 127) / 128;
  const int n_items = nkb * BH;
  const int G = bwd_head_group(p.N, D, BH);
  const int nq = (p.N + BQ - 1) / BQ;
  const WaitCtl wc{p.wait.status, p.wait.limit_ns};

  // The work item with index `item`.
  struct Item {
    int jblk, bh, b, h, k0, i_begin, n_it;
  };
  auto decode = [&](int item) -> Item {
    Item it;
    const int grp = item / (G * nkb), r_in = item % (G * nkb);
    const int gsize = min(G, BH - grp * G);  // the last group may be smaller
    it.jblk = r_in / gsize;
    it.bh = grp * G + r_in % gsize;
    it.b = it.bh / p.H;
    it.h = it.bh % p.H;
    it.k0 = it.jblk * 128;
    it.i_begin = p.causal ? it.k0 / BQ : 0;
    it.n_it = nq - it.i_begin;
    return it;
  };

  auto bar = [&](int i) -> uint32_t { return base + L::kBar + 8u * i; };
  auto q_addr = [&](int st) -> uint32_t { return base + L::kStage0 + st * 2 * L::kQT; };
  auto do_addr = [&](int st) -> uint32_t { return q_addr(st) + L::kQT; };
  volatile int* item_slot = reinterpret_cast<volatile int*>(sbase + L::kItemSlot);

  uint32_t* qbits = reinterpret_cast<uint32_t*>(sbase + L::kQBits);
  int* npos_s = reinterpret_cast<int*>(sbase + L::kNPos);
  // (SPARSE: one item per CTA) step `it` of the item (query rows
  // (i_begin + it) * BQ ..) is visited unless masked
  auto step_ok = [&](const Item& I, int it) -> bool {
    if constexpr (!SPARSE) return true;
    const int qb = ((I.i_begin + it) * BQ) >> 7;
    return ((qbits[qb >> 5] >> (qb & 31)) & 1u) != 0;
  };
  auto next_step = [&](const Item& I, int it) -> int {  // the next visited step after `it` (n_it: none)
    ++it;
    if constexpr (SPARSE) {
      while (it < I.n_it && !step_ok(I, it)) ++it;
    }
    return it;
  };
  // visited steps of an item
  auto n_pos_of = [&](const Item& I) -> int { return SPARSE ? npos_s[0] : I.n_it; };

  // Stage loads are numbered by the CTA's step counter g (stage = g %
  // kStages, across items).
  auto load_stage = [&](const Item& I, int g, int it) {
    const int st = g % L::kStages;
    const int q0 = (I.i_begin + it) * BQ;
    const uint32_t fb = bar(L::kBarQFull + st);
    mbar_expect_tx(fb, 2 * L::kQT + 2 * BQ * 4);
    for (int s = 0; s < L::kNSub; ++s) {
      tma_load_4d(q_addr(st) + s * L::kSubQ, &p.tm_q, fb, s * 64, I.h, q0, I.b);
      tma_load_4d(do_addr(st) + s * L::kSubQ, &p.tm_do, fb, s * 64, I.h, q0, I.b);
    }
    const size_t row0 = (size_t)I.bh * p.Npad + q0;
    bulk_load(base + L::kLse + st * BQ * 4, p.lse2 + row0, BQ * 4, fb);
    bulk_load(base + L::kDv + st * BQ * 4, p.dvec + row0, BQ * 4, fb);
  };
  auto load_kv = [&](const Item& I) {
    mbar_expect_tx(bar(L::kBarKV), 2 * L::kKV);
    for (int s = 0; s < L::kNSub; ++s) {
      tma_load_4d(base + L::kK + s * L::kSubKV, &p.tm_k, bar(L::kBarKV), s * 64, I.h, I.k0, I.b);
      tma_load_4d(base + L::kV + s * L::kSubKV, &p.tm_v, bar(L::kBarKV), s * 64, I.h, I.k0, I.b);
    }
  };

  if (SPARSE && warp == kWarpProducer) {
    // The producer warp reads this key block's column of the mask (all
    // loads in flight at once), packs it with ballots and counts the
    // visited steps.
    const Item I = decode(blockIdx.x);
    constexpr int kW = kMaxSparseTiles / 32;
    const uint8_t* mk = p.bmask + (size_t)I.h * nkb * nkb + I.jblk;
    uint8_t v[kW];
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const int qb = w * 32 + lane;
      v[w] = qb < nkb ? mk[(size_t)qb * nkb] : 0;
    }
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const uint32_t bits = __ballot_sync(0xffffffffu, v[w] != 0);
      if (lane == 0) qbits[w] = bits;
    }
    __syncwarp();
    int c = 0;
    for (int it = lane; it < I.n_it; it += 32) c += step_ok(I, it) ? 1 : 0;
    c = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0) npos_s[0] = c;
    __syncwarp();
  }
  if (warp == kWarpProducer && lane == 0) {
    mbar_init(bar(L::kBarKV), 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::kBarQFull + s), 1);
      mbar_init(bar(L::kBarQEmpty + s), kPdsThreads);  // released by the P/dS warps
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kBarSFull + s), 1);
      mbar_init(bar(L::kBarPFull + s), kPdsThreads);
      mbar_init(bar(L::kBarItemFull + s), 1);
      mbar_init(bar(L::kBarItemEmpty + s), R::kPds + 6);  // one arrival per consumer warp
    }
    mbar_init(bar(L::kBarDPFull), 1);
    mbar_init(bar(L::kBarDSFull), kPdsThreads);
    mbar_init(bar(L::kBarDSSmem + 0), kPdsThreads);
    mbar_init(bar(L::kBarDSSmem + 1), kPdsThreads);
    mbar_init(bar(L::kBarDQFull), 1);
    mbar_init(bar(L::kBarDQEmpty), 128);
    mbar_init(bar(L::kBarDKV), 1);
    mbar_init(bar(L::kBarKTmem), 128);
    mbar_init(bar(L::kBarDVEmpty), kPdsThreads);
    mbar_init(bar(L::kBarDKEmpty), 128);
    mbar_init(bar(L::kBarDrain), 1);
    fence_mbar_init();
    tma_prefetch(&p.tm_q);
    tma_prefetch(&p.tm_k);
    tma_prefetch(&p.tm_v);
    tma_prefetch(&p.tm_do);
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

  // Consumers: the item of position n in the CTA's sequence (-1: no more),
  // or -2 if the wait gave up.  Every lane of the calling warp waits; lane
  // 0 then frees the slot for the producer.
  auto take_item = [&](int n) -> int {
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarItemFull + (n & 1)), (n >> 1) & 1, wc));
    int item = -2;
    if (ok) item = item_slot[n & 1];
    __syncwarp();
    if (ok && lane == 0) mbar_arrive(bar(L::kBarItemEmpty + (n & 1)));
    return item;
  };

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    // Claims items, publishes them, and issues every load: for each item a
    // few of its Q/dO stages first (their slots are freed by the previous
    // item's steps), then K and V once the previous item's MMAs have all
    // completed, then the rest of its stages.
    if (lane == 0) {
      int g = 0;        // stage loads issued
      int n = 0;        // items published
      bool ok = true;
      bool kv_inflight = false;
      for (;; ++n) {
        int item;
        if (n == 0) item = blockIdx.x;
        else if (SPARSE) item = -1;
        else item = gridDim.x + (int)atomicAdd(p.sched, 1u);
        if (item >= n_items) item = -1;
        // the slot's previous item (n - 2) has been read by every consumer
        if (!mbar_wait(bar(L::kBarItemEmpty + (n & 1)), ((n >> 1) & 1) ^ 1, wc)) {
          ok = false;
          break;
        }
        item_slot[n & 1] = item;
        mbar_arrive(bar(L::kBarItemFull + (n & 1)));  // release: the slot is visible to the waiters
        if (item < 0) break;
        const Item I = decode(item);
        const int n_pos = n_pos_of(I);
        if (n_pos == 0) continue;  // (SPARSE) a key block with no visited step loads nothing
        if (p.debug_flags & 2) {   // (timeout test: K and V, but no query step)
          load_kv(I);
          kv_inflight = true;
          break;
        }
        const int n_pre = min(L::kStages - 1, n_pos);
        int pos = 0, it = next_step(I, -1);
        for (; pos < n_pre && ok; ++pos, it = next_step(I, it), ++g) {
          if (!(ok = mbar_wait(bar(L::kBarQEmpty + g % L::kStages), ((g / L::kStages) & 1) ^ 1, wc))) break;
          load_stage(I, g, it);
        }
        // K and V: every MMA of the previous item (the last readers of
        // both) has completed
        if (ok && n > 0) ok = mbar_wait(bar(L::kBarDKV), (n - 1) & 1, wc);
        if (!ok) break;
        load_kv(I);
        for (; pos < n_pos && ok; ++pos, it = next_step(I, it), ++g) {
          if (!(ok = mbar_wait(bar(L::kBarQEmpty + g % L::kStages), ((g / L::kStages) & 1) ^ 1, wc))) break;
          load_stage(I, g, it);
        }
        if (!ok) break;
      }
      if (!ok || kv_inflight) {
        // Let every copy already issued land before shared memory goes away.
        mbar_wait_drain(bar(L::kBarKV), n & 1, wc.limit_ns);
        for (int i = max(0, g - L::kStages); i < g; ++i)
          mbar_wait_drain(bar(L::kBarQFull + i % L::kStages), (i / L::kStages) & 1, wc.limit_ns);
      }
      if (!SPARSE) {
        // The last CTA to finish zeroes the item counter for the next launch
        // (every CTA has claimed its last, out-of-range item by now).
        __threadfence();
        if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
          p.sched[0] = 0u;
          p.sched[1] = 0u;
          __threadfence();
        }
      }
    }
  } else if (warp == kWarpWaiter) {
    // ------------------------------------------------------------ waiter
    // Performs every mbarrier wait the MMA issuer depends on, in the issuer's
    // order, and hands each one over at a named barrier (see named_bar_and).
    // The MMA warp reads the item from the slot after the item's first
    // hand-off (H0).
    auto w = [&](int i, uint32_t parity) { return mbar_wait(bar(i), parity, wc); };
    bool ok = true;
    int g = 0;
    for (int n = 0; ok; ++n) {
      const int item = take_item(n);
      if (item == -2) {
        named_bar_and(kHandoffBar, 64, false);
        break;
      }
      if (item == -1) {  // no more items: H0 with the flag up, the issuer reads -1
        named_bar_and(kHandoffBar, 64, true);
        break;
      }
      const Item I = decode(item);
      const int n_pos = n_pos_of(I);
      if (n_pos == 0) {  // (SPARSE) nothing to issue; the issuer still takes H0
        ok = named_bar_and(kHandoffBar, 64, true);
        continue;
      }
      // H0: K, V loaded, K in TMEM, the item's first stage loaded.
      int qst = g % L::kStages;                 // stage of step g
      uint32_t qph = (g / L::kStages) & 1;      // its QFull parity
      ok = named_bar_and(kHandoffBar, 64,
                         __all_sync(0xffffffffu, w(L::kBarKV, n & 1) && w(L::kBarKTmem, n & 1) &&
                                                     w(L::kBarQFull + qst, qph)));
      // The step loop is the critical path of every hand-off: its waits are
      // addressed incrementally, and the item's first step, which also waits
      // for the previous item's dV and dK stores (the columns its first dV
      // and dK MMAs start over), is peeled off.  Hand-offs of step g:
      //   H1: P_g and the next Q/dO stage;  H2: dS_g in TMEM;
      //   H3: dS_g in shared memory, dQ_{g-1} drained.
      auto h3 = [&](uint32_t b1, uint32_t p2) {
        return named_bar_and(kHandoffBar, 64,
                             __all_sync(0xffffffffu, w(L::kBarDSSmem + b1, p2) && w(L::kBarDQEmpty, b1 ^ 1)));
      };
      if (ok) {  // first step of the item
        if (++qst == L::kStages) {
          qst = 0;
          qph ^= 1u;
        }
        const uint32_t b1 = g & 1, p2 = (g >> 1) & 1;
        bool r = w(L::kBarPFull + b1, p2);
        if (n_pos > 1) r = r && w(L::kBarQFull + qst, qph);
        if (n > 0) r = r && w(L::kBarDVEmpty, (n - 1) & 1);
        ok = named_bar_and(kHandoffBar, 64, __all_sync(0xffffffffu, r));
        if (ok) {
          r = w(L::kBarDSFull, b1);
          if (n > 0) r = r && w(L::kBarDKEmpty, (n - 1) & 1);
          ok = named_bar_and(kHandoffBar, 64, __all_sync(0xffffffffu, r));
        }
        if (ok) ok = h3(b1, p2);
        ++g;
      }
      for (int it = 1; ok && it < n_pos; ++it, ++g) {
        if (++qst == L::kStages) {  // stage and parity of step g + 1
          qst = 0;
          qph ^= 1u;
        }
        const uint32_t b1 = g & 1, p2 = (g >> 1) & 1;
        bool r = w(L::kBarPFull + b1, p2);
        if (it + 1 < n_pos) r = r && w(L::kBarQFull + qst, qph);
        ok = named_bar_and(kHandoffBar, 64, __all_sync(0xffffffffu, r));
        if (!ok) break;
        ok = named_bar_and(kHandoffBar, 64, __all_sync(0xffffffffu, w(L::kBarDSFull, b1)));
        if (!ok) break;
        ok = h3(b1, p2);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the schedule, converged; one elected lane
    // issues (MMAs and commits inside elect.sync, no branch around them).
    // This warp waits on no mbarrier: it learns that operands are ready at
    // the named-barrier hand-offs with the waiter warp.  It reads an item's
    // slot only at the item's H0, when no MMA of the previous item is in
    // flight.
    constexpr uint32_t idesc_s = make_idesc(BF16, 128, BQ, false, false);
    constexpr uint32_t idesc_g = make_idesc(BF16, 128, D, false, true);
    constexpr uint32_t idesc_q = make_idesc(BF16, 128, BQ, true, true);
    // V x dO^T over d -> 128 x BQ in TMEM (both operands in shared memory).
    auto issue_st = [&](uint32_t d_t, uint32_t a_tile, uint32_t b_tile) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t ao = (ks >> 2) * L::kSubKV + (ks & 3) * 32;
        const uint32_t bo = (ks >> 2) * L::kSubQ + (ks & 3) * 32;
        mma_ss(d_t, make_sdesc(a_tile + ao, 16, 1024), make_sdesc(b_tile + bo, 16, 1024), idesc_s,
               ks > 0);
      }
    };
    // S^T = K Q^T over d, with K read from TMEM (copied there once per
    // item): only Q is read from shared memory.
    auto issue_s = [&](uint32_t d_t, uint32_t b_tile) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t bo = (ks >> 2) * L::kSubQ + (ks & 3) * 32;
        mma_ts(d_t, tmem + L::kColK + ks * 8, make_sdesc(b_tile + bo, 16, 1024), idesc_s, ks > 0);
      }
    };
    // [P^T or dS^T](TMEM, packed per warpgroup) x [dO or Q] over BQ queries -> 128 x d.
    auto issue_grad = [&](uint32_t d_t, uint32_t a_buf, uint32_t b_tile, bool acc) {
#pragma unroll
      for (int ks = 0; ks < BQ / 16; ++ks)
        mma_ts(d_t, a_buf + L::packed_col(ks * 16), make_sdesc(b_tile + ks * 2048, L::kSubQ, 1024),
               idesc_g, (acc || ks > 0) ? 1u : 0u);
    };
    // dQ^T = K^T dS^T over the 128 keys, dS^T from shared-memory buffer
    // `buf`: A = K (MN-major, M = 128 rows of d), B = dS^T (MN-major).  For
    // d = 64 the K tile has one 64-column block; a zero block offset makes
    // A's rows 64-127 repeat rows 0-63, and TMEM lanes 64-127 of dQ^T are a
    // copy the drain ignores.
    auto issue_dq = [&](int buf) {
      const uint32_t kt = base + L::kK, ds = base + L::kDS + buf * L::kDSBytes;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_ss(tmem + L::kColDQ, make_sdesc(kt + ks * 2048, D == 128 ? L::kSubKV : 0, 1024),
               make_sdesc(ds + ks * 2048, L::kDSsub, 1024), idesc_q, ks > 0);
    };
    // Per step g, three hand-offs (each lets the tensor pipe drain, so the
    // schedule groups as many MMAs behind each as the dependencies allow):
    //   H1 [P_g, next stage]                  : dV_g, S_{g+1}
    //   H2 [dS_g in TMEM]                      : dK_g, dP_{g+1}
    //   H3 [dS_g in smem, dQ_{g-1} drained]    : dQ_g
    // (S and dP of an item's first step are issued at its H0.)  In-order
    // execution keeps every TMEM / shared-memory reuse behind the MMA that
    // last read it, within an item and across items.
    bool ok = true;
    int g = 0;
    for (int n = 0; ok; ++n) {
      ok = named_bar_and(kHandoffBar, 64, true);  // H0
      if (!ok) break;
      const int item = item_slot[n & 1];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kBarItemEmpty + (n & 1)));
      if (item < 0) break;
      const Item I = decode(item);
      const int n_pos = n_pos_of(I);
      if (n_pos == 0) continue;
      int st = g % L::kStages;  // stage of step g (advanced incrementally)
      tc_fence_after();
      issue_s(tmem + L::kColS, q_addr(st));
      tc_commit(bar(L::kBarSFull));
      issue_st(tmem + L::kColDP, base + L::kV, do_addr(st));
      tc_commit(bar(L::kBarDPFull));
      for (int it = 0; ok && it < n_pos; ++it, ++g, st = (st + 1 == L::kStages) ? 0 : st + 1) {
        const int nst = (st + 1 == L::kStages) ? 0 : st + 1;
        const bool has_next = it + 1 < n_pos;
        ok = named_bar_and(kHandoffBar, 64, true);  // H1
        if (!ok) break;
        tc_fence_after();
        issue_grad(tmem + L::kColDV, tmem + L::kColS, do_addr(st), it > 0);
        if (has_next) {
          issue_s(tmem + L::kColS, q_addr(nst));
          tc_commit(bar(L::kBarSFull));
        }
        ok = named_bar_and(kHandoffBar, 64, true);  // H2
        if (!ok) break;
        tc_fence_after();
        issue_grad(tmem + L::kColDK, tmem + L::kColDP, q_addr(st), it > 0);
        if (has_next) {
          issue_st(tmem + L::kColDP, base + L::kV, do_addr(nst));
          tc_commit(bar(L::kBarDPFull));
        }
        ok = named_bar_and(kHandoffBar, 64, true);  // H3
        if (!ok) break;
        tc_fence_after();
        issue_dq(g & 1);
        tc_commit(bar(L::kBarDQFull));
      }
      // every MMA of the item completes before this arrives: the dK, dV
      // stores and the next item's K/V load wait for it
      if (ok) tc_commit(bar(L::kBarDKV));
    }
    // Every MMA issued above completes before tensor memory is released.
    tc_commit(bar(L::kBarDrain));
    mbar_wait_drain(bar(L::kBarDrain), 0, wc.limit_ns);
  } else if (warp < kWarpDrain0) {
    // ------------------------------------------------ P^T and dS^T (key rows)
    // NWG warpgroups on the same 128 key rows (TMEM lanes), each owning CW of
    // the BQ query columns: warpgroup hf has columns [hf CW, hf CW + CW).
    // Each writes its 16-bit P^T / dS^T only into its own column range.
    const int hf = warp >> 2, qd = warp & 3;
    const int kl = qd * 32 + lane;  // key row within the block = TMEM lane
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const float c = p.scale * kLog2e;
    const float2 c2 = make_float2(c, c);
    const int cbase = hf * CW;  // first query column of this warpgroup
    // Every named barrier of these warps is met by all of them: a wait that
    // gives up in one warp travels to the others through named_bar_and (at
    // an item's start and after its steps), never by leaving the loop alone.
    bool ok = true;
    int g = 0;
    for (int n = 0; ok; ++n) {
      const int item = take_item(n);
      if (!named_bar_and(kPdsBar, kPdsThreads, item != -2)) {
        ok = false;
        break;
      }
      if (item < 0) break;  // (-1: no more items, read alike by every warp from the slot)
      const Item I = decode(item);
      const int n_pos = n_pos_of(I);
      const int key = I.k0 + kl;
      const bool key_ok = key < p.N;
      const float slope2 = ALIBI ? p.alibi[I.h] * kLog2e : 0.f;  // ALiBi slope, log2 units
      if (hf == 0 && n_pos > 0) {
        // K row kl -> TMEM lane kl as the 16-bit A operand of S^T = K Q^T:
        // column c holds d elements 2c, 2c+1 (the row's own 32-bit words).
        // The previous item's MMAs, the last readers of these columns, have
        // completed (this warpgroup waited for them before its dV stores).
        ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarKV), n & 1, wc));
      }
      if (hf == 0 && n_pos > 0 && ok) {
        uint32_t kw[D / 2];
#pragma unroll
        for (int sub = 0; sub < D / 64; ++sub)
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint4 v = *reinterpret_cast<const uint4*>(sbase + L::kK + sub * L::kSubKV + kl * 128 +
                                                            ((ch ^ (kl & 7)) * 16));
            kw[sub * 32 + ch * 4 + 0] = v.x;
            kw[sub * 32 + ch * 4 + 1] = v.y;
            kw[sub * 32 + ch * 4 + 2] = v.z;
            kw[sub * 32 + ch * 4 + 3] = v.w;
          }
#pragma unroll
        for (int cc = 0; cc < D / 2; cc += 32) tmem_st32(tmem + lane_off + L::kColK + cc, kw + cc);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(L::kBarKTmem));
      }
      // it: position in the item; step: the query step it visits; g: the
      // CTA's step counter (stages, buffers and barrier parities).
      for (int it = 0, step = next_step(I, -1); ok && it < n_pos; ++it, step = next_step(I, step), ++g) {
        const int st = g % L::kStages;
        const int q0 = (I.i_begin + step) * BQ;
        // dropout: bit i keeps score (query q0 + cbase + i, this key)
        uint32_t keepw = 0xffffffffu;
        if constexpr (DROPOUT) {
          static_assert(CW == 16, "lane l draws query l % 16 of key group l / 16");
          // Lane l: the 16 decisions of query q0 + cbase + l % 16 for the
          // warp's key group g0 + l / 16, at bits 16 (l / 16) .. of its word.
          // After the transpose, bit l of lane m is bit m of lane l's word: the
          // decision of query l % 16 for key m when l / 16 = m / 16.
          const int gsel = lane >> 4;
          const uint32_t g0 = (uint32_t)(key - lane) >> 4;  // the warp's first 16-key group
          const uint32_t qrow = (uint32_t)(q0 + cbase + (lane & 15));
          const uint32_t t = warp_transpose32(keep_bits16(p.drop, I.bh, qrow, g0 + gsel) << (16 * gsel), lane);
          keepw = (t >> (16 * gsel)) & 0xffffu;
        }
        ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarQFull + st), (g / L::kStages) & 1, wc));
        if (!ok) break;
        // -LSE * log2(e) of this warpgroup's queries, read before waiting on S^T.
        float lv[CW];
        {
          const float4* l4 = reinterpret_cast<const float4*>(sbase + L::kLse + st * BQ * 4 + cbase * 4);
#pragma unroll
          for (int i4 = 0; i4 < CW / 4; ++i4) {
            const float4 v = l4[i4];
            lv[4 * i4] = v.x; lv[4 * i4 + 1] = v.y; lv[4 * i4 + 2] = v.z; lv[4 * i4 + 3] = v.w;
          }
        }
        if constexpr (ALIBI) {
          // lv[i] <- lv[i] - m |query - key| for the warpgroup's query columns;
          // linear in i unless the columns straddle this thread's key.
          const int d0 = q0 + cbase - key;  // query - key at column 0
          const bool ge = __all_sync(0xffffffffu, d0 >= 0), le = __all_sync(0xffffffffu, d0 + CW - 1 <= 0);
          if (ge || le) {
            const float k1 = ge ? -slope2 : slope2, k0 = k1 * (float)d0;
#pragma unroll
            for (int i = 0; i < CW; ++i) lv[i] = fmaf((float)i, k1, lv[i] + k0);
          } else {
#pragma unroll
            for (int i = 0; i < CW; ++i) lv[i] -= slope2 * fabsf((float)(d0 + i));
          }
        }
        ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarSFull), g & 1, wc));
        if (!ok) break;
        tc_fence_after();
        const uint32_t tS = tmem + lane_off + L::kColS;
        const float4* dvec = reinterpret_cast<const float4*>(sbase + L::kDv + st * BQ * 4 + cbase * 4);
        // visible(q) = key < N && (!causal || key <= q): column i of this
        // warpgroup is visible iff i >= vis_from (vis_from > CW: none).
        const int vis_from = !key_ok ? CW + 1 : (p.causal ? max(0, key - (q0 + cbase)) : 0);
        const bool warp_all_vis = __all_sync(0xffffffffu, vis_from == 0);
        float pr[CW];
#pragma unroll
        for (int cc = 0; cc < CW; cc += CH) {
          uint32_t r[CH];
          tmem_ld_w<CH>(tS + cbase + cc, r);
          tmem_ld_wait();
          reg_fence<CH>(r);
          uint32_t pk[CH / 2];
          if (warp_all_vis) {  // common case: no masking in this warp
#pragma unroll
            for (int i = 0; i < CH; i += 2) {
              const float2 x = fma2(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), c2,
                                    make_float2(lv[cc + i], lv[cc + i + 1]));
              pr[cc + i] = ex2(x.x);
              pr[cc + i + 1] = ex2(x.y);
            }
          } else {
#pragma unroll
            for (int i = 0; i < CH; ++i) {
              const float e = ex2(fmaf(__uint_as_float(r[i]), c, lv[cc + i]));
              pr[cc + i] = (cc + i >= vis_from) ? e : 0.f;
            }
          }
#pragma unroll
          for (int i = 0; i < CH / 2; ++i) {
            if constexpr (DROPOUT) {  // P of the kept scores only
              const int b0 = cc + 2 * i;
              pk[i] = pack2<BF16>(((keepw >> b0) & 1u) ? pr[cc + 2 * i] : 0.f,
                                  ((keepw >> (b0 + 1)) & 1u) ? pr[cc + 2 * i + 1] : 0.f);
            } else {
              pk[i] = pack2<BF16>(pr[cc + 2 * i], pr[cc + 2 * i + 1]);
            }
          }
          tmem_st_w<CH / 2>(tS + cbase + cc / 2, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(L::kBarPFull + (g & 1)));

        float dv[CW];  // D of this warpgroup's queries, read before waiting on dP^T
#pragma unroll
        for (int i4 = 0; i4 < CW / 4; ++i4) {
          const float4 d4 = dvec[i4];
          dv[4 * i4] = d4.x; dv[4 * i4 + 1] = d4.y; dv[4 * i4 + 2] = d4.z; dv[4 * i4 + 3] = d4.w;
        }
        ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarDPFull), g & 1, wc));
        if (!ok) break;
        // dP^T of this step was issued after the dK (and dV) of the previous
        // step (in this item or the previous one), so that step's Q/dO stage
        // is no longer read: hand it back to the producer.
        if (g > 0) mbar_arrive(bar(L::kBarQEmpty + (g - 1) % L::kStages));
        tc_fence_after();
        const uint32_t tDP = tmem + lane_off + L::kColDP;
        uint32_t dsk[CW / 2];  // packed 16-bit dS^T of this row
#pragma unroll
        for (int cc = 0; cc < CW; cc += CH) {
          uint32_t r[CH];
          tmem_ld_w<CH>(tDP + cbase + cc, r);
          tmem_ld_wait();
          reg_fence<CH>(r);
#pragma unroll
          for (int i = 0; i < CH / 2; ++i) {
            float2 dp = make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
            if constexpr (DROPOUT) {  // dP of a kept score times 256 / t, of a dropped one 0
              const int b0 = cc + 2 * i;
              dp = mul2(dp, make_float2(((keepw >> b0) & 1u) ? p.drop.scale : 0.f,
                                        ((keepw >> (b0 + 1)) & 1u) ? p.drop.scale : 0.f));
            }
            const float2 ds = mul2(make_float2(pr[cc + 2 * i], pr[cc + 2 * i + 1]),
                                   sub2(dp, make_float2(dv[cc + 2 * i], dv[cc + 2 * i + 1])));
            dsk[cc / 2 + i] = pack2<BF16>(ds.x, ds.y);
          }
          tmem_st_w<CH / 2>(tDP + cbase + cc / 2, dsk + cc / 2);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(L::kBarDSFull));  // dK and the next dP^T may go ahead
        // dS^T row into shared-memory buffer g & 1 (128-byte swizzle): 16-byte
        // chunk j of this row goes to chunk j ^ (row % 8) of its 128-byte line.
        // The dQ that read this buffer two steps ago has completed: it was
        // issued before the dP^T whose completion this warpgroup waited for.
        uint8_t* ds_row = sbase + L::kDS + (g & 1) * L::kDSBytes + kl * 128;
#pragma unroll
        for (int g4 = 0; g4 < CW / 8; ++g4) {
          const int gc = cbase / 8 + g4;  // 16-byte chunk index along the queries
          const int sub = gc >> 3;        // 64-query sub-tile
          uint4* dst = reinterpret_cast<uint4*>(ds_row + sub * L::kDSsub + (((gc & 7) ^ (kl & 7)) * 16));
          *dst = make_uint4(dsk[4 * g4], dsk[4 * g4 + 1], dsk[4 * g4 + 2], dsk[4 * g4 + 3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(L::kBarDSSmem + (g & 1)));
      }
      ok = named_bar_and(kPdsBar, kPdsThreads, ok);  // (a warp that gave up in the steps)
      if (!ok) break;
      uint8_t* dst = reinterpret_cast<uint8_t*>(p.dv) +
                     ((((size_t)I.b * p.N + (key_ok ? key : 0)) * p.H + I.h) * D) * 2;
      if (n_pos > 0) {
        // (every P/dS warp takes the same branch: the TMA store below meets
        // at a named barrier)
        ok = named_bar_and(kPdsBar, kPdsThreads, __all_sync(0xffffffffu, mbar_wait(bar(L::kBarDKV), n & 1, wc)));
        if (!ok) break;
        tc_fence_after();
        // warpgroup hf stores columns [hf D / NWG, (hf + 1) D / NWG) of dV
        if constexpr (ACC) {
          acc_row_from_tmem<D / NWG>(tmem + lane_off + L::kColDV, hf * (D / NWG), 1.f, key_ok,
                                     (p.kv_flags & kAccFirst) != 0,
                                     p.dv_acc + (((size_t)I.b * p.N + (key_ok ? key : 0)) * p.H + I.h) * D);
          tc_fence_before();
          mbar_arrive(bar(L::kBarDVEmpty));  // the next item's first dV may overwrite the columns
        } else {
          // Through shared memory and one TMA store per 64-column box (the
          // dS buffers are free: the item's last dQ MMA has completed); rows
          // past N are clipped by the store.
          stage_row_from_tmem<D / NWG, BF16>(tmem + lane_off + L::kColDV, hf * (D / NWG),
                                             DROPOUT ? p.drop.scale : 1.f, kl, sbase + L::kDS);
          tc_fence_before();
          mbar_arrive(bar(L::kBarDVEmpty));  // the next item's first dV may overwrite the columns
          fence_proxy_async_smem();
          named_bar_sync(kPdsBar, kPdsThreads);
          if (warp == 0 && lane == 0) {
            for (int bx = 0; bx < D / 64; ++bx)
              tma_store_4d(&p.tm_dv, base + L::kDS + bx * 16384, bx * 64, I.h, I.k0, I.b);
            bulk_commit();
            bulk_wait_read_all();  // the buffers are written again by the next item's dS
          }
          named_bar_sync(kPdsBar, kPdsThreads);
        }
      } else if (SPARSE && key_ok) {
        store_zero_row<D / NWG>(dst + hf * (D / NWG) * 2);  // no visited query: dV = 0
      }
    }
    if (!ACC && warp == 0 && lane == 0) bulk_wait_all();  // the dV stores have landed
  } else {
    // ------------------------------------------------ dQ drain (warps 8-11)
    // TMEM -> registers -> shared memory (the accumulator's row-major tile
    // layout) -> bulk reduce-adds into the accumulator; after an item's last
    // step, its dK stores.
    const int qd = warp & 3;
    const int ln = qd * 32 + lane;  // TMEM lane: d index of dQ^T (d=64: lanes >= 64 repeat)
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    float* sdq = reinterpret_cast<float*>(sbase + L::kDQ);
    const bool leader = (warp == kWarpDrain0 && lane == 0);
    bool ok = true;
    int g = 0;
    for (int n = 0; ok; ++n) {
      const int item = take_item(n);
      if (!named_bar_and(kDrainBar, 128, item != -2)) {  // (the four warps decide together)
        ok = false;
        break;
      }
      if (item < 0) break;
      const Item I = decode(item);
      const int n_pos = n_pos_of(I);
      for (int it = 0, step = next_step(I, -1); ok && it < n_pos; ++it, step = next_step(I, step), ++g) {
        const int q0 = (I.i_begin + step) * BQ;
        // The four warps meet at named barriers below: the give-up flag of a
        // bounded wait travels through the first one so they branch together.
        ok = named_bar_and(kDrainBar, 128,
                           __all_sync(0xffffffffu, mbar_wait(bar(L::kBarDQFull), g & 1, wc)));
        if (!ok) break;
        tc_fence_after();
        uint32_t r[64];
        tmem_ld32(tmem + lane_off + L::kColDQ, r);
        tmem_ld32(tmem + lane_off + L::kColDQ + 32, r + 32);
        tmem_ld_wait();
        reg_fence<64>(r);
        tc_fence_before();
        mbar_arrive(bar(L::kBarDQEmpty));
        // The tile goes out in two halves of BQ/2 rows, each with its own bulk
        // reduce-add, so that staging one half overlaps the copy engine's read
        // of the other (the reduce path of one SM moves about 20 bytes/clk).
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          if (leader) bulk_wait_read_but_last();  // this half's previous reduce has read it
          named_bar_sync(kDrainBar, 128);
          if (ln < D) {
            // r[c] = dQ[q0 + c][ln]: row c of the tile, column ln (128-byte rows per warp).
#pragma unroll
            for (int cq = 32 * hh; cq < 32 * hh + 32; ++cq) sdq[cq * D + ln] = __uint_as_float(r[cq]);
          }
          fence_proxy_async_smem();
          named_bar_sync(kDrainBar, 128);
          if (leader) {
            bulk_reduce_add_f32(p.dqacc + ((size_t)I.bh * p.Npad + q0 + hh * (BQ / 2)) * D,
                                base + L::kDQ + hh * (L::kDQBytes / 2), L::kDQBytes / 2);
            bulk_commit();
          }
        }
      }
      if (!ok) break;
      const int key = I.k0 + ln;
      const bool key_ok = key < p.N;
      uint8_t* dst = reinterpret_cast<uint8_t*>(p.dk) +
                     ((((size_t)I.b * p.N + (key_ok ? key : 0)) * p.H + I.h) * D) * 2;
      if (n_pos > 0) {
        // (the four drain warps take the same branch: they meet at named
        // barriers below)
        ok = named_bar_and(kDrainBar, 128, __all_sync(0xffffffffu, mbar_wait(bar(L::kBarDKV), n & 1, wc)));
        if (!ok) break;
        tc_fence_after();
        if constexpr (ACC) {
          acc_row_from_tmem<D>(tmem + lane_off + L::kColDK, 0, p.scale, key_ok, (p.kv_flags & kAccFirst) != 0,
                               p.dk_acc + (((size_t)I.b * p.N + (key_ok ? key : 0)) * p.H + I.h) * D);
          tc_fence_before();
          mbar_arrive(bar(L::kBarDKEmpty));  // the next item's first dK may overwrite the columns
        } else {
          // Through the dQ staging tile (once the last dQ reduce has read it)
          // and one TMA store per 64-column box.
          if (leader) bulk_wait_read_all();
          named_bar_sync(kDrainBar, 128);
          stage_row_from_tmem<D, BF16>(tmem + lane_off + L::kColDK, 0, p.scale, ln, sbase + L::kDQ);
          tc_fence_before();
          mbar_arrive(bar(L::kBarDKEmpty));  // the next item's first dK may overwrite the columns
          fence_proxy_async_smem();
          named_bar_sync(kDrainBar, 128);
          if (leader) {
            for (int bx = 0; bx < D / 64; ++bx)
              tma_store_4d(&p.tm_dk, base + L::kDQ + bx * 16384, bx * 64, I.h, I.k0, I.b);
            bulk_commit();
            bulk_wait_read_all();  // the next item's dQ is staged here
          }
          named_bar_sync(kDrainBar, 128);
        }
      } else if (SPARSE && key_ok) {
        store_zero_row<D>(dst);  // no visited query: dK = 0 (lane ln is key k0 + ln here)
      }
    }
    if (leader) bulk_wait_all();
  }

  if (threadIdx.x == 0) griddep_launch_dependents();  // (this CTA has no more items; see launch_pdl)
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpProducer) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- pre / post
// Memory-bound helpers, sized to the SM count and written as grid-stride
// loops with several 16-byte loads in flight per thread: one wave of four
// 256-thread blocks per SM (at most 64 registers a thread), 128 KB of loads
// in flight per SM.
constexpr int kAuxThreads = 256;
constexpr int kAuxBlocksPerSm = 4;

// (1) D_r = sum_c dO[r][c] O[r][c] for every row r = (b, n, h) of the
//     [B, N, H, d] tensors, in their memory order: one row is 16 lanes
//     (d=128) or 8 lanes (d=64) of 16 bytes each; a warp takes kU groups of
//     rows with all loads issued before the arithmetic.
// (2) lse2 = -LSE * log2(e) per (b, h, n < Npad), -inf on the padding rows,
//     whose D is 0 (their P is then exactly 0).
// (3) The fp32 dQ accumulator is cleared.
// (4) The main kernel's work counter is zeroed.
// Row indices are split into (b, n, h) or (b h, n) with 32-bit divisions
// (U = unsigned) when B H Npad < 2^31, else 64-bit ones (a 64-bit division
// is a long instruction sequence, which dominated these kernels' time).
template <int D, bool BF16, typename U>
__global__ void __launch_bounds__(kAuxThreads, kAuxBlocksPerSm) attn_bwd_pre_kernel(const __grid_constant__ BwdArgs p) {
  griddep_wait();  // (programmatic serialization: see griddep_wait)
  constexpr int kLanesPerRow = D * 2 / 16;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  constexpr int kU = 4;
  const int lane = threadIdx.x & 31;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nwarps = nthreads >> 5, gw = tid >> 5;

  const long long rows = (long long)p.B * p.N * p.H;
  const long long groups = (rows + kRowsPerWarp - 1) / kRowsPerWarp;
  const int sub = lane / kLanesPerRow, part = lane % kLanesPerRow;
  for (long long g0 = gw * kU; g0 < groups; g0 += nwarps * kU) {
    uint4 ov[kU], gv[kU];
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const long long r = (g0 + j) * kRowsPerWarp + sub;
      if (r < rows) {
        ov[j] = reinterpret_cast<const uint4*>(p.o)[r * kLanesPerRow + part];
        gv[j] = reinterpret_cast<const uint4*>(p.dO)[r * kLanesPerRow + part];
      } else {
        ov[j] = make_uint4(0, 0, 0, 0);
        gv[j] = ov[j];
      }
    }
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const uint32_t* ow = &ov[j].x;
      const uint32_t* gwv = &gv[j].x;
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float2 x = unpack2<BF16>(ow[w]), y = unpack2<BF16>(gwv[w]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
#pragma unroll
      for (int off = kLanesPerRow / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      const long long r = (g0 + j) * kRowsPerWarp + sub;
      if (part == 0 && r < rows) {
        const U ur = (U)r, bn = ur / (U)p.H;
        const U h = ur - bn * (U)p.H, b = bn / (U)p.N, n = bn - b * (U)p.N;
        p.dvec[((size_t)b * p.H + h) * p.Npad + n] = acc;
      }
    }
  }

  const long long nrow_ws = (long long)p.B * p.H * p.Npad;
  for (long long i = tid; i < nrow_ws; i += nthreads) {
    const U bh = (U)i / (U)p.Npad, n = (U)i - bh * (U)p.Npad;
    if (n < (U)p.N) {
      // A row that sees no key (LSE = -inf, block-sparse masks) gets -inf
      // too: its P would be exactly 0 if it were visited.
      const float l = p.lse[bh * p.N + n];
      p.lse2[i] = l == -INFINITY ? -INFINITY : -l * kLog2e;
    } else {
      p.lse2[i] = -INFINITY;
      p.dvec[i] = 0.f;
    }
  }

  float4* z = reinterpret_cast<float4*>(p.dqacc);
  const long long nz = nrow_ws * D / 4;
  for (long long i = tid; i < nz; i += nthreads) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (tid == 0) {  // (4) the main kernel's work counter
    p.sched[0] = 0u;
    p.sched[1] = 0u;
  }
  griddep_launch_dependents();  // (see launch_pdl)
}

// dQ = scale * accumulator, to 16-bit, [B, N, H, d]: one thread per 8
// consecutive outputs, kU of them (a grid stride apart) in flight.  (U: the
// index type of the row split, as in the preprocess kernel.)
template <int D, bool BF16, typename U>
__global__ void __launch_bounds__(kAuxThreads, kAuxBlocksPerSm) attn_dq_post_kernel(const __grid_constant__ BwdArgs p) {
  griddep_wait();  // (programmatic serialization: see griddep_wait)
  constexpr int kU = 4;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  const long long total = (long long)p.B * p.N * p.H * D / 8;
  const float s = p.scale;
  for (long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += kU * nthreads) {
    float4 x[kU], y[kU];
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const long long idx = i0 + j * nthreads;
      if (idx < total) {
        const int c = (int)(idx % (D / 8)) * 8;  // idx = r d / 8 + c / 8, r = (b N + n) H + h
        const U r = (U)(idx / (D / 8)), bn = r / (U)p.H;
        const U h = r - bn * (U)p.H, b = bn / (U)p.N, n = bn - b * (U)p.N;
        const float4* src = reinterpret_cast<const float4*>(
            p.dqacc + (((size_t)b * p.H + h) * p.Npad + n) * D + c);
        x[j] = src[0];
        y[j] = src[1];
      }
    }
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const long long idx = i0 + j * nthreads;
      if (idx < total)
        reinterpret_cast<uint4*>(p.dq)[idx] =
            make_uint4(pack2<BF16>(x[j].x * s, x[j].y * s), pack2<BF16>(x[j].z * s, x[j].w * s),
                       pack2<BF16>(y[j].x * s, y[j].y * s), pack2<BF16>(y[j].z * s, y[j].w * s));
    }
  }
  griddep_launch_dependents();  // (see launch_pdl)
}

template <int D, bool BF16, bool ALIBI, bool SPARSE, bool DROPOUT, bool ACC = false>
cudaError_t launch_main_t(const BwdArgs& a, cudaStream_t stream) {
  using L = BwdLayout<D, BwdNwg<DROPOUT>::value>;
  auto* k = attn_bwd_main_kernel<D, BF16, ALIBI, SPARSE, DROPOUT, ACC>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
  if (e != cudaSuccess) return e;
  // one CTA per item (block-sparse), else a persistent grid of one CTA per SM
  const long long items = (long long)((a.N + 127) / 128) * a.B * a.H;
  const unsigned grid = (unsigned)(SPARSE ? items : (items < a.sms ? items : a.sms));
  e = launch_pdl(k, grid, BwdRoles<BwdNwg<DROPOUT>::value>::kThreads, L::kSmem, stream, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int bwd_q_rows(int d) { return d == 128 ? BwdLayout<128>::BQ : BwdLayout<64>::BQ; }
int bwd_smem_bytes(int d) { return d == 128 ? BwdLayout<128>::kSmem : BwdLayout<64>::kSmem; }

// Whether the row splits of the pre / post kernels fit 32-bit indices
// (debug flag bit 3 takes the 64-bit form regardless, for tests).
static bool aux_narrow(const BwdArgs& a) {
  return (long long)a.B * a.H * a.Npad < (1ll << 31) && !(a.debug_flags & 8);
}

template <typename U>
cudaError_t launch_bwd_pre_u(const BwdArgs& a, unsigned grid, cudaStream_t stream) {
  if (a.d == 128)
    return a.bf16 ? launch_pdl(attn_bwd_pre_kernel<128, true, U>, grid, kAuxThreads, 0, stream, a)
                  : launch_pdl(attn_bwd_pre_kernel<128, false, U>, grid, kAuxThreads, 0, stream, a);
  return a.bf16 ? launch_pdl(attn_bwd_pre_kernel<64, true, U>, grid, kAuxThreads, 0, stream, a)
                : launch_pdl(attn_bwd_pre_kernel<64, false, U>, grid, kAuxThreads, 0, stream, a);
}

cudaError_t launch_bwd_pre(const BwdArgs& a, cudaStream_t stream) {
  const unsigned grid = (unsigned)(a.sms * kAuxBlocksPerSm);
  return aux_narrow(a) ? launch_bwd_pre_u<unsigned>(a, grid, stream)
                       : launch_bwd_pre_u<unsigned long long>(a, grid, stream);
}

template <bool ALIBI, bool SPARSE, bool DROPOUT>
cudaError_t launch_main_v(const BwdArgs& a, cudaStream_t stream) {
  if (a.d == 128)
    return a.bf16 ? launch_main_t<128, true, ALIBI, SPARSE, DROPOUT>(a, stream)
                  : launch_main_t<128, false, ALIBI, SPARSE, DROPOUT>(a, stream);
  return a.bf16 ? launch_main_t<64, true, ALIBI, SPARSE, DROPOUT>(a, stream)
                : launch_main_t<64, false, ALIBI, SPARSE, DROPOUT>(a, stream);
}

template <bool DROPOUT>
cudaError_t launch_main_d(const BwdArgs& a, cudaStream_t stream) {
  if (a.bmask)
    return a.alibi ? launch_main_v<true, true, DROPOUT>(a, stream) : launch_main_v<false, true, DROPOUT>(a, stream);
  return a.alibi ? launch_main_v<true, false, DROPOUT>(a, stream) : launch_main_v<false, false, DROPOUT>(a, stream);
}

cudaError_t launch_bwd_main(const BwdArgs& a, cudaStream_t stream) {
  return a.drop.t < 256 ? launch_main_d<true>(a, stream) : launch_main_d<false>(a, stream);
}

cudaError_t launch_bwd_main_acc(const BwdArgs& a, cudaStream_t stream) {
  if (a.d == 128)
    return a.bf16 ? launch_main_t<128, true, false, false, false, true>(a, stream)
                  : launch_main_t<128, false, false, false, false, true>(a, stream);
  return a.bf16 ? launch_main_t<64, true, false, false, false, true>(a, stream)
                : launch_main_t<64, false, false, false, false, true>(a, stream);
}

// out[i] = RNE(mul * acc[i]) as 16-bit, eight values per thread and pass.
template <bool BF16>
__global__ void __launch_bounds__(kAuxThreads, kAuxBlocksPerSm) attn_cast_acc_kernel(const float* __restrict__ acc,
                                                                    uint4* __restrict__ out, long long n8,
                                                                    float mul) {
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += nthreads) {
    const float4 x = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 y = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    out[i] = make_uint4(pack2<BF16>(x.x * mul, x.y * mul), pack2<BF16>(x.z * mul, x.w * mul),
                        pack2<BF16>(y.x * mul, y.y * mul), pack2<BF16>(y.z * mul, y.w * mul));
  }
}

cudaError_t launch_cast_acc(const float* acc, void* out, long long n, float mul, int bf16, int sms,
                            cudaStream_t stream) {
  const long long n8 = n / 8;
  long long blocks = (n8 + kAuxThreads - 1) / kAuxThreads;
  const long long cap = (long long)sms * kAuxBlocksPerSm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (bf16)
    attn_cast_acc_kernel<true><<<(unsigned)blocks, kAuxThreads, 0, stream>>>(acc, static_cast<uint4*>(out), n8, mul);
  else
    attn_cast_acc_kernel<false><<<(unsigned)blocks, kAuxThreads, 0, stream>>>(acc, static_cast<uint4*>(out), n8, mul);
  return cudaGetLastError();
}

template <typename U>
cudaError_t launch_dq_post_u(const BwdArgs& a, unsigned grid, cudaStream_t stream) {
  if (a.d == 128)
    return a.bf16 ? launch_pdl(attn_dq_post_kernel<128, true, U>, grid, kAuxThreads, 0, stream, a)
                  : launch_pdl(attn_dq_post_kernel<128, false, U>, grid, kAuxThreads, 0, stream, a);
  return a.bf16 ? launch_pdl(attn_dq_post_kernel<64, true, U>, grid, kAuxThreads, 0, stream, a)
                : launch_pdl(attn_dq_post_kernel<64, false, U>, grid, kAuxThreads, 0, stream, a);
}

cudaError_t launch_dq_post(const BwdArgs& a, cudaStream_t stream) {
  const unsigned grid = (unsigned)(a.sms * kAuxBlocksPerSm);
  return aux_narrow(a) ? launch_dq_post_u<unsigned>(a, grid, stream)
                       : launch_dq_post_u<unsigned long long>(a, grid, stream);
}

}  // namespace attn
