// attn_decode.cu -- decoding against a key/value cache for sm_103a.
//
// Nq query rows, the last Nq positions of a sequence of Nk keys (the KV-cache
// decoding of page "FlashAttention技术解析：如何让GPT训练速度提升5-9倍",
// section 4.1, and page "突破单卡显存极限：FlashAttention-2技术解析与实战指南",
// section 3.2 on vLLM inference): O = softmax(s q K^T [end-aligned causal
// mask]) V and LSE per query row.  Under the causal mask query i sees keys
// j <= Nk - Nq + i.
//
// With few query rows the work is the stream of K and V: each key costs
// 4 d bytes of HBM traffic and 4 Nq d FLOPs, so the path is bound by HBM
// bandwidth, not by the tensor core.  The key range of every (b, h) is split
// into contiguous chunks, one CTA each (enough CTAs to fill the GPU even at
// B*H = 1), and every CTA runs the forward's tile loop on its chunk:
//   S = q K_j^T (tcgen05, the Nq rows padded to one 128-row tile by TMA's
//   zero fill), the running max / running sum recurrence of page
//   "突破单卡显存极限", section 2.1, O += P V_j with P from TMEM,
// and writes its unnormalised O, its reference max m and its sum l to the
// workspace.  A second kernel merges the chunks with the same recurrence:
//   M = max_c m_c,  L = sum_c 2^(m_c - M) l_c,  O = sum_c 2^(m_c - M) O_c / L,
//   LSE = ln 2 (M + log2 L).
//
// sm_103a mapping of the chunk kernel:
//   warps 0-3  softmax: one thread per (padded) query row = TMEM lane;
//   warp 4     TMA producer: q once, K_j and V_j through a ring of slots;
//   warp 5     MMA warp: S_{j+1} into the second S buffer while the softmax
//              works on S_j, then O += P_j V_j; it waits on mbarriers
//              itself (the path is HBM-bound, the MMA time is a fraction
//              of the load time).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kDecThreads = 192;
constexpr int kWarpDecProducer = 4;
constexpr int kWarpDecMma = 5;
constexpr float kDecTau = 8.0f;
constexpr float kDecLn2 = 0.69314718055994530942f;
constexpr float kDecLog2e = 1.44269504088896340736f;

template <int D>
struct DecLayout {
  static constexpr int kSub = 128 * 128;    // one 64-column box: 128 rows x 128 B
  static constexpr int kNSub = D / 64;
  static constexpr int kTile = 128 * D * 2;  // 128 rows of q, K or V
  static constexpr int kSlots = D == 128 ? 6 : 12;
  static constexpr int kQ = 0;
  static constexpr int kSlot0 = kTile;
  static constexpr int kBar = kSlot0 + kSlots * kTile;
  static constexpr int kBarQFull = 0;
  static constexpr int kBarKVFull = 1;
  static constexpr int kBarKVEmpty = kBarKVFull + kSlots;
  static constexpr int kBarSFull = kBarKVEmpty + kSlots;  // [2]
  static constexpr int kBarPFull = kBarSFull + 2;         // [2]
  static constexpr int kBarPVDone = kBarPFull + 2;        // one phase per O += P V_j
  static constexpr int kBarOFull = kBarPVDone + 1;
  static constexpr int kBarDrain = kBarOFull + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kBytes = kTmemSlot + 16;
  static constexpr int kSmem = kBytes + 1024;
  // TMEM columns: two S buffers and O
  static constexpr int kColS0 = 0, kColS1 = 128, kColO = 256;
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

// ALIBI: the scores carry the linear bias -m_h |pos_i - j| (m_h = p.alibi[h],
// pos_i = Nk - Nq + i the query's position), as in the forward.
template <int D, bool BF16, bool ALIBI>
__global__ void __launch_bounds__(kDecThreads, 1)
    attn_decode_split_kernel(const __grid_constant__ DecArgs p) {
  using L = DecLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x % p.n_split;
  const int bh = blockIdx.x / p.n_split;
  const int b = bh / p.H, h = bh % p.H;
  // this CTA's keys [k_lo, k_hi): whole 128-key tiles except at the end
  const int k_lo = split * p.keys_per_split;
  const int k_hi = min(p.Nk, k_lo + p.keys_per_split);
  const int n = k_hi > k_lo ? (k_hi - k_lo + 127) / 128 : 0;
  const WaitCtl wc{p.wait.status, p.wait.limit_ns};

  auto bar = [&](int i) -> uint32_t { return base + L::kBar + 8u * i; };
  auto slot_addr = [&](int s) -> uint32_t { return base + L::kSlot0 + s * L::kTile; };
  // load index of K_j is 2j, of V_j 2j + 1
  auto kv_slot = [&](int i) { return i % L::kSlots; };
  auto kv_par = [&](int i) { return (uint32_t)((i / L::kSlots) & 1); };

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kBarQFull), 1);
    for (int s = 0; s < L::kSlots; ++s) {
      mbar_init(bar(L::kBarKVFull + s), 1);
      mbar_init(bar(L::kBarKVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(L::kBarSFull + t), 1);
      mbar_init(bar(L::kBarPFull + t), 128);
    }
    mbar_init(bar(L::kBarPVDone), 1);
    mbar_init(bar(L::kBarOFull), 1);
    mbar_init(bar(L::kBarDrain), 1);
    fence_mbar_init();
  }
  if (warp == kWarpDecProducer) {
    tmem_alloc(base + L::kTmemSlot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sbase + L::kTmemSlot);

  if (warp == kWarpDecProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0 && !(p.debug_flags & 4)) {
      tma_prefetch(&p.tm_q);
      tma_prefetch(&p.tm_k);
      tma_prefetch(&p.tm_v);
      mbar_expect_tx(bar(L::kBarQFull), L::kTile);
      for (int s = 0; s < L::kNSub; ++s)
        tma_load_4d(base + L::kQ + s * L::kSub, &p.tm_q, bar(L::kBarQFull), s * 64, h, 0, b);
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < n && ok; ++j) {
        for (int kind = 0; kind < 2; ++kind) {
          const int slot = kv_slot(issued);
          if (!mbar_wait(bar(L::kBarKVEmpty + slot), kv_par(issued) ^ 1, wc)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar(L::kBarKVFull + slot), L::kTile);
          const CUtensorMap* m = kind ? &p.tm_v : &p.tm_k;
          for (int s = 0; s < L::kNSub; ++s)
            tma_load_4d(slot_addr(slot) + s * L::kSub, m, bar(L::kBarKVFull + slot), s * 64, h,
                        k_lo + j * 128, b);
          ++issued;
        }
      }
      if (!ok) {
        mbar_wait_drain(bar(L::kBarQFull), 0, wc.limit_ns);
        for (int i = max(0, issued - L::kSlots); i < issued; ++i)
          mbar_wait_drain(bar(L::kBarKVFull + kv_slot(i)), kv_par(i), wc.limit_ns);
      }
    }
  } else if (warp == kWarpDecMma) {
    // ------------------------------------------------------------ MMA warp
    // Converged warp, one elected lane issues.  Order per key tile j:
    //   S_{j+1} = q K_{j+1}^T into buffer (j+1) & 1 (that buffer's P_{j-1}
    //   was read by O += P_{j-1} V_{j-1}, issued before it), then
    //   O += P_j V_j, whose completion releases K_j and V_j.
    constexpr uint32_t idesc_s = make_idesc(BF16, 128, 128, false, false);
    constexpr uint32_t idesc_o = make_idesc(BF16, 128, D, false, true);
    auto w = [&](int i, uint32_t parity) { return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, wc)); };
    auto issue_s = [&](int j) {
      const uint32_t kaddr = slot_addr(kv_slot(2 * j));
      const uint32_t dS = tmem + ((j & 1) ? L::kColS1 : L::kColS0);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t off = (ks >> 2) * L::kSub + (ks & 3) * 32;
        mma_ss(dS, make_sdesc(base + L::kQ + off, 16, 1024), make_sdesc(kaddr + off, 16, 1024),
               idesc_s, ks > 0);
      }
    };
    bool ok = n > 0 && w(L::kBarQFull, 0) && w(L::kBarKVFull + kv_slot(0), kv_par(0));
    if (ok) {
      tc_fence_after();
      issue_s(0);
      tc_commit(bar(L::kBarSFull + 0));
    }
    for (int j = 0; ok && j < n; ++j) {
      if (j + 1 < n) {
        ok = w(L::kBarKVFull + kv_slot(2 * j + 2), kv_par(2 * j + 2));
        if (!ok) break;
        tc_fence_after();
        issue_s(j + 1);
        tc_commit(bar(L::kBarSFull + ((j + 1) & 1)));
      }
      ok = w(L::kBarPFull + (j & 1), (j >> 1) & 1) && w(L::kBarKVFull + kv_slot(2 * j + 1), kv_par(2 * j + 1));
      if (!ok) break;
      tc_fence_after();
      const uint32_t vaddr = slot_addr(kv_slot(2 * j + 1));
      const uint32_t aP = tmem + ((j & 1) ? L::kColS1 : L::kColS0);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_ts(tmem + L::kColO, aP + ks * 8, make_sdesc(vaddr + ks * 2048, L::kSub, 1024), idesc_o,
               (j > 0 || ks > 0) ? 1u : 0u);
      tc_commit(bar(L::kBarPVDone));
      tc_commit(bar(L::kBarKVEmpty + kv_slot(2 * j)));
      tc_commit(bar(L::kBarKVEmpty + kv_slot(2 * j + 1)));
    }
    if (ok && n > 0) tc_commit(bar(L::kBarOFull));
    tc_commit(bar(L::kBarDrain));
    mbar_wait_drain(bar(L::kBarDrain), 0, wc.limit_ns);
  } else {
    // ------------------------------------------------------------ softmax
    const int qd = warp & 3;
    const int row = qd * 32 + lane;  // query row (rows >= Nq are TMA zero fill)
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const uint32_t tO = tmem + lane_off + L::kColO;
    const float c = p.scale * kDecLog2e;
    // keys < lim are visible to this row
    const int lim = p.causal ? min(k_hi, p.Nk - p.Nq + row + 1) : k_hi;
    const int lim_warp_min = p.causal ? min(k_hi, p.Nk - p.Nq + qd * 32 + 1) : k_hi;
    const float slope2 = ALIBI ? p.alibi[h] * kDecLog2e : 0.f;  // ALiBi slope, log2 units
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarSFull + (j & 1)), (j >> 1) & 1, wc));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + ((j & 1) ? L::kColS1 : L::kColS0);
      uint32_t s[128];
      tmem_ld32(tS + 0, s);
      tmem_ld32(tS + 32, s + 32);
      tmem_ld32(tS + 64, s + 64);
      tmem_ld32(tS + 96, s + 96);
      tmem_ld_wait();
      reg_fence<128>(s);
      const int kv0 = k_lo + j * 128;
      if (kv0 + 128 > lim_warp_min) {
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (kv0 + i >= lim) s[i] = __float_as_uint(-INFINITY);
      }
      if constexpr (ALIBI) {
        // s <- s * scale * log2(e) - m |pos - key|, linear in the column
        // unless the tile straddles the row's position.
        const int r0 = p.Nk - p.Nq + row - kv0;
        const bool left = __all_sync(0xffffffffu, r0 >= 127), right = __all_sync(0xffffffffu, r0 <= 0);
        if (left || right) {
          const float k1 = left ? slope2 : -slope2, k0 = -k1 * (float)r0;
#pragma unroll
          for (int i = 0; i < 128; ++i)
            s[i] = __float_as_uint(fmaf(__uint_as_float(s[i]), c, fmaf((float)i, k1, k0)));
        } else {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            s[i] = __float_as_uint(
                fmaf(__uint_as_float(s[i]), c, -slope2 * fabsf((float)(r0 - i))));
        }
      }
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
      const float m_tile =
          max3(max3(mk[0], mk[1], mk[2]), max3(mk[3], mk[4], mk[5]), fmaxf(mk[6], mk[7])) *
          (ALIBI ? 1.f : c);  // with ALiBi the scale is already applied
      float alpha = 1.f;
      if (m_tile > m_ref + kDecTau) {  // move the reference only by more than 2^tau
        alpha = ex2(m_ref - m_tile);    // 0 on the first visible tile
        m_ref = m_tile;
      }
      const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O <- alpha O once O += P_{j-1} V_{j-1} has completed (S_j was
        // issued before it, so S_j complete does not imply it).
        ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarPVDone), (j - 1) & 1, wc));
        if (!ok) break;
        tc_fence_after();
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
      const float2 c2 = make_float2(c, c), neg2 = make_float2(neg, neg);
      float2 sk[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};
      uint32_t pk[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const float2 sv = make_float2(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
        const float2 x = ALIBI ? add2(sv, neg2) : fma2(sv, c2, neg2);
        const float2 e = make_float2(ex2(x.x), ex2(x.y));
        sk[i & 3] = add2(sk[i & 3], e);
        pk[i] = pack2<BF16>(e.x, e.y);
      }
      tmem_st32(tS, pk);
      tmem_st32(tS + 32, pk + 32);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(L::kBarPFull + (j & 1)));
      const float2 s01 = add2(add2(sk[0], sk[1]), add2(sk[2], sk[3]));
      l = l * alpha + (s01.x + s01.y);
    }
    if (n > 0 && ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarOFull), 0, wc));
    // Partial results of this chunk; rows past Nq (TMA zero fill) are not
    // written, but their lanes take part in the warp-wide TMEM loads.
    const size_t part = ((size_t)bh * p.n_split + split) * p.Nq + row;
    const bool have = ok && n > 0;  // warp-uniform
    if (have) {
      tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < D; cc += 32) {
        uint32_t o[32];
        tmem_ld32(tO + cc, o);
        tmem_ld_wait();
        reg_fence<32>(o);
        if (row < p.Nq) {
          float4* dst = reinterpret_cast<float4*>(p.ws_o + part * D + cc);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                                 __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
        }
      }
    }
    if (row < p.Nq) {
      // a chunk without a visible key (or one that gave up) contributes nothing
      p.ws_ml[part * 2 + 0] = have ? m_ref : -INFINITY;
      p.ws_ml[part * 2 + 1] = have ? l : 0.f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpDecProducer) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// One warp per (b, h, query row): merges the chunks of that row.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_decode_merge_kernel(const __grid_constant__ DecArgs p) {
  const long long wg = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)p.B * p.H * p.Nq;
  if (wg >= rows) return;
  const int bh = (int)(wg / p.Nq), row = (int)(wg % p.Nq);
  const int b = bh / p.H, h = bh % p.H;
  constexpr int kPer = D / 32;  // output columns per lane
  float M = -INFINITY;
  for (int c = 0; c < p.n_split; ++c)
    M = fmaxf(M, p.ws_ml[(((size_t)bh * p.n_split + c) * p.Nq + row) * 2]);
  float Lsum = 0.f;
  float acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  for (int c = 0; c < p.n_split; ++c) {
    const size_t part = ((size_t)bh * p.n_split + c) * p.Nq + row;
    const float mc = p.ws_ml[part * 2], lc = p.ws_ml[part * 2 + 1];
    if (mc == -INFINITY) continue;  // no visible key in this chunk
    const float wgt = ex2(mc - M);
    Lsum = fmaf(wgt, lc, Lsum);
    const float* oc = p.ws_o + part * D + lane * kPer;
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = fmaf(wgt, oc[i], acc[i]);
  }
  const float inv = 1.f / Lsum;
  uint32_t wv[kPer / 2];
#pragma unroll
  for (int i = 0; i < kPer / 2; ++i) wv[i] = pack2<BF16>(acc[2 * i] * inv, acc[2 * i + 1] * inv);
  uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) + ((((size_t)b * p.Nq + row) * p.H + h) * D + lane * kPer) * 2;
  if constexpr (kPer == 4)
    *reinterpret_cast<uint2*>(orow) = make_uint2(wv[0], wv[1]);
  else
    *reinterpret_cast<uint32_t*>(orow) = wv[0];
  if (lane == 0) p.lse[(size_t)bh * p.Nq + row] = (M + __log2f(Lsum)) * kDecLn2;
}

template <int D, bool BF16, bool ALIBI>
cudaError_t launch_split_t(const DecArgs& a, cudaStream_t stream) {
  using L = DecLayout<D>;
  auto* k = attn_decode_split_kernel<D, BF16, ALIBI>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)((long long)a.B * a.H * a.n_split);
  k<<<grid, kDecThreads, L::kSmem, stream>>>(a);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_merge_t(const DecArgs& a, cudaStream_t stream) {
  const long long warps = (long long)a.B * a.H * a.Nq;
  const unsigned grid = (unsigned)((warps + 7) / 8);
  attn_decode_merge_kernel<D, BF16><<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

int decode_n_split(int B, int H, int Nk) {
  // Chunks of whole 128-key tiles, at least two tiles each, about two CTAs
  // per SM of a GB300 (152 SMs) in total, at most kDecodeMaxSplit per head;
  // then as few chunks as the resulting chunk length needs (none empty).
  const int tiles = (Nk + 127) / 128;
  const long long bh = (long long)B * H;
  long long want = (2 * 152 + bh - 1) / bh;
  if (want > (tiles + 1) / 2) want = (tiles + 1) / 2;
  if (want > kDecodeMaxSplit) want = kDecodeMaxSplit;
  if (want < 1) want = 1;
  const long long per = (tiles + want - 1) / want;
  return (int)((tiles + per - 1) / per);
}

int decode_smem_bytes(int d) { return d == 128 ? DecLayout<128>::kSmem : DecLayout<64>::kSmem; }

int decode_keys_per_split(int Nk, int n_split) {
  const int tiles = (Nk + 127) / 128;
  return (tiles + n_split - 1) / n_split * 128;
}

cudaError_t launch_decode_split(const DecArgs& a, cudaStream_t stream) {
  if (a.alibi) {
    if (a.d == 128) return a.bf16 ? launch_split_t<128, true, true>(a, stream) : launch_split_t<128, false, true>(a, stream);
    return a.bf16 ? launch_split_t<64, true, true>(a, stream) : launch_split_t<64, false, true>(a, stream);
  }
  if (a.d == 128) return a.bf16 ? launch_split_t<128, true, false>(a, stream) : launch_split_t<128, false, false>(a, stream);
  return a.bf16 ? launch_split_t<64, true, false>(a, stream) : launch_split_t<64, false, false>(a, stream);
}

cudaError_t launch_decode_merge(const DecArgs& a, cudaStream_t stream) {
  if (a.d == 128) return a.bf16 ? launch_merge_t<128, true>(a, stream) : launch_merge_t<128, false>(a, stream);
  return a.bf16 ? launch_merge_t<64, true>(a, stream) : launch_merge_t<64, false>(a, stream);
}

}  // namespace attn
