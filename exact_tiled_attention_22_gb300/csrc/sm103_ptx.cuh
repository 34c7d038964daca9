// sm103_ptx.cuh -- thin inline-PTX wrappers for the sm_103a features the
// attention kernels use: mbarriers, TMA (cp.async.bulk.tensor), tcgen05 MMA
// with TMEM accumulators, TMEM loads/stores, and bounded waits.
//
// Written from the public PTX ISA descriptions of these instructions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

namespace attn {

// Device status codes written into the per-device status word.
constexpr int kDevOk = 0;
constexpr int kDevTimeout = 1;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- launches
// Programmatic dependent launch: a kernel launched with the programmatic
// stream serialization attribute may start while the kernel before it on the
// stream is still running.  griddep_wait() blocks the calling thread until
// that kernel has completed and its memory operations are visible (a no-op
// without the attribute); every thread calls it before its first access to
// global memory.  griddep_launch_dependents() lets the next kernel be
// scheduled once every CTA of this grid has called it (or exited).
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// `count` arrivals at once (count >= 1).
__device__ __forceinline__ void mbar_arrive_n(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P1;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P1;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok;
}

// Everything a bounded wait needs: the device status word and the limit.
struct WaitCtl {
  int* status;         // per-device status word (global memory)
  uint64_t limit_ns;   // give up after this long
};

// Waits for the phase of parity `parity` of barrier `bar` to complete.
// Returns false if the wait gave up: either the time limit ran out (the
// status word is then set to kDevTimeout) or another wait on the device had
// already given up (status word nonzero).  Never traps.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          const WaitCtl& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 31u) == 0) {
      if (*reinterpret_cast<volatile int*>(w.status) != kDevOk) return false;
      if (globaltimer_ns() - t0 > w.limit_ns) {
        atomicCAS(w.status, kDevOk, kDevTimeout);
        return false;
      }
    }
  }
}

// Same, but ignores the status word: used only on the way out of a kernel
// that already gave up, to let asynchronous copies and MMAs it issued land
// before shared memory and tensor memory are released.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity,
                                                uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map))
               : "memory");
}

// 4-D tiled load into shared memory; completion is signalled on `bar`
// through the transaction count.  c0 is the innermost coordinate.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map,
                                            uint32_t bar, int c0, int c1, int c2,
                                            int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3)
      : "memory");
}

// 4-D tiled store shared -> global, tracked by bulk groups (bulk_commit /
// bulk_wait_*).  c0 is the innermost coordinate (c0 * element size a
// multiple of 16 bytes); rows outside the tensor are not written.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2,
                                             int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// Plain bulk copy global -> shared (both 16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src,
                                          uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Barrier over `count` threads (a multiple of 32, whole warps) on hardware
// barrier `id` that also ANDs a flag across them: every participant gets the
// same answer, so code after it can branch uniformly (for example on whether
// a bounded wait gave up).  Used as the hand-off between the warp that waits
// on mbarriers and the warp that issues tcgen05.mma: an mbarrier wait (or any
// shared-memory access) in the issuing thread holds it until its in-flight
// MMAs drain, while a named barrier does not.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Barrier over `count` threads (whole warps) on hardware barrier `id`.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Bulk reduction shared -> global: dst[i] += src[i] for `bytes` / 4 fp32
// values (both 16-byte aligned, bytes % 16 == 0), tracked by bulk groups.
__device__ __forceinline__ void bulk_reduce_add_f32(float* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile(
      "cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
          reinterpret_cast<uint64_t>(gdst)),
      "r"(ssrc), "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until all but the most recently committed bulk group of this thread
// have finished reading their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read_but_last() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Waits until every committed bulk group of this thread has finished
// reading its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Makes this thread's generic-proxy shared-memory writes visible to the
// async proxy (tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// The MMA and commit wrappers below are warp-collective: every lane of a
// converged warp calls them with the same arguments, and one lane, chosen by
// elect.sync (the same lane each time in a fully converged warp), issues the
// instruction.  Keeping the issuing warp converged matters: a thread that
// leaves a divergent branch around its MMAs and reconverges with its warp
// waits for the tensor pipe to take them, which idles the pipe at every such
// point and makes the issue rate sensitive to the arithmetic of other warps
// on the same scheduler.
//
// Arrives once on `bar` when every tcgen05 operation issued before it by the
// elected thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// D(tmem) (+)= A(smem desc) * B(smem desc) per the instruction descriptor;
// accumulate when acc != 0.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
// Same with the A operand read from tensor memory.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                       uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

// Instruction descriptor for kind::f16 with fp32 accumulation.
//   bits 4-5 D type (1 = f32); 7-9 A type, 10-12 B type (0 f16, 1 bf16);
//   15 / 16: A / B MN-major; 17-22 N >> 3; 24-28 M >> 4.
__host__ __device__ constexpr uint32_t make_idesc(bool bf16, int M, int N, bool a_mn,
                                                  bool b_mn) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle, version 1.
//   bits 0-13 start >> 4; 16-29 leading byte offset >> 4;
//   32-45 stride byte offset >> 4; 46-47 version (1); 61-63 layout (2 = 128B).
// Tiles are stored as 8-row x 128-byte swizzle atoms, atoms of consecutive
// rows 1024 bytes apart (SBO = 1024).  LBO is the distance between 64-element
// column blocks and matters only for MN-major operands wider than 64.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo,
                                               uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) |
         ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// ---- TMEM loads / stores: 32 lanes x 32-bit, one lane (row) per thread.
// Warp w of a warpgroup may touch lanes [32*(w%4), 32*(w%4)+32).
#define ATTN_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                   "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define ATTN_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                   "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : ATTN_R8(0), ATTN_R8(8), ATTN_R8(16), ATTN_R8(24)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      ATTN_W8(0), ATTN_W8(8), ATTN_W8(16), ATTN_W8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      ATTN_W8(0), ATTN_W8(8)
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : ATTN_R8(0), ATTN_R8(8)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               ATTN_W8(0)
               : "memory");
}
// 32 or 16 columns of this thread's TMEM lane, by width
template <int W>
__device__ __forceinline__ void tmem_ld_w(uint32_t taddr, uint32_t* r) {
  static_assert(W == 32 || W == 16, "width");
  if constexpr (W == 32) tmem_ld32(taddr, r); else tmem_ld16(taddr, r);
}
template <int W>
__device__ __forceinline__ void tmem_st_w(uint32_t taddr, const uint32_t* r) {
  static_assert(W == 16 || W == 8, "width");
  if constexpr (W == 16) tmem_st16(taddr, r); else tmem_st8(taddr, r);
}
#undef ATTN_R8
#undef ATTN_W8

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// After tmem_ld_wait(): ties the loaded registers to this point so the
// compiler cannot move their first use above the wait.
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t* r) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i])::"memory");
}

// ---------------------------------------------------------------- math
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- Paired fp32 arithmetic: one instruction on two independent lanes of a
// float2, each lane rounded exactly like the scalar operation (the .rn forms
// of fma/add/sub/mul on f32x2 operands).
#define ATTN_F2_IN(v) "f"((v).x), "f"((v).y)
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : ATTN_F2_IN(a), ATTN_F2_IN(b), ATTN_F2_IN(c));
  return d;
}
#define ATTN_F2_BINOP(name, op)                                                   \
  __device__ __forceinline__ float2 name(float2 a, float2 b) {                   \
    float2 d;                                                                     \
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"                                         \
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t" op                   \
        " rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"                               \
        : "=f"(d.x), "=f"(d.y) : ATTN_F2_IN(a), ATTN_F2_IN(b));                   \
    return d;                                                                     \
  }
ATTN_F2_BINOP(add2, "add.rn.f32x2")
ATTN_F2_BINOP(sub2, "sub.rn.f32x2")
ATTN_F2_BINOP(mul2, "mul.rn.f32x2")
#undef ATTN_F2_BINOP

// Three-input maximum.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packs two fp32 values into one 32-bit word of 16-bit floats (RNE):
// `lo` in bits 0-15 (the lower column / k index), `hi` in bits 16-31.
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  if constexpr (BF16) {
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  }
  return r;
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  float2 f;
  if constexpr (BF16) {
    f.x = __uint_as_float(w << 16);
    f.y = __uint_as_float(w & 0xFFFF0000u);
  } else {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    f = __half22float2(h);
  }
  return f;
}

}  // namespace attn
