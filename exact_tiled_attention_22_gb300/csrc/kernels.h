// kernels.h -- internal interface between the C-ABI host layer and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace attn {

// Kernel ids used by the per-kernel timing of attn_profile_*.
enum KernelId {
  kKFwd = 0, kKBwdPre = 1, kKBwdMain = 2, kKDqPost = 3, kKDecSplit = 4, kKDecMerge = 5, kKNum = 6
};

struct WaitCtlHost {
  int* status;
  unsigned long long limit_ns;
};

// Dropout of the attention probabilities (see dropout.cuh): Philox4x32-10
// key (k0, k1) = the seed's low and high words, counter word 3 = offset;
// a score is kept iff its byte is below t, cmp = (256 - t) * 0x00010001;
// kept probabilities are multiplied by scale = 256 / t.  t = 256: no dropout.
// Philox4x32-10 key schedule (Salmon et al., SC 2011): the round key is
// (k0, k1) advanced by these Weyl increments once per round.
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u, kPhiloxW1 = 0xBB67AE85u;

struct DropoutArgs {
  uint32_t k0, k1;
  uint32_t offset;
  uint32_t cmp;
  float scale;
  int t;
  // round keys of rounds 0..9: rk[2r] = k0 + r W0, rk[2r + 1] = k1 + r W1
  // (mod 2^32), filled on the host so that each round's key xor reads a
  // kernel parameter instead of an addition per call
  uint32_t rk[20];
};

// Accumulation flags of attn_fwd_acc / attn_bwd_acc (values of attn.h).
constexpr int kAccFirst = 1;  // no earlier partial: start the accumulators
constexpr int kAccLast = 2;   // final partial: write the 16-bit result

// Forward: one CTA per (pair of 128-row query tiles, b, h).
struct FwdArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // [B,N,H,d], boxes of 64 columns x 128 rows
  CUtensorMap tm_o;              // the store of O, same boxes
  void* o;
  float* lse;
  // Accumulating variant (attn_fwd_acc): o_acc fp32 [B,N,H,d] and lse the
  // running natural-log LSE; o written (16-bit) on the last partial only.
  float* o_acc;
  int acc_flags;
  const float* alibi;  // ALiBi slope per head [H] (device), or null
  const uint8_t* bmask;  // block-sparse mask [H][nb][nb], nb = ceil(N/128) (device), or null
  DropoutArgs drop;
  int B, H, N, d;
  int causal;
  float scale;
  int bf16;
  int debug_flags;
  WaitCtlHost wait;
};
int fwd_smem_bytes(int d);
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);

// Largest N / 128 the block-sparse variants take.
constexpr int kMaxSparseTiles = 512;

// Backward.  Workspace regions (fp32): lse2 [BH][Npad] (-LSE * log2 e),
// dvec [BH][Npad] (D = rowsum(dO * O)), dqacc [BH][Npad][d], Npad = N
// rounded up to 128; then 256 bytes holding the main kernel's work counter.
struct BwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // q/do boxes of bwd_q_rows(d) rows, k/v 128 rows
  CUtensorMap tm_dk, tm_dv;             // stores of dK, dV: boxes of 64 columns x 128 rows
  const void* o;
  const void* dO;
  const float* lse;
  const float* alibi;  // ALiBi slope per head [H] (device), or null
  const uint8_t* bmask;  // block-sparse mask [H][nb][nb] (device), or null
  DropoutArgs drop;
  float* lse2;
  float* dvec;
  float* dqacc;
  unsigned* sched;  // [2] item counter of the persistent main kernel and its exit count
  void* dq;
  void* dk;
  void* dv;
  // Accumulating variant (attn_bwd_acc): dK and dV are added into these fp32
  // [B,N,H,d] accumulators (stored instead when kv_flags has kAccFirst)
  // instead of being written as 16-bit dk, dv.
  float* dk_acc;
  float* dv_acc;
  int kv_flags;
  int B, H, N, Npad, d;
  int causal;
  float scale;
  int bf16;
  int sms;  // SM count of the device (grid size of the memory-bound kernels)
  int debug_flags;  // bit 1: the main kernel loads K and V but no query steps (timeout tests);
                   // bit 3: 64-bit row splits in the pre / post kernels
  WaitCtlHost wait;
};
int bwd_q_rows(int d);
int bwd_smem_bytes(int d);
cudaError_t launch_bwd_pre(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_main_acc(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_fwd_acc(const FwdArgs& a, cudaStream_t stream);
// 16-bit out[i] = RNE(mul * acc[i]) for n fp32 values (n % 8 == 0).
cudaError_t launch_cast_acc(const float* acc, void* out, long long n, float mul, int bf16, int sms,
                            cudaStream_t stream);
cudaError_t launch_bwd_main(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_dq_post(const BwdArgs& a, cudaStream_t stream);

// Decoding against a key/value cache: q, o [B, Nq, H, d], k, v [B, Nk, H, d],
// lse [B, H, Nq].  Workspace (fp32): ws_o [B*H*n_split][Nq][d] (unnormalised
// chunk outputs), ws_ml [B*H*n_split][Nq][2] (reference max in log2 units,
// sum).
constexpr int kDecodeMaxSplit = 64;
struct DecArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // boxes of 64 columns x 128 rows
  void* o;
  float* lse;
  const float* alibi;  // ALiBi slope per head [H] (device), or null
  float* ws_o;
  float* ws_ml;
  int B, H, Nq, Nk, d;
  int n_split, keys_per_split;
  int causal;
  float scale;
  int bf16;
  int debug_flags;  // bit 2: the chunk kernel loads nothing (timeout tests)
  WaitCtlHost wait;
};
int decode_n_split(int B, int H, int Nk);
int decode_keys_per_split(int Nk, int n_split);
int decode_smem_bytes(int d);
cudaError_t launch_decode_split(const DecArgs& a, cudaStream_t stream);
cudaError_t launch_decode_merge(const DecArgs& a, cudaStream_t stream);

// Id of the calling thread's current CUDA context (unique for the life of
// the process, unlike the CUcontext handle, which a new context may reuse).
// The thread must have a current context (the runtime binds the device's
// primary context on cudaSetDevice or any runtime call that needs one).
cudaError_t current_context_id(unsigned long long* id);

// Launches `kernel` on `stream` with programmatic stream serialization, so
// that it can start (and wait in griddep_wait) while the kernel before it
// finishes.  Every kernel of the library lets its dependents be scheduled
// only at its end (griddep_launch_dependents after its last work): with the
// trigger at the start, the next kernel's CTAs became resident early and a
// back-to-back fwd+bwd step ran 1-2 % slower at N = 8192 and 32768; at the
// end the launch latency is still hidden (10 % on the encoder shape against
// plain launches).
template <typename Arg>
cudaError_t launch_pdl(void (*kernel)(Arg), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                       const Arg& arg) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, arg);
}

// Sets the calling thread's attn_last_error_string() text (printf format).
void set_last_error(const char* fmt, ...) __attribute__((format(printf, 1, 2)));

}  // namespace attn
