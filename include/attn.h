/*
 * attn.h -- C ABI of the exact tiled attention library for NVIDIA GB300
 * (sm_103a).  Library: exact_tiled_attention_22_gb300/libattn.so.
 *
 * What is computed.  For every batch b and head h, with one scale s:
 *
 *   S = s * Q K^T,  P = softmax_row(S) (keys j > query i removed when causal),
 *   O = P V,        LSE_i = log sum_j exp(S_ij)   (natural log)
 *
 * i.e. standard attention as written in page "突破单卡显存极限：FlashAttention-2
 * 技术解析与实战指南", section 1 (S = Q @ K.T, P = softmax(S), P @ V), with the
 * scale and causal switch of the call in page "Flash Attention V2大模型时代的算力
 * 救星", section 4.2 (flash_attention(q, k, v, softmax_scale=1.0/sqrt(d_k),
 * causal=...)).  The forward is computed tile by tile with the running max / running
 * sum recurrence of page "突破单卡显存极限", section 2.1, so no N x N matrix
 * is ever stored; only the per-row statistic LSE is kept (page "Flash
 * Attention V2大模型时代的算力救星", section 3.2: keep the softmax normalisation
 * statistics, not the matrix).  The backward recomputes P from LSE (same
 * section; page "突破单卡显存极限", section 2.2) and returns the gradients of
 * L = sum(O * dO):
 *
 *   dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic,  dS = P * (dP - D),
 *   dQ = s dS K,  dK = s dS^T Q.
 *
 * The result is exact attention up to floating-point rounding (fp32
 * accumulation; P and dS are rounded to the input type before the second
 * matrix product of each pair).
 *
 * Layout.  Q, K, V, O, dO, dQ, dK, dV: contiguous row-major [B, N, H, d]
 * arrays of `dtype` (element (b, n, h, c) at ((b*N + n)*H + h)*d + c) -- the
 * sequence-major layout recommended in page "Flash Attention V2大模型时代的算力
 * 救星", section 5.2.  LSE: contiguous fp32 [B, H, N].
 *
 * Pointers.  All pointers are device pointers, 16-byte aligned.  The caller
 * owns every buffer, including the backward workspace; the library allocates
 * nothing in these calls and does not synchronise the stream, so the calls
 * can be issued back to back or captured.  Outputs and workspaces must not
 * overlap one another or any input (the ALiBi slopes and the block mask
 * included); a call in which they do is refused with ATTN_ERR_INVALID.
 *
 * Streams.  `stream` is a cudaStream_t (NULL = legacy default stream).  Work
 * is enqueued on it; host-side argument errors return before anything is
 * enqueued.  Device-side errors (a bounded wait that expired) are recorded
 * in a per-device status word that attn_status() reads.
 *
 * Threads.  Any host thread may call; the calls act on the thread's current
 * device and make its primary context current on the thread if none is.
 *
 * Supported: d in {64, 128}; dtype fp16 or bf16; B, H, N >= 1 with
 * B*H*ceil(N/128) < 2^31, B*H < 2^25 and B*H*N*d < 2^40 (tensors may hold
 * more than 2^31 elements); any N (tails are masked in-kernel, no padding
 * needed);
 * scale finite and > 0.  Devices other than compute capability 10.3 are
 * rejected with ATTN_ERR_UNSUPPORTED: there is no fallback path.
 */
#ifndef EXACT_TILED_ATTENTION_ATTN_H
#define EXACT_TILED_ATTENTION_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTN_F16 = 0, ATTN_BF16 = 1 } attn_dtype_t;

#define ATTN_OK 0
#define ATTN_ERR_INVALID -1     /* null pointer, B/H/N < 1, size overflow,
                                   scale not finite or <= 0, aliasing */
#define ATTN_ERR_UNSUPPORTED -2 /* d not in {64,128}, unknown dtype, or the
                                   current device is not sm_103 */
#define ATTN_ERR_ALIGN -3       /* a pointer is not 16-byte aligned */
#define ATTN_ERR_CUDA -4        /* a CUDA runtime/driver call failed */
#define ATTN_ERR_TIMEOUT -5     /* a device-side bounded wait expired
                                   (reported by attn_status) */
#define ATTN_ERR_WORKSPACE -6   /* backward workspace missing or too small */

/*
 * attn_fwd -- forward pass.
 *   q, k, v : [B, N, H, d] inputs (read only).
 *   o       : [B, N, H, d] output, same dtype.
 *   lse     : [B, H, N] fp32 output, natural-log logsumexp of the scaled,
 *             masked scores of each query row.
 *   scale   : the score scale s (usually 1/sqrt(d)).
 *   causal  : nonzero removes keys j > i from query row i.
 * Returns ATTN_OK or a negative ATTN_ERR_* code (nothing enqueued on error).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int H, int N, int d, float scale, int causal,
             attn_dtype_t dtype, void* stream);

/*
 * attn_bwd_workspace_size -- bytes of device workspace attn_bwd needs:
 * fp32 D and scaled LSE rows plus an fp32 dQ accumulator, each over
 * B*H*Npad rows with Npad = N rounded up to 128, and 256 bytes for the
 * work counter of the backward's persistent main kernel; linear in N (no
 * N x N term).  Returns 0 for invalid sizes.
 */
size_t attn_bwd_workspace_size(int B, int H, int N, int d);

/*
 * attn_bwd -- backward pass.
 *   q, k, v, o, lse : the forward's inputs and outputs (o and lse exactly as
 *                     attn_fwd wrote them).
 *   dO              : [B, N, H, d] gradient of the loss w.r.t. o.
 *   dq, dk, dv      : [B, N, H, d] outputs.
 *   workspace       : device buffer of at least
 *                     attn_bwd_workspace_size(B, H, N, d) bytes, 256-byte
 *                     aligned, owned by the caller; its contents on entry do
 *                     not matter and on return are unspecified.
 * The dQ partial sums of the key blocks are added into an fp32 accumulator
 * in whatever order the blocks finish, so dq may differ in the last bits
 * between runs.  Returns ATTN_OK or a negative ATTN_ERR_* code.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o,
             const float* lse, const void* dO, void* dq, void* dk, void* dv,
             int B, int H, int N, int d, float scale, int causal,
             attn_dtype_t dtype, void* workspace, size_t workspace_bytes,
             void* stream);

/*
 * attn_bwd_noalloc -- attn_bwd for callers that cannot allocate device memory.
 *
 * The pages describe no such call; it is an interface addition of this
 * library.  It exists for callers that have no way to hand attn_bwd a
 * workspace: plain C code embedded in a host program or plugin that owns no
 * CUDA memory pool and gets no allocator handle, and latency-critical loops
 * that must not call cudaMalloc because it can synchronise the device.
 *
 * Arguments, layout, results and error codes are those of attn_bwd, minus
 * the workspace: the scratch lives in a file-scope __device__ array of
 * ATTN_NOALLOC_WORKSPACE_BYTES (32 MiB) owned by the library, present on
 * every GPU that loads the library's device code and held until the process
 * exits.  No cudaMalloc, cudaFree or other allocating routine is called.
 *   - Shapes whose attn_bwd_workspace_size(B, H, N, d) exceeds
 *     ATTN_NOALLOC_WORKSPACE_BYTES are rejected with ATTN_ERR_WORKSPACE
 *     (B*H*Npad <= 64512 rows at d = 128 and <= 126976 rows at d = 64,
 *     Npad = N rounded up to 128).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current), which may load the
 *     library's device code there; make that first call before any stream
 *     capture.  The address is kept per device and per context: a call made
 *     in another context of the device looks it up again.
 *   - Every call on a device shares the one array.  Each call rewrites the
 *     part it uses (the dQ accumulator is zeroed, D and the scaled LSE are
 *     overwritten), so results never depend on an earlier call, but calls
 *     whose kernels overlap on the GPU (e.g. on two streams) race on it.
 */
#define ATTN_NOALLOC_WORKSPACE_BYTES (32u * 1024u * 1024u)
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dO, void* dq, void* dk,
                     void* dv, int B, int H, int N, int d, float scale,
                     int causal, attn_dtype_t dtype, void* stream);

/*
 * ALiBi variants (page "FlashAttention技术解析：如何让GPT训练速度提升5-9倍",
 * section 4.1, names Attention with Linear Biases for long contexts).  Same
 * arguments as attn_fwd / attn_bwd / attn_decode plus
 *   alibi_slopes : device pointer to fp32 [H], the slope m_h of each head
 *                  (finite, >= 0), or NULL for no bias (the plain call).
 * The scores become S_ij = s * <q_i, k_j> - m_h |pos_i - j|, pos_i the
 * query's position in the sequence (i for attn_fwd/attn_bwd, Nk - Nq + i
 * for attn_decode); LSE is of these biased scores, and attn_bwd_alibi must be
 * given the forward's o and lse from attn_fwd_alibi with the same slopes.
 * The slopes are read on the device; nothing checks their values.
 */
int attn_fwd_alibi(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int N, int d, float scale, int causal,
                   const float* alibi_slopes, attn_dtype_t dtype, void* stream);
int attn_bwd_alibi(const void* q, const void* k, const void* v, const void* o,
                   const float* lse, const void* dO, void* dq, void* dk, void* dv,
                   int B, int H, int N, int d, float scale, int causal,
                   const float* alibi_slopes, attn_dtype_t dtype, void* workspace,
                   size_t workspace_bytes, void* stream);
int attn_decode_alibi(const void* q, const void* k, const void* v, void* o,
                      float* lse, int B, int H, int Nq, int Nk, int d, float scale,
                      int causal, const float* alibi_slopes, attn_dtype_t dtype,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * Block-sparse variants (page "FlashAttention技术解析：如何让GPT训练速度提升5-9倍",
 * section 5.2, names Block-Sparse FlashAttention: tiles whose mask block is
 * zero are skipped, so the work scales with the kept blocks).  Same arguments
 * as attn_fwd_alibi / attn_bwd_alibi (alibi_slopes may be NULL) plus
 *   block_mask : device pointer to uint8 [H][nb][nb], nb = ceil(N / 128),
 *                or NULL (then identical to the ALiBi call).  Entry
 *                block_mask[h][qb][kb] = 0 removes every score S_ij of head h
 *                with i in rows [128 qb, 128 qb + 128) and j in keys
 *                [128 kb, 128 kb + 128); any non-zero byte keeps the block.
 *                The mask combines with causal masking (both must allow S_ij).
 * A query row left with no key gets O = 0, LSE = -inf and dQ = 0; a key that
 * no query sees gets dK = dV = 0.  attn_bwd_sparse must be given the same
 * mask, slopes and causal flag as the attn_fwd_sparse that made o and lse.
 * The mask is read on the device by every block (no copy is kept).
 * Errors as attn_fwd / attn_bwd, plus ATTN_ERR_INVALID for N > 65536 when a
 * mask is given.
 */
int attn_fwd_sparse(const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int H, int N, int d, float scale, int causal,
                    const float* alibi_slopes, const uint8_t* block_mask,
                    attn_dtype_t dtype, void* stream);
int attn_bwd_sparse(const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const void* dO, void* dq, void* dk, void* dv,
                    int B, int H, int N, int d, float scale, int causal,
                    const float* alibi_slopes, const uint8_t* block_mask,
                    attn_dtype_t dtype, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * Dropout of the attention probabilities, with every option (page "Flash
 * Attention V2大模型时代的算力救星", section 4.2: the dropout_p argument of the
 * call; page "FlashAttention-2：GPU利用率从50%干到90%", improvement 2: dropout
 * done inside the kernel).  Same arguments as attn_fwd_sparse /
 * attn_bwd_sparse (alibi_slopes and block_mask may be NULL) plus
 *   dropout_p : probability of dropping a score, 0 <= dropout_p < 1; it is
 *               used as the keep threshold t = floor(256 (1 - dropout_p) +
 *               1/2) of 256 levels (t = 256, i.e. dropout_p < 1/512: no
 *               dropout; t = 0 is refused)
 *   seed      : 64-bit key of the generator
 *   offset    : 32-bit counter word, to draw a new mask per call (e.g. a
 *               training step) with the same seed
 * O_i = sum_j Z_ij P_ij v_j * 256 / t, where P = softmax of the scores and
 * Z_ij = 1 iff byte (j mod 16) of Philox4x32-10 (Salmon et al., SC 2011) at
 * counter (i, j / 16, b * H + h, offset) and key (seed & 0xffffffff,
 * seed >> 32), bytes taken from its four 32-bit output words in order,
 * least significant first, is below t.  LSE is of the scores before dropout.
 * attn_bwd_ex redraws the same decisions: it must be given the forward's
 * dropout_p, seed and offset (and mask, slopes and causal flag); it returns
 * the gradients of the dropped-out attention.  No mask is stored.
 * Errors as attn_fwd_sparse / attn_bwd_sparse, plus ATTN_ERR_INVALID for a
 * dropout_p outside [0, 1) or above 1 - 1/512.
 */
int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                int B, int H, int N, int d, float scale, int causal,
                const float* alibi_slopes, const uint8_t* block_mask,
                float dropout_p, uint64_t seed, uint32_t offset,
                attn_dtype_t dtype, void* stream);
int attn_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                const float* lse, const void* dO, void* dq, void* dk, void* dv,
                int B, int H, int N, int d, float scale, int causal,
                const float* alibi_slopes, const uint8_t* block_mask,
                float dropout_p, uint64_t seed, uint32_t offset,
                attn_dtype_t dtype, void* workspace, size_t workspace_bytes,
                void* stream);

/*
 * Partial attention over a range of keys, accumulated across calls -- the
 * single-GPU building blocks of sequence (context) parallelism, where a long
 * sequence is split over devices and each device's queries meet the other
 * devices' keys and values one block at a time (page "Flash Attention V2大模型
 * 时代的算力救星", section 6, sequence parallelism across GPUs).  A call takes
 * queries and one block of keys/values of the same length N (element (b, n, h)
 * of q is query n of the call's query range, of k and v key n of its key
 * range); `causal` masks key n > query n (the block on the diagonal: the two
 * ranges are the same positions) and causal = 0 keeps every key (a key
 * block entirely before the query range).  A block entirely after the query
 * range is simply not passed.
 *
 * attn_fwd_acc -- merges this block's attention into running accumulators:
 *   o_acc : fp32 [B, N, H, d], the softmax-weighted mean over the keys seen
 *           so far (read unless FIRST; written unless LAST; may be NULL when
 *           flags has both FIRST and LAST)
 *   lse   : fp32 [B, H, N], the natural-log LSE over the keys seen so far
 *           (read unless FIRST, always written: after the LAST call it is
 *           the LSE of the whole key range)
 *   o     : [B, N, H, d] of dtype, written with the merged output on the
 *           LAST call only (may be NULL otherwise)
 *   flags : ATTN_ACC_FIRST (no earlier block: the accumulators' contents are
 *           ignored), ATTN_ACC_LAST (the final block), both, or 0.
 * With L = log(e^lse + e^lse_blk), o_acc becomes (e^lse o_acc +
 * e^lse_blk O_blk) / e^L and lse becomes L: the blockwise recurrence of page
 * "突破单卡显存极限：FlashAttention-2技术解析与实战指南", section 2.1, applied
 * to whole key blocks, so the result after the last block is the exact
 * attention over all of them (up to rounding), whatever their order.
 *
 * attn_bwd_acc -- the backward pass of one query range against one key block,
 * summed over calls.  o and lse are the FINAL forward output and LSE of the
 * query range (over all its key blocks), so P is recomputed exactly; dO its
 * gradient.
 *   dq       : [B, N, H, d] of dtype, written on the dq_flags LAST call: dQ of
 *              the query range over every key block passed with it.  The sum
 *              runs in the workspace (fp32): pass the same workspace from the
 *              FIRST call to the LAST for one query range (the FIRST call
 *              computes D = rowsum(dO * O) and clears the sum there).
 *   dk_acc, dv_acc : fp32 [B, N, H, d] accumulators of dK and dV of the key
 *              block, added to (overwritten when kv_flags is ATTN_ACC_FIRST);
 *              after the last query range they hold dK (scale included) and
 *              dV; attn_cast_acc turns them into 16-bit.
 *   dq_flags : ATTN_ACC_FIRST and/or ATTN_ACC_LAST (or 0) for the query range;
 *   kv_flags : ATTN_ACC_FIRST or 0 for the key block.
 * Errors as attn_fwd / attn_bwd, plus ATTN_ERR_INVALID for bad flags or a
 * missing pointer that the flags require.
 *
 * attn_cast_acc -- out[i] = RNE(mul * acc[i]) as 16-bit `dtype`, for n fp32
 * values (n a multiple of 8; both pointers 16-byte aligned, not overlapping).
 */
#define ATTN_ACC_FIRST 1
#define ATTN_ACC_LAST 2
int attn_fwd_acc(const void* q, const void* k, const void* v, float* o_acc,
                 float* lse, void* o, int B, int H, int N, int d, float scale,
                 int causal, int flags, attn_dtype_t dtype, void* stream);
int attn_bwd_acc(const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const void* dO, void* dq, float* dk_acc,
                 float* dv_acc, int B, int H, int N, int d, float scale,
                 int causal, int dq_flags, int kv_flags, attn_dtype_t dtype,
                 void* workspace, size_t workspace_bytes, void* stream);
int attn_cast_acc(const float* acc, void* out, size_t n, float mul,
                  attn_dtype_t dtype, void* stream);

/*
 * Decoding against a key/value cache (the KV-cache decoding of page
 * "FlashAttention技术解析：如何让GPT训练速度提升5-9倍", section 4.1, and page
 * "突破单卡显存极限", section 3.2): Nq query rows that are the LAST Nq positions
 * of a sequence of Nk keys.
 *
 *   S = s * q K^T (query i sees keys j <= Nk - Nq + i when causal),
 *   O = softmax_row(S) V,  LSE_i = log sum_j exp(S_ij)   (natural log)
 *
 * i.e. the last Nq rows of attn_fwd over the whole sequence.  The key range of
 * every (b, h) is split into chunks that run as separate blocks; their
 * partial results (unnormalised O, running max, running sum) go to the
 * workspace and a second kernel merges them, so the result is exact up to
 * floating-point rounding and does not depend on the chunking.
 *
 *   q, o : [B, Nq, H, d]  (dtype), 1 <= Nq <= 128
 *   k, v : [B, Nk, H, d]  (dtype), the cache, Nk >= 1 (Nk >= Nq when causal)
 *   lse  : [B, H, Nq] fp32 output
 * Errors as attn_fwd; ATTN_ERR_UNSUPPORTED for Nq > 128, ATTN_ERR_INVALID for
 * causal with Nq > Nk, ATTN_ERR_WORKSPACE for a missing or short workspace.
 */
size_t attn_decode_workspace_size(int B, int H, int Nq, int Nk, int d);
int attn_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                int B, int H, int Nq, int Nk, int d, float scale, int causal,
                attn_dtype_t dtype, void* workspace, size_t workspace_bytes,
                void* stream);

/*
 * attn_philox4x32_10 -- diagnostic: the dropout decisions' generator itself.
 * Runs the kernels' Philox4x32-10 (Salmon et al., SC 2011, section 3.2; the
 * generator named under attn_fwd_ex) on n caller-given inputs, one GPU thread
 * each, so that it can be checked against the algorithm's published
 * known-answer vectors on the device.
 *   in  : device pointer, uint32 [n][6]: counter words 0-3, then key words 0-1
 *   out : device pointer, uint32 [n][4]: the four output words, in order
 *   n   : 1 <= n <= 2^24
 * Both 4-byte aligned, not overlapping.  Asynchronous on `stream`.  Returns
 * ATTN_OK, ATTN_ERR_INVALID (null, n out of range, overlap), ATTN_ERR_ALIGN
 * or ATTN_ERR_CUDA (launch failed).
 */
int attn_philox4x32_10(const uint32_t* in, uint32_t* out, int n, void* stream);

/*
 * attn_status -- synchronises `stream`, then reads and clears the current
 * device's status word.  Returns ATTN_OK, ATTN_ERR_TIMEOUT if a kernel gave up
 * on a bounded wait since the last call (its outputs are then garbage), or
 * ATTN_ERR_CUDA if the synchronisation itself failed.  While the word is set,
 * kernels on that device give up at their first wait, so a caller that sees a
 * timeout must call attn_status before trusting later results.
 */
int attn_status(void* stream);

/* Text of the last host-side error on the calling thread ("" if none). */
const char* attn_last_error_string(void);

/*
 * attn_set_wait_limit -- testing knob.  Sets the time limit, in nanoseconds,
 * of every device-side wait of later launches (default 2e9, i.e. 2 s;
 * 0 restores the default), and debug flags that make a kernel's load warp
 * hold back its copies, so that its consumers' waits run out (used to test
 * the timeout path without faulting the GPU): bit 0 the forward (no loads),
 * bit 1 the backward main kernel (K and V, but no query steps), bit 2 the
 * decoding chunk kernel (no loads).  Bit 3 changes no result: the
 * backward's preprocess and dQ conversion kernels split row indices with
 * 64-bit arithmetic, the form they take by themselves only when
 * B * H * N (N rounded up to 128) reaches 2^31.  Process-wide.
 */
int attn_set_wait_limit(unsigned long long limit_ns, int debug_flags);

/*
 * Per-kernel timing on the launch stream, for benchmarks.  Between
 * attn_profile_begin() and attn_profile_end(), every kernel launched by this
 * library is bracketed by CUDA events on its stream.  attn_profile_end()
 * synchronises those events and fills, for kernel ids 0..n-1
 * (0 forward, 1 backward preprocess, 2 backward main, 3 dQ conversion,
 * 4 decode chunks, 5 decode merge),
 * the number of launches and their summed device time in milliseconds.
 * Returns the number of kernel ids filled, or a negative ATTN_ERR_* code.
 */
int attn_profile_begin(void);
int attn_profile_end(int* launches, double* total_ms, int n);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_TILED_ATTENTION_ATTN_H */
