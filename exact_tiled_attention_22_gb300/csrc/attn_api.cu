// attn_api.cu -- the C ABI (include/attn.h): argument checks, TMA tensor-map
// encoding, launch geometry, the device status word and per-kernel timing.
// The kernels themselves live in attn_fwd.cu and attn_bwd.cu.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "attn.h"
#include "kernels.h"

namespace {

// Per-device status word read by attn_status(); kernels set it when a bounded
// wait runs out.  One copy per device (module globals are per context).
__device__ int g_attn_status;

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s

thread_local std::string t_err;

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int sms = 0;
  int* status = nullptr;            // device address of g_attn_status ...
  unsigned long long status_ctx = 0;  // ... in the context with this id
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
unsigned long long g_wait_ns = kDefaultWaitNs;
int g_debug_flags = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
std::once_flag g_ctx_once;

// Looks up the current device: architecture and SM count once per device,
// the status word's address once per context.
int current_device(DeviceInfo** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device %d out of range", dev);
  // Binds the device's primary context to this thread: the tensor-map
  // encoding is a driver call, and a thread that has made no runtime call
  // yet (e.g. a framework's backward worker) has no current context.
  if ((e = cudaSetDevice(dev)) != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    d.supported = (major == 10 && minor == 3);
    d.sms = sms;
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.ready = true;
  }
  if (!d.supported)
    return fail(ATTN_ERR_UNSUPPORTED, "device %d is not sm_103 (GB300); no other path exists", dev);
  // The status word's address belongs to the context the module was loaded
  // in: look it up again whenever the thread's current context is another
  // one (a context torn down by cudaDeviceReset and created anew included;
  // context ids are never reused within a process).
  unsigned long long ctx = 0;
  if (attn::current_context_id(&ctx) != cudaSuccess)
    return fail(ATTN_ERR_CUDA, "cannot identify the current CUDA context");
  if (!d.status || d.status_ctx != ctx) {
    void* ptr = nullptr;
    if ((e = cudaGetSymbolAddress(&ptr, g_attn_status)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(status)");
    d.status = static_cast<int*>(ptr);
    d.status_ctx = ctx;
  }
  *out = &d;
  return ATTN_OK;
}

// A [B, N, H, d] 16-bit tensor as a 4-D TMA map (d, H, N, B), 128-byte
// swizzle, boxes of 64 columns x `rows` sequence rows of one (b, h).
int encode_bnhd(CUtensorMap* m, const void* ptr, int B, int N, int H, int d, int rows, bool bf16) {
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2, (cuuint64_t)N * H * d * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                        const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

struct Range {
  uintptr_t lo, hi;
};
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }
Range rng(const void* p, size_t bytes) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return {a, a + bytes};
}

// Bytes of a block mask [H][nb][nb], nb = ceil(N / 128).
size_t mask_bytes(int H, int N) {
  const size_t nb = ((size_t)N + 127) / 128;
  return (size_t)H * nb * nb;
}

// The block-sparse variants keep one 128-row block list per CTA in shared
// memory: N / 128 is bounded.
int check_block_mask(int N) {
  if ((N + 127) / 128 > attn::kMaxSparseTiles)
    return fail(ATTN_ERR_INVALID, "block_mask supports N <= %d, got %d", attn::kMaxSparseTiles * 128, N);
  return ATTN_OK;
}

// Dropout probability -> keep threshold and the kernels' constants (t = 256:
// no dropout).  p must lie in [0, 1) and keep a threshold of at least 1.
int make_dropout(float dropout_p, uint64_t seed, uint32_t offset, attn::DropoutArgs* out) {
  const double p = (double)dropout_p;
  if (!(p >= 0.0 && p < 1.0))
    return fail(ATTN_ERR_INVALID, "dropout_p must be in [0, 1), got %g", p);
  const int t = (int)std::floor(256.0 * (1.0 - p) + 0.5);
  if (t < 1) return fail(ATTN_ERR_INVALID, "dropout_p %g keeps no score (256 (1 - p) < 1/2)", p);
  out->k0 = (uint32_t)(seed & 0xFFFFFFFFull);
  out->k1 = (uint32_t)(seed >> 32);
  out->offset = offset;
  out->t = t;
  out->cmp = (uint32_t)(256 - t) * 0x00010001u;
  out->scale = 256.0f / (float)t;
  for (int r = 0; r < 10; ++r) {
    out->rk[2 * r] = out->k0 + (uint32_t)r * attn::kPhiloxW0;
    out->rk[2 * r + 1] = out->k1 + (uint32_t)r * attn::kPhiloxW1;
  }
  return ATTN_OK;
}

int check_common(int B, int H, int N, int d, float scale, attn_dtype_t dtype) {
  if (B < 1 || H < 1 || N < 1) return fail(ATTN_ERR_INVALID, "B, H, N must be >= 1 (got %d, %d, %d)", B, H, N);
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim d=%d not supported (64 or 128)", d);
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return fail(ATTN_ERR_UNSUPPORTED, "unknown dtype %d", (int)dtype);
  // Kernels index tensors with 64-bit offsets; what must fit in 31 bits is
  // B*H and the grids (at most ceil(N/128) blocks per head, 64 per head
  // when decoding).
  const long long bh = (long long)B * H;
  if (bh * (((long long)N + 127) / 128) >= (1ll << 31) || bh * 64 >= (1ll << 31))
    return fail(ATTN_ERR_INVALID, "B*H*ceil(N/128) = %lld blocks too many (< 2^31, and B*H < 2^25)",
                bh * (((long long)N + 127) / 128));
  const long long elems = bh * N * d;
  if (elems >= (1ll << 40)) return fail(ATTN_ERR_INVALID, "B*H*N*d = %lld too large (< 2^40)", elems);
  if (!std::isfinite(scale) || !(scale > 0.f)) return fail(ATTN_ERR_INVALID, "scale must be finite and > 0");
  return ATTN_OK;
}

// ---------------------------------------------------------------- profiling
struct ProfState {
  bool on = false;
  std::vector<cudaEvent_t> pool;
  size_t used = 0;
  std::vector<int> kind;  // one per event pair
};
ProfState g_prof;
std::mutex g_prof_mu;
constexpr size_t kProfPairs = 8192;

// Runs `launch` bracketed by events when profiling is on.
template <typename F>
cudaError_t timed(int kind, cudaStream_t stream, F&& launch) {
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (g_prof.on && g_prof.used + 2 <= g_prof.pool.size()) {
      e0 = g_prof.pool[g_prof.used];
      e1 = g_prof.pool[g_prof.used + 1];
      g_prof.used += 2;
      g_prof.kind.push_back(kind);
    }
  }
  if (e0) cudaEventRecord(e0, stream);
  cudaError_t e = launch();
  if (e1) cudaEventRecord(e1, stream);
  return e;
}

}  // namespace

namespace attn {
cudaError_t current_context_id(unsigned long long* id) {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<CtxGetIdFn>(fn);
  });
  if (!g_ctx_current || !g_ctx_id) return cudaErrorNotSupported;
  CUcontext c = nullptr;
  if (g_ctx_current(&c) != CUDA_SUCCESS || !c) return cudaErrorDeviceUninitialized;
  return g_ctx_id(c, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

void set_last_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_err = buf;
}
}  // namespace attn

extern "C" {

const char* attn_last_error_string(void) { return t_err.c_str(); }

int attn_set_wait_limit(unsigned long long limit_ns, int debug_flags) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_wait_ns = limit_ns ? limit_ns : kDefaultWaitNs;
  g_debug_flags = debug_flags;
  return ATTN_OK;
}

int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                int d, float scale, int causal, const float* alibi_slopes, const uint8_t* block_mask,
                float dropout_p, uint64_t seed, uint32_t offset, attn_dtype_t dtype, void* stream) {
  t_err.clear();
  if (!q || !k || !v || !o || !lse) return fail(ATTN_ERR_INVALID, "null pointer argument");
  if (alibi_slopes && !aligned4(alibi_slopes)) return fail(ATTN_ERR_ALIGN, "alibi_slopes must be 4-byte aligned");
  int rc = check_common(B, H, N, d, scale, dtype);
  if (rc) return rc;
  if (block_mask && (rc = check_block_mask(N))) return rc;
  attn::DropoutArgs drop;
  if ((rc = make_dropout(dropout_p, seed, offset, &drop))) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(ATTN_ERR_ALIGN, "all pointers must be 16-byte aligned");
  const size_t tb = (size_t)B * N * H * d * 2, lb = (size_t)B * H * N * 4;
  const Range outs[2] = {rng(o, tb), rng(lse, lb)};
  const Range ins[5] = {rng(q, tb), rng(k, tb), rng(v, tb), rng(alibi_slopes, alibi_slopes ? (size_t)H * 4 : 0),
                        rng(block_mask, block_mask ? mask_bytes(H, N) : 0)};
  if (overlap(outs[0], outs[1])) return fail(ATTN_ERR_INVALID, "o and lse overlap");
  for (const Range& a : outs)
    for (const Range& b : ins)
      if (overlap(a, b)) return fail(ATTN_ERR_INVALID, "an output overlaps an input");

  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev))) return rc;
  attn::FwdArgs a;
  std::memset(&a, 0, sizeof a);
  const bool bf16 = dtype == ATTN_BF16;
  if ((rc = encode_bnhd(&a.tm_q, q, B, N, H, d, 128, bf16)) ||
      (rc = encode_bnhd(&a.tm_k, k, B, N, H, d, 128, bf16)) ||
      (rc = encode_bnhd(&a.tm_v, v, B, N, H, d, 128, bf16)) ||
      (rc = encode_bnhd(&a.tm_o, o, B, N, H, d, 128, bf16)))
    return rc;
  a.o = o;
  a.lse = lse;
  a.alibi = alibi_slopes;
  a.bmask = block_mask;
  a.drop = drop;
  a.B = B; a.H = H; a.N = N; a.d = d;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  a.bf16 = bf16;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    a.debug_flags = g_debug_flags;
    a.wait.limit_ns = g_wait_ns;
  }
  a.wait.status = dev->status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = timed(attn::kKFwd, s, [&] { return attn::launch_fwd(a, s); });
  if (e != cudaSuccess) return cuda_fail(e, "attn_fwd launch");
  return ATTN_OK;
}

int attn_fwd_sparse(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                    int d, float scale, int causal, const float* alibi_slopes, const uint8_t* block_mask,
                    attn_dtype_t dtype, void* stream) {
  return attn_fwd_ex(q, k, v, o, lse, B, H, N, d, scale, causal, alibi_slopes, block_mask, 0.f, 0, 0, dtype,
                     stream);
}

int attn_fwd_alibi(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                   int d, float scale, int causal, const float* alibi_slopes, attn_dtype_t dtype,
                   void* stream) {
  return attn_fwd_ex(q, k, v, o, lse, B, H, N, d, scale, causal, alibi_slopes, nullptr, 0.f, 0, 0, dtype,
                     stream);
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
             float scale, int causal, attn_dtype_t dtype, void* stream) {
  return attn_fwd_ex(q, k, v, o, lse, B, H, N, d, scale, causal, nullptr, nullptr, 0.f, 0, 0, dtype, stream);
}

size_t attn_decode_workspace_size(int B, int H, int Nq, int Nk, int d) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || (d != 64 && d != 128)) return 0;
  const size_t parts = (size_t)B * H * attn::decode_n_split(B, H, Nk) * Nq;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  return up(parts * d * 4) + up(parts * 2 * 4);
}

int attn_decode_alibi(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                      int Nq, int Nk, int d, float scale, int causal, const float* alibi_slopes,
                      attn_dtype_t dtype, void* workspace, size_t workspace_bytes, void* stream) {
  t_err.clear();
  if (!q || !k || !v || !o || !lse) return fail(ATTN_ERR_INVALID, "null pointer argument");
  if (alibi_slopes && !aligned4(alibi_slopes)) return fail(ATTN_ERR_ALIGN, "alibi_slopes must be 4-byte aligned");
  if (Nq < 1 || Nk < 1) return fail(ATTN_ERR_INVALID, "Nq, Nk must be >= 1 (got %d, %d)", Nq, Nk);
  if (Nq > 128) return fail(ATTN_ERR_UNSUPPORTED, "decode takes at most 128 query rows (got %d)", Nq);
  if (causal && Nq > Nk) return fail(ATTN_ERR_INVALID, "causal decode needs Nq <= Nk (got %d > %d)", Nq, Nk);
  int rc = check_common(B, H, Nk, d, scale, dtype);
  if (rc) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(ATTN_ERR_ALIGN, "all pointers must be 16-byte aligned");
  const size_t need = attn_decode_workspace_size(B, H, Nq, Nk, d);
  if (!workspace || workspace_bytes < need)
    return fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(ATTN_ERR_ALIGN, "workspace must be 256-byte aligned");
  const size_t qb = (size_t)B * Nq * H * d * 2, kb = (size_t)B * Nk * H * d * 2, lb = (size_t)B * H * Nq * 4;
  const Range outs[3] = {rng(o, qb), rng(lse, lb), rng(workspace, need)};
  const Range ins[4] = {rng(q, qb), rng(k, kb), rng(v, kb), rng(alibi_slopes, alibi_slopes ? (size_t)H * 4 : 0)};
  for (int i = 0; i < 3; ++i)
    for (int j = i + 1; j < 3; ++j)
      if (overlap(outs[i], outs[j])) return fail(ATTN_ERR_INVALID, "outputs or workspace overlap");
  for (const Range& a : outs)
    for (const Range& b : ins)
      if (overlap(a, b)) return fail(ATTN_ERR_INVALID, "an output overlaps an input");

  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev))) return rc;
  attn::DecArgs a;
  std::memset(&a, 0, sizeof a);
  const bool bf16 = dtype == ATTN_BF16;
  if ((rc = encode_bnhd(&a.tm_q, q, B, Nq, H, d, 128, bf16)) ||
      (rc = encode_bnhd(&a.tm_k, k, B, Nk, H, d, 128, bf16)) ||
      (rc = encode_bnhd(&a.tm_v, v, B, Nk, H, d, 128, bf16)))
    return rc;
  a.o = o;
  a.lse = lse;
  a.alibi = alibi_slopes;
  a.B = B; a.H = H; a.Nq = Nq; a.Nk = Nk; a.d = d;
  a.n_split = attn::decode_n_split(B, H, Nk);
  a.keys_per_split = attn::decode_keys_per_split(Nk, a.n_split);
  const size_t parts = (size_t)B * H * a.n_split * Nq;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.ws_o = reinterpret_cast<float*>(ws);
  a.ws_ml = reinterpret_cast<float*>(ws + (parts * d * 4 + 255) / 256 * 256);
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  a.bf16 = bf16;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    a.debug_flags = g_debug_flags;
    a.wait.limit_ns = g_wait_ns;
  }
  a.wait.status = dev->status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = timed(attn::kKDecSplit, s, [&] { return attn::launch_decode_split(a, s); });
  if (e != cudaSuccess) return cuda_fail(e, "attn_decode chunk launch");
  e = timed(attn::kKDecMerge, s, [&] { return attn::launch_decode_merge(a, s); });
  if (e != cudaSuccess) return cuda_fail(e, "attn_decode merge launch");
  return ATTN_OK;
}

int attn_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                int Nk, int d, float scale, int causal, attn_dtype_t dtype, void* workspace,
                size_t workspace_bytes, void* stream) {
  return attn_decode_alibi(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, nullptr, dtype, workspace,
                           workspace_bytes, stream);
}

size_t attn_bwd_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
  const size_t npad = ((size_t)N + 127) / 128 * 128;
  const size_t rows = (size_t)B * H * npad;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  return up(rows * 4) * 2 + up(rows * d * 4) + 256;
}

int attn_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
                const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                int causal, const float* alibi_slopes, const uint8_t* block_mask, float dropout_p,
                uint64_t seed, uint32_t offset, attn_dtype_t dtype, void* workspace,
                size_t workspace_bytes, void* stream) {
  t_err.clear();
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv)
    return fail(ATTN_ERR_INVALID, "null pointer argument");
  if (alibi_slopes && !aligned4(alibi_slopes)) return fail(ATTN_ERR_ALIGN, "alibi_slopes must be 4-byte aligned");
  int rc = check_common(B, H, N, d, scale, dtype);
  if (rc) return rc;
  if (block_mask && (rc = check_block_mask(N))) return rc;
  attn::DropoutArgs drop;
  if ((rc = make_dropout(dropout_p, seed, offset, &drop))) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dO) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(ATTN_ERR_ALIGN, "all pointers must be 16-byte aligned");
  const size_t need = attn_bwd_workspace_size(B, H, N, d);
  if (!workspace || workspace_bytes < need)
    return fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(ATTN_ERR_ALIGN, "workspace must be 256-byte aligned");
  const size_t tb = (size_t)B * N * H * d * 2, lb = (size_t)B * H * N * 4;
  const Range outs[4] = {rng(dq, tb), rng(dk, tb), rng(dv, tb), rng(workspace, need)};
  const Range ins[8] = {rng(q, tb), rng(k, tb), rng(v, tb), rng(o, tb), rng(lse, lb), rng(dO, tb),
                        rng(alibi_slopes, alibi_slopes ? (size_t)H * 4 : 0),
                        rng(block_mask, block_mask ? mask_bytes(H, N) : 0)};
  for (int i = 0; i < 4; ++i) {
    for (int j = i + 1; j < 4; ++j)
      if (overlap(outs[i], outs[j])) return fail(ATTN_ERR_INVALID, "output buffers overlap");
    for (const Range& b : ins)
      if (overlap(outs[i], b)) return fail(ATTN_ERR_INVALID, "an output or the workspace overlaps an input");
  }

  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev))) return rc;
  attn::BwdArgs a;
  std::memset(&a, 0, sizeof a);
  const bool bf16 = dtype == ATTN_BF16;
  const int qrows = attn::bwd_q_rows(d);
  if ((rc = encode_bnhd(&a.tm_q, q, B, N, H, d, qrows, bf16)) ||
      (rc = encode_bnhd(&a.tm_k, k, B, N, H, d, 128, bf16)) ||
      (rc = encode_bnhd(&a.tm_v, v, B, N, H, d, 128, bf16)) ||
      (rc = encode_bnhd(&a.tm_do, dO, B, N, H, d, qrows, bf16)) ||
      (rc = encode_bnhd(&a.tm_dk, dk, B, N, H, d, 128, bf16)) ||
      (rc = encode_bnhd(&a.tm_dv, dv, B, N, H, d, 128, bf16)))
    return rc;
  const int npad = (N + 127) / 128 * 128;
  const size_t rows = (size_t)B * H * npad;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.o = o;
  a.dO = dO;
  a.lse = lse;
  a.alibi = alibi_slopes;
  a.bmask = block_mask;
  a.drop = drop;
  a.lse2 = reinterpret_cast<float*>(ws);
  a.dvec = reinterpret_cast<float*>(ws + up(rows * 4));
  a.dqacc = reinterpret_cast<float*>(ws + 2 * up(rows * 4));
  a.sched = reinterpret_cast<unsigned*>(ws + 2 * up(rows * 4) + up(rows * (size_t)d * 4));
  a.dq = dq; a.dk = dk; a.dv = dv;
  a.B = B; a.H = H; a.N = N; a.Npad = npad; a.d = d;
  a.sms = dev->sms;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  a.bf16 = bf16;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    a.debug_flags = g_debug_flags;
    a.wait.limit_ns = g_wait_ns;
  }
  a.wait.status = dev->status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = timed(attn::kKBwdPre, s, [&] { return attn::launch_bwd_pre(a, s); });
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd preprocess launch");
  e = timed(attn::kKBwdMain, s, [&] { return attn::launch_bwd_main(a, s); });
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd main launch");
  e = timed(attn::kKDqPost, s, [&] { return attn::launch_dq_post(a, s); });
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd dQ conversion launch");
  return ATTN_OK;
}

int attn_bwd_sparse(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                    int causal, const float* alibi_slopes, const uint8_t* block_mask, attn_dtype_t dtype,
                    void* workspace, size_t workspace_bytes, void* stream) {
  return attn_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, alibi_slopes, block_mask, 0.f,
                     0, 0, dtype, workspace, workspace_bytes, stream);
}

int attn_bwd_alibi(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                   int causal, const float* alibi_slopes, attn_dtype_t dtype, void* workspace,
                   size_t workspace_bytes, void* stream) {
  return attn_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, alibi_slopes, nullptr, 0.f,
                     0, 0, dtype, workspace, workspace_bytes, stream);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
             void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
             attn_dtype_t dtype, void* workspace, size_t workspace_bytes, void* stream) {
  return attn_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, nullptr, nullptr, 0.f, 0, 0,
                     dtype, workspace, workspace_bytes, stream);
}

int attn_fwd_acc(const void* q, const void* k, const void* v, float* o_acc, float* lse, void* o, int B, int H,
                 int N, int d, float scale, int causal, int flags, attn_dtype_t dtype, void* stream) {
  t_err.clear();
  if (flags < 0 || flags > (ATTN_ACC_FIRST | ATTN_ACC_LAST))
    return fail(ATTN_ERR_INVALID, "flags must be a combination of ATTN_ACC_FIRST and ATTN_ACC_LAST");
  const bool first = (flags & ATTN_ACC_FIRST) != 0, last = (flags & ATTN_ACC_LAST) != 0;
  if (!q || !k || !v || !lse) return fail(ATTN_ERR_INVALID, "null pointer argument");
  if (!(first && last) && !o_acc) return fail(ATTN_ERR_INVALID, "o_acc is needed unless flags has FIRST and LAST");
  if (last && !o) return fail(ATTN_ERR_INVALID, "o is needed with ATTN_ACC_LAST");
  int rc = check_common(B, H, N, d, scale, dtype);
  if (rc) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(lse) || !aligned16(o_acc) || !aligned16(o))
    return fail(ATTN_ERR_ALIGN, "all pointers must be 16-byte aligned");
  const size_t tb = (size_t)B * N * H * d * 2, lb = (size_t)B * H * N * 4;
  const Range outs[3] = {rng(o_acc, (first && last) ? 0 : 2 * tb), rng(lse, lb), rng(o, last ? tb : 0)};
  const Range ins[3] = {rng(q, tb), rng(k, tb), rng(v, tb)};
  for (int i = 0; i < 3; ++i) {
    for (int j = i + 1; j < 3; ++j)
      if (overlap(outs[i], outs[j])) return fail(ATTN_ERR_INVALID, "output buffers overlap");
    for (const Range& b : ins)
      if (overlap(outs[i], b)) return fail(ATTN_ERR_INVALID, "an output overlaps an input");
  }
  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev))) return rc;
  attn::FwdArgs a;
  std::memset(&a, 0, sizeof a);
  const bool bf16 = dtype == ATTN_BF16;
  if ((rc = encode_bnhd(&a.tm_q, q, B, N, H, d, 128, bf16)) ||
      (rc = encode_bnhd(&a.tm_k, k, B, N, H, d, 128, bf16)) ||
      (rc = encode_bnhd(&a.tm_v, v, B, N, H, d, 128, bf16)))
    return rc;
  a.o = o;
  a.lse = lse;
  a.o_acc = o_acc;
  a.acc_flags = flags;
  if ((rc = make_dropout(0.f, 0, 0, &a.drop))) return rc;
  a.B = B; a.H = H; a.N = N; a.d = d;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  a.bf16 = bf16;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    a.debug_flags = g_debug_flags;
    a.wait.limit_ns = g_wait_ns;
  }
  a.wait.status = dev->status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = timed(attn::kKFwd, s, [&] { return attn::launch_fwd_acc(a, s); });
  if (e != cudaSuccess) return cuda_fail(e, "attn_fwd_acc launch");
  return ATTN_OK;
}

int attn_bwd_acc(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                 void* dq, float* dk_acc, float* dv_acc, int B, int H, int N, int d, float scale, int causal,
                 int dq_flags, int kv_flags, attn_dtype_t dtype, void* workspace, size_t workspace_bytes,
                 void* stream) {
  t_err.clear();
  const int all = ATTN_ACC_FIRST | ATTN_ACC_LAST;
  if (dq_flags < 0 || dq_flags > all || kv_flags < 0 || kv_flags > ATTN_ACC_FIRST)
    return fail(ATTN_ERR_INVALID, "dq_flags: FIRST and/or LAST; kv_flags: 0 or ATTN_ACC_FIRST");
  const bool dq_last = (dq_flags & ATTN_ACC_LAST) != 0;
  if (!q || !k || !v || !o || !lse || !dO || !dk_acc || !dv_acc || (dq_last && !dq))
    return fail(ATTN_ERR_INVALID, "null pointer argument");
  int rc = check_common(B, H, N, d, scale, dtype);
  if (rc) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dO) ||
      !aligned16(dq) || !aligned16(dk_acc) || !aligned16(dv_acc))
    return fail(ATTN_ERR_ALIGN, "all pointers must be 16-byte aligned");
  const size_t need = attn_bwd_workspace_size(B, H, N, d);
  if (!workspace || workspace_bytes < need)
    return fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(ATTN_ERR_ALIGN, "workspace must be 256-byte aligned");
  const size_t tb = (size_t)B * N * H * d * 2, lb = (size_t)B * H * N * 4;
  const Range outs[4] = {rng(dq, dq_last ? tb : 0), rng(dk_acc, 2 * tb), rng(dv_acc, 2 * tb), rng(workspace, need)};
  const Range ins[6] = {rng(q, tb), rng(k, tb), rng(v, tb), rng(o, tb), rng(lse, lb), rng(dO, tb)};
  for (int i = 0; i < 4; ++i) {
    for (int j = i + 1; j < 4; ++j)
      if (overlap(outs[i], outs[j])) return fail(ATTN_ERR_INVALID, "output buffers overlap");
    for (const Range& b : ins)
      if (overlap(outs[i], b)) return fail(ATTN_ERR_INVALID, "an output or the workspace overlaps an input");
  }
  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev))) return rc;
  attn::BwdArgs a;
  std::memset(&a, 0, sizeof a);
  const bool bf16 = dtype == ATTN_BF16;
  const int qrows = attn::bwd_q_rows(d);
  if ((rc = encode_bnhd(&a.tm_q, q, B, N, H, d, qrows, bf16)) ||
      (rc = encode_bnhd(&a.tm_k, k, B, N, H, d, 128, bf16)) ||
      (rc = encode_bnhd(&a.tm_v, v, B, N, H, d, 128, bf16)) ||
      (rc = encode_bnhd(&a.tm_do, dO, B, N, H, d, qrows, bf16)))
    return rc;
  const int npad = (N + 127) / 128 * 128;
  const size_t rows = (size_t)B * H * npad;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.o = o;
  a.dO = dO;
  a.lse = lse;
  if ((rc = make_dropout(0.f, 0, 0, &a.drop))) return rc;
  a.lse2 = reinterpret_cast<float*>(ws);
  a.dvec = reinterpret_cast<float*>(ws + up(rows * 4));
  a.dqacc = reinterpret_cast<float*>(ws + 2 * up(rows * 4));
  a.sched = reinterpret_cast<unsigned*>(ws + 2 * up(rows * 4) + up(rows * (size_t)d * 4));
  a.dq = dq;
  a.dk_acc = dk_acc;
  a.dv_acc = dv_acc;
  a.kv_flags = kv_flags;
  a.B = B; a.H = H; a.N = N; a.Npad = npad; a.d = d;
  a.sms = dev->sms;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  a.bf16 = bf16;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    a.debug_flags = g_debug_flags;
    a.wait.limit_ns = g_wait_ns;
  }
  a.wait.status = dev->status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (dq_flags & ATTN_ACC_FIRST) {
    e = timed(attn::kKBwdPre, s, [&] { return attn::launch_bwd_pre(a, s); });
    if (e != cudaSuccess) return cuda_fail(e, "attn_bwd_acc preprocess launch");
  }
  e = timed(attn::kKBwdMain, s, [&] { return attn::launch_bwd_main_acc(a, s); });
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd_acc main launch");
  if (dq_last) {
    e = timed(attn::kKDqPost, s, [&] { return attn::launch_dq_post(a, s); });
    if (e != cudaSuccess) return cuda_fail(e, "attn_bwd_acc dQ conversion launch");
  }
  return ATTN_OK;
}

int attn_cast_acc(const float* acc, void* out, size_t n, float mul, attn_dtype_t dtype, void* stream) {
  t_err.clear();
  if (!acc || !out) return fail(ATTN_ERR_INVALID, "null pointer argument");
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return fail(ATTN_ERR_UNSUPPORTED, "unknown dtype %d", (int)dtype);
  if (n == 0 || n % 8 != 0 || n >= (1ull << 40))
    return fail(ATTN_ERR_INVALID, "n must be a positive multiple of 8 below 2^40 (got %zu)", n);
  if (!std::isfinite(mul)) return fail(ATTN_ERR_INVALID, "mul must be finite");
  if (!aligned16(acc) || !aligned16(out)) return fail(ATTN_ERR_ALIGN, "all pointers must be 16-byte aligned");
  if (overlap(rng(acc, n * 4), rng(out, n * 2))) return fail(ATTN_ERR_INVALID, "out overlaps acc");
  DeviceInfo* dev = nullptr;
  int rc = current_device(&dev);
  if (rc) return rc;
  cudaError_t e = attn::launch_cast_acc(acc, out, (long long)n, mul, dtype == ATTN_BF16, dev->sms,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attn_cast_acc launch");
  return ATTN_OK;
}

int attn_status(void* stream) {
  t_err.clear();
  DeviceInfo* dev = nullptr;
  int rc = current_device(&dev);
  if (rc) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int h = 0;
  if ((e = cudaMemcpyFromSymbol(&h, g_attn_status, sizeof h)) != cudaSuccess)
    return cuda_fail(e, "read status word");
  if (h != 0) {
    const int zero = 0;
    if ((e = cudaMemcpyToSymbol(g_attn_status, &zero, sizeof zero)) != cudaSuccess)
      return cuda_fail(e, "clear status word");
    return fail(ATTN_ERR_TIMEOUT, "a device-side wait ran out of time (status %d)", h);
  }
  return ATTN_OK;
}

int attn_profile_begin(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (g_prof.pool.empty()) {
    g_prof.pool.resize(2 * kProfPairs);
    for (auto& ev : g_prof.pool) {
      cudaError_t e = cudaEventCreate(&ev);
      if (e != cudaSuccess) {
        g_prof.pool.clear();
        return cuda_fail(e, "cudaEventCreate");
      }
    }
  }
  g_prof.used = 0;
  g_prof.kind.clear();
  g_prof.on = true;
  return ATTN_OK;
}

int attn_profile_end(int* launches, double* total_ms, int n) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof.on = false;
  const int m = n < attn::kKNum ? n : attn::kKNum;
  for (int i = 0; i < m; ++i) {
    if (launches) launches[i] = 0;
    if (total_ms) total_ms[i] = 0.0;
  }
  for (size_t i = 0; i < g_prof.kind.size(); ++i) {
    cudaEvent_t e0 = g_prof.pool[2 * i], e1 = g_prof.pool[2 * i + 1];
    cudaError_t e = cudaEventSynchronize(e1);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
    float ms = 0.f;
    if ((e = cudaEventElapsedTime(&ms, e0, e1)) != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
    const int k = g_prof.kind[i];
    if (k < m) {
      if (launches) launches[k] += 1;
      if (total_ms) total_ms[k] += ms;
    }
  }
  g_prof.kind.clear();
  g_prof.used = 0;
  return m;
}

}  // extern "C"
