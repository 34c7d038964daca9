// attn_noalloc.cu -- attn_bwd_noalloc: the backward pass for callers that
// cannot allocate device memory.
//
// attn_bwd needs a scratch workspace (per-row D and scaled LSE, and an fp32
// dQ accumulator).  Some callers have no way to provide one: plain C code
// embedded in a host program or plugin that owns no CUDA memory pool and
// gets no allocator handle, or latency-critical loops that must not call
// cudaMalloc because it can synchronise the whole device.  For them this
// entry point uses a fixed scratch array that the library itself owns: a
// file-scope __device__ array, created on each GPU when the library's device
// code is loaded there and held until the process exits.
//
// The array is shared by every call on a device.  Each call rewrites all of
// the part it uses (the preprocess kernel zeroes the dQ accumulator and
// overwrites D and the scaled LSE), so nothing carries over between calls,
// but two calls whose kernels overlap on the GPU (for example on two
// streams) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "attn.h"
#include "kernels.h"

namespace {

// Scratch for attn_bwd_noalloc; ATTN_NOALLOC_WORKSPACE_BYTES in attn.h.
constexpr size_t kScratchBytes = ATTN_NOALLOC_WORKSPACE_BYTES;
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_mu;
// Device address of g_bwd_scratch per device, and the id of the context it
// was looked up in: module globals live in a context, so a device whose
// context was torn down (cudaDeviceReset) and created anew has the array at
// a new address.
void* g_scratch_addr[kMaxDev] = {};
unsigned long long g_scratch_ctx[kMaxDev] = {};

}  // namespace

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                int B, int H, int N, int d, float scale, int causal,
                                attn_dtype_t dtype, void* stream) {
  const size_t need = attn_bwd_workspace_size(B, H, N, d);
  if (need > kScratchBytes) {
    attn::set_last_error("attn_bwd_noalloc: this shape needs %zu bytes of scratch, more than "
                         "the %zu-byte library-owned array; use attn_bwd with a workspace",
                         need, kScratchBytes);
    return ATTN_ERR_WORKSPACE;
  }
  if (need == 0)  // invalid sizes: let attn_bwd report which argument
    return attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, dtype, nullptr, 0,
                    stream);
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    attn::set_last_error("attn_bwd_noalloc: no current device (%s)", cudaGetErrorString(e));
    return ATTN_ERR_CUDA;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    attn::set_last_error("attn_bwd_noalloc: cannot query device %d", dev);
    return ATTN_ERR_CUDA;
  }
  if (major != 10 || minor != 3) {
    attn::set_last_error("attn_bwd_noalloc: device %d is not sm_103 (GB300)", dev);
    return ATTN_ERR_UNSUPPORTED;
  }
  // Makes the device's primary context current on this thread if none is.
  if ((e = cudaSetDevice(dev)) != cudaSuccess) {
    attn::set_last_error("attn_bwd_noalloc: cudaSetDevice failed: %s", cudaGetErrorString(e));
    return ATTN_ERR_CUDA;
  }
  unsigned long long ctx = 0;
  if (attn::current_context_id(&ctx) != cudaSuccess) {
    attn::set_last_error("attn_bwd_noalloc: cannot identify the current CUDA context");
    return ATTN_ERR_CUDA;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx) {
      // In host code g_bwd_scratch only names a host-side stand-in; the
      // device address comes from the runtime, once per device and context,
      // with that device current.
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
      if (e != cudaSuccess || !ptr) {
        attn::set_last_error("attn_bwd_noalloc: cudaGetSymbolAddress failed: %s",
                             cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
      }
      g_scratch_addr[dev] = ptr;
      g_scratch_ctx[dev] = ctx;
    }
    scratch = g_scratch_addr[dev];
  }
  return attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, dtype, scratch,
                  kScratchBytes, stream);
}
