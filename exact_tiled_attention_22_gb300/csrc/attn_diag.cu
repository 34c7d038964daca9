// attn_diag.cu -- attn_philox4x32_10: runs the dropout generator of the
// kernels (dropout.cuh) on caller-given counters and keys, so that a test can
// hold it against the published known-answer vectors of Philox4x32-10
// (Salmon et al., SC 2011) on the GPU itself.
#include <cuda_runtime.h>

#include <cstdint>

#include "attn.h"
#include "dropout.cuh"
#include "kernels.h"

namespace {

// One thread per vector: in[6 i .. 6 i + 5] = counter words 0-3, key words
// 0-1; out[4 i .. 4 i + 3] = the four output words.
__global__ void philox_diag_kernel(const uint32_t* __restrict__ in, uint32_t* __restrict__ out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint32_t* c = in + 6 * (size_t)i;
  const uint4 x = attn::philox4x32_10(make_uint4(c[0], c[1], c[2], c[3]), c[4], c[5]);
  uint32_t* o = out + 4 * (size_t)i;
  o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w;
}

}  // namespace

extern "C" int attn_philox4x32_10(const uint32_t* in, uint32_t* out, int n, void* stream) {
  if (!in || !out || n < 1 || n > (1 << 24)) {
    attn::set_last_error("attn_philox4x32_10: null pointer or n outside [1, 2^24] (n = %d)", n);
    return ATTN_ERR_INVALID;
  }
  if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 3u) {
    attn::set_last_error("attn_philox4x32_10: pointers must be 4-byte aligned");
    return ATTN_ERR_ALIGN;
  }
  const uintptr_t ilo = reinterpret_cast<uintptr_t>(in), ihi = ilo + 24 * (size_t)n;
  const uintptr_t olo = reinterpret_cast<uintptr_t>(out), ohi = olo + 16 * (size_t)n;
  if (ilo < ohi && olo < ihi) {
    attn::set_last_error("attn_philox4x32_10: out overlaps in");
    return ATTN_ERR_INVALID;
  }
  philox_diag_kernel<<<(n + 127) / 128, 128, 0, static_cast<cudaStream_t>(stream)>>>(in, out, n);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    attn::set_last_error("attn_philox4x32_10 launch: %s", cudaGetErrorString(e));
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}
