// Sampled decode output with the workspaces in the library's own device
// memory (attn_skip_santa_decode_noalloc).
//
// attn_skip_santa_decode needs two workspaces, the per-key score stash and
// the per-tile (max, sum) pairs, and expects the caller to allocate them.
// Some callers cannot: a host runtime whose plugin interface hands over only
// input and output pointers, an engine that reserved all the device memory it
// will use before the first step, or a decode loop that cannot afford the
// device-wide synchronisation cudaMalloc and cudaFree imply.  For them this
// file keeps one fixed scratch array in the library's device memory and runs
// the same two kernels with both workspaces placed in it.
//
// The array is a file-scope __device__ variable: every GPU on which the
// library is loaded holds it (16.25 MiB) until the process exits.  In host
// code its name is only a host-side stand-in, never a device address, so each
// call looks up the device address with cudaGetSymbolAddress, for the context
// current on the calling thread, and passes it to the kernels.  The look-up is
// a host-side table read once the library's device code is loaded in that
// context; the first call in a context may load it.  No address is cached
// across calls: after cudaDeviceReset, or with another context made current
// on the same device, the array lives at a new address (or in another module
// instance), and a cached one would point at memory that is gone.
#include <cuda_runtime.h>

#include "attn_skip.h"

namespace {

constexpr size_t kScoreFloats = size_t(4) << 20;  // score stash: 4,194,304 floats
constexpr size_t kStatFloats = size_t(64) << 10;  // tile statistics: 65,536 floats
static __device__ __align__(256) float g_santa_scratch[kScoreFloats + kStatFloats];

// Device address of g_santa_scratch in the context current on this thread.
cudaError_t scratch_address(float **out) {
  void *sym = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&sym, g_santa_scratch);
  if (e != cudaSuccess) return e;
  *out = static_cast<float *>(sym);
  return cudaSuccess;
}

}  // namespace

extern "C" attn_status attn_skip_santa_decode_noalloc(
    const void *q, const void *k, const void *v, attn_dtype dt, int B, int Hq, int Hkv, int L,
    int dk, int dv, int64_t k_row_stride, int64_t v_row_stride, float scale, int n_samples,
    attn_santa_mode mode, const float *u, int n_tiles, attn_dtype out_dt, void *o, int32_t *idx,
    void *stream) {
  if (B <= 0 || Hq <= 0 || L <= 0 || n_tiles <= 0) return ATTN_EINVAL;
  // Compared in double so that no product of the int arguments can wrap.
  const double keys = (double)B * (double)Hq * (double)(((long)L + 127) / 128) * 128.0;
  const double stats = (double)B * (double)Hq * (double)n_tiles * 2.0;
  if (keys > (double)kScoreFloats || stats > (double)kStatFloats) return ATTN_EINVAL;
  float *scratch = nullptr;
  const cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    cudaGetLastError();  // clear the error so the caller can continue
    return ATTN_ECUDA;
  }
  // Both parts are written in full by the score pass before the sampling
  // pass reads them, so nothing left over from an earlier call is read and
  // nothing needs clearing.
  return attn_skip_santa_decode(q, k, v, dt, B, Hq, Hkv, L, dk, dv, k_row_stride, v_row_stride,
                                scale, n_samples, mode, u, n_tiles, scratch,
                                scratch + kScoreFloats, out_dt, o, idx, stream);
}
