// jl_bifocal_decode_noalloc: the decode entry point for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand the library a workspace: a plugin inside
// a host framework that owns every device allocation and exposes no
// allocator, or a runtime that forbids allocation on its serving path.  For
// them this entry point runs the same split-K decode kernels as
// jl_bifocal_decode, with the per-slice partial results kept in a fixed
// scratch array that is part of the library image instead of a caller
// workspace.
//
// The array (kScratchBytes, 16 MiB) is a file-scope __device__ variable:
// every GPU on which the library is loaded holds it until the process exits.
// A call needs min(SMs, 512) * B * Hq * (d + 2) * 4 bytes of it (one fp32
// partial per key slice and query head), so on a 148-SM B300 it serves
// B * Hq <= 218 at d = 128 and B * Hq <= 425 at d = 64.  Host
// code cannot use the array's name as a device address, so the first call
// on each device (with that device current) resolves the address with
// cudaGetSymbolAddress and caches it; that first call should therefore be
// made before any stream capture begins.  Nothing in the array needs to
// start at zero: each call writes every slot it later reads.  All calls share
// the one array, so calls whose kernels overlap on the GPU (different
// streams, or threads without ordering) race and corrupt each other.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "../../include/jetlong.h"
#include "internal.h"

namespace jl {
namespace {

// 16 MiB: the per-slice partials of B * Hq <= 218 query heads at d = 128 on
// a 148-SM GPU (one fp32 partial of d + 2 values per key slice and head).
constexpr size_t kScratchBytes = size_t(16) << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (resolved once).
void* scratch_on_current_device(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

}  // namespace jl

extern "C" {

size_t jl_bifocal_decode_noalloc_scratch_bytes(void) { return jl::kScratchBytes; }

int jl_bifocal_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, int L, int Lcap,
                              void* o, float* lse, int B, int Hq, int Hkv, int d, int w0,
                              int w_pretrained, double rope_theta, float softmax_scale,
                              void* cuda_stream) {
  using namespace jl;
  set_error(JL_OK, "");
  // The same argument checks, in the same order, as jl_bifocal_decode; only
  // then the size limit of the fixed array.
  int rc = check_decode_args("decode_noalloc", q, k_cache, v_cache, L, Lcap, o, B, Hq, Hkv, d, w0, w_pretrained,
                             rope_theta);
  if (rc != JL_OK) return rc;
  const size_t need = decode_scratch_bytes(B, Hq, d);
  if (need > kScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "decode_noalloc: B=%d Hq=%d d=%d needs %zu bytes of scratch; the fixed array holds %zu",
             B, Hq, d, need, kScratchBytes);
    return set_error(JL_ERR_UNSUPPORTED, msg);
  }
  cudaError_t err = cudaSuccess;
  void* scratch = scratch_on_current_device(&err);
  if (scratch == nullptr) {
    char msg[200];
    snprintf(msg, sizeof(msg), "decode_noalloc: cannot resolve the scratch array: %s",
             cudaGetErrorString(err));
    return set_error(JL_ERR_CUDA, msg);
  }
  // The kernels of jl_bifocal_decode, with the partials in the fixed array.
  return decode_call("decode_noalloc", q, k_cache, v_cache, nullptr, L, Lcap, o, lse, B, Hq, Hkv, d, w0,
                     w_pretrained, rope_theta, softmax_scale, static_cast<float*>(scratch), cuda_stream);
}

}  // extern "C"
