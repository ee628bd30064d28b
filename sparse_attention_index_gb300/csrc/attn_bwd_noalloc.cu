// dsa_sparse_attn_bwd_noalloc: the sparse-attention backward for callers that
// cannot allocate device memory.
//
// Some callers are handed their input and output buffers by a host program
// and have no way to obtain more device memory: a plugin running inside a
// runtime that owns every device allocation through its own pool, or code
// that must not call cudaMalloc once it is running because an allocation can
// fail or stall the device at that point. Such callers cannot supply the fp32
// dK/dV accumulator that dsa_sparse_attn_bwd asks for. This entry point runs
// the same kernels with that accumulator in a fixed array that lives in the
// library itself.
//
// The array is a file-scope __device__ variable of kNoallocMaxFloats floats
// (32 MiB). Every GPU that loads the library holds it until the process
// exits. Host code may not use its name as a device address (on the host the
// name refers to a host-side shadow, which a kernel cannot use), so the first
// call on each device looks up its device address with cudaGetSymbolAddress,
// with that device current, and caches it. That first call should therefore
// come before any stream capture. No call allocates or frees anything.

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/dsa.h"
#include "dsa_internal.h"

namespace {

constexpr size_t kNoallocMaxFloats = DSA_NOALLOC_BWD_MAX_FLOATS;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_bwd_scratch[kNoallocMaxFloats];

std::mutex g_setup_mutex;
float* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device; set up once per device.
float* scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    float* ptr = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_bwd_scratch) !=
        cudaSuccess)
      return nullptr;
    g_scratch_addr[dev] = ptr;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" int dsa_sparse_attn_bwd_noalloc(const void* Q, const void* K, const void* V,
                                           const int32_t* idx, const void* O, const float* lse,
                                           const void* dO, int B, int S, int H, int Hkv, int Dqk,
                                           int Dv, int k, float scale, void* dQ, void* dK,
                                           void* dV, void* stream) {
  // the same argument checks as dsa_sparse_attn_bwd
  const int rc = dsa::attn_bwd_args_status(Q, K, V, idx, O, lse, dO, B, S, H, Hkv, Dqk, Dv, k,
                                           dQ, dK, dV);
  if (rc != DSA_OK) return rc;
  // per-head K/V runs on the dense-tile kernels, whose scratch this entry point lacks
  if (Hkv != 1) return DSA_ERR_UNSUPPORTED;
  // the accumulator needs one fp32 row of Dqk + Dv per key
  const unsigned long long need =
      static_cast<unsigned long long>(B) * S * Hkv * (static_cast<unsigned>(Dqk) + Dv);
  if (need > kNoallocMaxFloats) return DSA_ERR_WORKSPACE;
  float* ws = scratch_for_current_device();
  if (ws == nullptr) return DSA_ERR_CUDA;
  // launch_attn_bwd zeroes the rows it uses (cudaMemsetAsync) before accumulating
  return dsa::launch_attn_bwd(Q, K, V, idx, O, lse, dO, B, S, H, Dqk, Dv, k, scale, dQ, dK, dV,
                              ws, static_cast<cudaStream_t>(stream), dsa::kBwdPathNoAlloc, 1,
                              nullptr);
}
