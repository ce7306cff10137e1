// Allocation-free decode entry point: moe_ffn_layer on the GEMV rail with its
// scratch in a statically sized device array owned by the library.
//
// Who needs it: callers that cannot call cudaMalloc at the point where they run
// the layer, for example a serving loop that must stay allocation-free after
// start-up (cudaMalloc and cudaFree can synchronise the device and stall other
// streams), or a plugin inside a host framework that hands over only a stream
// and its tensors. They pass inputs and outputs as usual; everything else the
// decode rail needs comes from this file's array.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/moe_mxfp4.h"
#include "moe_internal.h"

namespace {

// Scratch of every decode call on a device. Device code could name it directly;
// host code only ever uses the address obtained below.
__device__ __align__(256) unsigned char g_decode_scratch[MOE_DECODE_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_decode_scratch on the current device, looked up once per
// device with that device current (and kept for the life of the process: the
// library is not meant to be used across cudaDeviceReset).
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) {
    moe::set_last_cuda_error((int)err);
    return MOE_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return MOE_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (err != cudaSuccess || p == nullptr) {
      moe::set_last_cuda_error((int)(err != cudaSuccess ? err : cudaErrorInvalidSymbol));
      return MOE_ECUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" int moe_ffn_layer_decode_static(const float* x, int T, int D, int F, int E, int k,
                                           const float* w_router, const float* b_router,
                                           const uint8_t* g_qs, const uint8_t* g_sc,
                                           const float* bg, const uint8_t* u_qs,
                                           const uint8_t* u_sc, const float* bu,
                                           const uint8_t* d_qs, const uint8_t* d_sc,
                                           const float* bd, float* y, int32_t* ids_out,
                                           float* weights_out, cudaStream_t stream) {
  if (T < 0 || T > MOE_GEMV_MAX_T) return MOE_EINVAL;
  const size_t need = moe_ffn_workspace_bytes(T, D, F, E, k, MOE_RAIL_GEMV);
  if (need == 0) return MOE_EINVAL;
  if (need > (size_t)MOE_DECODE_SCRATCH_BYTES) return MOE_ESCRATCH;
  if (T == 0) return MOE_OK;
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != MOE_OK) return rc;
  return moe_ffn_layer(x, T, D, F, E, k, w_router, b_router, g_qs, g_sc, bg, u_qs, u_sc, bu, d_qs,
                       d_sc, bd, MOE_RAIL_GEMV, scratch, (size_t)MOE_DECODE_SCRATCH_BYTES, y,
                       ids_out, weights_out, stream);
}
