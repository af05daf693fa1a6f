// muon_newton_schulz_noalloc: Newton-Schulz without a caller workspace.
//
// Some callers cannot hand this library device memory.  A framework whose
// caching allocator owns the device's memory does not want foreign
// cudaMalloc calls carving pieces out of the pool it has reserved; cudaFree
// synchronises the whole device, which a latency-sensitive training loop
// cannot afford between steps; and a plugin running inside a host
// application may have no allocator at all.  For them this entry point
// takes its scratch from one fixed array compiled into the library, so the
// call itself allocates nothing.
//
// The array lives in device memory of every GPU that loads the library, for
// the life of the process.  Its size caps the problems this entry point
// accepts (see MC_NOALLOC_SCRATCH_BYTES); larger requests are rejected with
// MC_ERR_WORKSPACE and must use muon_newton_schulz with a workspace.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/muonclip.h"
#include "kernels.h"

namespace {

static_assert(MC_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");

// The scratch.  In host code `g_noalloc_scratch` is only a host-side
// stand-in for the symbol: the device address comes from
// cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch on the current device (set-up on first use,
// then kept: a cudaDeviceReset would invalidate it, which the header rules
// out for callers of this entry point).
mc_status scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return mc::record_error(MC_ERR_CUDA, "muon_newton_schulz_noalloc: cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices)
    return mc::record_error(MC_ERR_UNSUPPORTED, "muon_newton_schulz_noalloc: device index too large");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      char msg[160];
      snprintf(msg, sizeof msg, "muon_newton_schulz_noalloc: cudaGetSymbolAddress failed: %s",
               cudaGetErrorString(e));
      return mc::record_error(MC_ERR_CUDA, msg);
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return MC_OK;
}

}  // namespace

extern "C" mc_status muon_newton_schulz_noalloc(const mc_mat* M, mc_mat* O, int32_t count,
                                                const mc_hparams* hp, int32_t* status,
                                                mc_stream_t stream) {
  size_t need = 0;
  mc_status st = mc_workspace_size(M, count, hp, &need);
  if (st != MC_OK) return st;
  if (need > (size_t)MC_NOALLOC_SCRATCH_BYTES) {
    char msg[200];
    snprintf(msg, sizeof msg,
             "muon_newton_schulz_noalloc: these matrices need %zu bytes of scratch; the static "
             "array holds %zu (use muon_newton_schulz with a workspace)",
             need, (size_t)MC_NOALLOC_SCRATCH_BYTES);
    return mc::record_error(MC_ERR_WORKSPACE, msg);
  }
  void* ws = nullptr;
  if ((st = scratch_address(&ws)) != MC_OK) return st;
  return muon_newton_schulz(M, O, count, hp, ws, (size_t)MC_NOALLOC_SCRATCH_BYTES, status, stream);
}
