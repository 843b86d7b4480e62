// gn_static_ws.cu -- gn_fwd_static_ws: the forward pass for callers that
// cannot allocate device memory.
//
// gn_fwd needs a caller-provided workspace.  Some callers cannot obtain one:
// code that runs under a fixed memory budget once it has started (serving
// loops that forbid allocation on the request path), plugins whose host
// framework hands them no allocator, and paths where calling cudaMalloc is
// not permitted at that point.  For them this file holds the workspace itself,
// in a statically sized device array, and the entry point below never calls
// cudaMalloc, cudaFree or any allocating routine.
//
// The array exists once per device that loads the library and stays reserved
// until the process exits.  Every call shares it, so calls that overlap on
// the GPU (two streams at once, or two host threads) race and must not be
// made.  Like any workspace it needs no clearing: each call zero-fills the
// counters it uses, on its own stream, before its kernels run.
#include <mutex>

#include "../../include/gn.h"
#include "gn_internal.h"

namespace {

constexpr size_t kStaticWsBytes = GN_STATIC_WS_BYTES;  // per device

// The scratch area.  In host code this name is only a stand-in for the
// device array: its device address is obtained with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_dev_ptr[kMaxDevices] = {};

// Device address of g_static_ws on the current device, looked up once per
// device (with that device current) and cached.
cudaError_t static_ws_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_dev_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess) return e;
    g_dev_ptr[dev] = p;
  }
  *out = g_dev_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

int gn_fwd_static_ws(const void* x, int64_t N, int64_t C, int64_t HW, int64_t G, int layout,
                     int dtype, const float* gamma, const float* beta, float eps, void* y,
                     float* mean, float* rstd, void* stream) {
  const size_t need = gn_workspace_size(GN_OP_FWD, N, C, HW, G, layout, dtype);
  if (need > kStaticWsBytes) return GN_ERR_WORKSPACE;  // larger than the static area
  if (need == 0)  // invalid or empty problem: gn_fwd reports it, touching no workspace
    return gn_fwd(x, N, C, HW, G, layout, dtype, gamma, beta, eps, y, mean, rstd, nullptr, 0,
                  stream);
  void* ws = nullptr;
  const cudaError_t e = static_ws_address(&ws);
  if (e != cudaSuccess) return gn::record_cuda_error(e);
  // gn_fwd validates every argument before it enqueues anything, and clears
  // the counters of the area at the start of its work on `stream`, so the
  // contents the previous call left do not matter.
  return gn_fwd(x, N, C, HW, G, layout, dtype, gamma, beta, eps, y, mean, rstd, ws,
                kStaticWsBytes, stream);
}

}  // extern "C"
