// gn_plan.cpp -- host-side work decomposition for one GroupNorm call.
//
// The plan depends only on the problem (N, C, HW, G, layout, dtype), on
// whether every data pointer is 16-byte aligned, and on the device's SM count,
// so the same call on the same device always runs the same reduction tree and
// gives bit-identical results.
#include <atomic>

#include "gn_internal.h"

namespace gn {
namespace {

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t rup(int64_t a, int64_t b) { return cdiv(a, b) * b; }
int64_t clamp64(int64_t v, int64_t lo, int64_t hi) { return v < lo ? lo : (v > hi ? hi : v); }
size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

constexpr int kMaxDevices = 64;
constexpr int64_t kCluster = 8;           // CTAs per cluster in the first kernels
constexpr double kKeepBytes = 64.0 * (1 << 20);  // input kept in L2 for the second kernel
std::atomic<int> g_sm_cache[kMaxDevices];

}  // namespace

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 152;  // no device visible: size plans for a full GB300
  }
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = g_sm_cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();
    return 152;
  }
  if (dev >= 0 && dev < kMaxDevices) g_sm_cache[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

Geom make_geom(int op, int64_t N, int64_t C, int64_t HW, int64_t G, int layout, int dtype,
               bool aligned, int sm_count) {
  Geom g{};
  g.N = N;
  g.C = C;
  g.HW = HW;
  g.G = G;
  g.Cg = C / G;
  g.layout = layout;
  g.dtype = dtype;
  const int esz = dtype == kF32 ? 4 : 2;
  const int vec = 16 / esz;
  // Two 512-thread CTAs are resident per SM; one item per CTA, one wave when
  // the problem is large enough to fill the device.
  const int64_t target = (int64_t)sm_count * 2;
  int64_t item_len = 0;  // rows (NHWC) or elements (NCHW mode 0) per item
  if (layout == kNHWC) {
    g.vw = (aligned && C % vec == 0) ? vec : 1;
    g.V = C / g.vw;
    g.ncb = (int)cdiv(g.V, 256);
    g.Wv = (int)cdiv(g.V, g.ncb);
    g.rpi = 512 / g.Wv;
    if (g.rpi < 1) g.rpi = 1;
    g.tpb = g.Wv * g.rpi;
    int64_t T = clamp64(cdiv(target, N * g.ncb), 1, cdiv(HW, g.rpi));
    if (T >= kCluster) T = rup(T, kCluster);
    g.rb = rup(cdiv(HW, T), g.rpi);
    g.T = T;  // trailing items may be empty when rb*T > HW
    g.cl = T % kCluster == 0 ? kCluster : 1;
    g.Tp = T / g.cl;
    g.cstride = 1;
    g.tstride = C;
    g.arrivals_per_n = g.Tp * g.ncb;
    g.items_per_n = T * g.ncb;
    item_len = g.rb;
  } else {
    g.vw = (aligned && HW % vec == 0) ? vec : 1;
    if (HW >= 2048) {
      g.mode = 0;
      g.tpb = 512;
      int64_t P = clamp64(cdiv(target, N * C), 1, cdiv(HW, (int64_t)g.tpb * g.vw));
      if (P >= kCluster) P = rup(P, kCluster);
      g.L = rup(cdiv(HW, P), g.vw);
      g.T = P;  // trailing chunks may be empty when L*P > HW
      g.cl = P % kCluster == 0 ? kCluster : 1;
      g.Tp = P / g.cl;
      g.cstride = g.Tp;
      g.tstride = 1;
      g.arrivals_per_n = C * g.Tp;
      g.items_per_n = C * P;
      item_len = g.L;
    } else {
      g.mode = 1;
      g.tpb = 256;
      g.RB = clamp64(cdiv(N * C, target), 8, C);
      g.T = 1;
      g.cl = 1;
      g.Tp = 1;
      g.cstride = 1;
      g.tstride = 1;
      g.items_per_n = cdiv(C, g.RB);
      g.arrivals_per_n = g.items_per_n;
    }
  }
  g.items = N * g.items_per_n;
  // The second kernel re-reads first what the first kernel read last: the
  // last kKeepBytes of input (spread over all items) are loaded with the L2
  // evict_last policy, the rest with evict_first.
  const double in_bytes = (double)N * C * HW * esz * (op == kBwd ? 2.0 : 1.0);
  const double keep_frac = in_bytes <= kKeepBytes ? 1.0 : kKeepBytes / in_bytes;
  if (g.layout == kNCHW && g.mode == 1)
    g.keep_from = keep_frac >= 1.0 ? 0 : 1;  // whole rows: all or nothing
  else
    g.keep_from = item_len - (int64_t)((double)item_len * keep_frac);
  return g;
}

WsLayout ws_layout(int op, const Geom& g) {
  WsLayout w{};
  size_t off = 0;
  w.tickets = off;
  off = align256(off + sizeof(unsigned) * (size_t)(g.N + 1));
  w.part = off;
  off = align256(off + 2 * sizeof(float) * (size_t)(g.N * g.C * g.Tp));
  w.chst = off;
  off = align256(off + 2 * sizeof(float) * (size_t)(g.N * g.C));
  w.coef = off;
  if (op == kBwd) off = align256(off + 2 * sizeof(float) * (size_t)(g.N * g.G));
  w.total = off;
  return w;
}

cudaError_t launch_first(const void* kernel, const KParams& p, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.g.items, 1, 1);
  cfg.blockDim = dim3((unsigned)p.g.tpb, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (p.g.cl > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.g.cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  void* args[] = {const_cast<KParams*>(&p)};
  return cudaLaunchKernelExC(&cfg, kernel, args);
}

}  // namespace gn
