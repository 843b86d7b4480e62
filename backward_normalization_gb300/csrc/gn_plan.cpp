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
  (void)op;
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
  // Four 512-thread CTAs fit on one SM; one item per CTA, one wave when the
  // problem is large enough to fill the device.
  const int64_t target = (int64_t)sm_count * 4;
  if (layout == kNHWC) {
    g.vw = (aligned && C % vec == 0) ? vec : 1;
    g.V = C / g.vw;
    g.ncb = (int)cdiv(g.V, 256);
    g.Wv = (int)cdiv(g.V, g.ncb);
    g.rpi = 512 / g.Wv;
    if (g.rpi < 1) g.rpi = 1;
    g.tpb = g.Wv * g.rpi;
    int64_t T = clamp64(cdiv(target, N * g.ncb), 1, cdiv(HW, g.rpi));
    g.rb = rup(cdiv(HW, T), g.rpi);
    g.T = cdiv(HW, g.rb);
    g.items_per_n = g.T * g.ncb;
    g.items = N * g.items_per_n;
    g.cstride = 1;
    g.tstride = C;
  } else {
    g.vw = (aligned && HW % vec == 0) ? vec : 1;
    if (HW >= 2048) {
      g.mode = 0;
      g.tpb = 512;
      const int64_t P = clamp64(cdiv(target, N * C), 1, cdiv(HW, (int64_t)g.tpb * g.vw));
      g.L = rup(cdiv(HW, P), g.vw);
      g.T = cdiv(HW, g.L);
      g.items_per_n = C * g.T;
      g.cstride = g.T;
      g.tstride = 1;
    } else {
      g.mode = 1;
      g.tpb = 256;
      g.RB = clamp64(cdiv(N * C, target), 8, C);
      g.T = 1;
      g.items_per_n = cdiv(C, g.RB);
      g.cstride = 1;
      g.tstride = 1;
    }
    g.items = N * g.items_per_n;
  }
  return g;
}

WsLayout ws_layout(int op, const Geom& g) {
  WsLayout w{};
  size_t off = 0;
  w.tickets = off;
  off = align256(off + sizeof(unsigned long long) * (size_t)(g.N + 1));
  w.err = off;
  off = align256(off + sizeof(unsigned));
  w.part = off;
  off = align256(off + 2 * sizeof(float) * (size_t)(g.N * g.C * g.T));
  w.chst = off;
  off = align256(off + 2 * sizeof(float) * (size_t)(g.N * g.C));
  w.coef = off;
  if (op == kBwd) off = align256(off + 2 * sizeof(float) * (size_t)(g.N * g.G));
  w.total = off;
  return w;
}

}  // namespace gn
