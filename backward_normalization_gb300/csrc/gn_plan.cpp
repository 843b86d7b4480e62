// gn_plan.cpp -- host-side work decomposition for one GroupNorm call.
//
// The plan depends only on the problem (N, C, HW, G, layout, dtype), on
// whether every data pointer is 16-byte aligned, and on the device's SM count,
// so the same call on the same device always runs the same reduction tree and
// gives bit-identical results.
#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "gn_internal.h"

namespace gn {
namespace {

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t rup(int64_t a, int64_t b) { return cdiv(a, b) * b; }
int64_t clamp64(int64_t v, int64_t lo, int64_t hi) { return v < lo ? lo : (v > hi ? hi : v); }
size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

constexpr int kMaxDevices = 64;
std::atomic<int> g_regime_override{kRegimeAuto};
constexpr int kGroup1 = 8;                // items per level-1 group (when an (n, c) has >= 16)
constexpr double kKeepBytes = 64.0 * (1 << 20);  // input kept in L2 for the second kernel
std::atomic<int> g_sm_cache[kMaxDevices];

}  // namespace

namespace {
// Co-resident CTAs of the op's first (second = 0) or second (second = 1)
// kernel, or an estimate when no device is visible (two 512-thread or four
// 256-thread CTAs per SM).
int64_t resident_or(const Geom& g, int op, int second, int sm_count) {
  const int64_t r = resident_ctas(g, op, second);
  if (r > 0) return r;
  const int64_t per_sm = g.tpb > 256 ? 2 : 4;
  return (int64_t)sm_count * per_sm;
}
}  // namespace

void set_regime_override(int regime) { g_regime_override.store(regime); }

cudaError_t prepare_smem(const void* kernel, size_t smem) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> done;  // (device, kernel) -> limit set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto it = done.find({dev, kernel});
  if (it != done.end() && it->second >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  done[{dev, kernel}] = smem;
  return cudaSuccess;
}

cudaError_t prepare_resident_kernel(const void* kernel, const Geom& g) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> done;  // (device, kernel) -> smem set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto it = done.find({dev, kernel});
  if (it != done.end() && it->second >= g.smem) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)g.smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  done[{dev, kernel}] = g.smem;
  return cudaSuccess;
}

namespace {
constexpr size_t kSmemPerCta = 227 * 1024 - 1024;  // dynamic smem budget (static use ~1 KB)
constexpr size_t kSmemPerSm = 228 * 1024;           // shared memory of one SM
constexpr size_t kSmallSlice = 88 * 1024;           // slice that lets two CTAs share an SM
constexpr int64_t kMaxUnitBytes = 16ll << 20;       // per-unit input (x, or x + dy)
constexpr int kRingDeep = 8;                        // ring slots when a slice streams

size_t a128(size_t v) { return (v + 127) & ~size_t(127); }
int64_t gcd64(int64_t a, int64_t b) { return b ? gcd64(b, a % b) : a; }

// Clusters of the resident kernel that fit on the device at once (0 if none,
// -1 when no device is visible).
int64_t resident_clusters(const Geom& g, int op) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  const void* fn = resident_kernel_ptr(g, op == kBwd);
  if (prepare_resident_kernel(fn, g) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)g.K, 1, 1);
  cfg.blockDim = dim3((unsigned)resident_threads(g), 1, 1);
  cfg.dynamicSmemBytes = g.smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)g.K;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int nc = 0;
  if (cudaOccupancyMaxActiveClusters(&nc, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return nc;
}

// The automatic choice, from measurements on GB300: the resident kernel wins
// for channels_last forwards and for small NCHW units; for large NCHW units
// and the channels_last backward the two-kernel path is faster today (the
// resident kernel cannot keep every SM streaming there).
bool resident_preferred(const Geom& g, int op) {
  const int esz = dtype_size(g.dtype);
  if (g.layout == kNHWC) return op == kFwd;
  return g.Cg * g.HW * esz <= (1 << 20);
}

// The automatic choice of the wave regime (where its plan fits), from
// measurements on GB300.  It reads each input once; with its pieces held in
// tensor memory and stage A and stage B on separate warps, it beats the
// two-kernel path on every NCHW problem measured from 64 MiB up, forward /
// backward in us against two-kernel: fp32 112x64x512x512 G8 2593 / 4176
// against 3191 / 5231; fp32 16x64x512x512 G64 (1 MiB units) 341 / 509
// against 476 / 784; fp32 32x64x256x256 G8 173 / 302 against 244 / 402;
// fp32 64x64x128x128 G8 (512 KiB units) 93 / 151 against 150 / 245; fp32
// 256x64x64x64 G8 (128 KiB units) 219 / 242 against 433 / 587; bf16
// 8x320x64x64 G32 NCHW 47 / 53 against 69 / 98; fp32 1x64x512x512 G8 (64 MiB)
// 39 / 54 against 37 / 60.  Smaller inputs are left to the resident and
// two-kernel paths.  The small channels-last workloads stay with the other
// families (bf16 8x320x64x64 G32: 50 / 55 us against 29 / 38 us; bf16
// 32x512x32x32 G32: 38 / 53 us against 32 / 38 us): with a handful of steps
// per CTA the cooperative launch and the pipeline's fill cost more than the
// second read they save.
bool wave_preferred(const Geom& g, int op) {
  (void)op;
  const int esz = dtype_size(g.dtype);
  return g.layout == kNCHW && g.Cg * g.HW * esz >= (64ll << 10) && g.N * g.C * g.HW * esz >= (32ll << 20);
}

// The automatic choice of the flat regime, from measurements on GB300 (L2
// flushed before each call): channels-last backwards whose x and dy hold
// 10-48 MiB together, where its one launch and minimal HBM traffic beat the
// two-kernel path (bf16 8x320x64x64 G32: 38.6 against 41.8 us; at N = 2,
// 26.0 against 35.1 us).  Larger backwards lose to the two-kernel path (at
// 64 MiB, 32x512x32x32: 53 against 38 us: pass 2 reads most chunks again
// and the merge and second barrier cost more than the saved launch), and
// forwards lose to the resident or two-kernel path (8x320x64x64: 34.7
// against 23.2 us resident).
bool flat_preferred(const Geom& g, int op) {
  const double in = 2.0 * (double)g.N * (double)g.C * (double)g.HW * dtype_size(g.dtype);
  return op == kBwd && g.layout == kNHWC && in >= 10.0 * (1 << 20) && in <= 48.0 * (1 << 20);
}

// Input that counts as tiny for the automatic choice (see plan_resident).
constexpr double kResidentTinyBytes = 1 << 20;

// Fills the resident-regime fields of g; false when the problem does not fit
// the regime (the two-kernel path then runs).  For the automatic choice
// (`auto_choice`) the regime is also declined unless one wave of clusters
// covers every unit, or the input is tiny: measured on GB300, a cluster's
// load / reduce / write phases barely overlap, so later waves cost nearly a
// whole cluster latency each (bf16 channels-last 8x320x64x64 G32: 22.3 us
// resident against 28.8 us two-kernel in one wave of 32 clusters, but 38.7
// against 34.9 us at N = 16 and 127.8 against 89.0 us at N = 64; fp32 NCHW
// 512x32x16x16 G8: 248 against 28 us).
bool plan_resident(Geom& g, int op, bool auto_choice) {
  const int esz = dtype_size(g.dtype);
  const int vec = 16 / esz;
  const int nten = op == kBwd ? 2 : 1;
  if (g.vw != vec || g.dtype == kF64) return false;  // f64: two-kernel path only
  Geom r = g;
  size_t red_f, xch_f, tot_f, grp_f;
  int64_t nch;  // chunks per slice
  if (g.layout == kNCHW) {
    if (g.Cg > 16) return false;
    if (g.Cg * g.HW * esz * nten > kMaxUnitBytes) return false;
    // large chunks: the per-chunk cost of the pipeline is then small
    const int64_t cbytes = op == kBwd ? 32 * 1024 : 64 * 1024;
    int64_t m = 16 / g.Cg;
    while (m > 1 && g.HW * esz / m < 2 * cbytes) m /= 2;
    r.m = m;
    r.K = (int)(g.Cg * m);
    r.tpb = 512;
    r.slice = rup(cdiv(g.HW, m), vec);
    r.chunk = cbytes / esz < r.slice ? cbytes / esz : r.slice;
    r.chunk_bytes = r.chunk * esz;
    r.units = g.N * g.G;
    nch = cdiv(r.slice, r.chunk);
    red_f = 2 * (size_t)resident_threads(r);
    xch_f = 2;
    tot_f = 0;
    grp_f = 2;
  } else {
    // channel block: whole groups, whole 16-byte vectors, at most 128 channels
    // when possible (TMA boxes hold at most 256 elements per dimension)
    const int64_t step = g.Cg / gcd64(g.Cg, vec) * vec;
    int64_t cb = 0;
    for (int64_t c = step; c <= g.C && c <= 256; c += step)
      if (g.C % c == 0 && (c <= 128 || cb == 0)) cb = c;
    if (cb == 0) return false;
    if (g.HW * cb * esz * nten > kMaxUnitBytes) return false;
    if (g.N * g.HW > 0x7fffffffLL) return false;  // TMA row coordinates are 32-bit
    r.Cb = cb;
    r.ncbu = g.C / cb;
    r.ncb = 1;
    r.Wv = (int)(cb / vec);
    r.rpi = 256 / r.Wv > 0 ? 256 / r.Wv : 1;
    r.tpb = r.Wv * r.rpi;
    const int64_t row_bytes = cb * esz;
    r.units = g.N * r.ncbu;
    r.K = 1;
    while (r.K < 16 && (size_t)(cdiv(g.HW, r.K) * row_bytes * nten) > kSmallSlice) r.K *= 2;
    r.slice = cdiv(g.HW, r.K);
    // chunks of at most 16 KB (and 256 rows, the TMA box limit) that tile the
    // slice evenly
    const int64_t max_rows = clamp64((16 * 1024) / row_bytes, 1, 256);
    nch = cdiv(r.slice, max_rows);
    r.chunk = cdiv(r.slice, nch);
    r.chunk_bytes = r.chunk * row_bytes;
    red_f = 2 * (size_t)vec * ((r.tpb + 31) / 32 * 32);
    if (red_f < 2 * (size_t)resident_threads(r)) red_f = 2 * (size_t)resident_threads(r);
    xch_f = 2 * (size_t)cb;
    tot_f = 2 * (size_t)cb;
    grp_f = 2 * (size_t)(cb / g.Cg);
  }
  const size_t fixed = a128(red_f * 4) + a128(xch_f * 4) + a128(tot_f * 4) + a128(grp_f * 4);
  r.ten_stride = (int64_t)a128((size_t)r.chunk_bytes);
  const size_t slot = (size_t)r.ten_stride * nten;
  if (kSmemPerCta < fixed + 1024) return false;
  const int64_t slots = (int64_t)((kSmemPerCta - fixed - 512) / (slot + 16));
  if (nch <= slots) {
    r.nres = (int)nch;
    r.S = 0;
  } else {
    if (slots < 3) return false;
    r.S = (int)(slots - 1 < kRingDeep ? slots - 1 : kRingDeep);
    r.nres = (int)(slots - r.S);
  }
  size_t off = 0;
  off += a128((size_t)r.nres * slot);
  r.off_ring = off;
  off += a128((size_t)r.S * slot);
  r.off_red = off;
  off += a128(red_f * 4);
  r.off_xch = off;
  off += a128(xch_f * 4);
  r.off_tot = off;
  off += a128(tot_f * 4);
  r.off_grp = off;
  off += a128(grp_f * 4);
  r.off_bar = off;
  off += a128(8 * (size_t)(r.nres + 2 * r.S));  // full barriers, and empty barriers for the ring
  r.smem = off + 128;  // slack for aligning the dynamic shared memory base
  if (r.smem > kSmemPerCta) return false;
  if (r.units * r.K > 0x7fffffffLL) return false;
  r.regime = kRegimeResident;
  r.T = 0;  // no two-kernel partial records
  r.l1 = 1;
  r.Tp = 0;
  r.groups1 = 0;
  const int64_t nc = resident_clusters(r, op);
  if (nc == 0) return false;
  if (auto_choice) {
    // co-resident clusters (an estimate when no device is visible: one or two
    // CTAs per SM by shared memory)
    const int64_t waves_of =
        nc > 0 ? nc : (int64_t)device_sm_count() * (r.smem <= kSmemPerSm / 2 ? 2 : 1) / r.K;
    const double in_bytes = (double)g.N * g.C * g.HW * esz * nten;
    if (r.units > waves_of && in_bytes > kResidentTinyBytes) return false;
  }
  g = r;
  return true;
}
}  // namespace

namespace {
// Pipelined regime (NCHW): every CTA takes one piece of every unit, in
// lockstep, so the input read between a unit's two passes is only the lag's
// D units; its chunks of at most kPipeChunkBytes per tensor stream through a
// ring of at least kPipeMinSlots slots in the CTA's share of shared memory.
#ifndef GN_PIPE_CHUNK_BYTES
#define GN_PIPE_CHUNK_BYTES (16 * 1024)
#endif
#ifndef GN_PIPE_LAG
#define GN_PIPE_LAG 2
#endif
#ifndef GN_PIPE_L2_BYTES
#define GN_PIPE_L2_BYTES (64ll << 20)
#endif
#ifndef GN_PIPE_MAX_SLOTS
#define GN_PIPE_MAX_SLOTS 16
#endif
#ifndef GN_PIPE_CTAS_PER_SM
#define GN_PIPE_CTAS_PER_SM 2
#endif
constexpr int64_t kPipeChunkBytes = GN_PIPE_CHUNK_BYTES;
constexpr int64_t kPipeLag = GN_PIPE_LAG;         // D: pass 2 of unit u runs in step u + D
constexpr int64_t kPipeL2Bytes = GN_PIPE_L2_BYTES;  // the D + 1 units in flight must fit
constexpr int kPipeMaxSlots = GN_PIPE_MAX_SLOTS;
constexpr int kPipeCtasPerSm = GN_PIPE_CTAS_PER_SM;
constexpr int kPipeMinSlots = 4;

// CTAs of the pipelined kernel that fit on the device at once, or an estimate
// (kPipeCtasPerSm per SM) when no device is visible; 0 if none fit.
int64_t pipelined_ctas(const Geom& g, int op, int sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return (int64_t)sm_count * kPipeCtasPerSm;
  }
  size_t smem = 0;
  const void* fn = nchw_pipelined_kernel(g, op == kBwd, &smem);
  int nb = 0;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, g.tpb, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return (int64_t)nb * sm_count;
}

// Fills the pipelined-regime fields of g (a two-kernel plan of the same
// problem); false when the problem does not fit the regime.
bool plan_pipelined(Geom& g, int op, int sm_count) {
  const int esz = dtype_size(g.dtype);
  const int vec = 16 / esz;
  const int nten = op == kBwd ? 2 : 1;
  if (g.layout != kNCHW || g.mode != 0 || g.vw != vec || g.dtype == kF64) return false;
  const int64_t unit_bytes = g.Cg * g.HW * esz * nten;
  if ((kPipeLag + 1) * unit_bytes > kPipeL2Bytes) return false;
  Geom r = g;
  r.regime = kRegimePipelined;
  r.tpb = 512 / kPipeCtasPerSm / 32 * 32;
  const size_t smem_cap = std::min(kSmemPerCta, kSmemPerSm / kPipeCtasPerSm - 2048);
  // ---- the ring
  const int64_t scratch = nchw_pipelined_scratch_floats(r);
  r.off_red = 0;
  const size_t fixed = a128((size_t)scratch * 4);
  const size_t overhead = kSlotHdrBytes + sizeof(uint64_t) + 128;  // header, mbarrier, padding
  if (smem_cap < fixed + 512 + kPipeMinSlots * overhead) return false;
  const int64_t fit = (int64_t)((smem_cap - fixed - 512) / kPipeMinSlots - overhead) / nten;
  const int64_t cbytes = std::min<int64_t>(kPipeChunkBytes, fit);
  r.chunk = cbytes / 128 * 128 / esz;  // elements (a multiple of the vector width)
  if (r.chunk < (int64_t)r.tpb * vec) return false;
  r.chunk_bytes = r.chunk * esz;
  r.ten_stride = (int64_t)a128((size_t)r.chunk_bytes);
  r.dy_in_ring = nten == 2 ? 1 : 0;
  const size_t slot = (size_t)r.ten_stride * nten;
  const size_t per_slot = slot + kSlotHdrBytes + sizeof(uint64_t);  // data, header, mbarrier
  r.S = (int)std::min<int64_t>(kPipeMaxSlots, (int64_t)((smem_cap - fixed - 512) / per_slot));
  r.off_tot = fixed;                                          // slot headers
  r.off_bar = r.off_tot + a128(kSlotHdrBytes * (size_t)r.S);  // mbarriers
  r.off_ring = r.off_bar + a128(8 * (size_t)r.S);
  r.smem = r.off_ring + (size_t)r.S * slot + 128;  // slack for aligning the dynamic smem base
  if (r.smem > smem_cap) return false;
  r.grid = pipelined_ctas(r, op, sm_count);
  if (r.grid < g.Cg) return false;
  // ---- the pieces: segments of each plane, one per CTA
  const int64_t m = r.grid / g.Cg;
  r.L = rup(cdiv(g.HW, m), vec);
  r.T = cdiv(g.HW, r.L);
  r.units_fin = g.N * g.G;
  r.unit_groups = 1;
  r.pieces = g.Cg * r.T;
  r.l1 = 1;  // the finaliser merges the Cg*T records of its unit directly
  r.Tp = r.T;
  r.groups1 = 0;
  r.cstride = r.T;
  r.tstride = 1;
  r.arrivals_per_n = g.Cg * r.T;
  r.items_per_n = g.C * r.T;
  r.items = g.N * r.items_per_n;
  r.keep_from = 0;
  r.lag = std::min<int64_t>(kPipeLag, r.units_fin);
  g = r;
  return true;
}
}  // namespace

namespace {
// Wave regime (gn_wave.cu): a unit's pieces are held by several CTAs at
// once, S slots each; S >= 2 (one piece in use, one landing).
#ifndef GN_WAVE_MIN_SLOTS
#define GN_WAVE_MIN_SLOTS 3
#endif
#ifndef GN_WAVE_MAX_SLOTS
#define GN_WAVE_MAX_SLOTS 8
#endif
#ifndef GN_WAVE_MAX_CB
#define GN_WAVE_MAX_CB 128
#endif
// Tensor-memory buffers a wave CTA may hold reduced pieces in (0: none).
#ifndef GN_WAVE_MAX_HOLD
#define GN_WAVE_MAX_HOLD 4
#endif
constexpr int kWaveMinSlots = GN_WAVE_MIN_SLOTS;
constexpr int kWaveMaxSlots = GN_WAVE_MAX_SLOTS;
constexpr int64_t kWaveMaxCb = GN_WAVE_MAX_CB;  // channels per NHWC unit (TMA box <= 256)
constexpr int64_t kWaveMaxHold = GN_WAVE_MAX_HOLD < kWaveMaxSlots - 1 ? GN_WAVE_MAX_HOLD : kWaveMaxSlots - 1;

// CTAs of the wave kernel that fit on the device at once with `smem` bytes of
// dynamic shared memory (an estimate when no device is visible).
int64_t wave_ctas(const Geom& g, int op, size_t smem, int sm_count, int want_per_sm) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return (int64_t)sm_count * want_per_sm;
  }
  const void* fn = wave_kernel_ptr(g, op == kBwd);
  int nb = 0;
  if (prepare_smem(fn, smem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, g.tpb, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return (int64_t)std::min(nb, want_per_sm) * sm_count;
}

// One candidate cut of a wave plan: pieces per unit P, values per piece R
// (elements of a plane, or rows), slots S, CTAs NC; `cost` estimates its
// time in microseconds.
struct WaveCut {
  int64_t P = 0, R = 0, m = 1, nb = 1, box = 0, Cb = 0, S = 0, steps = 0, H = 0, T4 = 0;
  bool fwd = false;
  double cost = 0.0;
  size_t slot = 0, out = 0;
};

// Stage A of a wave step runs this many pieces ahead of stage B: with
// tensor-memory buffers, one less than their number; else one when a third
// slot lets a piece land while two are in use.
int64_t wave_ahead(int64_t H, int64_t S) { return H > 0 ? H - 1 : (S >= 3 ? 1 : 0); }

// Cost model of a wave cut, in microseconds, fitted to measurements on
// GB300.  t_io is a step's data at 45 GB/s per SM (in + out), shared by the
// CTAs on it.  With pieces held in tensor memory and warp specialisation, a
// step costs about 1.75 us plus half of t_io: the stages overlap the copies,
// and most of a step is the chain of barriers, record exchange and merge
// (fp32 NCHW forward, per step: 13.8 KB pieces 2.0 us, 26 KB 2.3, 32 KB 2.3,
// 52 KB 3.0, 55 KB 3.0).  With only two hold buffers stage A runs one step
// ahead, and every step waits for the unit's slowest CTA: about 0.4 us more,
// plus up to 1 us as the unit spreads over all CTAs (backward: 55 KB pieces
// over 19 CTAs 4.0 us, over 152 CTAs 5.0 us).  A unit over a small share of
// the CTAs straddling two steps costs nothing measurable there.  Without hold buffers: t_io plus 0.4 us a
// step, 0.3 us more for a unit split over CTAs, about 1 us more when the
// wait for a unit is exposed (two slots), and a piece time more when a unit
// straddles two steps.
#ifndef GN_WAVE_FORCE_CB
#define GN_WAVE_FORCE_CB 0
#endif
#ifndef GN_WAVE_FORCE_P
#define GN_WAVE_FORCE_P 0
#endif
double wave_cost(const WaveCut& c, int64_t NC) {
  const double t_io = (double)(c.slot + c.out) * kWaveCtasPerSm / 45.0e3;
  double per_step;
  if (c.H > 0 && kWaveWs) {
    per_step = 1.75 + 0.5 * t_io;
    if (c.H < 3) per_step += 0.4 + (double)std::min(c.P, NC) / (double)NC;
    // forward: a unit over more than half of the CTAs that straddles two
    // steps holds up the merge of most CTAs (fp32 NCHW 112x64x512x512 G8:
    // 104 pieces per unit 4.4 us a step, 152 pieces 2.9 us).  The backward
    // measured the other way (bf16 NCHW 32x64x512x512 G8: 104 pieces 4.05
    // us a step for 121 KB, 152 pieces 3.24 us for 83 KB).
    if (c.fwd && c.P > NC / 2 && NC % c.P != 0) per_step += 0.3 * t_io;
  } else {
    per_step = t_io + 0.4 + (c.P > 1 ? 0.3 : 0.0) + (wave_ahead(c.H, c.S) < 1 ? 1.0 : 0.0);
    if (c.P > 1 && NC % c.P != 0) per_step += t_io;
  }
  return (double)c.steps * per_step + t_io;
}

// Shared memory of a wave plan besides its slots: the records and CTA sums,
// the per-channel and per-group values, the mbarriers.
int64_t wave_red_floats(const Geom& g, int64_t P, int64_t Cb, int vec, int64_t H) {
  // the unit's records, then the CTA sums: per-thread partials, the shifts
  // and the per-(column, value) totals of NHWC pieces, or a block-sum scratch
  const int64_t nch = g.layout == kNHWC ? Cb : 1;
  // gathered, or the CTA's own for the pieces between stages A and B
  const int64_t recs = P > 1 ? P * nch : std::max<int64_t>(2, H) * nch;
  const int64_t red = 2 * recs + (g.layout == kNHWC ? 2 * vec * kWaveThreads + 3 * Cb : 64);
  return std::max<int64_t>(red, 2 * kWaveThreads);
}

size_t wave_fixed_bytes(const Geom& g, int64_t P, int64_t Cb, int vec, int64_t H) {
  const int64_t red = wave_red_floats(g, P, Cb, vec, H);
  const int64_t grp = g.layout == kNHWC ? Cb / g.Cg : 1;
  Geom t = g;
  t.Cb = Cb;
  const size_t cst = (size_t)wave_cst_floats(t) * 4 * kWaveMaxSlots;  // per-piece constants (H + 1 <= max slots)
  const size_t tab = (size_t)2 * P * 4;                                 // piece counts, planes
  return a128((size_t)red * 4) + a128(tab) + a128(cst) + a128((size_t)grp * 8) +
         a128(8 * (kWaveMaxSlots + 3 * kWaveMaxHold));
}

// Threads of one stage of a wave CTA: half of it with warp specialisation.
int64_t wave_stage_threads(bool ws) { return ws ? kWaveThreads / 2 : kWaveThreads; }

// Tensor-memory buffers for the reduced pieces of a cut (c.H, 0 when fewer
// than two fit) and the 16-byte vectors a thread keeps per tensor (c.T4, a
// multiple of 4).  Thread t of a stage keeps its vectors -- the ones it
// reduces in stage A and writes in stage B -- in lane 32*(warp % 4) + t % 32
// of every buffer; without warp specialisation warps w and w + 4 share a lane,
// at column offsets 0 and 4*nten*T4.
void wave_hold(const Geom& g, WaveCut& c, int nten, int vec) {
  c.H = c.T4 = 0;
#if defined(GN_WAVE_TMEM) && GN_WAVE_TMEM == 0
  return;
#endif
  const int64_t nthr = wave_stage_threads(kWaveWs);
  int64_t per;  // vectors per thread and tensor
  if (g.layout == kNCHW) {
    per = cdiv(c.R / vec, nthr);
  } else {
    const int64_t wv = c.Cb / vec;
    if (wv < 1 || wv > nthr) return;
    per = cdiv(c.R, nthr / wv);
  }
  const int64_t T4 = rup(std::max<int64_t>(per, 1), 4);
  const int64_t cols = 4 * nten * T4 * (nthr / 128);  // columns of one buffer
  const int64_t H = std::min<int64_t>(kWaveMaxHold, kWaveTmemCols / cols);
  if (H < 2) return;
  c.H = H;
  c.T4 = T4;
}

// Fills the wave-regime fields of g; false when the problem does not fit.
bool plan_wave(Geom& g, int op, int sm_count) {
  const int esz = dtype_size(g.dtype);
  const int vec = 16 / esz;
  const int nten = op == kBwd ? 2 : 1;
  if (g.vw != vec || g.dtype == kF64) return false;
  const size_t budget = kWaveCtasPerSm == 1 ? kSmemPerCta : kSmemPerSm / kWaveCtasPerSm - 1024;
  const int64_t NC = (int64_t)sm_count * kWaveCtasPerSm;
  WaveCut best;
  auto consider = [&](WaveCut c, int64_t units) {
    if (c.P < 1 || c.P > NC) return;
    // every thread of stage B polls at most 32 of a unit's records
    if (c.P * (g.layout == kNHWC ? c.Cb : 1) > 32 * wave_stage_threads(kWaveWs)) return;
    if (GN_WAVE_FORCE_CB > 0 && g.layout == kNHWC && c.Cb != GN_WAVE_FORCE_CB) return;
    if (GN_WAVE_FORCE_P > 0 && c.P != GN_WAVE_FORCE_P) return;
    c.fwd = op == kFwd;
    wave_hold(g, c, nten, vec);
    const size_t fixed = wave_fixed_bytes(g, c.P, c.Cb, vec, c.H);
    if (fixed + 128 + 2 * c.slot > budget) return;
    c.S = std::min<int64_t>(kWaveMaxSlots, (int64_t)((budget - fixed - 128) / c.slot));
    if (c.S < 2) return;
    c.steps = cdiv(units * c.P, NC);
    c.cost = wave_cost(c, NC);
    // the cheapest cut; at equal cost one whose stage A runs ahead, then
    // the one with more slots, then wider rows
    auto key = [&](const WaveCut& w) {
      return std::make_tuple(-w.cost, wave_ahead(w.H, w.S) >= 1, w.S >= kWaveMinSlots, w.Cb);
    };
    if (best.P == 0 || key(c) > key(best)) best = c;
  };
  if (g.layout == kNCHW) {
    if ((g.HW * esz) % 16 != 0) return false;
    for (int64_t m = 1; m * g.Cg <= NC; ++m) {
      WaveCut c;
      c.R = rup(cdiv(g.HW, m), vec);
      c.m = cdiv(g.HW, c.R);
      if (c.m != m) continue;
      c.P = g.Cg * m;
      c.slot = a128((size_t)(c.R * esz)) * nten;
      c.out = (size_t)(c.R * esz);
      consider(c, g.N * g.G);
    }
  } else {
    if (g.N * g.HW > 0x7fffffffLL) return false;  // TMA row coordinates are 32-bit
    const int64_t step = g.Cg / gcd64(g.Cg, vec) * vec;
    for (int64_t cb = step; cb <= g.C && cb <= kWaveMaxCb; cb += step) {
      if (g.C % cb != 0) continue;
      const int64_t rowb = cb * esz;
      for (int64_t P = 1; P <= NC && P <= g.HW; ++P) {
        WaveCut c;
        c.Cb = cb;
        int64_t R = cdiv(g.HW, P);
        if (R > 256) R = rup(R, 256);
        if (cdiv(g.HW, R) != P) continue;  // another P gives this cut
        c.P = P;
        c.R = R;
        c.box = R > 256 ? 256 : R;
        c.nb = R / c.box;
        c.slot = a128((size_t)(R * rowb)) * nten;
        c.out = (size_t)(R * rowb);
        consider(c, g.N * (g.C / cb));
      }
    }
  }
  if (best.P == 0) return false;
  Geom r = g;
  r.regime = kRegimeWave;
  r.tpb = kWaveThreads;  // (NCHW with warp specialisation: + the merge warp, below)
  r.wP = best.P;
  r.wR = best.R;
  r.wm = best.m;
  r.S = (int)best.S;
  r.wH = best.H;
  r.wT = best.T4;
  r.wB = best.H > 0 ? best.H + 1 : best.S;  // constants live from stage A to stage B
  r.wWs = best.H > 0 && kWaveWs ? 1 : 0;
  if (r.wWs && g.layout == kNCHW) r.tpb = kWaveThreads + 32;
  if (g.layout == kNHWC) {
    r.Cb = best.Cb;
    r.ncbu = g.C / best.Cb;
    r.units = g.N * r.ncbu;
    r.chunk = best.box;
    r.wnb = best.nb;
    r.wcols = r.ncbu;
    r.Tp = best.P;  // records per (n, c): one per piece
  } else {
    r.Cb = 0;
    r.units = g.N * g.G;
    r.chunk = 0;
    r.wnb = 1;
    r.wcols = g.G;
    r.Tp = best.m;  // records per (n, c): one per segment of the plane
  }
  r.ten_stride = (int64_t)(best.slot / nten);
  r.T = 0;
  r.l1 = 1;
  r.units_fin = 0;  // no counters: records are polled, the parameter step follows a grid barrier
  r.groups1 = 0;
  r.unit_groups = 0;
  size_t off = 0;
  r.off_ring = off;
  off += (size_t)r.S * best.slot;
  const int64_t red = wave_red_floats(g, r.wP, r.Cb, vec, r.wH);
  r.off_red = off;
  off += a128((size_t)red * 4);
  r.off_tot = off;  // piece counts (and NCHW planes) of a unit
  off += a128((size_t)2 * r.wP * 4);
  r.off_xch = off;  // per-piece constants
  off += a128((size_t)wave_cst_floats(r) * 4 * r.wB);
  r.off_grp = off;  // per-group results of a unit (NCHW merge warp: one per hold buffer)
  off += a128((size_t)std::max<int64_t>(g.layout == kNHWC ? r.Cb / g.Cg : 1, r.wH) * 8);
  // slots' mbarriers, then (warp specialisation) the hold buffers' full,
  // empty and merged ones
  r.off_bar = off;
  off += a128(8 * (size_t)(r.S + 3 * r.wH));
  r.smem = off + 128;  // slack for aligning the dynamic shared memory base
  // a CTA that allocates tensor memory takes more than half of an SM's shared
  // memory, so that no other CTA of the kernel can share its SM (and wait
  // there for the columns it holds)
  if (r.wH > 0) r.smem = std::max<size_t>(r.smem, kSmemPerSm / (kWaveCtasPerSm + 1) + 1024);
  if (r.smem > budget) return false;
  const int64_t nc = wave_ctas(r, op, r.smem, sm_count, kWaveCtasPerSm);
  if (nc < r.wP) return false;  // a unit's pieces must be co-resident
  if (r.units * r.wP > 0x7fffffffLL || g.N * g.C * r.Tp > 0x7fffffffLL) return false;  // 32-bit indices
  r.grid = std::min<int64_t>(nc, r.units * r.wP);
  g = r;
  return true;
}

// Co-resident CTAs of a flat-regime plan (one per SM at most); the SM count
// when no device is visible.
int64_t flat_ctas(const Geom& g, int op, int sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return sm_count;
  }
  const void* fn = flat_kernel_ptr(g, op == kBwd);
  int nb = 0;
  if (prepare_smem(fn, g.smem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, g.tpb, g.smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return (int64_t)std::min(nb, 1) * sm_count;
}

// Slot bytes per tensor of a flat-regime ring, and the chunks of a run that
// the forward keeps when the whole run fits in shared memory.
constexpr int64_t kFlatSlotBytes = 16 << 10;
constexpr int64_t kFlatWholeChunks = 8;

// Fills the flat-regime fields of g (gn_flat.cu); false when the problem does
// not fit the regime: dense, 16-byte aligned channels-last fp32 / fp16 / bf16
// data of at most kFlatThreads 16-byte columns per row, and per-segment
// tables that fit in shared memory.  One CTA per SM takes an equal run of the
// N*HW rows.  The forward keeps its whole run in shared memory when it fits
// (kFlatWholeChunks chunks); otherwise, and for the backward, the run streams
// through a ring of as many kFlatSlotBytes slots (per tensor) as fit.
bool plan_flat(Geom& g, int op, int sm_count) {
  const int esz = dtype_size(g.dtype);
  const int vec = 16 / esz;
  if (g.layout != kNHWC || g.dtype == kF64 || g.vw != vec) return false;
  const int64_t V = g.C / vec;
  if (V > kFlatThreads) return false;
  const int64_t R = g.N * g.HW;
  const int64_t NB = std::min<int64_t>(sm_count, R);
  if (NB < 1) return false;
  const bool bwd = op == kBwd;
  const int nten = bwd ? 2 : 1;
  Geom r = g;
  r.regime = kRegimeFlat;
  r.V = V;
  r.Wv = (int)V;
  r.ncb = 1;
  r.rpi = (int)std::max<int64_t>(1, kFlatThreads / V);
  r.tpb = r.rpi * r.Wv;
  int64_t segmax = 0, ngv = 0;
  for (int64_t b = 0; b < NB; ++b) {
    const int64_t a = b * R / NB, z = (b + 1) * R / NB;
    segmax = std::max(segmax, (z - 1) / g.HW - a / g.HW + 1);
  }
  for (int64_t j = 0; j < V; ++j)
    ngv = std::max(ngv, (j * vec + vec - 1) / g.Cg - j * vec / g.Cg + 1);
  r.fSeg = segmax;
  r.fNgv = (int)ngv;
  const int64_t rowb = g.C * esz;
  const int64_t rmax = cdiv(R, NB);
  const int64_t sgn = segmax * g.G;
  const size_t red = bwd ? (size_t)2 * vec * (r.tpb + 1) * 4 : (size_t)ngv * r.tpb * 8;
  const size_t tab = 4 * (bwd ? (size_t)(4 * sgn + 2 * g.C) : (size_t)(2 * sgn + g.G));
  const size_t runs = a128((size_t)(NB + 1) * 8) + a128((size_t)NB * 8);  // run table
  const size_t fixed = a128(red) + a128(tab) + runs + a128(kFlatBookBytes) + 128;
  if (fixed + 1024 > kSmemPerCta || tab > (32u << 10)) return false;
  const int64_t whole = cdiv(rmax, kFlatWholeChunks);
  const size_t whole_slot = a128((size_t)(whole * rowb));
  int64_t chunk, S;
  if (!bwd && fixed + (size_t)cdiv(rmax, whole) * whole_slot <= kSmemPerCta) {
    chunk = whole;
    S = cdiv(rmax, whole);
  } else {
    chunk = std::max<int64_t>(1, kFlatSlotBytes / rowb);
    const size_t slot = a128((size_t)(chunk * rowb)) * nten;
    S = std::min<int64_t>((int64_t)((kSmemPerCta - fixed) / slot), kFlatMaxSlots);
    S = std::min<int64_t>(S, cdiv(rmax, chunk));
    if (S < 2 && cdiv(rmax, chunk) > 1) return false;
  }
  if (chunk * rowb * nten >= (1 << 20)) return false;  // one mbarrier phase's byte count
  r.chunk = chunk;
  r.S = (int)S;
  r.ten_stride = (int64_t)a128((size_t)(chunk * rowb));
  size_t off = 0;
  r.off_ring = off;
  off += (size_t)S * (size_t)r.ten_stride * nten;
  r.off_red = off;
  off += a128(red);
  r.off_grp = off;
  off += a128(tab);
  r.off_tot = off;
  off += runs;
  r.off_bar = off;
  off += a128(kFlatBookBytes);
  r.smem = off + 128;  // slack for aligning the dynamic shared memory base
  if (r.smem > kSmemPerCta) return false;
  // records: one per (CTA, segment) and group (forward) or channel (backward),
  // in the workspace's partial-sum region
  const int64_t recs = NB * segmax * (bwd ? g.C : g.G);
  r.l1 = 1;
  r.Tp = cdiv(recs, g.N * g.C);
  r.T = r.Tp;
  r.groups1 = 0;
  r.units_fin = 0;
  r.unit_groups = 0;
  r.fin2 = 0;
  r.grid = NB;
  if (flat_ctas(r, op, sm_count) < NB) return false;
  g = r;
  return true;
}
}  // namespace

int64_t plan_max_clusters(const Geom& g, int op) {
  if (g.regime == kRegimeResident) return resident_clusters(g, op);
  const int64_t r = resident_ctas(g, op, 0);
  return r > 0 ? r : -1;
}

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

int64_t resident_ctas(const Geom& g, int op, int second) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  size_t smem = 0;
  const void* fn = g.layout == kNHWC ? nhwc_kernel(g, op == kBwd, second, &smem)
                                     : nchw_kernel(g, op == kBwd, second, &smem);
  using Key = std::tuple<int, const void*, int, size_t>;
  static std::mutex mu;
  static std::map<Key, int64_t> cache;
  const Key key{dev, fn, g.tpb, smem};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int64_t r = 0;
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, g.tpb, smem) == cudaSuccess)
    r = (int64_t)nb * device_sm_count();
  cudaGetLastError();
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = r;
  return r;
}

namespace {
#ifndef GN_FIN2_BYTES
#define GN_FIN2_BYTES (4 * 1024)
#endif
// Records one second-kernel CTA may read to finalise its groups itself, and
// the most shared memory that finalisation may take (the default dynamic
// limit, so the second kernels need no opt-in and keep two CTAs per SM).
// Every CTA of a sample repeats that work, so it pays only while the records
// are few: measured on GB300, NCHW planes (Cg records per CTA) gain, while
// channels-last rows (4608 records per CTA at 512 channels) lost more in the
// second kernel than the chain costs the first.
constexpr int64_t kFin2Bytes = GN_FIN2_BYTES;
constexpr int64_t kFin2SmemBytes = 48 * 1024;

// Most channels, extended to whole groups, that one second-kernel CTA covers:
// an NCHW plane (mode 0) or block of RB planes (mode 1).
int64_t fin2_channels(const Geom& g) {
  if (g.mode == 0) return g.Cg;
  const int64_t blk = g.RB, nblk = g.items_per_n;
  int64_t best = 0;
  for (int64_t b = 0; b < nblk; ++b) {
    const int64_t lo = b * blk, hi = std::min(g.C, lo + blk);
    if (lo >= hi) continue;
    best = std::max(best, cdiv(hi, g.Cg) * g.Cg - lo / g.Cg * g.Cg);
  }
  return best;
}

// Moves the finalisation of an NCHW plan into the second kernel when each of
// its CTAs reads at most kFin2Bytes of records: with every item record (no
// chain at all in the first kernel) if they are few enough, else with
// level-1 records (the first kernel keeps only the level-1 merge).
// Otherwise the plan is left as it is.  Channels-last CTAs cover whole rows
// of C channels, far more records than the budget at the shapes here, so
// that layout keeps the chain (its kernels carry no second-kernel
// finalisation at all).
void plan_fin2(Geom& g) {
  if (g.layout != kNCHW) return;
  const int64_t mc = fin2_channels(g);
  for (int l1 : {1, kGroup1}) {
    if (l1 > 1 && g.T < 2 * kGroup1) break;
    const int64_t Tp = cdiv(g.T, l1);
    if (mc * Tp * (int64_t)sizeof(float) * 2 > kFin2Bytes) continue;
    Geom f = g;
    f.fin2 = 1;
    f.maxch2 = mc;
    f.nsl2 = (int)clamp64(g.tpb / mc, 1, Tp);
    f.Tp = Tp;
    if (fin2_smem_floats(f) * (int64_t)sizeof(float) > kFin2SmemBytes) continue;
    g.fin2 = 1;
    g.maxch2 = mc;
    g.nsl2 = f.nsl2;
    g.l1 = l1;
    g.Tp = Tp;
    g.groups1 = l1 > 1 ? g.N * g.C * Tp : 0;
    if (g.mode == 0) {
      g.cstride = Tp;
      g.arrivals_per_n = g.C * Tp;
    }
    return;
  }
}

Geom plan_geom(int op, int64_t N, int64_t C, int64_t HW, int64_t G, int layout, int dtype,
               bool aligned, bool dense) {
  const int sm_count = device_sm_count();
  Geom g{};
  g.N = N;
  g.C = C;
  g.HW = HW;
  g.G = G;
  g.Cg = C / G;
  g.layout = layout;
  g.dtype = dtype;
  const int esz = dtype_size(dtype);
  const int vec = 16 / esz;
  // One item per CTA of the first kernel, and as many items as fit on the
  // device at once (one wave) unless the problem needs more.
  int64_t item_len = 0;  // rows (NHWC) or elements (NCHW mode 0) per item
  if (layout == kNHWC) {
    g.vw = (aligned && C % vec == 0) ? vec : 1;
    g.V = C / g.vw;
    g.ncb = (int)cdiv(g.V, 256);
    g.Wv = (int)cdiv(g.V, g.ncb);
    g.rpi = 512 / g.Wv;
    if (g.rpi < 1) g.rpi = 1;
    g.tpb = g.Wv * g.rpi;
    // One wave: as many row blocks per (n, cb) as CTAs fit on the device.
    const int64_t units = N * g.ncb;
    const int64_t T = clamp64(resident_or(g, op, 0, sm_count) / units, 1, cdiv(HW, g.rpi));
    g.rb = rup(cdiv(HW, T), g.rpi);
    g.T = T;  // trailing items may be empty when rb*T > HW
    g.l1 = T >= 2 * kGroup1 ? kGroup1 : 1;
    g.Tp = cdiv(T, g.l1);
    g.groups1 = g.l1 > 1 ? units * g.Tp : 0;
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
      const int64_t pmax = cdiv(HW, (int64_t)g.tpb * g.vw);
      const int64_t P = clamp64(resident_or(g, op, 0, sm_count) / (N * C), 1, pmax);
      g.L = rup(cdiv(HW, P), g.vw);
      g.T = P;  // trailing chunks may be empty when L*P > HW
      g.l1 = P >= 2 * kGroup1 ? kGroup1 : 1;
      g.Tp = cdiv(P, g.l1);
      g.groups1 = g.l1 > 1 ? N * C * g.Tp : 0;
      g.cstride = g.Tp;
      g.tstride = 1;
      g.arrivals_per_n = C * g.Tp;
      g.items_per_n = C * P;
      item_len = g.L;
    } else {
      g.mode = 1;
      g.tpb = 256;
      g.RB = clamp64(cdiv(N * C, resident_or(g, op, 0, sm_count)), 8, C);
      g.T = 1;
      g.l1 = 1;
      g.Tp = 1;
      g.groups1 = 0;
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
  g.units_fin = N;  // the two-kernel path finalises per sample
  g.unit_groups = 0;
  g.regime = kRegimeGeneric;
  // strided views run on the two-kernel path only
  const int ov = dense ? g_regime_override.load() : kRegimeGeneric;
  if (ov == kRegimeResident) {
    plan_resident(g, op, false);  // wherever the problem fits the regime
  } else if (ov == kRegimePipelined) {
    plan_pipelined(g, op, sm_count);
  } else if (ov == kRegimeWave) {
    plan_wave(g, op, sm_count);
  } else if (ov == kRegimeFlat) {
    plan_flat(g, op, sm_count);
  } else if (ov == kRegimeAuto && wave_preferred(g, op) && plan_wave(g, op, sm_count)) {
    // taken
  } else if (ov == kRegimeAuto && flat_preferred(g, op) && plan_flat(g, op, sm_count)) {
    // taken
  } else if (ov == kRegimeAuto && resident_preferred(g, op)) {
    // measured on GB300: the pipelined kernel moves the minimal traffic but is
    // slower than these families on every workload here (its steps are
    // latency-bound), so it runs only when asked for
    plan_resident(g, op, true);
  }
  if (g.regime == kRegimeGeneric) plan_fin2(g);
  const int64_t pipe = g.regime == kRegimePipelined ? 2 * g.units_fin + 3 : 0;
  g.counters = g.units_fin + 1 + g.groups1 + pipe;  // resident: units_fin = N, groups1 = 0
  return g;
}

// Plans are cached per (device, regime override, op, problem, alignment):
// building one queries occupancy, and every call (and every workspace layout,
// which looks at the plans of both ops) needs them.
using PlanKey = std::tuple<int, int, int, int64_t, int64_t, int64_t, int64_t, int, int, int, int>;
std::mutex g_plan_mu;
std::map<PlanKey, Geom> g_plan_cache;
constexpr size_t kPlanCacheMax = 4096;
}  // namespace

Geom make_geom(int op, int64_t N, int64_t C, int64_t HW, int64_t G, int layout, int dtype,
               bool aligned, bool dense) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = -1;
  }
  const PlanKey key{dev, g_regime_override.load(), op, N, C, HW, G, layout, dtype, aligned ? 1 : 0,
                    dense ? 1 : 0};
  {
    std::lock_guard<std::mutex> lock(g_plan_mu);
    auto it = g_plan_cache.find(key);
    if (it != g_plan_cache.end()) return it->second;
  }
  const Geom g = plan_geom(op, N, C, HW, G, layout, dtype, aligned, dense);
  std::lock_guard<std::mutex> lock(g_plan_mu);
  if (g_plan_cache.size() >= kPlanCacheMax) g_plan_cache.clear();
  g_plan_cache.emplace(key, g);
  return g;
}

int64_t problem_counters(const Geom& g) {
  int64_t c = 0;
  for (int op = 0; op < 2; ++op)
    for (int a = 0; a < 2; ++a)
      for (int d = 0; d < 2; ++d) {
        const Geom o = make_geom(op, g.N, g.C, g.HW, g.G, g.layout, g.dtype, a != 0, d != 0);
        if (o.counters > c) c = o.counters;
      }
  return c;
}

WsLayout ws_layout(int op, const Geom& g) {
  WsLayout w{};
  // the error word first, then the counters; every call clears [0, clear) on
  // its stream before its kernels run.  The counter region is the same for
  // both ops and both alignments of a problem, so that a forward and its
  // backward lay it out alike.
  (void)op;
  w.err = 0;
  w.tickets = 16;
  w.clear = w.tickets + sizeof(unsigned) * (size_t)problem_counters(g);
  size_t off = align256(w.clear);
  w.part0 = off;
  if (g.l1 > 1) off = align256(off + 2 * sizeof(float) * (size_t)(g.N * g.C * g.T));
  w.part = off;
  off = align256(off + 2 * sizeof(float) * (size_t)(g.N * g.C * g.Tp));
  w.chst = off;
  off = align256(off + 2 * sizeof(float) * (size_t)(g.N * g.C));
  w.coef = off;
  if (op == kBwd) off = align256(off + 2 * sizeof(float) * (size_t)(g.N * g.G));
  w.total = off;
  return w;
}

}  // namespace gn
