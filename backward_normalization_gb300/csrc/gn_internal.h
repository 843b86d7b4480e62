// gn_internal.h -- plan (work decomposition) and kernel parameter block shared
// by the C-ABI layer and the kernels.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gn {

enum Layout { kNCHW = 0, kNHWC = 1 };
enum DType { kF32 = 0, kF16 = 1, kBF16 = 2 };
enum Op { kFwd = 0, kBwd = 1 };

// Regimes (which kernel family runs a call).
enum Regime {
  kRegimeAuto = -1,
  kRegimeGeneric = 0,   // stats/reduce kernel + apply/dx kernel, any shape
  kRegimeResident = 1,  // one kernel: a cluster holds a unit in shared memory
};

// How one call is cut into "items" (one CTA each).  Both kernels of an op use
// the same items; the second kernel walks them in reverse so that the data the
// first kernel read last is still in L2 when it is needed again.
struct Geom {
  int64_t N, C, HW, G, Cg;
  int layout, dtype;
  int vw;    // elements per access: the 16-byte vector width, or 1 (scalar path)
  int tpb;   // threads per CTA
  // NHWC: a row is one (n, hw) position holding C channels; a thread owns a
  // fixed column of vw channels and walks rows.
  int64_t V;     // columns per row (C / vw)
  int Wv;        // columns per column block
  int ncb;       // column blocks per row
  int rpi;       // rows handled concurrently by one CTA (row lanes)
  int64_t rb;    // rows per item
  // NCHW: a row is one (n, c) channel plane of HW elements.
  int mode;      // 0: item = (row, chunk) walked by the whole CTA; 1: item = block of rows, one warp per row
  int64_t L;     // mode 0: chunk length (multiple of vw)
  int64_t RB;    // mode 1: rows per item
  // common
  int64_t T;     // items per (n, column block) (NHWC) or per row (NCHW)
  int cl;        // CTAs per thread-block cluster of the first kernel (1 or 8);
                 // a cluster = cl consecutive items that merge their partials through DSMEM
  int64_t Tp;    // partial records per (n, c) = T / cl
  int64_t cstride, tstride;  // partial index = n*C*Tp + c*cstride + t'*tstride
  int64_t arrivals_per_n;    // cluster-level partials that complete sample n
  int64_t items_per_n;       // NCHW mode 1: items per sample
  int64_t items;
  int64_t keep_from;  // item-relative row/element index from which the first kernel
                      // loads with the L2 evict_last policy (the part read again first)
  // resident regime (gn_resident.cu)
  int regime;
  int K;               // CTAs per unit (cluster size)
  int64_t m;           // NCHW: pieces per channel plane (K = Cg*m)
  int64_t units;       // clusters: N*G (NCHW) or N (NHWC)
  int64_t slice;       // NCHW: elements per piece; NHWC: rows per CTA
  int64_t chunk;       // NCHW: elements per chunk; NHWC: rows per chunk (TMA box rows)
  int64_t Cb;          // NHWC: channels per unit (whole groups); a unit is (n, channel block)
  int64_t ncbu;        // NHWC: channel blocks per sample (C / Cb)
  int64_t chunk_bytes; // bytes of one tensor's chunk (the TMA transfer)
  int64_t ten_stride;  // bytes between a slot's x and dy parts (chunk_bytes rounded up to 128)
  int nres, S;         // resident chunk slots, ring slots
  size_t smem;         // dynamic shared memory bytes
  size_t off_ring, off_red, off_xch, off_tot, off_grp, off_bar;
};

// Workspace layout (byte offsets, each 256-byte aligned).
struct WsLayout {
  size_t tickets;  // (N + 1) uint32 arrival counters: one per sample, one global
  size_t err;      // uint32 error word (a bounded wait ran out)
  size_t part;     // N*C*Tp float2 partial sums
  size_t chst;     // N*C float2 per-channel results of the finalisation
  size_t coef;     // N*G float2 dx coefficients (backward only)
  size_t total;
};

struct KParams {
  CUtensorMap tmx;   // resident NHWC: 2-D [N*HW, C] views of x and dy for TMA tiles
  CUtensorMap tmdy;
  Geom g;
  const void* x;
  const void* dy;
  void* out;  // y (forward) or dx (backward)
  const float* gamma;
  const float* beta;
  float* mean;   // forward: written; backward: read
  float* rstd;
  float* dgamma;
  float* dbeta;
  float eps;
  unsigned* tickets;
  unsigned* err;
  float2* part;
  float2* chst;
  float2* coef;
};

// plan.cpp
int device_sm_count();
// Co-resident clusters of the plan's first (or only) kernel (-1: no device).
int64_t plan_max_clusters(const Geom& g, int op);
// Test hook: force a regime (kRegimeAuto = automatic choice).
void set_regime_override(int regime);
// CTAs of the op's first kernel that fit on the current device at once when
// launched with g.tpb threads in clusters of `cl` CTAs (0: no device).
int64_t resident_first_ctas(const Geom& g, int op, int cl);
Geom make_geom(int op, int64_t N, int64_t C, int64_t HW, int64_t G, int layout,
               int dtype, bool aligned);
WsLayout ws_layout(int op, const Geom& g);

// Events recorded around/between the kernels of a call (benchmark hook; the
// launchers record the non-null ones on the call's stream).
struct TimingEvents {
  cudaEvent_t begin, mid, end;
};
const TimingEvents& timing_events();

// Launches the first kernel of an op (one CTA per item, clusters of g.cl CTAs).
cudaError_t launch_first(const void* kernel, const KParams& p, size_t smem, cudaStream_t s);

// kernels (gn_nhwc.cu / gn_nchw.cu): enqueue the two kernels of an op.
cudaError_t launch_nhwc(const KParams& p, cudaStream_t s, bool bwd);
cudaError_t launch_nchw(const KParams& p, cudaStream_t s, bool bwd);
// The first kernel's function and dynamic shared memory for a plan.
const void* nhwc_first_kernel(const Geom& g, bool bwd, size_t* smem);
const void* nchw_first_kernel(const Geom& g, bool bwd, size_t* smem);
// gn_resident.cu
const void* resident_kernel_ptr(const Geom& g, bool bwd);
cudaError_t launch_resident(const KParams& p, cudaStream_t s, bool bwd);
// Threads of a resident CTA: the consumer warps plus one producer warp.
inline int resident_threads(const Geom& g) { return (g.tpb + 31) / 32 * 32 + 32; }
// Sets the kernel attributes a resident launch needs (large shared memory,
// 16-CTA clusters); idempotent.
cudaError_t prepare_resident_kernel(const void* kernel, const Geom& g);

}  // namespace gn
