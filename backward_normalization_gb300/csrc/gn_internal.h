// gn_internal.h -- plan (work decomposition) and kernel parameter block shared
// by the C-ABI layer and the kernels.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gn {

enum Layout { kNCHW = 0, kNHWC = 1 };
enum DType { kF32 = 0, kF16 = 1, kBF16 = 2, kF64 = 3 };

// Bytes per stored element.  Every dtype is computed in fp32; f64 is a
// storage type (16-byte vectors of two doubles, converted on load and store).
__host__ __device__ inline int dtype_size(int dtype) {
  return dtype == kF64 ? 8 : dtype == kF32 ? 4 : 2;
}
enum Op { kFwd = 0, kBwd = 1 };

// Regimes (which kernel family runs a call).
enum Regime {
  kRegimeAuto = -1,
  kRegimeGeneric = 0,   // stats/reduce kernel + apply/dx kernel, any shape
  kRegimeResident = 1,  // one kernel: a cluster holds a unit in shared memory
  kRegimePipelined = 2, // one persistent kernel: pass-1 and pass-2 tasks of
                        // units in flight, the second pass reading from L2
  kRegimeWave = 3,      // one persistent kernel: every piece of a unit stays on
                        // chip (shared or tensor memory) until the unit's
                        // statistics are known
  kRegimeFlat = 4,      // one cooperative kernel (channels-last): every SM holds an
                        // equal run of rows, one grid barrier between the passes
};

// How one call is cut into "items" for the two-kernel path.  Both kernels
// run one CTA per item (one wave when the problem allows).  Each item's
// partial sums go to a fixed slot, groups of l1 consecutive items are merged
// by the group's last CTA, and the last group of a sample finalises it --
// every sum in a fixed order, whichever CTA runs it.  The second kernel is
// elementwise and walks the items in reverse order (the data the first kernel
// read last is still in L2).
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
  int l1;        // items per level-1 group (1: no level-1 merge)
  int64_t Tp;    // level-1 records per (n, c) = ceil(T / l1)
  int64_t groups1;           // level-1 groups in the call
  int64_t cstride, tstride;  // level-1 record index = n*C*Tp + c*cstride + t1*tstride
  int64_t arrivals_per_n;    // records that complete a finalisation unit
  int64_t units_fin;         // finalisation units: N (a unit is a sample) or N*G
  int unit_groups;           // 1: a unit is one (sample, group) (pipelined NCHW)
  int64_t items_per_n;       // NCHW mode 1: items per sample
  int64_t items;
  int64_t keep_from;  // item-relative row/element index from which the first kernel
                      // loads with the L2 evict_last policy (the part read again first)
  // Finalisation in the second kernel (NCHW two-kernel path, when the
  // records are few): the first kernel ends with its item records (and at
  // most the level-1 merge); every CTA of the second kernel sums the Tp
  // records of the channels of its groups itself, in one fixed order, and
  // the parameter gradients are spread over its CTAs by channel.  Otherwise
  // the last arrival of a sample finalises it in the first kernel.
  int fin2;
  int nsl2;        // fixed slices per channel in those sums
  int64_t maxch2;  // most channels (whole groups) that one second-kernel CTA covers
  // pipelined regime: units_fin units of `pieces` pass-1 and `pieces` pass-2
  // tasks each (a piece is item u*T + q: NHWC, or plane q/T of the unit's
  // group, segment q%T: NCHW); pass-2 tasks trail pass-1 tasks by `lag` units
  int64_t pieces, lag;
  int64_t grid;        // persistent CTAs (all co-resident)
  int64_t counters;    // uint32 counter slots this plan uses at the start of the workspace
  int dy_in_ring;      // pipelined backward: each ring slot holds a dy chunk after the x chunk
  // pipelined: S ring slots of ten_stride bytes per tensor; a chunk is `chunk`
  // elements (NCHW) or rows (NHWC); slot headers at off_tot, mbarriers at
  // off_bar, reduction scratch at off_red; smem bytes in all
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
  // wave regime (gn_wave.cu): units (`units`) of wP pieces; a piece is wR
  // elements of one channel plane (NCHW; wm pieces per plane) or wR rows of
  // Cb channels (NHWC, read as wnb TMA boxes of `chunk` rows); `grid` CTAs
  // hold S slots of ten_stride bytes per tensor; wcols parameter columns
  // (channel blocks of a sample) finish dgamma/dbeta.  wH > 0: a reduced
  // piece waits for its unit's statistics in one of wH tensor-memory
  // buffers (wT 16-byte vectors per thread and tensor), which frees its slot
  // for the next copy at once; wH = 0: it waits in its slot.  wB buffers of
  // per-piece constants.  wWs = 1: stage A and stage B run on separate halves
  // of the CTA (warp specialisation), handing pieces over through mbarriers.
  int64_t wP, wR, wm, wnb, wcols, wH, wT, wB, wWs;
  // flat regime (gn_flat.cu): `grid` CTAs take equal runs of the N*HW rows,
  // read as chunks of `chunk` rows into S slots of ten_stride bytes per
  // tensor.  fSeg: most samples one CTA's run touches (its segments);
  // fNgv: most groups one 16-byte column spans.
  int64_t fSeg;
  int fNgv;
};

// Bytes reserved per ring-slot header of the pipelined kernel (the header
// struct of gn_tasks.cuh is checked against it at compile time).
constexpr size_t kSlotHdrBytes = 112;

// Shared memory of a fin2 second kernel's finalisation (NCHW), in floats
// from the 16-byte aligned base: the staged records (one run, channel-major,
// copied from an even record index, so with up to one extra record at each
// end), the slice sums, the per-channel stage, the per-group values and
// per-warp sums of the parameter step.
struct Fin2Smem {
  int64_t recs, part, stage, grp, wpart, total;
};
__host__ __device__ inline Fin2Smem fin2_smem(const Geom& g) {
  Fin2Smem s{};
  if (!g.fin2) return s;
  const int64_t run = (g.maxch2 * g.Tp + 3) & ~int64_t(1);
  const int64_t pairs = (int64_t)g.nsl2 * g.maxch2;
  s.recs = 0;
  s.part = s.recs + 2 * run;
  s.stage = s.part + 2 * (pairs > 64 ? pairs : 64);
  s.grp = s.stage + 2 * g.maxch2;
  s.wpart = s.grp + 2 * (g.maxch2 / g.Cg + 1);
  s.total = s.wpart + 64;
  return s;
}
__host__ __device__ inline int64_t fin2_smem_floats(const Geom& g) { return fin2_smem(g).total; }

// Workspace layout (byte offsets; the scratch regions are 256-byte aligned).
struct WsLayout {
  size_t err;      // uint32 error word at offset 0 (a bounded wait ran out)
  size_t tickets;  // uint32 counters at offset 16: one per finalisation unit, 1 global, one
                   // per level-1 group; pipelined: then (8-byte aligned) a 64-bit ready
                   // record per unit and the count of CTAs done.  Sized by
                   // problem_counters(), whichever op and alignment the call has.
  size_t clear;    // bytes [0, clear) that every call zero-fills before its kernels
  size_t part0;    // N*C*T float2 item partial sums (when l1 > 1)
  size_t part;     // N*C*Tp float2 level-1 partial sums
  size_t chst;     // N*C float2 per-channel results of the finalisation
  size_t coef;     // N*G float2 dx coefficients (backward only)
  size_t total;
};

struct KParams {
  CUtensorMap tmx;   // resident / wave NHWC: 2-D [N*HW, C] views of x and dy for TMA tiles
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
  unsigned* tickets;  // [0, units_fin) per unit, [units_fin] global
  unsigned* cnt1;     // per level-1 group
  unsigned* ready;    // pipelined: per unit a 64-bit ready record (8-byte aligned)
  unsigned* queue;    // pipelined: [0] CTAs done
  // Element strides of the views (two-kernel path; the other regimes take
  // dense tensors only): per sample (s_n) and per channel plane (NCHW) or
  // spatial row (NHWC) (s_r).  Dense NCHW: C*HW, HW; dense NHWC: HW*C, C.
  int64_t xs_n, xs_r;   // x
  int64_t ds_n, ds_r;   // dy
  int64_t os_n, os_r;   // y or dx
  unsigned* err;
  int clear_words;    // uint32 words at the start of the workspace cleared before the kernels
  int stall_unit;     // fault injection: a unit whose arrival is withheld (-1: none)
  float2* part0;      // item partials (== part when l1 == 1)
  float2* part;
  float2* chst;
  float2* coef;
  float* kst;         // forward with fin2: the per-(n, c) shifts x(n, c, hw = 0), saved by
                      // the first kernel (the second may overwrite x in place); aliases chst
};

// gn_api.cu: records e as this thread's last CUDA error (gn_last_cuda_error),
// clears the runtime's sticky launch error and returns GN_ERR_CUDA.
int record_cuda_error(cudaError_t e);

// plan.cpp
int device_sm_count();
// Co-resident clusters of the plan's first (or only) kernel (-1: no device).
int64_t plan_max_clusters(const Geom& g, int op);
// Test hook: force a regime (kRegimeAuto = automatic choice).
void set_regime_override(int regime);
// CTAs of the op's first (second = 0) or second (second = 1) two-kernel-path
// kernel that fit on the current device at once (0: no device visible).
int64_t resident_ctas(const Geom& g, int op, int second);
// `dense`: every view is densely packed in its layout; strided views run on
// the two-kernel path only.
Geom make_geom(int op, int64_t N, int64_t C, int64_t HW, int64_t G, int layout,
               int dtype, bool aligned, bool dense = true);
WsLayout ws_layout(int op, const Geom& g);
// Counter slots of a problem: the most that any plan of it (either op, either
// alignment, dense or strided views) uses; the workspace layout reserves this
// many for every call.
int64_t problem_counters(const Geom& g);

// Events recorded around/between the kernels of a call (benchmark hook; the
// launchers record the non-null ones on the call's stream).
struct TimingEvents {
  cudaEvent_t begin, mid, end;
};
const TimingEvents& timing_events();


// kernels (gn_nhwc.cu / gn_nchw.cu): enqueue the two kernels of an op.
cudaError_t launch_nhwc(const KParams& p, cudaStream_t s, bool bwd);
cudaError_t launch_nchw(const KParams& p, cudaStream_t s, bool bwd);
// The pipelined regime's kernel (NCHW; one launch, cooperative).
cudaError_t launch_nchw_pipelined(const KParams& p, cudaStream_t s, bool bwd);
const void* nchw_pipelined_kernel(const Geom& g, bool bwd, size_t* smem);
int64_t nchw_pipelined_scratch_floats(const Geom& g);
// The first (second = 0) or second (second = 1) kernel's function and its
// dynamic shared memory for a plan.
const void* nhwc_kernel(const Geom& g, bool bwd, int second, size_t* smem);
const void* nchw_kernel(const Geom& g, bool bwd, int second, size_t* smem);
// gn_wave.cu
const void* wave_kernel_ptr(const Geom& g, bool bwd);
cudaError_t launch_wave(const KParams& p, cudaStream_t s, bool bwd);
// Floats of one wave-regime slot's constants (prefetched with the piece):
// NHWC, gamma and beta (forward) or gamma, then mean and rstd of its groups
// (backward) of the unit's Cb channels; NCHW, gamma of the group's Cg
// channels, then beta of the piece's channel (forward) or the unit's mean and
// rstd (backward).  Rounded up to 4 floats.
__host__ __device__ inline int wave_cst_floats(const Geom& g) {
  const int64_t n = g.layout == kNHWC ? 2 * g.Cb + 2 * (g.Cb / g.Cg) : g.Cg + 2;
  return (int)((n + 3) & ~int64_t(3));
}

// Threads of a wave-regime CTA, and such CTAs that share an SM (several
// independent CTAs per SM overlap one another's barrier-bound phases).
#ifndef GN_WAVE_THREADS
#define GN_WAVE_THREADS 256
#endif
#ifndef GN_WAVE_CTAS_PER_SM
#define GN_WAVE_CTAS_PER_SM 1
#endif
constexpr int kWaveThreads = GN_WAVE_THREADS;
constexpr int kWaveCtasPerSm = GN_WAVE_CTAS_PER_SM;
// Wave plans that hold pieces in tensor memory run stage A and stage B on
// separate halves of the CTA (1) or both on the whole CTA in turn (0).
#ifndef GN_WAVE_WS
#define GN_WAVE_WS 1
#endif
constexpr bool kWaveWs = GN_WAVE_WS != 0;
// Tensor-memory columns one wave CTA allocates (its share of the SM's 512).
constexpr int kWaveTmemCols = 512 / GN_WAVE_CTAS_PER_SM;
static_assert(kWaveTmemCols >= 32 && (kWaveTmemCols & (kWaveTmemCols - 1)) == 0,
              "a tensor-memory allocation is a power of two of at least 32 columns");
static_assert(kWaveThreads % 128 == 0, "whole warp quarters share the tensor-memory lanes");
// gn_flat.cu
const void* flat_kernel_ptr(const Geom& g, bool bwd);
cudaError_t launch_flat(const KParams& p, cudaStream_t s, bool bwd);
// Most ring slots of a flat-regime CTA, and the bytes its shared-memory
// bookkeeping (mbarriers, fill counts, flags) takes after the tables.
constexpr int kFlatMaxSlots = 32;
constexpr size_t kFlatBookBytes = 8 * kFlatMaxSlots + 4 * 2 * kFlatMaxSlots + 16;
// Threads of a flat-regime CTA at most (a whole number of row lanes of C/vw columns).
constexpr int kFlatThreads = 512;
// gn_resident.cu
// [N*HW, C] view of an NHWC tensor for TMA, boxes of [g.chunk rows, g.Cb channels].
cudaError_t encode_nhwc_map(CUtensorMap* map, const void* base, const Geom& g);
const void* resident_kernel_ptr(const Geom& g, bool bwd);
cudaError_t launch_resident(const KParams& p, cudaStream_t s, bool bwd);
// Threads of a resident CTA: the consumer warps plus one producer warp.
inline int resident_threads(const Geom& g) { return (g.tpb + 31) / 32 * 32 + 32; }
// Raises a kernel's dynamic shared memory limit to at least `smem` bytes on
// the current device; remembered per (device, kernel), so that launches after
// the first make no attribute call.
cudaError_t prepare_smem(const void* kernel, size_t smem);
// Sets the kernel attributes a resident launch needs (large shared memory,
// 16-CTA clusters); idempotent.
cudaError_t prepare_resident_kernel(const void* kernel, const Geom& g);

}  // namespace gn
