// gn_api.cu -- the C ABI declared in include/gn.h: argument validation
// (before anything is enqueued), planning and kernel dispatch.
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "../../include/gn.h"
#include "gn_device.cuh"

namespace {

thread_local int t_last_cuda_error = 0;
thread_local gn::TimingEvents t_events = {nullptr, nullptr, nullptr};

// Fault injection (test hook).  GN_FAULT_LAUNCH makes every call fail with
// GN_ERR_CUDA after validation and before anything is enqueued, as a failed
// launch would; GN_FAULT_STALL makes the next wave-regime call withhold one
// arrival (the next flat-regime call one chunk copy), so that the bounded
// waits on it run out.  The environment
// variable GN_FAULT_INJECT=launch sets GN_FAULT_LAUNCH at the first call.
std::atomic<int> g_fault{-1};  // -1: not read from the environment yet

int fault_mode() {
  int f = g_fault.load(std::memory_order_relaxed);
  if (f >= 0) return f;
  const char* e = std::getenv("GN_FAULT_INJECT");
  f = (e && std::strcmp(e, "launch") == 0) ? GN_FAULT_LAUNCH : GN_FAULT_NONE;
  int expect = -1;
  g_fault.compare_exchange_strong(expect, f);
  return g_fault.load(std::memory_order_relaxed);
}

// GN_FAULT_STALL applies to one call: the unit whose arrival that call
// withholds (unit 0), then the mode returns to GN_FAULT_NONE.
int take_stall() {
  int f = GN_FAULT_STALL;
  return g_fault.compare_exchange_strong(f, GN_FAULT_NONE) ? 0 : -1;
}

int elem_size(int dtype) { return gn::dtype_size(dtype); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [a, a+na) and [b, b+nb) share a byte.
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

int check_problem(int64_t N, int64_t C, int64_t HW, int64_t G, int layout, int dtype) {
  if (layout != GN_LAYOUT_NCHW && layout != GN_LAYOUT_NHWC) return GN_ERR_UNSUPPORTED;
  if (dtype != GN_DTYPE_F32 && dtype != GN_DTYPE_F16 && dtype != GN_DTYPE_BF16 &&
      dtype != GN_DTYPE_F64)
    return GN_ERR_UNSUPPORTED;
  if (N < 0 || C < 0 || HW < 0 || G <= 0) return GN_ERR_INVALID;
  if (C % G != 0) return GN_ERR_INVALID;
  // element offsets and per-call counts must stay far from int64 overflow
  if (N > 0 && C > 0 && HW > 0) {
    const double e = (double)N * (double)C * (double)HW;
    if (e > 4.0e18) return GN_ERR_UNSUPPORTED;
  }
  return GN_OK;
}

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = (int)e;
  cudaGetLastError();  // a failed launch must not poison the caller's next CUDA call
  return GN_ERR_CUDA;
}

// Plan + workspace check shared by both ops.
int prepare(int op, int64_t N, int64_t C, int64_t HW, int64_t G, int layout, int dtype,
            bool aligned, bool dense, void* workspace, size_t workspace_bytes, gn::KParams* p) {
  std::memset(p, 0, sizeof(*p));
  p->stall_unit = -1;
  p->g = gn::make_geom(op, N, C, HW, G, layout, dtype, aligned, dense);
  if (p->g.regime == gn::kRegimeGeneric && (p->g.items <= 0 || p->g.items > 0x7fffffffLL))
    return GN_ERR_UNSUPPORTED;
  const gn::WsLayout w = gn::ws_layout(op, p->g);
  if (!workspace || workspace_bytes < w.total || !aligned16(workspace)) return GN_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  p->tickets = reinterpret_cast<unsigned*>(ws + w.tickets);
  p->err = reinterpret_cast<unsigned*>(ws + w.err);
  p->clear_words = (int)(w.clear / sizeof(unsigned));
  // counters: one per unit, the global one, one per level-1 group, then (pipelined)
  // a 64-bit ready record per unit and the count of CTAs done
  const int64_t U = p->g.units_fin;
  p->cnt1 = p->tickets + U + 1;
  if (p->g.regime == gn::kRegimePipelined) {
    const int64_t r = U + 1 + p->g.groups1;
    p->ready = p->tickets + (r + 1) / 2 * 2;  // 8-byte aligned records
    p->queue = p->ready + 2 * U;
  }
  p->part = reinterpret_cast<float2*>(ws + w.part);
  p->part0 = p->g.l1 > 1 ? reinterpret_cast<float2*>(ws + w.part0) : p->part;
  p->chst = reinterpret_cast<float2*>(ws + w.chst);
  p->kst = reinterpret_cast<float*>(ws + w.chst);
  p->coef = reinterpret_cast<float2*>(ws + w.coef);
  return GN_OK;
}

// Zero-fills the workspace's error word and counters ([0, clear_words)) on
// the call's stream.  Launched with programmatic stream serialisation: it may
// be scheduled while the previous work on the stream runs, waits for that
// work to complete before it writes (the previous call may still use the same
// workspace), and the call's first kernel waits for it in turn.
__global__ void __launch_bounds__(256) ws_clear(unsigned* ws, int words) {
  gn::grid_launch_dependents();
  gn::grid_dependency_wait();
  for (int i = threadIdx.x; i < words; i += blockDim.x) ws[i] = 0u;
}

// Enqueues the workspace clear, then the plan's kernel(s).  The wave and
// flat regimes' kernels clear what they use themselves (ordered by a grid
// barrier of their cooperative launch) and need no separate clear.
cudaError_t launch(const gn::KParams& p, cudaStream_t s, bool bwd) {
  const bool nhwc = p.g.layout == GN_LAYOUT_NHWC;
  const gn::TimingEvents& ev = gn::timing_events();
  if (ev.begin) cudaEventRecord(ev.begin, s);
  if (p.g.regime != gn::kRegimeWave && p.g.regime != gn::kRegimeFlat) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, ws_clear, p.err, p.clear_words);
    if (e != cudaSuccess) return e;
  }
  switch (p.g.regime) {
    case gn::kRegimeResident: return gn::launch_resident(p, s, bwd);
    case gn::kRegimePipelined: return gn::launch_nchw_pipelined(p, s, bwd);
    case gn::kRegimeWave: return gn::launch_wave(p, s, bwd);
    case gn::kRegimeFlat: return gn::launch_flat(p, s, bwd);
    default: return nhwc ? gn::launch_nhwc(p, s, bwd) : gn::launch_nchw(p, s, bwd);
  }
}

size_t ws_size_any_alignment(int op, int64_t N, int64_t C, int64_t HW, int64_t G, int layout,
                             int dtype) {
  // Large enough for either op, either alignment and dense or strided views,
  // so that one workspace serves a forward and the following backward.
  (void)op;
  size_t best = 0;
  for (int o = 0; o < 2; ++o)
    for (int a = 0; a < 2; ++a)
      for (int d = 0; d < 2; ++d) {
        const gn::Geom g = gn::make_geom(o, N, C, HW, G, layout, dtype, a != 0, d != 0);
        const size_t t = gn::ws_layout(o, g).total;
        if (t > best) best = t;
      }
  return best;
}

// A view's element strides: per sample (sn) and per channel plane (NCHW) or
// spatial row (NHWC) (sr); within a plane (NCHW) or a row (NHWC) elements
// are contiguous.
struct View {
  int64_t sn, sr;
};

View dense_view(int64_t N, int64_t C, int64_t HW, int layout) {
  (void)N;
  return layout == GN_LAYOUT_NCHW ? View{C * HW, HW} : View{HW * C, C};
}

bool is_dense(const View& v, int64_t N, int64_t C, int64_t HW, int layout) {
  const View d = dense_view(N, C, HW, layout);
  return (v.sn == d.sn || N == 1) && (v.sr == d.sr || (layout == GN_LAYOUT_NCHW ? C : HW) == 1);
}

// The strides keep distinct elements apart: planes (rows) are contiguous runs
// of HW (C) elements, laid out sample-major or plane(row)-major without
// overlap.  An extent of 1 leaves its stride free.
bool view_ok(const View& v, int64_t N, int64_t C, int64_t HW, int layout) {
  const int64_t run = layout == GN_LAYOUT_NCHW ? HW : C;    // contiguous elements
  const int64_t cnt = layout == GN_LAYOUT_NCHW ? C : HW;    // runs per sample
  if (v.sn < 0 || v.sr < 0) return false;
  const int64_t sr = cnt > 1 ? v.sr : run, sn = N > 1 ? v.sn : run * cnt;
  if (sr < run || sn < run) return false;
  return sn >= cnt * sr || sr >= N * sn;
}

// Bytes from a view's first element to one past its last.
size_t view_span(const View& v, int64_t N, int64_t C, int64_t HW, int layout, int esz) {
  const int64_t run = layout == GN_LAYOUT_NCHW ? HW : C;
  const int64_t cnt = layout == GN_LAYOUT_NCHW ? C : HW;
  return (size_t)((N - 1) * v.sn + (cnt - 1) * v.sr + run) * (size_t)esz;
}

// The vector path needs the view's planes (rows) to start on 16-byte boundaries.
bool view_aligned(const void* base, const View& v, int64_t N, int64_t C, int64_t HW, int layout,
                  int esz) {
  if (!aligned16(base)) return false;
  const int64_t cnt = layout == GN_LAYOUT_NCHW ? C : HW;
  if (N > 1 && (v.sn * esz) % 16 != 0) return false;
  if (cnt > 1 && (v.sr * esz) % 16 != 0) return false;
  return true;
}

void set_views(gn::KParams* p, const View& xv, const View& dv, const View& ov) {
  p->xs_n = xv.sn;
  p->xs_r = xv.sr;
  p->ds_n = dv.sn;
  p->ds_r = dv.sr;
  p->os_n = ov.sn;
  p->os_r = ov.sr;
}

int fwd_impl(const void* x, View xv, int64_t N, int64_t C, int64_t HW, int64_t G, int layout,
             int dtype, const float* gamma, const float* beta, float eps, void* y, View yv,
             float* mean, float* rstd, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_problem(N, C, HW, G, layout, dtype);
  if (rc != GN_OK) return rc;
  if (N == 0 || C == 0 || HW == 0) return GN_OK;
  if (!x || !y || !mean || !rstd) return GN_ERR_INVALID;
  if (!(eps >= 0.0f)) return GN_ERR_INVALID;  // rejects NaN and negative eps
  if (!view_ok(xv, N, C, HW, layout) || !view_ok(yv, N, C, HW, layout)) return GN_ERR_INVALID;
  const int esz = elem_size(dtype);
  const size_t xb = view_span(xv, N, C, HW, layout, esz), yb = view_span(yv, N, C, HW, layout, esz);
  const size_t sbytes = sizeof(float) * (size_t)(N * G);
  const bool same = y == x && xv.sn == yv.sn && xv.sr == yv.sr;  // in place
  if (!same && overlap(y, yb, x, xb)) return GN_ERR_INVALID;
  if (overlap(mean, sbytes, x, xb) || overlap(mean, sbytes, y, yb) ||
      overlap(rstd, sbytes, x, xb) || overlap(rstd, sbytes, y, yb) ||
      overlap(mean, sbytes, rstd, sbytes))
    return GN_ERR_INVALID;
  const bool dense = is_dense(xv, N, C, HW, layout) && is_dense(yv, N, C, HW, layout);
  const bool aligned = view_aligned(x, xv, N, C, HW, layout, esz) &&
                       view_aligned(y, yv, N, C, HW, layout, esz);
  gn::KParams p;
  rc = prepare(GN_OP_FWD, N, C, HW, G, layout, dtype, aligned, dense, workspace, workspace_bytes,
               &p);
  if (rc != GN_OK) return rc;
  set_views(&p, xv, xv, yv);
  p.x = x;
  p.out = y;
  p.gamma = gamma;
  p.beta = beta;
  p.mean = mean;
  p.rstd = rstd;
  p.eps = eps;
  if (fault_mode() == GN_FAULT_LAUNCH) return cuda_fail(cudaErrorLaunchFailure);
  p.stall_unit = take_stall();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = launch(p, s, false);
  return e == cudaSuccess ? GN_OK : cuda_fail(e);
}

int bwd_impl(const void* dy, View dyv, const void* x, View xv, const float* mean,
             const float* rstd, const float* gamma, int64_t N, int64_t C, int64_t HW, int64_t G,
             int layout, int dtype, void* dx, View dxv, float* dgamma, float* dbeta,
             void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_problem(N, C, HW, G, layout, dtype);
  if (rc != GN_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (C == 0) return GN_OK;
  if (N == 0 || HW == 0) {
    // empty sums: the parameter gradients are zero
    if ((dgamma || dbeta) && fault_mode() == GN_FAULT_LAUNCH)
      return cuda_fail(cudaErrorLaunchFailure);
    if (dgamma) {
      const cudaError_t e = cudaMemsetAsync(dgamma, 0, sizeof(float) * (size_t)C, s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    if (dbeta) {
      const cudaError_t e = cudaMemsetAsync(dbeta, 0, sizeof(float) * (size_t)C, s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return GN_OK;
  }
  if (!dy || !x || !mean || !rstd || !dx) return GN_ERR_INVALID;
  if (!view_ok(dyv, N, C, HW, layout) || !view_ok(xv, N, C, HW, layout) ||
      !view_ok(dxv, N, C, HW, layout))
    return GN_ERR_INVALID;
  const int esz = elem_size(dtype);
  const size_t xb = view_span(xv, N, C, HW, layout, esz);
  const size_t db = view_span(dyv, N, C, HW, layout, esz);
  const size_t ob = view_span(dxv, N, C, HW, layout, esz);
  const size_t cbytes = sizeof(float) * (size_t)C;
  const bool on_dy = dx == dy && dxv.sn == dyv.sn && dxv.sr == dyv.sr;
  const bool on_x = dx == x && dxv.sn == xv.sn && dxv.sr == xv.sr;
  if (!on_dy && !on_x && (overlap(dx, ob, dy, db) || overlap(dx, ob, x, xb)))
    return GN_ERR_INVALID;
  if (overlap(dgamma, cbytes, dx, ob) || overlap(dbeta, cbytes, dx, ob) ||
      overlap(dgamma, cbytes, dbeta, cbytes))
    return GN_ERR_INVALID;
  const bool dense = is_dense(dyv, N, C, HW, layout) && is_dense(xv, N, C, HW, layout) &&
                     is_dense(dxv, N, C, HW, layout);
  const bool aligned = view_aligned(x, xv, N, C, HW, layout, esz) &&
                       view_aligned(dy, dyv, N, C, HW, layout, esz) &&
                       view_aligned(dx, dxv, N, C, HW, layout, esz);
  gn::KParams p;
  rc = prepare(GN_OP_BWD, N, C, HW, G, layout, dtype, aligned, dense, workspace, workspace_bytes,
               &p);
  if (rc != GN_OK) return rc;
  set_views(&p, xv, dyv, dxv);
  p.x = x;
  p.dy = dy;
  p.out = dx;
  p.gamma = gamma;
  p.mean = const_cast<float*>(mean);
  p.rstd = const_cast<float*>(rstd);
  p.dgamma = dgamma;
  p.dbeta = dbeta;
  if (fault_mode() == GN_FAULT_LAUNCH) return cuda_fail(cudaErrorLaunchFailure);
  p.stall_unit = take_stall();
  const cudaError_t e = launch(p, s, true);
  return e == cudaSuccess ? GN_OK : cuda_fail(e);
}

}  // namespace

namespace gn {
const TimingEvents& timing_events() { return t_events; }
int record_cuda_error(cudaError_t e) { return cuda_fail(e); }
}  // namespace gn

extern "C" {

size_t gn_workspace_size(int op, int64_t N, int64_t C, int64_t HW, int64_t G, int layout,
                         int dtype) {
  if (op != GN_OP_FWD && op != GN_OP_BWD) return 0;
  if (check_problem(N, C, HW, G, layout, dtype) != GN_OK) return 0;
  if (N == 0 || C == 0 || HW == 0) return 0;
  return ws_size_any_alignment(op, N, C, HW, G, layout, dtype);
}

int gn_fwd(const void* x, int64_t N, int64_t C, int64_t HW, int64_t G, int layout, int dtype,
           const float* gamma, const float* beta, float eps, void* y, float* mean, float* rstd,
           void* workspace, size_t workspace_bytes, void* stream) {
  const View d = dense_view(N, C, HW, layout);
  return fwd_impl(x, d, N, C, HW, G, layout, dtype, gamma, beta, eps, y, d, mean, rstd, workspace,
                  workspace_bytes, stream);
}

int gn_fwd_ex(const void* x, int64_t x_sn, int64_t x_sr, int64_t N, int64_t C, int64_t HW,
              int64_t G, int layout, int dtype, const float* gamma, const float* beta, float eps,
              void* y, int64_t y_sn, int64_t y_sr, float* mean, float* rstd, void* workspace,
              size_t workspace_bytes, void* stream) {
  return fwd_impl(x, View{x_sn, x_sr}, N, C, HW, G, layout, dtype, gamma, beta, eps, y,
                  View{y_sn, y_sr}, mean, rstd, workspace, workspace_bytes, stream);
}

int gn_bwd(const void* dy, const void* x, const float* mean, const float* rstd,
           const float* gamma, int64_t N, int64_t C, int64_t HW, int64_t G, int layout,
           int dtype, void* dx, float* dgamma, float* dbeta, void* workspace,
           size_t workspace_bytes, void* stream) {
  const View d = dense_view(N, C, HW, layout);
  return bwd_impl(dy, d, x, d, mean, rstd, gamma, N, C, HW, G, layout, dtype, dx, d, dgamma,
                  dbeta, workspace, workspace_bytes, stream);
}

int gn_bwd_ex(const void* dy, int64_t dy_sn, int64_t dy_sr, const void* x, int64_t x_sn,
              int64_t x_sr, const float* mean, const float* rstd, const float* gamma, int64_t N,
              int64_t C, int64_t HW, int64_t G, int layout, int dtype, void* dx, int64_t dx_sn,
              int64_t dx_sr, float* dgamma, float* dbeta, void* workspace,
              size_t workspace_bytes, void* stream) {
  return bwd_impl(dy, View{dy_sn, dy_sr}, x, View{x_sn, x_sr}, mean, rstd, gamma, N, C, HW, G,
                  layout, dtype, dx, View{dx_sn, dx_sr}, dgamma, dbeta, workspace,
                  workspace_bytes, stream);
}

const char* gn_status_string(int status) {
  switch (status) {
    case GN_OK: return "GN_OK";
    case GN_ERR_INVALID: return "GN_ERR_INVALID: invalid problem or buffers";
    case GN_ERR_UNSUPPORTED: return "GN_ERR_UNSUPPORTED: unsupported layout, dtype or size";
    case GN_ERR_WORKSPACE: return "GN_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case GN_ERR_CUDA: return "GN_ERR_CUDA: a CUDA call failed";
    case GN_ERR_TIMEOUT:
      return "GN_ERR_TIMEOUT: a bounded wait in a kernel ran out; that call's outputs are not valid";
    default: return "unknown gn_status";
  }
}

int gn_last_cuda_error(void) { return t_last_cuda_error; }

int gn_set_fault_injection(int mode) {
  if (mode != GN_FAULT_NONE && mode != GN_FAULT_LAUNCH && mode != GN_FAULT_STALL)
    return GN_ERR_INVALID;
  g_fault.store(mode);
  return GN_OK;
}

int gn_workspace_status(const void* workspace, void* stream) {
  if (!workspace || !aligned16(workspace)) return GN_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  return word ? GN_ERR_TIMEOUT : GN_OK;
}

int gn_set_regime(int regime) {
  if (regime != GN_REGIME_AUTO && regime != GN_REGIME_TWO_KERNEL && regime != GN_REGIME_RESIDENT &&
      regime != GN_REGIME_PIPELINED && regime != GN_REGIME_WAVE && regime != GN_REGIME_FLAT)
    return GN_ERR_INVALID;
  gn::set_regime_override(regime);
  return GN_OK;
}

int gn_set_timing_events(void* ev_begin, void* ev_mid, void* ev_end) {
  t_events.begin = static_cast<cudaEvent_t>(ev_begin);
  t_events.mid = static_cast<cudaEvent_t>(ev_mid);
  t_events.end = static_cast<cudaEvent_t>(ev_end);
  return GN_OK;
}

int gn_plan_info(int op, int64_t N, int64_t C, int64_t HW, int64_t G, int layout, int dtype,
                 int aligned, gn_plan_desc* out) {
  if (!out) return GN_ERR_INVALID;
  if (op != GN_OP_FWD && op != GN_OP_BWD) return GN_ERR_INVALID;
  const int rc = check_problem(N, C, HW, G, layout, dtype);
  if (rc != GN_OK) return rc;
  std::memset(out, 0, sizeof(*out));
  if (N == 0 || C == 0 || HW == 0) return GN_OK;
  const gn::Geom g = gn::make_geom(op, N, C, HW, G, layout, dtype, aligned != 0);
  out->regime = g.regime;
  // the plan's kernels, plus the workspace clear that precedes every regime
  // but the wave and flat regimes (whose kernels clear what they use)
  const bool self_clear = g.regime == gn::kRegimeWave || g.regime == gn::kRegimeFlat;
  out->launches = (g.regime == gn::kRegimeGeneric ? 2 : 1) + (self_clear ? 0 : 1);
  out->vector_width = g.vw;
  out->threads = g.tpb;
  const bool persistent = g.regime == gn::kRegimePipelined || g.regime == gn::kRegimeWave ||
                          g.regime == gn::kRegimeFlat;
  out->ctas = g.regime == gn::kRegimeResident ? g.units * g.K : persistent ? g.grid : g.items;
  out->partials = g.N * g.C * (g.T + (g.l1 > 1 ? g.Tp : 0));
  out->workspace_bytes = gn::ws_layout(op, g).total;
  out->err_offset = gn::ws_layout(op, g).err;
  out->clear_bytes = gn::ws_layout(op, g).clear;
  out->cluster_ctas = g.regime == gn::kRegimeResident ? g.K : 1;
  out->finalise_second = g.fin2;
  out->level1_items = g.l1 > 1 ? g.l1 : 1;
  const int64_t mc = gn::plan_max_clusters(g, op);
  out->max_clusters = mc > 0 ? (int)mc : 0;
  // item / piece shape (the boundaries the parity tests sample)
  out->slots = g.regime == gn::kRegimeGeneric ? 0 : g.S;
  out->hold_buffers = g.regime == gn::kRegimeWave ? (int)g.wH : 0;
  if (g.regime == gn::kRegimeWave) {
    out->piece_elems = g.wR;
    out->pieces_per_unit = g.wP;
  } else if (g.regime == gn::kRegimeFlat) {
    const int64_t R = g.N * g.HW, run = (R + g.grid - 1) / g.grid;
    out->piece_elems = g.chunk;
    out->pieces_per_unit = (run + g.chunk - 1) / g.chunk;
  } else if (g.regime == gn::kRegimeResident) {
    out->piece_elems = g.slice;
    out->pieces_per_unit = g.K;
  } else if (g.layout == GN_LAYOUT_NHWC) {
    out->piece_elems = g.rb;
    out->pieces_per_unit = g.T;
  } else if (g.mode == 0) {
    out->piece_elems = g.L;
    out->pieces_per_unit = g.T;
  } else {
    out->piece_elems = g.RB * g.HW;
    out->pieces_per_unit = g.items_per_n;
  }
  if (g.regime == gn::kRegimeResident) {
    out->smem_bytes = g.smem;
  } else if (persistent) {
    out->smem_bytes = g.smem;
  } else {
    size_t sm = 0;
    if (g.layout == GN_LAYOUT_NHWC)
      gn::nhwc_kernel(g, op == GN_OP_BWD, 0, &sm);
    else
      gn::nchw_kernel(g, op == GN_OP_BWD, 0, &sm);
    out->smem_bytes = sm;
  }
  return GN_OK;
}

}  // extern "C"
