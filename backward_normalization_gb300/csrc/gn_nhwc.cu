// gn_nhwc.cu -- two-kernel GroupNorm path for channels_last activations.
//
// Memory: element (n, c, hw) sits at (n*HW + hw)*C + c, so one spatial
// position ("row") holds the C channels contiguously and a group is a run of
// Cg channels inside every row.  An item = (sample n, column block cb, block
// t of rb consecutive rows), numbered ((n*ncb + cb)*T + t); each thread owns
// one column of vw channels (one 16-byte vector) and walks the item's rows
// with stride rpi, so every warp issues coalesced 16-byte loads and a
// thread's channels (and their group constants) never change.
//
// Forward : nhwc_fwd_stats  -> per-(item, channel) shifted sums; groups of l1
//                              items, then the sample, are merged by their
//                              last CTA into mean/rstd per group
//           nhwc_fwd_apply  -> y = (x - mean) * rstd*gamma + beta
// Backward: nhwc_bwd_reduce -> per-(item, channel) sum(dy), sum(dy*(x-mean));
//                              merged the same way into the dx coefficients
//           nhwc_bwd_dx     -> dx = rstd*gamma*dy + B*(x - mean) + D; its first
//                              CTA forms dgamma/dbeta
// The second kernel of each op walks items and rows in the reverse order of
// the first, so it starts on the data the first kernel left in L2.
#include "gn_finalize.cuh"

namespace gn {
namespace {

struct NhwcItem {
  int64_t n, t, cb, col, row0, row1;
  int j, r;
  bool active;
};

__device__ __forceinline__ NhwcItem nhwc_item(const Geom& g, int64_t item) {
  NhwcItem it;
  const int tid = threadIdx.x;
  it.j = tid % g.Wv;
  it.r = tid / g.Wv;
  it.t = item % g.T;
  item /= g.T;
  it.cb = item % g.ncb;
  it.n = item / g.ncb;
  it.col = it.cb * g.Wv + it.j;
  it.active = (it.r < g.rpi) && (it.col < g.V);
  it.row0 = it.t * g.rb;
  it.row1 = (it.row0 + g.rb < g.HW) ? it.row0 + g.rb : g.HW;  // may be <= row0: empty item
  return it;
}

// Values that depend only on the group, for the vw channels of a thread's
// vector: NG = 1 when the vector lies inside one group (vw divides Cg, or
// vw = 1), else NG = vw values, one per channel.  The single value keeps the
// per-thread constants of the wide vectors in few registers.
template <int VW, int NG>
struct PerGroup {
  float v[NG];
  __device__ __forceinline__ float operator[](int e) const { return v[NG == 1 ? 0 : e]; }
};

// Whether a plan's vectors lie inside one group each.
inline bool one_group_per_vector(const Geom& g) { return g.vw == 1 || g.Cg % g.vw == 0; }

// Tail of both first kernels.  CTA sums: each (column, value) pair adds its
// rpi row lanes in lane order (one barrier, no tree).  Then the item record
// part0[n][t][c], and the arrival chain (group of l1 items, sample).
template <typename T, int VW, bool kBwd>
__device__ __forceinline__ void publish_nhwc(const KParams& p, const NhwcItem& it, float* red,
                                             const float (&acc)[2 * VW]) {
  const Geom& g = p.g;
  const int tid = threadIdx.x, tpb = blockDim.x;
#pragma unroll
  for (int q = 0; q < 2 * VW; ++q) red[q * tpb + tid] = acc[q];
  __syncthreads();
  float* rec = reinterpret_cast<float*>(p.part0 + it.n * g.C * g.T + it.t * g.C);
  for (int pi = tid; pi < g.Wv * 2 * VW; pi += tpb) {
    const int q = pi / g.Wv, j = pi % g.Wv;
    const int64_t col = it.cb * g.Wv + j;
    if (col >= g.V) continue;
    float s = 0.f;
    for (int r = 0; r < g.rpi; ++r) s += red[q * tpb + r * g.Wv + j];
    rec[2 * (col * VW + q / 2) + (q & 1)] = s;
  }
  const int64_t t1 = it.t / g.l1;
  const int64_t tlo = t1 * g.l1;
  const unsigned gsize = (unsigned)((tlo + g.l1 < g.T) ? g.l1 : g.T - tlo);
  auto merge = [&]() {
    // group record of the column block's channels: its items' records in item order
    const int64_t c0 = it.cb * g.Wv * VW;
    const int64_t c1 = (c0 + (int64_t)g.Wv * VW < g.C) ? c0 + (int64_t)g.Wv * VW : g.C;
    for (int64_t c = c0 + tid; c < c1; c += tpb) {
      float ax = 0.f, ay = 0.f;
      sum_records(p.part0 + it.n * g.C * g.T + tlo * g.C + c, g.C, 0, 1, gsize, ax, ay);
      p.part[it.n * g.C * g.Tp + t1 * g.C + c] = make_float2(ax, ay);
    }
  };
  arrive_and_finalize<T, kBwd>(p, unit_of(p, it.n, 0), (it.n * g.ncb + it.cb) * g.Tp + t1, gsize,
                               merge, red, (int64_t)2 * VW * tpb);
}

// Forward pass 1 of one item: per-channel shifted sums, then publish.
template <typename T, int VW>
__device__ __forceinline__ void stats_item(const KParams& p, int64_t item, float* red) {
  const Geom& g = p.g;
  const NhwcItem it = nhwc_item(g, item);
  float acc[2 * VW];
#pragma unroll
  for (int q = 0; q < 2 * VW; ++q) acc[q] = 0.f;
  if (it.active && it.row0 < it.row1) {
    const T* xn = static_cast<const T*>(p.x) + it.n * p.xs_n + it.col * VW;
    const int64_t xr = p.xs_r;
    const uint64_t pfirst = policy_evict_first(), plast = policy_evict_last();
    const int64_t keep = it.row0 + g.keep_from;  // rows from here on are read again first
    float K[VW];
    Access<T, VW>::load(xn, K, pfirst);  // row 0 of the sample: the per-channel shift
    const int64_t step = g.rpi;
    int64_t row = it.row0 + it.r;
    using Raw = typename Access<T, VW>::Raw;
    constexpr int U = 8;  // rows in flight per thread
    for (; row + (U - 1) * step < it.row1; row += U * step) {
      const uint64_t pol = row >= keep ? plast : pfirst;
      Raw raw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) raw[u] = Access<T, VW>::load_raw(xn + (row + u * step) * xr, pol);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float v[VW];
        Access<T, VW>::unpack(raw[u], v);
#pragma unroll
        for (int k = 0; k < VW; ++k) {
          const float d = v[k] - K[k];
          acc[2 * k] += d;
          acc[2 * k + 1] = fmaf(d, d, acc[2 * k + 1]);
        }
      }
    }
    if (row < it.row1) {  // the last (< U) rows: one predicated batch, not a row at a time
      const uint64_t pol = row >= keep ? plast : pfirst;
      Raw raw[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        raw[u] = row + u * step < it.row1 ? Access<T, VW>::load_raw(xn + (row + u * step) * xr, pol)
                                          : Raw{};
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (row + u * step >= it.row1) break;
        float v[VW];
        Access<T, VW>::unpack(raw[u], v);
#pragma unroll
        for (int k = 0; k < VW; ++k) {
          const float d = v[k] - K[k];
          acc[2 * k] += d;
          acc[2 * k + 1] = fmaf(d, d, acc[2 * k + 1]);
        }
      }
    }
  }
  publish_nhwc<T, VW, false>(p, it, red, acc);
}

template <typename T, int VW>
__global__ void __launch_bounds__(512, 2) nhwc_fwd_stats(const __grid_constant__ KParams p) {
  grid_dependency_wait();  // the previous kernel's results (and x, dy) are complete
  grid_launch_dependents();
  extern __shared__ float red[];
  stats_item<T, VW>(p, blockIdx.x, red);
}

// Backward pass 1 of one item: per-channel sum(dy), sum(dy*(x-mean)), then publish.
template <typename T, int VW, int NG>
__device__ __forceinline__ void reduce_item(const KParams& p, int64_t item, float* red) {
  const Geom& g = p.g;
  const NhwcItem it = nhwc_item(g, item);
  float acc[2 * VW];
#pragma unroll
  for (int q = 0; q < 2 * VW; ++q) acc[q] = 0.f;
  if (it.active && it.row0 < it.row1) {
    PerGroup<VW, NG> mu;
#pragma unroll
    for (int k = 0; k < NG; ++k) mu.v[k] = __ldg(p.mean + it.n * g.G + (it.col * VW + k) / g.Cg);
    const T* xn = static_cast<const T*>(p.x) + it.n * p.xs_n + it.col * VW;
    const T* dyn = static_cast<const T*>(p.dy) + it.n * p.ds_n + it.col * VW;
    const int64_t xr = p.xs_r, dr = p.ds_r;
    const uint64_t pfirst = policy_evict_first(), plast = policy_evict_last();
    const int64_t keep = it.row0 + g.keep_from;
    const int64_t step = g.rpi;
    int64_t row = it.row0 + it.r;
    using Raw = typename Access<T, VW>::Raw;
    constexpr int U = 4;  // rows in flight per thread (x and dy each)
    for (; row + (U - 1) * step < it.row1; row += U * step) {
      const uint64_t pol = row >= keep ? plast : pfirst;
      Raw rx[U], rd[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        rx[u] = Access<T, VW>::load_raw(xn + (row + u * step) * xr, pol);
        rd[u] = Access<T, VW>::load_raw(dyn + (row + u * step) * dr, pol);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float xv[VW], dv[VW];
        Access<T, VW>::unpack(rx[u], xv);
        Access<T, VW>::unpack(rd[u], dv);
#pragma unroll
        for (int k = 0; k < VW; ++k) {
          acc[2 * k] += dv[k];
          acc[2 * k + 1] = fmaf(dv[k], xv[k] - mu[k], acc[2 * k + 1]);
        }
      }
    }
    if (NG > 1) {  // per-channel group constants: a predicated batch would spill here
      for (; row < it.row1; row += step) {
        const uint64_t pol = row >= keep ? plast : pfirst;
        float xv[VW], dv[VW];
        Access<T, VW>::load(xn + row * xr, xv, pol);
        Access<T, VW>::load(dyn + row * dr, dv, pol);
#pragma unroll
        for (int k = 0; k < VW; ++k) {
          acc[2 * k] += dv[k];
          acc[2 * k + 1] = fmaf(dv[k], xv[k] - mu[k], acc[2 * k + 1]);
        }
      }
    } else if (row < it.row1) {  // the last (< U) rows: one predicated batch (masked rows add 0)
      const uint64_t pol = row >= keep ? plast : pfirst;
      Raw rx[U], rd[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const bool in = row + u * step < it.row1;
        rx[u] = in ? Access<T, VW>::load_raw(xn + (row + u * step) * xr, pol) : Raw{};
        rd[u] = in ? Access<T, VW>::load_raw(dyn + (row + u * step) * dr, pol) : Raw{};
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (row + u * step >= it.row1) break;
        float xv[VW], dv[VW];
        Access<T, VW>::unpack(rx[u], xv);
        Access<T, VW>::unpack(rd[u], dv);
#pragma unroll
        for (int k = 0; k < VW; ++k) {
          acc[2 * k] += dv[k];
          acc[2 * k + 1] = fmaf(dv[k], xv[k] - mu[k], acc[2 * k + 1]);
        }
      }
    }
  }
  publish_nhwc<T, VW, true>(p, it, red, acc);
}

template <typename T, int VW, int NG>
__global__ void __launch_bounds__(512, 2) nhwc_bwd_reduce(const __grid_constant__ KParams p) {
  grid_dependency_wait();  // the previous kernel's results (and x, dy) are complete
  grid_launch_dependents();
  extern __shared__ float red[];
  reduce_item<T, VW, NG>(p, blockIdx.x, red);
}

// Forward pass 2 of one item: y = (x - mean) * rstd*gamma + beta, rows last to first.
template <typename T, int VW, int NG>
__device__ __forceinline__ void apply_item(const KParams& p, int64_t item) {
  const Geom& g = p.g;
  const NhwcItem it = nhwc_item(g, item);
  if (!it.active) return;
  const int64_t cnt = it.row1 - it.row0 - it.r;  // rows of this lane: r, r+step, ...
  if (cnt <= 0) return;
  PerGroup<VW, NG> mu;
  float a[VW], b[VW];
#pragma unroll
  for (int k = 0; k < VW; ++k) {
    const int64_t c = it.col * VW + k;
    const int64_t ng = it.n * g.G + c / g.Cg;
    const float r = __ldcg(p.rstd + ng);  // written earlier in this call: not the read-only path
    a[k] = p.gamma ? r * __ldg(p.gamma + c) : r;
    b[k] = p.beta ? __ldg(p.beta + c) : 0.f;
    if (NG > 1 || k == 0) mu.v[NG > 1 ? k : 0] = __ldcg(p.mean + ng);
  }
  const T* xn = static_cast<const T*>(p.x) + it.n * p.xs_n + it.col * VW;
  T* yn = static_cast<T*>(p.out) + it.n * p.os_n + it.col * VW;
  const int64_t xr = p.xs_r, yr = p.os_r;
  const uint64_t pol = policy_evict_first();
  const int64_t step = g.rpi;
  int64_t row = it.row0 + it.r + ((cnt - 1) / step) * step;  // last row of the lane
  for (; row - 3 * step >= it.row0; row -= 4 * step) {
    float v[4][VW];
#pragma unroll
    for (int u = 0; u < 4; ++u) Access<T, VW>::load(xn + (row - u * step) * xr, v[u], pol);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll
      for (int k = 0; k < VW; ++k) v[u][k] = fmaf(v[u][k] - mu[k], a[k], b[k]);
      Access<T, VW>::store(yn + (row - u * step) * yr, v[u], pol);
    }
  }
  for (; row >= it.row0; row -= step) {
    float v[VW];
    Access<T, VW>::load(xn + row * xr, v, pol);
#pragma unroll
    for (int k = 0; k < VW; ++k) v[k] = fmaf(v[k] - mu[k], a[k], b[k]);
    Access<T, VW>::store(yn + row * yr, v, pol);
  }
}

// Backward pass 2 of one item: dx = rstd*gamma*dy + B*(x - mean) + D, rows last to first.
template <typename T, int VW, int NG>
__device__ __forceinline__ void dx_item(const KParams& p, int64_t item) {
  const Geom& g = p.g;
  const NhwcItem it = nhwc_item(g, item);
  if (!it.active) return;
  const int64_t cnt = it.row1 - it.row0 - it.r;
  if (cnt <= 0) return;
  PerGroup<VW, NG> mu, B, D;
  float A[VW];
#pragma unroll
  for (int k = 0; k < VW; ++k) {
    const int64_t c = it.col * VW + k;
    const int64_t ng = it.n * g.G + c / g.Cg;
    const float r = __ldg(p.rstd + ng);
    A[k] = p.gamma ? r * __ldg(p.gamma + c) : r;
    if (NG > 1 || k == 0) {
      const float2 cf = __ldcg(p.coef + ng);
      mu.v[NG > 1 ? k : 0] = __ldg(p.mean + ng);
      B.v[NG > 1 ? k : 0] = cf.x;
      D.v[NG > 1 ? k : 0] = cf.y;
    }
  }
  const T* xn = static_cast<const T*>(p.x) + it.n * p.xs_n + it.col * VW;
  const T* dyn = static_cast<const T*>(p.dy) + it.n * p.ds_n + it.col * VW;
  T* dxn = static_cast<T*>(p.out) + it.n * p.os_n + it.col * VW;
  const int64_t xr = p.xs_r, dr = p.ds_r, orr = p.os_r;
  const uint64_t pol = policy_evict_first();
  const int64_t step = g.rpi;
  int64_t row = it.row0 + it.r + ((cnt - 1) / step) * step;
  using Raw = typename Access<T, VW>::Raw;
  for (; row - step >= it.row0; row -= 2 * step) {
    Raw rx[2], rd[2];  // packed until used: fewer live registers
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      rx[u] = Access<T, VW>::load_raw(xn + (row - u * step) * xr, pol);
      rd[u] = Access<T, VW>::load_raw(dyn + (row - u * step) * dr, pol);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float xv[VW], dv[VW];
      Access<T, VW>::unpack(rx[u], xv);
      Access<T, VW>::unpack(rd[u], dv);
#pragma unroll
      for (int k = 0; k < VW; ++k) xv[k] = fmaf(A[k], dv[k], fmaf(B[k], xv[k] - mu[k], D[k]));
      Access<T, VW>::store(dxn + (row - u * step) * orr, xv, pol);
    }
  }
  for (; row >= it.row0; row -= step) {
    float xv[VW], dv[VW];
    Access<T, VW>::load(xn + row * xr, xv, pol);
    Access<T, VW>::load(dyn + row * dr, dv, pol);
#pragma unroll
    for (int k = 0; k < VW; ++k) xv[k] = fmaf(A[k], dv[k], fmaf(B[k], xv[k] - mu[k], D[k]));
    Access<T, VW>::store(dxn + row * orr, xv, pol);
  }
}

template <typename T, int VW, int NG>
__global__ void __launch_bounds__(512, 2) nhwc_fwd_apply(const __grid_constant__ KParams p) {
  grid_dependency_wait();  // the previous kernel's results (and x, dy) are complete
  grid_launch_dependents();
  apply_item<T, VW, NG>(p, p.g.items - 1 - (int64_t)blockIdx.x);
}

template <typename T, int VW, int NG>
__global__ void __launch_bounds__(512, 2) nhwc_bwd_dx(const __grid_constant__ KParams p) {
  extern __shared__ float sm[];
  grid_dependency_wait();
  grid_launch_dependents();
  // the first CTA also adds up dgamma / dbeta: every channel's sums are
  // complete once the first kernel is
  if (blockIdx.x == 0) finalize_params(p, sm);
  dx_item<T, VW, NG>(p, p.g.items - 1 - (int64_t)blockIdx.x);
}

template <typename T, int VW, int NG>
cudaError_t run_op(const KParams& p, cudaStream_t s, bool bwd) {
  const Geom& g = p.g;
  const size_t sm1 = sizeof(float) * 2 * VW * g.tpb;
  const TimingEvents& ev = timing_events();
  cudaError_t e = bwd ? launch_pdl(nhwc_bwd_reduce<T, VW, NG>, g.items, g.tpb, sm1, s, p)
                      : launch_pdl(nhwc_fwd_stats<T, VW>, g.items, g.tpb, sm1, s, p);
  if (e != cudaSuccess) return e;
  if (ev.mid) cudaEventRecord(ev.mid, s);
  e = bwd ? launch_pdl(nhwc_bwd_dx<T, VW, NG>, g.items, g.tpb, sizeof(float) * 2 * g.tpb, s, p)
          : launch_pdl(nhwc_fwd_apply<T, VW, NG>, g.items, g.tpb, 0, s, p);
  if (ev.end) cudaEventRecord(ev.end, s);
  return e;
}

template <typename T>
cudaError_t dispatch_vw(const KParams& p, cudaStream_t s, bool bwd) {
  constexpr int V = Elem<T>::VEC;
  if (p.g.vw == 1) return run_op<T, 1, 1>(p, s, bwd);
  return one_group_per_vector(p.g) ? run_op<T, V, 1>(p, s, bwd) : run_op<T, V, V>(p, s, bwd);
}

template <typename T, int VW, int NG>
const void* kernel_t(const Geom& g, bool bwd, int second, size_t* smem) {
  *smem = second ? (bwd ? sizeof(float) * 2 * g.tpb : 0) : sizeof(float) * 2 * VW * g.tpb;
  if (second)
    return bwd ? (const void*)nhwc_bwd_dx<T, VW, NG> : (const void*)nhwc_fwd_apply<T, VW, NG>;
  return bwd ? (const void*)nhwc_bwd_reduce<T, VW, NG> : (const void*)nhwc_fwd_stats<T, VW>;
}

template <typename T>
const void* kernel_vw(const Geom& g, bool bwd, int second, size_t* smem) {
  constexpr int V = Elem<T>::VEC;
  if (g.vw == 1) return kernel_t<T, 1, 1>(g, bwd, second, smem);
  return one_group_per_vector(g) ? kernel_t<T, V, 1>(g, bwd, second, smem)
                                 : kernel_t<T, V, V>(g, bwd, second, smem);
}

}  // namespace

const void* nhwc_kernel(const Geom& g, bool bwd, int second, size_t* smem) {
  switch (g.dtype) {
    case kF32: return kernel_vw<float>(g, bwd, second, smem);
    case kF16: return kernel_vw<__half>(g, bwd, second, smem);
    case kF64: return kernel_vw<double>(g, bwd, second, smem);
    default: return kernel_vw<__nv_bfloat16>(g, bwd, second, smem);
  }
}

cudaError_t launch_nhwc(const KParams& p, cudaStream_t s, bool bwd) {
  switch (p.g.dtype) {
    case kF32: return dispatch_vw<float>(p, s, bwd);
    case kF16: return dispatch_vw<__half>(p, s, bwd);
    case kF64: return dispatch_vw<double>(p, s, bwd);
    default: return dispatch_vw<__nv_bfloat16>(p, s, bwd);
  }
}

}  // namespace gn
