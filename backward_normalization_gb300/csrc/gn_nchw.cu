// gn_nchw.cu -- GroupNorm for NCHW activations: the two-kernel path and the
// pipelined kernel.
//
// Memory: element (n, c, hw) sits at (n*C + c)*HW + hw, so each (n, c)
// channel plane ("row") is HW contiguous elements and a group is Cg
// consecutive planes.  Two item shapes:
//   mode 0 (large planes): item = (row, chunk of L elements), numbered
//          row*T + chunk; the whole CTA strides the chunk with 16-byte loads
//          and writes one record; groups of l1 chunks of a row are merged by
//          their last CTA.
//   mode 1 (small planes): item = RB consecutive rows of one sample; each warp
//          takes whole rows; one record per row.
// In the two-kernel path the elementwise second kernels walk the items (and
// the elements of a chunk) in reverse order, starting on the data the first
// kernel left in L2.  When a second-kernel CTA's groups have few records
// (g.fin2), that CTA derives their statistics (or dx coefficients) from the
// records itself and the first kernel ends with its records; otherwise the
// first kernel's last arrival of a sample finalises it.  The
// pipelined kernel (mode-0 shapes, 16-byte vectors) runs the lockstep
// schedule of gn_tasks.cuh over (sample, group) units, fed by bulk copies.
#include "gn_tasks.cuh"

namespace gn {
namespace {

// Dynamic shared memory of the first kernels, in floats: reduction scratch
// plus room to stage the per-channel results of the finalisation.
__host__ __device__ __forceinline__ int64_t nchw_smem_floats(const Geom& g) {
  const int64_t stage = 2 * g.C <= 8192 ? 2 * g.C : 0;
  return 2 * (int64_t)g.tpb + stage;
}

template <int VW>
__device__ __forceinline__ void acc_shifted(const float (&v)[VW], float K, float& s, float& q) {
#pragma unroll
  for (int k = 0; k < VW; ++k) {
    const float d = v[k] - K;
    s += d;
    q = fmaf(d, d, q);
  }
}

template <int VW>
__device__ __forceinline__ void acc_grad(const float (&xv)[VW], const float (&dv)[VW], float mu,
                                         float& s1, float& s2) {
#pragma unroll
  for (int k = 0; k < VW; ++k) {
    s1 += dv[k];
    s2 = fmaf(dv[k], xv[k] - mu, s2);
  }
}

struct Chunk {
  int64_t row, ch, h0, h1;
};

__device__ __forceinline__ Chunk chunk_of(const Geom& g, int64_t item) {
  Chunk c;
  c.row = item / g.T;
  c.ch = item % g.T;
  c.h0 = c.ch * g.L;
  c.h1 = (c.h0 + g.L < g.HW) ? c.h0 + g.L : g.HW;  // may be <= h0: empty chunk
  return c;
}

// Mode-0 tail of pass 1: CTA sum, the chunk's record, the arrival chain
// (group of l1 chunks of the row, then the chunk's unit).
template <typename T, bool kBwd>
__device__ __forceinline__ void publish_chunk(const KParams& p, const Chunk& k, float a, float b,
                                              float* sm) {
  const Geom& g = p.g;
  const float2 tot = block_sum2_t0(a, b, sm);
  if (threadIdx.x == 0) p.part0[k.row * g.T + k.ch] = tot;
  const int64_t t1 = k.ch / g.l1;
  const int64_t tlo = t1 * g.l1;
  const unsigned gsize = (unsigned)((tlo + g.l1 < g.T) ? g.l1 : g.T - tlo);
  auto merge = [&]() {
    if (threadIdx.x != 0) return;
    float ax = 0.f, ay = 0.f;
    sum_records(p.part0 + k.row * g.T + tlo, 1, 0, 1, gsize, ax, ay);
    p.part[k.row * g.Tp + t1] = make_float2(ax, ay);
  };
  if (g.fin2) {  // the second kernel finalises: at most the level-1 merge here
    if (g.l1 > 1) arrive_level1(p, k.row * g.Tp + t1, gsize, merge);
    return;
  }
  arrive_and_finalize<T, kBwd>(p, unit_of(p, k.row / g.C, k.row % g.C), k.row * g.Tp + t1, gsize,
                               merge, sm, nchw_smem_floats(g));
}

// ---------------------------------------------------------- mode 0 (chunks)
// Forward pass 1 of one chunk: shifted sums with K = x(n, c, 0).
template <typename T, int VW>
__device__ __forceinline__ void stats_chunk(const KParams& p, int64_t item, float* sm) {
  const Geom& g = p.g;
  const int tid = threadIdx.x;
  const uint64_t pfirst = policy_evict_first(), plast = policy_evict_last();
  const Chunk k = chunk_of(g, item);
  const T* xr = static_cast<const T*>(p.x) + plane_offset(g, k.row, p.xs_n, p.xs_r);
  const float K = Elem<T>::to_f(xr[0]);
  if (g.fin2 && k.ch == 0 && tid == 0) p.kst[k.row] = K;  // for the second kernel
  const int64_t keep = k.h0 + g.keep_from;
  float s = 0.f, q = 0.f;
  const int64_t st = (int64_t)blockDim.x * VW;
  int64_t h = k.h0 + (int64_t)tid * VW;
  for (; h + 3 * st < k.h1; h += 4 * st) {
    const uint64_t pol = h >= keep ? plast : pfirst;
    float v[4][VW];
#pragma unroll
    for (int u = 0; u < 4; ++u) Access<T, VW>::load(xr + h + u * st, v[u], pol);
#pragma unroll
    for (int u = 0; u < 4; ++u) acc_shifted<VW>(v[u], K, s, q);
  }
  for (; h < k.h1; h += st) {
    float v[VW];
    Access<T, VW>::load(xr + h, v, h >= keep ? plast : pfirst);
    acc_shifted<VW>(v, K, s, q);
  }
  publish_chunk<T, false>(p, k, s, q, sm);
}

// Backward pass 1 of one chunk: sum(dy), sum(dy*(x-mean)).
template <typename T, int VW>
__device__ __forceinline__ void reduce_chunk(const KParams& p, int64_t item, float* sm) {
  const Geom& g = p.g;
  const int tid = threadIdx.x;
  const uint64_t pfirst = policy_evict_first(), plast = policy_evict_last();
  const Chunk k = chunk_of(g, item);
  const int64_t n = k.row / g.C;
  const float mu = __ldg(p.mean + n * g.G + (k.row % g.C) / g.Cg);
  const T* xr = static_cast<const T*>(p.x) + plane_offset(g, k.row, p.xs_n, p.xs_r);
  const T* dr = static_cast<const T*>(p.dy) + plane_offset(g, k.row, p.ds_n, p.ds_r);
  const int64_t keep = k.h0 + g.keep_from;
  float s1 = 0.f, s2 = 0.f;
  const int64_t st = (int64_t)blockDim.x * VW;
  int64_t h = k.h0 + (int64_t)tid * VW;
  for (; h + st < k.h1; h += 2 * st) {
    const uint64_t pol = h >= keep ? plast : pfirst;
    float xv[2][VW], dv[2][VW];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      Access<T, VW>::load(xr + h + u * st, xv[u], pol);
      Access<T, VW>::load(dr + h + u * st, dv[u], pol);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) acc_grad<VW>(xv[u], dv[u], mu, s1, s2);
  }
  for (; h < k.h1; h += st) {
    const uint64_t pol = h >= keep ? plast : pfirst;
    float xv[VW], dv[VW];
    Access<T, VW>::load(xr + h, xv, pol);
    Access<T, VW>::load(dr + h, dv, pol);
    acc_grad<VW>(xv, dv, mu, s1, s2);
  }
  publish_chunk<T, true>(p, k, s1, s2, sm);
}

// Forward pass 2 of one chunk, last vector to first.  grp (fin2 plans): the
// chunk's group (mean, rstd) in shared memory.
template <typename T, int VW>
__device__ __forceinline__ void apply_chunk(const KParams& p, int64_t item, const float2* grp) {
  const Geom& g = p.g;
  const int tid = threadIdx.x;
  const uint64_t pol = policy_evict_first();
  const Chunk k = chunk_of(g, item);
  if (k.h0 >= k.h1) return;
  const int64_t n = k.row / g.C, c = k.row % g.C, ng = n * g.G + c / g.Cg;
  // mean/rstd may have been written earlier in this launch: coherent loads
  const float2 mr = grp ? grp[0] : make_float2(__ldcg(p.mean + ng), __ldcg(p.rstd + ng));
  const float r = mr.y, mu = mr.x;
  const float a = p.gamma ? r * __ldg(p.gamma + c) : r;
  const float b = p.beta ? __ldg(p.beta + c) : 0.f;
  const T* xr = static_cast<const T*>(p.x) + plane_offset(g, k.row, p.xs_n, p.xs_r) + k.h0;
  T* yr = static_cast<T*>(p.out) + plane_offset(g, k.row, p.os_n, p.os_r) + k.h0;
  const int64_t nv = (k.h1 - k.h0) / VW;
  const int64_t st = blockDim.x;
  int64_t i = nv - 1 - tid;
  for (; i - 3 * st >= 0; i -= 4 * st) {
    float v[4][VW];
#pragma unroll
    for (int u = 0; u < 4; ++u) Access<T, VW>::load(xr + (i - u * st) * VW, v[u], pol);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll
      for (int e = 0; e < VW; ++e) v[u][e] = fmaf(v[u][e] - mu, a, b);
      Access<T, VW>::store(yr + (i - u * st) * VW, v[u], pol);
    }
  }
  for (; i >= 0; i -= st) {
    float v[VW];
    Access<T, VW>::load(xr + i * VW, v, pol);
#pragma unroll
    for (int e = 0; e < VW; ++e) v[e] = fmaf(v[e] - mu, a, b);
    Access<T, VW>::store(yr + i * VW, v, pol);
  }
}

// Backward pass 2 of one chunk, last vector to first.  grp (fin2 plans): the
// chunk's group (B, D) in shared memory.
template <typename T, int VW>
__device__ __forceinline__ void dx_chunk(const KParams& p, int64_t item, const float2* grp) {
  const Geom& g = p.g;
  const int tid = threadIdx.x;
  const uint64_t pol = policy_evict_first();
  const Chunk k = chunk_of(g, item);
  if (k.h0 >= k.h1) return;
  const int64_t n = k.row / g.C, c = k.row % g.C, ng = n * g.G + c / g.Cg;
  const float r = __ldg(p.rstd + ng), mu = __ldg(p.mean + ng);
  const float A = p.gamma ? r * __ldg(p.gamma + c) : r;
  const float2 cf = grp ? grp[0] : __ldcg(p.coef + ng);
  const T* xr = static_cast<const T*>(p.x) + plane_offset(g, k.row, p.xs_n, p.xs_r) + k.h0;
  const T* dr = static_cast<const T*>(p.dy) + plane_offset(g, k.row, p.ds_n, p.ds_r) + k.h0;
  T* outr = static_cast<T*>(p.out) + plane_offset(g, k.row, p.os_n, p.os_r) + k.h0;
  const int64_t nv = (k.h1 - k.h0) / VW;
  const int64_t st = blockDim.x;
  int64_t i = nv - 1 - tid;
  for (; i - st >= 0; i -= 2 * st) {
    float xv[2][VW], dv[2][VW];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      Access<T, VW>::load(xr + (i - u * st) * VW, xv[u], pol);
      Access<T, VW>::load(dr + (i - u * st) * VW, dv[u], pol);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
#pragma unroll
      for (int e = 0; e < VW; ++e) xv[u][e] = fmaf(A, dv[u][e], fmaf(cf.x, xv[u][e] - mu, cf.y));
      Access<T, VW>::store(outr + (i - u * st) * VW, xv[u], pol);
    }
  }
  for (; i >= 0; i -= st) {
    float xv[VW], dv[VW];
    Access<T, VW>::load(xr + i * VW, xv, pol);
    Access<T, VW>::load(dr + i * VW, dv, pol);
#pragma unroll
    for (int e = 0; e < VW; ++e) xv[e] = fmaf(A, dv[e], fmaf(cf.x, xv[e] - mu, cf.y));
    Access<T, VW>::store(outr + i * VW, xv, pol);
  }
}

// ------------------------------------------------------- mode 1 (row blocks)
struct RowBlock {
  int64_t n, c0, c1;
};
__device__ __forceinline__ RowBlock rows_of(const Geom& g, int64_t item) {
  RowBlock b;
  b.n = item / g.items_per_n;
  b.c0 = (item % g.items_per_n) * g.RB;
  b.c1 = (b.c0 + g.RB < g.C) ? b.c0 + g.RB : g.C;
  return b;
}

template <typename T, int VW>
__device__ __forceinline__ void stats_rows(const KParams& p, int64_t item, float* sm) {
  const Geom& g = p.g;
  const RowBlock rb = rows_of(g, item);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const uint64_t pol = g.keep_from == 0 ? policy_evict_last() : policy_evict_first();
  for (int64_t c = rb.c0 + warp; c < rb.c1; c += nwarps) {
    const int64_t row = rb.n * g.C + c;
    const T* xr = static_cast<const T*>(p.x) + rb.n * p.xs_n + c * p.xs_r;
    const float K = Elem<T>::to_f(xr[0]);
    if (g.fin2 && lane == 0) p.kst[row] = K;  // for the second kernel
    float s = 0.f, q = 0.f;
    for (int64_t h = (int64_t)lane * VW; h < g.HW; h += 32 * VW) {
      float v[VW];
      Access<T, VW>::load(xr + h, v, pol);
      acc_shifted<VW>(v, K, s, q);
    }
    s = warp_sum_lane0(s);
    q = warp_sum_lane0(q);
    if (lane == 0) p.part[row] = make_float2(s, q);
  }
  if (!g.fin2)
    arrive_and_finalize<T, false>(p, unit_of(p, rb.n, 0), 0, 1, [] {}, sm, nchw_smem_floats(g));
}

template <typename T, int VW>
__device__ __forceinline__ void reduce_rows(const KParams& p, int64_t item, float* sm) {
  const Geom& g = p.g;
  const RowBlock rb = rows_of(g, item);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const uint64_t pol = g.keep_from == 0 ? policy_evict_last() : policy_evict_first();
  for (int64_t c = rb.c0 + warp; c < rb.c1; c += nwarps) {
    const int64_t row = rb.n * g.C + c;
    const float mu = __ldg(p.mean + rb.n * g.G + c / g.Cg);
    const T* xr = static_cast<const T*>(p.x) + rb.n * p.xs_n + c * p.xs_r;
    const T* dr = static_cast<const T*>(p.dy) + rb.n * p.ds_n + c * p.ds_r;
    float s1 = 0.f, s2 = 0.f;
    for (int64_t h = (int64_t)lane * VW; h < g.HW; h += 32 * VW) {
      float xv[VW], dv[VW];
      Access<T, VW>::load(xr + h, xv, pol);
      Access<T, VW>::load(dr + h, dv, pol);
      acc_grad<VW>(xv, dv, mu, s1, s2);
    }
    s1 = warp_sum_lane0(s1);
    s2 = warp_sum_lane0(s2);
    if (lane == 0) p.part[row] = make_float2(s1, s2);
  }
  if (!g.fin2)
    arrive_and_finalize<T, true>(p, unit_of(p, rb.n, 0), 0, 1, [] {}, sm, nchw_smem_floats(g));
}

// grp (fin2 plans): (mean, rstd) of groups g0, g0 + 1, ... in shared memory.
template <typename T, int VW>
__device__ __forceinline__ void apply_rows(const KParams& p, int64_t item, const float2* grp,
                                           int64_t g0) {
  const Geom& g = p.g;
  const RowBlock rb = rows_of(g, item);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const uint64_t pol = policy_evict_first();
  for (int64_t c = rb.c0 + warp; c < rb.c1; c += nwarps) {
    const int64_t ng = rb.n * g.G + c / g.Cg;
    const float2 mr = grp ? grp[c / g.Cg - g0] : make_float2(__ldcg(p.mean + ng), __ldcg(p.rstd + ng));
    const float r = mr.y, mu = mr.x;
    const float a = p.gamma ? r * __ldg(p.gamma + c) : r;
    const float b = p.beta ? __ldg(p.beta + c) : 0.f;
    const T* xr = static_cast<const T*>(p.x) + rb.n * p.xs_n + c * p.xs_r;
    T* yr = static_cast<T*>(p.out) + rb.n * p.os_n + c * p.os_r;
    for (int64_t h = (int64_t)lane * VW; h < g.HW; h += 32 * VW) {
      float v[VW];
      Access<T, VW>::load(xr + h, v, pol);
#pragma unroll
      for (int e = 0; e < VW; ++e) v[e] = fmaf(v[e] - mu, a, b);
      Access<T, VW>::store(yr + h, v, pol);
    }
  }
}

// grp (fin2 plans): (B, D) of groups g0, g0 + 1, ... in shared memory.
template <typename T, int VW>
__device__ __forceinline__ void dx_rows(const KParams& p, int64_t item, const float2* grp,
                                        int64_t g0) {
  const Geom& g = p.g;
  const RowBlock rb = rows_of(g, item);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const uint64_t pol = policy_evict_first();
  for (int64_t c = rb.c0 + warp; c < rb.c1; c += nwarps) {
    const int64_t ng = rb.n * g.G + c / g.Cg;
    const float r = __ldg(p.rstd + ng), mu = __ldg(p.mean + ng);
    const float A = p.gamma ? r * __ldg(p.gamma + c) : r;
    const float2 cf = grp ? grp[c / g.Cg - g0] : __ldcg(p.coef + ng);
    const T* xr = static_cast<const T*>(p.x) + rb.n * p.xs_n + c * p.xs_r;
    const T* dr = static_cast<const T*>(p.dy) + rb.n * p.ds_n + c * p.ds_r;
    T* outr = static_cast<T*>(p.out) + rb.n * p.os_n + c * p.os_r;
    for (int64_t h = (int64_t)lane * VW; h < g.HW; h += 32 * VW) {
      float xv[VW], dv[VW];
      Access<T, VW>::load(xr + h, xv, pol);
      Access<T, VW>::load(dr + h, dv, pol);
#pragma unroll
      for (int e = 0; e < VW; ++e) xv[e] = fmaf(A, dv[e], fmaf(cf.x, xv[e] - mu, cf.y));
      Access<T, VW>::store(outr + h, xv, pol);
    }
  }
}

// ------------------------------------------------------- two-kernel kernels
template <typename T, int VW>
__global__ void __launch_bounds__(512) nchw_fwd_stats(const __grid_constant__ KParams p) {
  grid_dependency_wait();  // the previous kernel's results (and x, dy) are complete
  grid_launch_dependents();
  extern __shared__ __align__(16) float sm[];
  if (p.g.mode == 0)
    stats_chunk<T, VW>(p, blockIdx.x, sm);
  else
    stats_rows<T, VW>(p, blockIdx.x, sm);
}

// fin2 plans: the channels a second-kernel item finalises (its plane's group,
// or its block of planes extended to whole groups) and the groups whose
// mean/rstd it writes (each group by the item holding its first plane's
// first chunk).
struct Fin2Range {
  int64_t n, ca, cb, wa, wb;
};
__device__ __forceinline__ Fin2Range nchw_fin2_range(const Geom& g, int64_t item) {
  Fin2Range r;
  if (g.mode == 0) {
    const Chunk k = chunk_of(g, item);
    const int64_t c = k.row % g.C, gi = c / g.Cg;
    r.n = k.row / g.C;
    r.ca = gi * g.Cg;
    r.cb = r.ca + g.Cg;
    const bool writer = k.ch == 0 && c == r.ca;
    r.wa = writer ? gi : 0;
    r.wb = writer ? gi + 1 : 0;
  } else {
    const RowBlock b = rows_of(g, item);
    r.n = b.n;
    r.ca = b.c0 / g.Cg * g.Cg;
    r.cb = (b.c1 + g.Cg - 1) / g.Cg * g.Cg;
    r.wa = (b.c0 + g.Cg - 1) / g.Cg;
    r.wb = (b.c1 + g.Cg - 1) / g.Cg;
  }
  return r;
}

// Dynamic shared memory of the second kernels, in bytes.
inline size_t second_smem(const Geom& g, bool bwd) {
  const int64_t f = fin2_smem_floats(g);
  const int64_t params = bwd ? 2 * (int64_t)g.tpb : 0;  // finalize_params scratch
  return sizeof(float) * (size_t)(f > params ? f : params);
}

template <typename T, int VW>
__global__ void __launch_bounds__(512) nchw_fwd_apply(const __grid_constant__ KParams p) {
  extern __shared__ __align__(16) float sm[];
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t item = p.g.items - 1 - (int64_t)blockIdx.x;
  const float2* grp = nullptr;
  int64_t g0 = 0;
  if (p.g.fin2) {
    const Fin2Range r = nchw_fin2_range(p.g, item);
    grp = fin2_groups<false>(p, r.n, r.ca, r.cb, r.wa, r.wb, sm);
    g0 = r.ca / p.g.Cg;
  }
  if (p.g.mode == 0)
    apply_chunk<T, VW>(p, item, grp);
  else
    apply_rows<T, VW>(p, item, grp, g0);
}

template <typename T, int VW>
__global__ void __launch_bounds__(512) nchw_bwd_reduce(const __grid_constant__ KParams p) {
  grid_dependency_wait();
  grid_launch_dependents();
  extern __shared__ __align__(16) float sm[];
  if (p.g.mode == 0)
    reduce_chunk<T, VW>(p, blockIdx.x, sm);
  else
    reduce_rows<T, VW>(p, blockIdx.x, sm);
}

template <typename T, int VW>
__global__ void __launch_bounds__(512) nchw_bwd_dx(const __grid_constant__ KParams p) {
  extern __shared__ __align__(16) float sm[];
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t item = p.g.items - 1 - (int64_t)blockIdx.x;
  const float2* grp = nullptr;
  int64_t g0 = 0;
  if (p.g.fin2) {
    const Fin2Range r = nchw_fin2_range(p.g, item);
    grp = fin2_groups<true>(p, r.n, r.ca, r.cb, 0, 0, sm);
    g0 = r.ca / p.g.Cg;
  } else if (blockIdx.x == 0) {
    // the first CTA adds up dgamma / dbeta: every channel's sums are
    // complete once the first kernel is
    finalize_params(p, sm);
  }
  if (p.g.mode == 0)
    dx_chunk<T, VW>(p, item, grp);
  else
    dx_rows<T, VW>(p, item, grp, g0);
}

// The pipelined regime (schedule in gn_tasks.cuh): a unit is one (sample n,
// group), its pieces the segments of its Cg planes (piece q: plane
// group*Cg + q/T, segment q%T), piece q of every unit streamed by CTA q in
// chunks of g.chunk elements; thread t takes the chunk's 16-byte vectors t,
// t + blockDim.x, ...  A pass-1 piece leaves one record (its shifted sums, or
// sum(dy) and sum(dy*(x - mean))); the unit's finaliser merges the Cg*T
// records as the two-kernel path does and publishes (mean, rstd) or (B, D).
template <typename T, int VW, bool kBwd>
__global__ void __launch_bounds__(512, 1) nchw_pipelined(const __grid_constant__ KParams p) {
  extern __shared__ __align__(128) char smem_raw[];
  char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const Geom& g = p.g;
  const RingSmem R = ring_smem(g, smem);
  float* sm = reinterpret_cast<float*>(smem + g.off_red);
  const int64_t sm_floats = nchw_smem_floats(g);
  unsigned long long* rec = reinterpret_cast<unsigned long long*>(p.ready);
  const int tid = threadIdx.x, nt = blockDim.x;
  float s1 = 0.f, s2 = 0.f, K = 0.f;               // pass-1 sums; shift (fwd) or mean (bwd)
  float ca = 0.f, cb = 0.f, cc = 0.f, cmu = 0.f;   // pass-2 constants
  bool ok = false;
  // piece of task t: plane a (channel e) of sample unit / G, segment b = [c, d)
  auto describe = [&](const Task& t, SlotHdr& h) {
    const int64_t n = t.unit / g.G, grp = t.unit % g.G;
    const int64_t plane = grp * g.Cg + t.piece / g.T, seg = t.piece % g.T;
    h.a = n * g.C + plane;
    h.b = seg;
    h.c = seg * g.L;
    h.d = (h.c + g.L < g.HW) ? h.c + g.L : g.HW;
    h.e = plane;
    h.nchunks = (int32_t)((h.d - h.c + g.chunk - 1) / g.chunk);
    // pass 1 brings along its shift: the plane's first element (forward) or
    // the group's mean (backward, when mean is 16-byte aligned)
    h.aux_off = 0;
    if (t.pass == 1) {
      if (!kBwd)
        h.aux_off = reinterpret_cast<int64_t>(static_cast<const T*>(p.x) + h.a * g.HW);
      else if ((reinterpret_cast<uintptr_t>(p.mean) & 15) == 0)
        h.aux_off = reinterpret_cast<int64_t>(p.mean + (t.unit & ~int64_t(3)));
    }
  };
  auto chunk_off = [&](const SlotHdr& h, int c, int32_t* bytes) {
    const int64_t e0 = h.c + (int64_t)c * g.chunk;
    *bytes = (int32_t)(((h.d - e0 < g.chunk) ? h.d - e0 : g.chunk) * (int64_t)sizeof(T));
    return h.a * g.HW + e0;
  };
  // finalisation of unit u by its designated CTA
  auto fin = [&](int64_t u) {
    const int64_t n = u / g.G, c0 = (u % g.G) * g.Cg;
    if (kBwd)
      finalize_bwd(p, n, c0, c0 + g.Cg, sm, sm_floats);
    else
      finalize_fwd<T>(p, n, c0, c0 + g.Cg, sm, sm_floats);
    __threadfence();
    __syncthreads();
    __shared__ int s_last;
    if (tid == 0) {
      atomicExch(p.tickets + u, 0u);
      if (kBwd) {
        const float2 cf = p.coef[u];
        put_record(rec + u, cf.x, cf.y);
        s_last = publish_and_arrive(p.tickets + g.units_fin, (unsigned)g.units_fin);
      } else {
        put_record(rec + u, p.mean[u], p.rstd[u]);
      }
    }
    if (!kBwd) return;
    __syncthreads();
    if (!s_last) return;
    finalize_params(p, sm);  // the last unit: dgamma, dbeta
    if (tid == 0) atomicExch(p.tickets + g.units_fin, 0u);
  };
  auto out_at = [&](const SlotHdr& h) {
    return static_cast<T*>(p.out) + h.a * g.HW + h.c + (int64_t)h.chunk * g.chunk;
  };
  auto consume = [&](const SlotHdr& h, char* sx, const char* sd) {
    const int c = h.chunk, nc = h.nchunks, bytes = h.bytes;
    if (c == 0 && (h.pass == 1 || h.step >= g.units_fin)) finalize_due(p, h.step, fin);
    const int64_t ch = h.e, ng = h.unit;
    const int nv = bytes / 16;
    uint4* vx = reinterpret_cast<uint4*>(sx);
    const uint4* vd = reinterpret_cast<const uint4*>(sd);
    if (h.pass == 1) {
      if (c == 0) {
        s1 = s2 = 0.f;
        if (!kBwd)
          K = Elem<T>::to_f(reinterpret_cast<const T*>(&h.aux)[0]);
        else
          K = h.aux_off ? reinterpret_cast<const float*>(&h.aux)[ng & 3] : __ldg(p.mean + ng);
      }
#pragma unroll 4
      for (int v = tid; v < nv; v += nt) {
        float xv[VW];
        Access<T, VW>::unpack(vx[v], xv);
        if (kBwd) {
          float dv[VW];
          Access<T, VW>::unpack(vd[v], dv);
          acc_grad<VW>(xv, dv, K, s1, s2);
        } else {
          acc_shifted<VW>(xv, K, s1, s2);
        }
      }
      if (c == nc - 1) {
        const float2 tot = block_sum2_t0(s1, s2, sm);
        if (tid == 0) {
          p.part[h.a * g.T + h.b] = tot;
          arrive_release(p, ng);
        }
      }
      return false;
    }
    if (c == 0) {
      float lo, hi;
      if (kBwd) {  // inputs: loaded before the wait, so the two latencies overlap
        const float r = __ldg(p.rstd + ng);
        ca = p.gamma ? r * __ldg(p.gamma + ch) : r;
        cmu = __ldg(p.mean + ng);
      } else {
        ca = p.gamma ? __ldg(p.gamma + ch) : 1.f;
        cb = p.beta ? __ldg(p.beta + ch) : 0.f;
      }
      ok = wait_record(rec + ng, p.err, &lo, &hi);
      if (kBwd) {
        cb = lo;
        cc = hi;
      } else {
        cmu = lo;
        ca *= hi;  // rstd * gamma
      }
    }
    if (ok) {  // the output replaces x in the slot; thread 0 stores it
#pragma unroll 4
      for (int v = tid; v < nv; v += nt) {
        float xv[VW];
        Access<T, VW>::unpack(vx[v], xv);
        if (kBwd) {
          float dv[VW];
          Access<T, VW>::unpack(vd[v], dv);
#pragma unroll
          for (int e = 0; e < VW; ++e) xv[e] = fmaf(ca, dv[e], fmaf(cb, xv[e] - cmu, cc));
        } else {
#pragma unroll
          for (int e = 0; e < VW; ++e) xv[e] = fmaf(xv[e] - cmu, ca, cb);
        }
        vx[v] = Access<T, VW>::pack(xv);
      }
    }
    return ok;
  };
  run_ring<kBwd>(p, R, describe, chunk_off, consume, out_at);
}

template <typename T, int VW>
cudaError_t run_op(const KParams& p, cudaStream_t s, bool bwd) {
  const Geom& g = p.g;
  const size_t sm1 = sizeof(float) * nchw_smem_floats(g);
  const TimingEvents& ev = timing_events();
  cudaError_t e = bwd ? launch_pdl(nchw_bwd_reduce<T, VW>, g.items, g.tpb, sm1, s, p)
                      : launch_pdl(nchw_fwd_stats<T, VW>, g.items, g.tpb, sm1, s, p);
  if (e != cudaSuccess) return e;
  if (ev.mid) cudaEventRecord(ev.mid, s);
  e = bwd ? launch_pdl(nchw_bwd_dx<T, VW>, g.items, g.tpb, second_smem(g, true), s, p)
          : launch_pdl(nchw_fwd_apply<T, VW>, g.items, g.tpb, second_smem(g, false), s, p);
  if (ev.end) cudaEventRecord(ev.end, s);
  return e;
}

template <typename T>
cudaError_t dispatch_vw(const KParams& p, cudaStream_t s, bool bwd) {
  return p.g.vw == 1 ? run_op<T, 1>(p, s, bwd) : run_op<T, Elem<T>::VEC>(p, s, bwd);
}

template <typename T, int VW>
const void* kernel_t(const Geom& g, bool bwd, int second, size_t* smem) {
  *smem = second ? second_smem(g, bwd) : sizeof(float) * nchw_smem_floats(g);
  if (second) return bwd ? (const void*)nchw_bwd_dx<T, VW> : (const void*)nchw_fwd_apply<T, VW>;
  return bwd ? (const void*)nchw_bwd_reduce<T, VW> : (const void*)nchw_fwd_stats<T, VW>;
}

template <typename T>
const void* kernel_vw(const Geom& g, bool bwd, int second, size_t* smem) {
  return g.vw == 1 ? kernel_t<T, 1>(g, bwd, second, smem)
                   : kernel_t<T, Elem<T>::VEC>(g, bwd, second, smem);
}

template <typename T>
const void* pipelined_t(const Geom& g, bool bwd, size_t* smem) {
  *smem = g.smem;
  constexpr int V = Elem<T>::VEC;
  return bwd ? (const void*)nchw_pipelined<T, V, true> : (const void*)nchw_pipelined<T, V, false>;
}

}  // namespace

const void* nchw_kernel(const Geom& g, bool bwd, int second, size_t* smem) {
  switch (g.dtype) {
    case kF32: return kernel_vw<float>(g, bwd, second, smem);
    case kF16: return kernel_vw<__half>(g, bwd, second, smem);
    case kF64: return kernel_vw<double>(g, bwd, second, smem);
    default: return kernel_vw<__nv_bfloat16>(g, bwd, second, smem);
  }
}

cudaError_t launch_nchw(const KParams& p, cudaStream_t s, bool bwd) {
  switch (p.g.dtype) {
    case kF32: return dispatch_vw<float>(p, s, bwd);
    case kF16: return dispatch_vw<__half>(p, s, bwd);
    case kF64: return dispatch_vw<double>(p, s, bwd);
    default: return dispatch_vw<__nv_bfloat16>(p, s, bwd);
  }
}

// Reduction scratch of the pipelined kernel (floats): the CTA sums and the
// per-channel staging of the finalisation.
int64_t nchw_pipelined_scratch_floats(const Geom& g) { return nchw_smem_floats(g); }

// The pipelined kernel of a plan (16-byte vectors only).
const void* nchw_pipelined_kernel(const Geom& g, bool bwd, size_t* smem) {
  switch (g.dtype) {
    case kF32: return pipelined_t<float>(g, bwd, smem);
    case kF16: return pipelined_t<__half>(g, bwd, smem);
    case kF64: return nullptr;  // f64 runs on the two-kernel path only
    default: return pipelined_t<__nv_bfloat16>(g, bwd, smem);
  }
}

cudaError_t launch_nchw_pipelined(const KParams& p, cudaStream_t s, bool bwd) {
  size_t smem = 0;
  const void* k = nchw_pipelined_kernel(p.g, bwd, &smem);
  return launch_cooperative(k, p, smem, s);
}

}  // namespace gn
