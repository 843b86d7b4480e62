// gn_nchw.cu -- two-kernel GroupNorm path for NCHW activations.
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
// As in gn_nhwc.cu, the last arrival of a sample finalises it, and the
// elementwise second kernels walk the items (and the elements of a chunk) in
// reverse order, starting on the data the first kernel left in L2.
#include "gn_finalize.cuh"

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

// Mode-0 tail of the first kernels: CTA sum, the chunk's record, the arrival
// chain (group of l1 chunks of the row, then the sample).
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
  arrive_and_finalize<T, kBwd>(p, k.row / g.C, k.row * g.Tp + t1, gsize, merge, sm,
                               nchw_smem_floats(g));
}

// ------------------------------------------------------------------ forward
template <typename T, int VW>
__global__ void __launch_bounds__(512) nchw_fwd_stats(const __grid_constant__ KParams p) {
  grid_dependency_wait();  // the previous kernel's results (and x, dy) are complete
  grid_launch_dependents();
  extern __shared__ float sm[];
  const Geom& g = p.g;
  const int tid = threadIdx.x;
  const T* x = static_cast<const T*>(p.x);
  const uint64_t pfirst = policy_evict_first(), plast = policy_evict_last();
  if (g.mode == 0) {
    const Chunk k = chunk_of(g, blockIdx.x);
    const T* xr = x + k.row * g.HW;
    const float K = Elem<T>::to_f(xr[0]);
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
  } else {
    const int64_t item = blockIdx.x;
    const int64_t n = item / g.items_per_n;
    const int64_t c0 = (item % g.items_per_n) * g.RB;
    const int64_t c1 = (c0 + g.RB < g.C) ? c0 + g.RB : g.C;
    const int lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const uint64_t pol = g.keep_from == 0 ? plast : pfirst;
    for (int64_t c = c0 + warp; c < c1; c += nwarps) {
      const int64_t row = n * g.C + c;
      const T* xr = x + row * g.HW;
      const float K = Elem<T>::to_f(xr[0]);
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
    arrive_and_finalize<T, false>(p, n, 0, 1, [] {}, sm, nchw_smem_floats(g));
  }
}

template <typename T, int VW>
__global__ void __launch_bounds__(512) nchw_fwd_apply(const __grid_constant__ KParams p) {
  grid_dependency_wait();  // the previous kernel's results (and x, dy) are complete
  grid_launch_dependents();
  const Geom& g = p.g;
  const int tid = threadIdx.x;
  const T* x = static_cast<const T*>(p.x);
  T* y = static_cast<T*>(p.out);
  const uint64_t pol = policy_evict_first();
  const int64_t item = g.items - 1 - (int64_t)blockIdx.x;
  if (g.mode == 0) {
    const Chunk k = chunk_of(g, item);
    if (k.h0 >= k.h1) return;
    const int64_t n = k.row / g.C, c = k.row % g.C, ng = n * g.G + c / g.Cg;
    const float r = __ldg(p.rstd + ng), mu = __ldg(p.mean + ng);
    const float a = p.gamma ? r * __ldg(p.gamma + c) : r;
    const float b = p.beta ? __ldg(p.beta + c) : 0.f;
    const T* xr = x + k.row * g.HW + k.h0;
    T* yr = y + k.row * g.HW + k.h0;
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
  } else {
    const int64_t n = item / g.items_per_n;
    const int64_t c0 = (item % g.items_per_n) * g.RB;
    const int64_t c1 = (c0 + g.RB < g.C) ? c0 + g.RB : g.C;
    const int lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    for (int64_t c = c0 + warp; c < c1; c += nwarps) {
      const int64_t row = n * g.C + c, ng = n * g.G + c / g.Cg;
      const float r = __ldg(p.rstd + ng), mu = __ldg(p.mean + ng);
      const float a = p.gamma ? r * __ldg(p.gamma + c) : r;
      const float b = p.beta ? __ldg(p.beta + c) : 0.f;
      const T* xr = x + row * g.HW;
      T* yr = y + row * g.HW;
      for (int64_t h = (int64_t)lane * VW; h < g.HW; h += 32 * VW) {
        float v[VW];
        Access<T, VW>::load(xr + h, v, pol);
#pragma unroll
        for (int e = 0; e < VW; ++e) v[e] = fmaf(v[e] - mu, a, b);
        Access<T, VW>::store(yr + h, v, pol);
      }
    }
  }
}

// ----------------------------------------------------------------- backward
template <typename T, int VW>
__global__ void __launch_bounds__(512) nchw_bwd_reduce(const __grid_constant__ KParams p) {
  grid_dependency_wait();  // the previous kernel's results (and x, dy) are complete
  grid_launch_dependents();
  extern __shared__ float sm[];
  const Geom& g = p.g;
  const int tid = threadIdx.x;
  const T* x = static_cast<const T*>(p.x);
  const T* dy = static_cast<const T*>(p.dy);
  const uint64_t pfirst = policy_evict_first(), plast = policy_evict_last();
  if (g.mode == 0) {
    const Chunk k = chunk_of(g, blockIdx.x);
    const int64_t n = k.row / g.C;
    const float mu = __ldg(p.mean + n * g.G + (k.row % g.C) / g.Cg);
    const T* xr = x + k.row * g.HW;
    const T* dr = dy + k.row * g.HW;
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
  } else {
    const int64_t item = blockIdx.x;
    const int64_t n = item / g.items_per_n;
    const int64_t c0 = (item % g.items_per_n) * g.RB;
    const int64_t c1 = (c0 + g.RB < g.C) ? c0 + g.RB : g.C;
    const int lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const uint64_t pol = g.keep_from == 0 ? plast : pfirst;
    for (int64_t c = c0 + warp; c < c1; c += nwarps) {
      const int64_t row = n * g.C + c;
      const float mu = __ldg(p.mean + n * g.G + c / g.Cg);
      const T* xr = x + row * g.HW;
      const T* dr = dy + row * g.HW;
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
    arrive_and_finalize<T, true>(p, n, 0, 1, [] {}, sm, nchw_smem_floats(g));
  }
}

template <typename T, int VW>
__global__ void __launch_bounds__(512) nchw_bwd_dx(const __grid_constant__ KParams p) {
  grid_dependency_wait();  // the previous kernel's results (and x, dy) are complete
  grid_launch_dependents();
  const Geom& g = p.g;
  const int tid = threadIdx.x;
  const T* x = static_cast<const T*>(p.x);
  const T* dy = static_cast<const T*>(p.dy);
  T* dx = static_cast<T*>(p.out);
  const uint64_t pol = policy_evict_first();
  const int64_t item = g.items - 1 - (int64_t)blockIdx.x;
  if (g.mode == 0) {
    const Chunk k = chunk_of(g, item);
    if (k.h0 >= k.h1) return;
    const int64_t n = k.row / g.C, c = k.row % g.C, ng = n * g.G + c / g.Cg;
    const float r = __ldg(p.rstd + ng), mu = __ldg(p.mean + ng);
    const float A = p.gamma ? r * __ldg(p.gamma + c) : r;
    const float2 cf = __ldcg(p.coef + ng);
    const T* xr = x + k.row * g.HW + k.h0;
    const T* dr = dy + k.row * g.HW + k.h0;
    T* outr = dx + k.row * g.HW + k.h0;
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
  } else {
    const int64_t n = item / g.items_per_n;
    const int64_t c0 = (item % g.items_per_n) * g.RB;
    const int64_t c1 = (c0 + g.RB < g.C) ? c0 + g.RB : g.C;
    const int lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    for (int64_t c = c0 + warp; c < c1; c += nwarps) {
      const int64_t row = n * g.C + c, ng = n * g.G + c / g.Cg;
      const float r = __ldg(p.rstd + ng), mu = __ldg(p.mean + ng);
      const float A = p.gamma ? r * __ldg(p.gamma + c) : r;
      const float2 cf = __ldcg(p.coef + ng);
      const T* xr = x + row * g.HW;
      const T* dr = dy + row * g.HW;
      T* outr = dx + row * g.HW;
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
}

template <typename T, int VW>
cudaError_t run_op(const KParams& p, cudaStream_t s, bool bwd) {
  const Geom& g = p.g;
  const size_t sm1 = sizeof(float) * nchw_smem_floats(g);
  const TimingEvents& ev = timing_events();
  if (ev.begin) cudaEventRecord(ev.begin, s);
  cudaError_t e = bwd ? launch_pdl(nchw_bwd_reduce<T, VW>, g.items, g.tpb, sm1, s, p)
                      : launch_pdl(nchw_fwd_stats<T, VW>, g.items, g.tpb, sm1, s, p);
  if (e != cudaSuccess) return e;
  if (ev.mid) cudaEventRecord(ev.mid, s);
  e = bwd ? launch_pdl(nchw_bwd_dx<T, VW>, g.items, g.tpb, 0, s, p)
          : launch_pdl(nchw_fwd_apply<T, VW>, g.items, g.tpb, 0, s, p);
  if (ev.end) cudaEventRecord(ev.end, s);
  return e;
}

template <typename T>
cudaError_t dispatch_vw(const KParams& p, cudaStream_t s, bool bwd) {
  return p.g.vw == 1 ? run_op<T, 1>(p, s, bwd) : run_op<T, Elem<T>::VEC>(p, s, bwd);
}

template <typename T, int VW>
const void* kernel_t(const Geom& g, bool bwd, int second, size_t* smem) {
  *smem = second ? 0 : sizeof(float) * nchw_smem_floats(g);
  if (second) return bwd ? (const void*)nchw_bwd_dx<T, VW> : (const void*)nchw_fwd_apply<T, VW>;
  return bwd ? (const void*)nchw_bwd_reduce<T, VW> : (const void*)nchw_fwd_stats<T, VW>;
}

template <typename T>
const void* kernel_vw(const Geom& g, bool bwd, int second, size_t* smem) {
  return g.vw == 1 ? kernel_t<T, 1>(g, bwd, second, smem)
                   : kernel_t<T, Elem<T>::VEC>(g, bwd, second, smem);
}

}  // namespace

const void* nchw_kernel(const Geom& g, bool bwd, int second, size_t* smem) {
  switch (g.dtype) {
    case kF32: return kernel_vw<float>(g, bwd, second, smem);
    case kF16: return kernel_vw<__half>(g, bwd, second, smem);
    default: return kernel_vw<__nv_bfloat16>(g, bwd, second, smem);
  }
}

cudaError_t launch_nchw(const KParams& p, cudaStream_t s, bool bwd) {
  switch (p.g.dtype) {
    case kF32: return dispatch_vw<float>(p, s, bwd);
    case kF16: return dispatch_vw<__half>(p, s, bwd);
    default: return dispatch_vw<__nv_bfloat16>(p, s, bwd);
  }
}

}  // namespace gn
