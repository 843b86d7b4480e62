// gn_nchw.cu -- GroupNorm kernels for NCHW activations.
//
// Memory: element (n, c, hw) sits at (n*C + c)*HW + hw, so each (n, c)
// channel plane ("row") is HW contiguous elements and a group is Cg
// consecutive planes.  Two item shapes:
//   mode 0 (large planes): item = (row, chunk of L elements); the whole CTA
//          strides the chunk with 16-byte loads; one partial per item.
//   mode 1 (small planes): item = RB consecutive rows of one sample; each warp
//          takes whole rows; one partial per row.
// The kernels mirror gn_nhwc.cu: stats/reduce kernels publish per-(n, c,
// chunk) partial sums and the last CTA of a sample finalises it; apply/dx
// kernels walk the items in reverse order.
#include "gn_finalize.cuh"

namespace gn {
namespace {

template <typename T, int VW>
__device__ __forceinline__ void acc_shifted(const float (&v)[VW], float K, float& s, float& q) {
#pragma unroll
  for (int k = 0; k < VW; ++k) {
    const float d = v[k] - K;
    s += d;
    q = fmaf(d, d, q);
  }
}

template <typename T, int VW>
__device__ __forceinline__ void acc_grad(const float (&xv)[VW], const float (&dv)[VW], float mu,
                                         float& s1, float& s2) {
#pragma unroll
  for (int k = 0; k < VW; ++k) {
    s1 += dv[k];
    s2 = fmaf(dv[k], xv[k] - mu, s2);
  }
}

// ------------------------------------------------------------------ forward
template <typename T, int VW>
__global__ void __launch_bounds__(512) nchw_fwd_stats(const __grid_constant__ KParams p) {
  extern __shared__ float sm[];
  const Geom& g = p.g;
  const int tid = threadIdx.x;
  const T* x = static_cast<const T*>(p.x);
  const uint64_t pol = policy_evict_last();
  int64_t n;
  if (g.mode == 0) {
    const int64_t item = blockIdx.x;
    const int64_t row = item / g.T, ch = item % g.T;
    n = row / g.C;
    const T* xr = x + row * g.HW;
    const int64_t h0 = ch * g.L;
    const int64_t h1 = (h0 + g.L < g.HW) ? h0 + g.L : g.HW;
    const float K = Elem<T>::to_f(xr[0]);
    float s = 0.f, q = 0.f;
    const int64_t st = (int64_t)blockDim.x * VW;
    int64_t h = h0 + (int64_t)tid * VW;
    for (; h + 3 * st < h1; h += 4 * st) {
      float v[4][VW];
#pragma unroll
      for (int u = 0; u < 4; ++u) Access<T, VW>::load(xr + h + u * st, v[u], pol);
#pragma unroll
      for (int u = 0; u < 4; ++u) acc_shifted<T, VW>(v[u], K, s, q);
    }
    for (; h < h1; h += st) {
      float v[VW];
      Access<T, VW>::load(xr + h, v, pol);
      acc_shifted<T, VW>(v, K, s, q);
    }
    const float2 tot = block_sum2_t0(s, q, sm);
    if (tid == 0) p.part[row * g.T + ch] = tot;
  } else {
    const int64_t item = blockIdx.x;
    n = item / g.items_per_n;
    const int64_t c0 = (item % g.items_per_n) * g.RB;
    const int64_t c1 = (c0 + g.RB < g.C) ? c0 + g.RB : g.C;
    const int lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    for (int64_t c = c0 + warp; c < c1; c += nwarps) {
      const int64_t row = n * g.C + c;
      const T* xr = x + row * g.HW;
      const float K = Elem<T>::to_f(xr[0]);
      float s = 0.f, q = 0.f;
      for (int64_t h = (int64_t)lane * VW; h < g.HW; h += 32 * VW) {
        float v[VW];
        Access<T, VW>::load(xr + h, v, pol);
        acc_shifted<T, VW>(v, K, s, q);
      }
      s = warp_sum_lane0(s);
      q = warp_sum_lane0(q);
      if (lane == 0) p.part[row] = make_float2(s, q);
    }
  }
  arrive_and_finalize<T, false>(p, n, sm);
}

template <typename T, int VW>
__global__ void __launch_bounds__(512) nchw_fwd_apply(const __grid_constant__ KParams p) {
  const Geom& g = p.g;
  const int tid = threadIdx.x;
  const T* x = static_cast<const T*>(p.x);
  T* y = static_cast<T*>(p.out);
  const uint64_t pol = policy_evict_first();
  const int64_t item = g.items - 1 - (int64_t)blockIdx.x;
  if (g.mode == 0) {
    const int64_t row = item / g.T, ch = item % g.T;
    const int64_t n = row / g.C, c = row % g.C, ng = n * g.G + c / g.Cg;
    const float r = __ldg(p.rstd + ng), mu = __ldg(p.mean + ng);
    const float a = p.gamma ? r * __ldg(p.gamma + c) : r;
    const float b = p.beta ? __ldg(p.beta + c) : 0.f;
    const T* xr = x + row * g.HW;
    T* yr = y + row * g.HW;
    const int64_t h0 = ch * g.L;
    const int64_t h1 = (h0 + g.L < g.HW) ? h0 + g.L : g.HW;
    const int64_t nv = (h1 - h0) / VW;
    const int64_t st = blockDim.x;
    int64_t k = nv - 1 - tid;
    for (; k - 3 * st >= 0; k -= 4 * st) {
      float v[4][VW];
#pragma unroll
      for (int u = 0; u < 4; ++u) Access<T, VW>::load(xr + h0 + (k - u * st) * VW, v[u], pol);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
#pragma unroll
        for (int e = 0; e < VW; ++e) v[u][e] = fmaf(v[u][e] - mu, a, b);
        Access<T, VW>::store(yr + h0 + (k - u * st) * VW, v[u], pol);
      }
    }
    for (; k >= 0; k -= st) {
      float v[VW];
      Access<T, VW>::load(xr + h0 + k * VW, v, pol);
#pragma unroll
      for (int e = 0; e < VW; ++e) v[e] = fmaf(v[e] - mu, a, b);
      Access<T, VW>::store(yr + h0 + k * VW, v, pol);
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
  extern __shared__ float sm[];
  const Geom& g = p.g;
  const int tid = threadIdx.x;
  const T* x = static_cast<const T*>(p.x);
  const T* dy = static_cast<const T*>(p.dy);
  const uint64_t pol = policy_evict_last();
  int64_t n;
  if (g.mode == 0) {
    const int64_t item = blockIdx.x;
    const int64_t row = item / g.T, ch = item % g.T;
    n = row / g.C;
    const float mu = __ldg(p.mean + n * g.G + (row % g.C) / g.Cg);
    const T* xr = x + row * g.HW;
    const T* dr = dy + row * g.HW;
    const int64_t h0 = ch * g.L;
    const int64_t h1 = (h0 + g.L < g.HW) ? h0 + g.L : g.HW;
    float s1 = 0.f, s2 = 0.f;
    const int64_t st = (int64_t)blockDim.x * VW;
    int64_t h = h0 + (int64_t)tid * VW;
    for (; h + st < h1; h += 2 * st) {
      float xv[2][VW], dv[2][VW];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        Access<T, VW>::load(xr + h + u * st, xv[u], pol);
        Access<T, VW>::load(dr + h + u * st, dv[u], pol);
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) acc_grad<T, VW>(xv[u], dv[u], mu, s1, s2);
    }
    for (; h < h1; h += st) {
      float xv[VW], dv[VW];
      Access<T, VW>::load(xr + h, xv, pol);
      Access<T, VW>::load(dr + h, dv, pol);
      acc_grad<T, VW>(xv, dv, mu, s1, s2);
    }
    const float2 tot = block_sum2_t0(s1, s2, sm);
    if (tid == 0) p.part[row * g.T + ch] = tot;
  } else {
    const int64_t item = blockIdx.x;
    n = item / g.items_per_n;
    const int64_t c0 = (item % g.items_per_n) * g.RB;
    const int64_t c1 = (c0 + g.RB < g.C) ? c0 + g.RB : g.C;
    const int lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
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
        acc_grad<T, VW>(xv, dv, mu, s1, s2);
      }
      s1 = warp_sum_lane0(s1);
      s2 = warp_sum_lane0(s2);
      if (lane == 0) p.part[row] = make_float2(s1, s2);
    }
  }
  arrive_and_finalize<T, true>(p, n, sm);
}

template <typename T, int VW>
__global__ void __launch_bounds__(512) nchw_bwd_dx(const __grid_constant__ KParams p) {
  const Geom& g = p.g;
  const int tid = threadIdx.x;
  const T* x = static_cast<const T*>(p.x);
  const T* dy = static_cast<const T*>(p.dy);
  T* dx = static_cast<T*>(p.out);
  const uint64_t pol = policy_evict_first();
  const int64_t item = g.items - 1 - (int64_t)blockIdx.x;
  if (g.mode == 0) {
    const int64_t row = item / g.T, ch = item % g.T;
    const int64_t n = row / g.C, c = row % g.C, ng = n * g.G + c / g.Cg;
    const float r = __ldg(p.rstd + ng), mu = __ldg(p.mean + ng);
    const float A = p.gamma ? r * __ldg(p.gamma + c) : r;
    const float2 cf = __ldcg(p.coef + ng);
    const T* xr = x + row * g.HW;
    const T* dr = dy + row * g.HW;
    T* outr = dx + row * g.HW;
    const int64_t h0 = ch * g.L;
    const int64_t h1 = (h0 + g.L < g.HW) ? h0 + g.L : g.HW;
    const int64_t nv = (h1 - h0) / VW;
    const int64_t st = blockDim.x;
    int64_t k = nv - 1 - tid;
    for (; k - st >= 0; k -= 2 * st) {
      float xv[2][VW], dv[2][VW];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        Access<T, VW>::load(xr + h0 + (k - u * st) * VW, xv[u], pol);
        Access<T, VW>::load(dr + h0 + (k - u * st) * VW, dv[u], pol);
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
#pragma unroll
        for (int e = 0; e < VW; ++e) xv[u][e] = fmaf(A, dv[u][e], fmaf(cf.x, xv[u][e] - mu, cf.y));
        Access<T, VW>::store(outr + h0 + (k - u * st) * VW, xv[u], pol);
      }
    }
    for (; k >= 0; k -= st) {
      float xv[VW], dv[VW];
      Access<T, VW>::load(xr + h0 + k * VW, xv, pol);
      Access<T, VW>::load(dr + h0 + k * VW, dv, pol);
#pragma unroll
      for (int e = 0; e < VW; ++e) xv[e] = fmaf(A, dv[e], fmaf(cf.x, xv[e] - mu, cf.y));
      Access<T, VW>::store(outr + h0 + k * VW, xv, pol);
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
cudaError_t fwd_t(const KParams& p, cudaStream_t s) {
  const Geom& g = p.g;
  const size_t sm1 = sizeof(float) * 2 * g.tpb;
  const TimingEvents& ev = timing_events();
  if (ev.begin) cudaEventRecord(ev.begin, s);
  nchw_fwd_stats<T, VW><<<(unsigned)g.items, g.tpb, sm1, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (ev.mid) cudaEventRecord(ev.mid, s);
  nchw_fwd_apply<T, VW><<<(unsigned)g.items, g.tpb, 0, s>>>(p);
  e = cudaGetLastError();
  if (ev.end) cudaEventRecord(ev.end, s);
  return e;
}

template <typename T, int VW>
cudaError_t bwd_t(const KParams& p, cudaStream_t s) {
  const Geom& g = p.g;
  const size_t sm1 = sizeof(float) * 2 * g.tpb;
  const TimingEvents& ev = timing_events();
  if (ev.begin) cudaEventRecord(ev.begin, s);
  nchw_bwd_reduce<T, VW><<<(unsigned)g.items, g.tpb, sm1, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (ev.mid) cudaEventRecord(ev.mid, s);
  nchw_bwd_dx<T, VW><<<(unsigned)g.items, g.tpb, 0, s>>>(p);
  e = cudaGetLastError();
  if (ev.end) cudaEventRecord(ev.end, s);
  return e;
}

template <typename T>
cudaError_t fwd_dispatch_vw(const KParams& p, cudaStream_t s) {
  return p.g.vw == 1 ? fwd_t<T, 1>(p, s) : fwd_t<T, Elem<T>::VEC>(p, s);
}
template <typename T>
cudaError_t bwd_dispatch_vw(const KParams& p, cudaStream_t s) {
  return p.g.vw == 1 ? bwd_t<T, 1>(p, s) : bwd_t<T, Elem<T>::VEC>(p, s);
}

}  // namespace

cudaError_t launch_nchw_fwd(const KParams& p, cudaStream_t s) {
  switch (p.g.dtype) {
    case kF32: return fwd_dispatch_vw<float>(p, s);
    case kF16: return fwd_dispatch_vw<__half>(p, s);
    default: return fwd_dispatch_vw<__nv_bfloat16>(p, s);
  }
}

cudaError_t launch_nchw_bwd(const KParams& p, cudaStream_t s) {
  switch (p.g.dtype) {
    case kF32: return bwd_dispatch_vw<float>(p, s);
    case kF16: return bwd_dispatch_vw<__half>(p, s);
    default: return bwd_dispatch_vw<__nv_bfloat16>(p, s);
  }
}

}  // namespace gn
