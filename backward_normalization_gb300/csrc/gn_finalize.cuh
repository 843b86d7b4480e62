// gn_finalize.cuh -- the cross-CTA steps of both ops, run by the CTA whose
// arrival completes a sample n (and, in the backward, by the CTA that
// completes the last sample).  All sums run in a fixed order, so results are
// bit-identical from run to run on the same device.
#pragma once

#include "gn_device.cuh"

namespace gn {

// For every channel c of sample n, sums the g.Tp partial records of (n, c)
// and calls fn(c, total) from one thread.  Threads are laid out as
// (slice, channel) with consecutive threads on consecutive channels; slice s
// adds records s, s + nsl, s + 2*nsl, ... (issued eight at a time so that the
// loads overlap), then the slice sums are added in slice order.
// `sm` holds at least 2 * blockDim.x floats.  Ends with __syncthreads().
template <typename Fn>
__device__ __forceinline__ void sum_channel_partials(const KParams& p, int64_t n, float* sm,
                                                     Fn fn) {
  const Geom& g = p.g;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int cpb = (int)(g.C < nt ? g.C : nt);
  int64_t nsl64 = nt / cpb;
  if (nsl64 > g.Tp) nsl64 = g.Tp;
  const int nsl = nsl64 < 1 ? 1 : (int)nsl64;
  const int cl = tid % cpb, sl = tid / cpb;
  const float2* base = p.part + n * g.C * g.Tp;
  for (int64_t c0 = 0; c0 < g.C; c0 += cpb) {
    const int64_t c = c0 + cl;
    float ax = 0.f, ay = 0.f;
    if (sl < nsl && c < g.C) {
      const float2* pc = base + c * g.cstride;
      const int64_t st = (int64_t)nsl * g.tstride;
      int64_t t = sl;
      for (; t + 7 * nsl < g.Tp; t += 8 * nsl) {
        float2 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __ldcg(pc + t * g.tstride + k * st);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          ax += v[k].x;
          ay += v[k].y;
        }
      }
      for (; t < g.Tp; t += nsl) {
        const float2 v = __ldcg(pc + t * g.tstride);
        ax += v.x;
        ay += v.y;
      }
    }
    if (sl < nsl) {
      sm[2 * (sl * cpb + cl)] = ax;
      sm[2 * (sl * cpb + cl) + 1] = ay;
    }
    __syncthreads();
    if (sl == 0 && c < g.C) {
      for (int s = 1; s < nsl; ++s) {
        ax += sm[2 * (s * cpb + cl)];
        ay += sm[2 * (s * cpb + cl) + 1];
      }
      fn(c, make_float2(ax, ay));
    }
    __syncthreads();
  }
}

// Offset of element (n, c, hw = 0): the per-channel shift of the forward sums.
__device__ __forceinline__ int64_t first_elem_offset(const Geom& g, int64_t n, int64_t c) {
  return g.layout == kNCHW ? (n * g.C + c) * g.HW : n * g.HW * g.C + c;
}

// Forward, sample n.  The partial records hold, per channel, S = sum(x - K_c)
// and Q = sum((x - K_c)^2) with K_c = x(n, c, hw = 0).  Each channel gives
// (mean_c, M2_c); the Cg channels of a group (HW elements each) merge into
//   mean_g = avg_c(mean_c),  M2_g = sum_c M2_c + HW * sum_c (mean_c - mean_g)^2,
// and var = M2_g / (Cg*HW) (biased), rstd = 1/sqrt(var + eps).
template <typename T>
__device__ void finalize_fwd(const KParams& p, int64_t n, float* sm) {
  const Geom& g = p.g;
  const T* x = static_cast<const T*>(p.x);
  const float hw = (float)g.HW;
  sum_channel_partials(p, n, sm, [&](int64_t c, float2 s) {
    const float K = Elem<T>::to_f(x[first_elem_offset(g, n, c)]);
    const float q = s.x / hw;
    const float m2 = fmaxf(fmaf(-s.x, q, s.y), 0.f);
    p.chst[n * g.C + c] = make_float2(K + q, m2);
  });
  const float cgf = (float)g.Cg;
  const float mf = (float)(g.Cg * g.HW);
  for (int64_t gi = threadIdx.x; gi < g.G; gi += blockDim.x) {
    const float2* cs = p.chst + n * g.C + gi * g.Cg;
    float s = 0.f;
    for (int64_t k = 0; k < g.Cg; ++k) s += __ldcg(cs + k).x;
    const float mg = s / cgf;
    float m2 = 0.f;
    for (int64_t k = 0; k < g.Cg; ++k) {
      const float2 v = __ldcg(cs + k);
      const float d = v.x - mg;
      m2 += fmaf(hw * d, d, v.y);
    }
    const float var = m2 / mf;
    p.mean[n * g.G + gi] = mg;
    p.rstd[n * g.G + gi] = 1.0f / sqrtf(var + p.eps);
  }
}

// Backward, sample n.  The partial records hold, per channel,
// S1 = sum(dy) and S2 = sum(dy * (x - mean_g)).  Per group:
//   c1 = sum_c gamma_c * S1_c          (= sum over the group of gamma*dy)
//   c2 = sum_c gamma_c * S2_c          (sum of gamma*dy*xhat = rstd * c2)
// and dx = rstd*gamma_c*dy + B*(x - mean) + D with
//   B = -rstd^3 * c2 / M,  D = -rstd * c1 / M,  M = Cg*HW.
// The per-channel (S1, S2) stay in chst for the dgamma/dbeta step.
__device__ __forceinline__ void finalize_bwd(const KParams& p, int64_t n, float* sm) {
  const Geom& g = p.g;
  sum_channel_partials(p, n, sm, [&](int64_t c, float2 s) { p.chst[n * g.C + c] = s; });
  const float mf = (float)(g.Cg * g.HW);
  for (int64_t gi = threadIdx.x; gi < g.G; gi += blockDim.x) {
    const float2* cs = p.chst + n * g.C + gi * g.Cg;
    float c1 = 0.f, c2 = 0.f;
    for (int64_t k = 0; k < g.Cg; ++k) {
      const float2 v = __ldcg(cs + k);
      const float gm = p.gamma ? __ldg(p.gamma + gi * g.Cg + k) : 1.0f;
      c1 = fmaf(gm, v.x, c1);
      c2 = fmaf(gm, v.y, c2);
    }
    const float r = __ldg(p.rstd + n * g.G + gi);
    p.coef[n * g.G + gi] = make_float2(-(r * r * r) * c2 / mf, -r * c1 / mf);
  }
}

// Level 2 of the parameter gradients, over samples in index order:
//   dbeta_c = sum_n S1[n, c],   dgamma_c = sum_n rstd[n, g(c)] * S2[n, c].
__device__ __forceinline__ void finalize_params(const KParams& p) {
  const Geom& g = p.g;
  if (!p.dgamma && !p.dbeta) return;
  for (int64_t c = threadIdx.x; c < g.C; c += blockDim.x) {
    const int64_t gi = c / g.Cg;
    float db = 0.f, dg = 0.f;
    for (int64_t n = 0; n < g.N; ++n) {
      const float2 v = __ldcg(p.chst + n * g.C + c);
      db += v.x;
      dg = fmaf(__ldg(p.rstd + n * g.G + gi), v.y, dg);
    }
    if (p.dbeta) p.dbeta[c] = db;
    if (p.dgamma) p.dgamma[c] = dg;
  }
}

// Tail of every CTA that published a cluster-level partial: arrive on the
// sample's counter and, if the sample is now complete, run its finalisation
// (and, in the backward, the parameter-gradient step once every sample is
// complete).  Must be reached by all threads of the CTA.
template <typename T, bool kBwd>
__device__ __forceinline__ void arrive_and_finalize(const KParams& p, int64_t n, float* sm) {
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) s_last = publish_and_arrive(p.tickets + n, (unsigned)p.g.arrivals_per_n);
  __syncthreads();
  if (!s_last) return;
  if (kBwd)
    finalize_bwd(p, n, sm);
  else
    finalize_fwd<T>(p, n, sm);
  __syncthreads();
  if (threadIdx.x == 0) atomicExch(p.tickets + n, 0u);
  if (!kBwd) return;
  if (threadIdx.x == 0) s_last = publish_and_arrive(p.tickets + p.g.N, (unsigned)p.g.N);
  __syncthreads();
  if (!s_last) return;
  finalize_params(p);
  __syncthreads();
  if (threadIdx.x == 0) atomicExch(p.tickets + p.g.N, 0u);
}

}  // namespace gn
