// gn_finalize.cuh -- the cross-CTA steps of both ops, run by the CTA whose
// arrival completes a unit (a sample, or in the pipelined NCHW kernel one
// (sample, group)) and, in the backward, by the CTA that completes the last
// unit.  All sums run in a fixed order, so results are bit-identical from run
// to run on the same device.
#pragma once

#include "gn_device.cuh"

namespace gn {

// Sums a strided run of float2 records into (ax, ay) in index order:
// records base[i*stride] for i = first, first + step, ... < count.  Loads are
// issued eight at a time (predicated), so a short run costs one round trip.
__device__ __forceinline__ void sum_records(const float2* base, int64_t stride, int64_t first,
                                            int64_t step, int64_t count, float& ax, float& ay) {
  for (int64_t i = first; i < count; i += 8 * step) {
    float2 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int64_t j = i + k * step;
      v[k] = j < count ? __ldcg(base + j * stride) : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      ax += v[k].x;
      ay += v[k].y;
    }
  }
}

// Threads as (slice, channel): consecutive threads on consecutive channels,
// nsl slices per channel block.
struct SliceLayout {
  int cpb, nsl, cl, sl;
};
__device__ __forceinline__ SliceLayout slice_layout(int64_t C, int64_t count) {
  SliceLayout L;
  const int nt = blockDim.x;
  L.cpb = (int)(C < nt ? C : nt);
  int64_t nsl = nt / L.cpb;
  if (nsl > count) nsl = count;
  L.nsl = nsl < 1 ? 1 : (int)nsl;
  L.cl = threadIdx.x % L.cpb;
  L.sl = threadIdx.x / L.cpb;
  return L;
}

// For every channel c in [ca, cb) of sample n, sums the g.Tp partial records
// of (n, c) and calls fn(c, total) from one thread.  Slice s adds records s,
// s + nsl, ... in order, then the slice sums are added in slice order.
// `sm` holds at least 2 * blockDim.x floats.  Ends with __syncthreads().
template <typename Fn>
__device__ __forceinline__ void sum_channel_partials(const KParams& p, int64_t n, int64_t ca,
                                                     int64_t cb, float* sm, Fn fn) {
  const Geom& g = p.g;
  const SliceLayout L = slice_layout(cb - ca, g.Tp);
  const float2* base = p.part + n * g.C * g.Tp;
  for (int64_t c0 = ca; c0 < cb; c0 += L.cpb) {
    const int64_t c = c0 + L.cl;
    float ax = 0.f, ay = 0.f;
    if (L.sl < L.nsl && c < cb)
      sum_records(base + c * g.cstride, g.tstride, L.sl, L.nsl, g.Tp, ax, ay);
    if (L.sl < L.nsl) {
      sm[2 * (L.sl * L.cpb + L.cl)] = ax;
      sm[2 * (L.sl * L.cpb + L.cl) + 1] = ay;
    }
    __syncthreads();
    if (L.sl == 0 && c < cb) {
      for (int s = 1; s < L.nsl; ++s) {
        ax += sm[2 * (s * L.cpb + L.cl)];
        ay += sm[2 * (s * L.cpb + L.cl) + 1];
      }
      fn(c, make_float2(ax, ay));
    }
    __syncthreads();
  }
}

// Where the finalising CTA keeps its per-channel results for the group step:
// in shared memory after the 2*blockDim.x floats used by the partial sums when
// the C records fit (sm_floats is the CTA's dynamic shared memory), else in
// the workspace.
__device__ __forceinline__ float2* channel_stage(const KParams& p, int64_t n, float* sm,
                                                 int64_t sm_floats) {
  const int64_t need = 2 * (int64_t)blockDim.x + 2 * p.g.C;
  return need <= sm_floats ? reinterpret_cast<float2*>(sm + 2 * blockDim.x) : p.chst + n * p.g.C;
}

// Offset of element (n, c, hw = 0): the per-channel shift of the forward sums.
__device__ __forceinline__ int64_t first_elem_offset(const Geom& g, int64_t n, int64_t c) {
  return g.layout == kNCHW ? (n * g.C + c) * g.HW : n * g.HW * g.C + c;
}

// Forward, channels [ca, cb) (whole groups) of sample n.  The partial records
// hold, per channel, S = sum(x - K_c)
// and Q = sum((x - K_c)^2) with K_c = x(n, c, hw = 0).  Each channel gives
// (mean_c, M2_c); the Cg channels of a group (HW elements each) merge into
//   mean_g = avg_c(mean_c),  M2_g = sum_c M2_c + HW * sum_c (mean_c - mean_g)^2,
// and var = M2_g / (Cg*HW) (biased), rstd = 1/sqrt(var + eps).
template <typename T>
__device__ void finalize_fwd(const KParams& p, int64_t n, int64_t ca, int64_t cb, float* sm,
                             int64_t sm_floats) {
  const Geom& g = p.g;
  const T* x = static_cast<const T*>(p.x);
  const float hw = (float)g.HW;
  float2* stage = channel_stage(p, n, sm, sm_floats);
  sum_channel_partials(p, n, ca, cb, sm, [&](int64_t c, float2 s) {
    const float K = Elem<T>::to_f(x[first_elem_offset(g, n, c)]);
    const float q = s.x / hw;
    const float m2 = fmaxf(fmaf(-s.x, q, s.y), 0.f);
    stage[c] = make_float2(K + q, m2);
  });
  const float cgf = (float)g.Cg;
  const float mf = (float)(g.Cg * g.HW);
  for (int64_t gi = ca / g.Cg + threadIdx.x; gi < cb / g.Cg; gi += blockDim.x) {
    const float2* cs = stage + gi * g.Cg;
    float s = 0.f;
    for (int64_t k = 0; k < g.Cg; ++k) s += cs[k].x;
    const float mg = s / cgf;
    float m2 = 0.f;
    for (int64_t k = 0; k < g.Cg; ++k) {
      const float2 v = cs[k];
      const float d = v.x - mg;
      m2 += fmaf(hw * d, d, v.y);
    }
    const float var = m2 / mf;
    p.mean[n * g.G + gi] = mg;
    p.rstd[n * g.G + gi] = 1.0f / sqrtf(var + p.eps);
  }
}

// Backward, channels [ca, cb) (whole groups) of sample n.  The partial
// records hold, per channel,
// S1 = sum(dy) and S2 = sum(dy * (x - mean_g)).  Per group:
//   c1 = sum_c gamma_c * S1_c          (= sum over the group of gamma*dy)
//   c2 = sum_c gamma_c * S2_c          (sum of gamma*dy*xhat = rstd * c2)
// and dx = rstd*gamma_c*dy + B*(x - mean) + D with
//   B = -rstd^3 * c2 / M,  D = -rstd * c1 / M,  M = Cg*HW.
// The per-channel (S1, S2) stay in chst for the dgamma/dbeta step.
__device__ __forceinline__ void finalize_bwd(const KParams& p, int64_t n, int64_t ca, int64_t cb,
                                             float* sm, int64_t sm_floats) {
  const Geom& g = p.g;
  float2* stage = channel_stage(p, n, sm, sm_floats);
  float2* chst = p.chst + n * g.C;
  sum_channel_partials(p, n, ca, cb, sm, [&](int64_t c, float2 s) {
    chst[c] = s;  // kept for the dgamma/dbeta step
    stage[c] = s;
  });
  const float mf = (float)(g.Cg * g.HW);
  for (int64_t gi = ca / g.Cg + threadIdx.x; gi < cb / g.Cg; gi += blockDim.x) {
    const float2* cs = stage + gi * g.Cg;
    float c1 = 0.f, c2 = 0.f;
    for (int64_t k = 0; k < g.Cg; ++k) {
      const float2 v = cs[k];
      const float gm = p.gamma ? __ldg(p.gamma + gi * g.Cg + k) : 1.0f;
      c1 = fmaf(gm, v.x, c1);
      c2 = fmaf(gm, v.y, c2);
    }
    const float r = __ldg(p.rstd + n * g.G + gi);
    p.coef[n * g.G + gi] = make_float2(-(r * r * r) * c2 / mf, -r * c1 / mf);
  }
}

// Level 2 of the parameter gradients:
//   dbeta_c = sum_n S1[n, c],   dgamma_c = sum_n rstd[n, g(c)] * S2[n, c],
// with the samples split into fixed slices (summed in order, then the slice
// sums in slice order).
__device__ __forceinline__ void finalize_params(const KParams& p, float* sm) {
  const Geom& g = p.g;
  if (!p.dgamma && !p.dbeta) return;
  const SliceLayout L = slice_layout(g.C, g.N);
  for (int64_t c0 = 0; c0 < g.C; c0 += L.cpb) {
    const int64_t c = c0 + L.cl;
    float db = 0.f, dg = 0.f;
    if (L.sl < L.nsl && c < g.C) {
      const int64_t gi = c / g.Cg;
      for (int64_t n = L.sl; n < g.N; n += 8 * L.nsl) {
        float2 v[8];
        float r[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int64_t j = n + k * L.nsl;
          v[k] = j < g.N ? __ldcg(p.chst + j * g.C + c) : make_float2(0.f, 0.f);
          r[k] = j < g.N ? __ldg(p.rstd + j * g.G + gi) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          db += v[k].x;
          dg = fmaf(r[k], v[k].y, dg);
        }
      }
    }
    if (L.sl < L.nsl) {
      sm[2 * (L.sl * L.cpb + L.cl)] = db;
      sm[2 * (L.sl * L.cpb + L.cl) + 1] = dg;
    }
    __syncthreads();
    if (L.sl == 0 && c < g.C) {
      for (int s = 1; s < L.nsl; ++s) {
        db += sm[2 * (s * L.cpb + L.cl)];
        dg += sm[2 * (s * L.cpb + L.cl) + 1];
      }
      if (p.dbeta) p.dbeta[c] = db;
      if (p.dgamma) p.dgamma[c] = dg;
    }
    __syncthreads();
  }
}

// A finalisation unit: the channels [c0, c1) (whole groups) of sample n,
// completed by `arrivals` arrivals on *ticket.  With a ready flag (pipelined
// kernel) the finaliser sets it once the unit's statistics are written.
struct Unit {
  int64_t n, c0, c1;
  unsigned* ticket;
  unsigned arrivals;
  unsigned* ready;
};

// The unit that channel c of sample n belongs to: the whole sample, or one
// (sample, group) when g.unit_groups is set.  Its ticket (and ready flag) is
// the unit's index n or n*G + c/Cg.
__device__ __forceinline__ Unit unit_of(const KParams& p, int64_t n, int64_t c) {
  const Geom& g = p.g;
  Unit u;
  u.n = n;
  int64_t id = n;
  if (g.unit_groups) {
    u.c0 = c / g.Cg * g.Cg;
    u.c1 = u.c0 + g.Cg;
    id = n * g.G + c / g.Cg;
  } else {
    u.c0 = 0;
    u.c1 = g.C;
  }
  u.ticket = p.tickets + id;
  u.arrivals = (unsigned)g.arrivals_per_n;
  u.ready = p.ready ? p.ready + id : nullptr;
  return u;
}

// Tail of every CTA that has written a partial record.  With level-1 groups
// (l1 > 1) the CTA arrives on its group's counter; the group's last CTA runs
// merge() (the group record from its item records, in item order) and
// arrives on the unit's counter.  The unit's last arrival runs its
// finalisation (and raises the unit's ready flag).  Every counter is reset by
// the CTA that completed it.  Must be reached by all threads of the CTA.
template <typename T, bool kBwd, typename Merge>
__device__ __forceinline__ void arrive_and_finalize(const KParams& p, const Unit& un,
                                                    int64_t group1, unsigned gsize, Merge merge,
                                                    float* sm, int64_t sm_floats) {
  __shared__ int s_last;
  __threadfence();  // this thread's record stores, before the CTA's arrival
  if (p.g.l1 > 1) {
    __syncthreads();
    if (threadIdx.x == 0) s_last = publish_and_arrive(p.cnt1 + group1, gsize);
    __syncthreads();
    if (!s_last) return;
    merge();
    __threadfence();
    if (threadIdx.x == 0) atomicExch(p.cnt1 + group1, 0u);
  }
  __syncthreads();
  if (threadIdx.x == 0) s_last = publish_and_arrive(un.ticket, un.arrivals);
  __syncthreads();
  if (!s_last) return;
  if (kBwd)
    finalize_bwd(p, un.n, un.c0, un.c1, sm, sm_floats);
  else
    finalize_fwd<T>(p, un.n, un.c0, un.c1, sm, sm_floats);
  __threadfence();  // the unit's statistics, before the ready flag and the next arrival
  __syncthreads();
  if (threadIdx.x == 0) {
    atomicExch(un.ticket, 0u);
    if (un.ready) atomicExch(un.ready, 1u);
  }
  // the backward's dgamma / dbeta are added up by the dx kernel, whose first
  // CTA finds every channel's sums complete when it starts
}

}  // namespace gn
