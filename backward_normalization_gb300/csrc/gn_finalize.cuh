// gn_finalize.cuh -- the cross-CTA steps of both ops: run by the CTA whose
// arrival completes a unit (a sample, or in the pipelined NCHW kernel one
// (sample, group)), the backward's parameter step by the dx kernel's first
// CTA; or, in NCHW plans with few records per group (fin2), by every CTA of
// the second kernel for its own groups, with the parameter step spread over
// its CTAs.  All sums run in a fixed order, so results are bit-identical from
// run to run on the same device.
#pragma once

#include "gn_device.cuh"

namespace gn {

// Sums a strided run of float2 records into (ax, ay) in index order:
// records base[i*stride] for i = first, first + step, ... < count.  Loads are
// issued B at a time (predicated), so a run of up to B costs one round trip.
template <int B = 8>
__device__ __forceinline__ void sum_records(const float2* base, int64_t stride, int64_t first,
                                            int64_t step, int64_t count, float& ax, float& ay) {
  for (int64_t i = first; i < count; i += B * step) {
    float2 v[B];
#pragma unroll
    for (int k = 0; k < B; ++k) {
      const int64_t j = i + k * step;
      v[k] = j < count ? __ldcg(base + j * stride) : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < B; ++k) {
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

// Offset of element (n, c, hw = 0) of x: the per-channel shift of the forward sums.
__device__ __forceinline__ int64_t first_elem_offset(const KParams& p, int64_t n, int64_t c) {
  return p.g.layout == kNCHW ? n * p.xs_n + c * p.xs_r : n * p.xs_n + c;
}

// Offset of channel plane `row` = n*C + c (NCHW) in a view with sample stride
// s_n and plane stride s_r.
__device__ __forceinline__ int64_t plane_offset(const Geom& g, int64_t row, int64_t s_n,
                                                int64_t s_r) {
  const int64_t n = row / g.C;
  return n * s_n + (row - n * g.C) * s_r;
}

// Forward statistics.  The partial records hold, per channel, S = sum(x - K_c)
// and Q = sum((x - K_c)^2) with K_c = x(n, c, hw = 0).  Each channel gives
// (mean_c, M2_c); the Cg channels of a group (HW elements each) merge into
//   mean_g = avg_c(mean_c),  M2_g = sum_c M2_c + HW * sum_c (mean_c - mean_g)^2,
// and var = M2_g / (Cg*HW) (biased), rstd = 1/sqrt(var + eps).
__device__ __forceinline__ float2 channel_moments(float K, float2 s, float hw) {
  const float q = s.x / hw;
  return make_float2(K + q, fmaxf(fmaf(-s.x, q, s.y), 0.f));  // (mean_c, M2_c)
}
// (mean_g, rstd_g) from the Cg (mean_c, M2_c) of a group.
__device__ __forceinline__ float2 group_moments(const float2* cs, const Geom& g, float eps) {
  const float hw = (float)g.HW;
  float s = 0.f;
  for (int64_t k = 0; k < g.Cg; ++k) s += cs[k].x;
  const float mg = s / (float)g.Cg;
  float m2 = 0.f;
  for (int64_t k = 0; k < g.Cg; ++k) {
    const float2 v = cs[k];
    const float d = v.x - mg;
    m2 += fmaf(hw * d, d, v.y);
  }
  const float var = m2 / (float)(g.Cg * g.HW);
  return make_float2(mg, 1.0f / sqrtf(var + eps));
}

// Backward coefficients.  The partial records hold, per channel,
// S1 = sum(dy) and S2 = sum(dy * (x - mean_g)).  Per group:
//   c1 = sum_c gamma_c * S1_c          (= sum over the group of gamma*dy)
//   c2 = sum_c gamma_c * S2_c          (sum of gamma*dy*xhat = rstd * c2)
// and dx = rstd*gamma_c*dy + B*(x - mean) + D with
//   B = -rstd^3 * c2 / M,  D = -rstd * c1 / M,  M = Cg*HW.
// Channel c's terms (gamma_c * S1_c, gamma_c * S2_c), formed per channel so
// that the gamma loads of a group run in parallel.
// The products are rounded on their own (never fused into the sums), so the
// terms formed ahead and the terms formed inside the group sum agree.
__device__ __forceinline__ float2 channel_terms(float gm, float2 s) {
  return make_float2(__fmul_rn(gm, s.x), __fmul_rn(gm, s.y));
}
__device__ __forceinline__ float2 coef_from(float c1, float c2, const Geom& g, float r) {
  const float mf = (float)(g.Cg * g.HW);
  return make_float2(-(r * r * r) * c2 / mf, -r * c1 / mf);
}
// (B, D) of a group from its Cg channel terms and its rstd r.
__device__ __forceinline__ float2 group_coef(const float2* cs, const Geom& g, float r) {
  float c1 = 0.f, c2 = 0.f;
  for (int64_t k = 0; k < g.Cg; ++k) {
    c1 += cs[k].x;
    c2 += cs[k].y;
  }
  return coef_from(c1, c2, g, r);
}
// The same from group gi's raw channel sums (S1_c, S2_c), its terms formed here.
__device__ __forceinline__ float2 group_coef_sums(const float2* cs, const KParams& p, int64_t gi,
                                                 float r) {
  const Geom& g = p.g;
  float c1 = 0.f, c2 = 0.f;
  for (int64_t k = 0; k < g.Cg; ++k) {
    const float2 t = channel_terms(p.gamma ? __ldg(p.gamma + gi * g.Cg + k) : 1.0f, cs[k]);
    c1 += t.x;
    c2 += t.y;
  }
  return coef_from(c1, c2, g, r);
}

// Forward, channels [ca, cb) (whole groups) of sample n: mean and rstd.
template <typename T>
__device__ void finalize_fwd(const KParams& p, int64_t n, int64_t ca, int64_t cb, float* sm,
                             int64_t sm_floats) {
  const Geom& g = p.g;
  const T* x = static_cast<const T*>(p.x);
  const float hw = (float)g.HW;
  float2* stage = channel_stage(p, n, sm, sm_floats);
  // the shift of this thread's first channel (ca + tid), requested with the records
  auto shift = [&](int64_t c) { return Elem<T>::to_f(x[first_elem_offset(p, n, c)]); };
  const int64_t c_pre = ca + threadIdx.x;
  const float k_pre = c_pre < cb ? shift(c_pre) : 0.f;
  sum_channel_partials(p, n, ca, cb, sm, [&](int64_t c, float2 s) {
    stage[c] = channel_moments(c == c_pre ? k_pre : shift(c), s, hw);
  });
  for (int64_t gi = ca / g.Cg + threadIdx.x; gi < cb / g.Cg; gi += blockDim.x) {
    const float2 mr = group_moments(stage + gi * g.Cg, g, p.eps);
    p.mean[n * g.G + gi] = mr.x;
    p.rstd[n * g.G + gi] = mr.y;
  }
}

// Backward, channels [ca, cb) (whole groups) of sample n: the dx coefficients.
// The per-channel (S1, S2) stay in chst for the dgamma/dbeta step (the stage
// may be chst itself, so it holds the same raw sums).
__device__ __forceinline__ void finalize_bwd(const KParams& p, int64_t n, int64_t ca, int64_t cb,
                                             float* sm, int64_t sm_floats) {
  const Geom& g = p.g;
  float2* stage = channel_stage(p, n, sm, sm_floats);
  float2* chst = p.chst + n * g.C;
  const bool terms = stage != chst;  // a stage of its own: the channel terms go there
  // gamma of this thread's first channel and rstd of its first group,
  // requested with the records
  auto gam = [&](int64_t c) { return p.gamma ? __ldg(p.gamma + c) : 1.0f; };
  const int64_t c_pre = ca + threadIdx.x, g_pre = ca / g.Cg + threadIdx.x;
  const float gam_pre = c_pre < cb ? gam(c_pre) : 0.f;
  const float r_pre = g_pre < cb / g.Cg ? __ldg(p.rstd + n * g.G + g_pre) : 0.f;
  sum_channel_partials(p, n, ca, cb, sm, [&](int64_t c, float2 s) {
    chst[c] = s;  // kept for the dgamma/dbeta step
    stage[c] = terms ? channel_terms(c == c_pre ? gam_pre : gam(c), s) : s;
  });
  for (int64_t gi = ca / g.Cg + threadIdx.x; gi < cb / g.Cg; gi += blockDim.x) {
    const float r = gi == g_pre ? r_pre : __ldg(p.rstd + n * g.G + gi);
    p.coef[n * g.G + gi] = terms ? group_coef(stage + gi * g.Cg, g, r)
                                 : group_coef_sums(stage + gi * g.Cg, p, gi, r);
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
  if (p.g.l1 > 1) {
    __syncthreads();  // the CTA's record stores, before thread 0's arrival
    if (threadIdx.x == 0) s_last = publish_and_arrive(p.cnt1 + group1, gsize);
    __syncthreads();
    if (!s_last) return;
    merge();
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
  __syncthreads();  // the unit's statistics, before the ready flag
  if (threadIdx.x == 0) {
    atomicExch(un.ticket, 0u);
    if (un.ready) {
      __threadfence();
      atomicExch(un.ready, 1u);
    }
  }
  // the backward's dgamma / dbeta are added up by the dx kernel, whose first
  // CTA finds every channel's sums complete when it starts
}

// ------------------------------------ finalisation in the second kernel (fin2)
// Tail of a first-kernel CTA of a fin2 plan with level-1 groups: the group's
// last CTA merges its item records into the level-1 record.  Nothing waits on
// it inside the launch; the second kernel reads the records after the launch
// boundary.  Must be reached by all threads of the CTA.
template <typename Merge>
__device__ __forceinline__ void arrive_level1(const KParams& p, int64_t group1, unsigned gsize,
                                              Merge merge) {
  __shared__ int s_last1;
  __syncthreads();  // the CTA's record stores, before thread 0's arrival
  if (threadIdx.x == 0) s_last1 = publish_and_arrive(p.cnt1 + group1, gsize);
  __syncthreads();
  if (!s_last1) return;
  merge();
  __syncthreads();
  if (threadIdx.x == 0) atomicExch(p.cnt1 + group1, 0u);
}

// Parameter gradients of a fin2 backward, spread over the second kernel's
// CTAs: CTA b takes channels b, b + gridDim.x, ... (at most kmax =
// ceil(C / gridDim.x)); its warps split into slots of wpc warps, slot k taking
// the CTA's k-th channel (in rounds when there are more channels than slots).
// Within a slot, thread i takes records f = i, i + 32*wpc, ... of the
// channel's N*Tp (record f = n*Tp + t1), each warp sums with a fixed tree and
// the slot's warps are added in warp order:
//   dbeta_c = sum S1,   dgamma_c = sum rstd[n, g(c)] * S2.
// Cheap to recompute (no state is kept across the steps).
struct ParamSplit {
  int wpc;    // warps per channel slot
  int nslot;  // channel slots per round
  int slot;   // this thread's slot
  int first;  // this thread's first record, and the stride between its records
  int step;
  int64_t kmax;  // channels of the most loaded CTA
};
__device__ __forceinline__ ParamSplit param_split(const Geom& g) {
  ParamSplit s;
  const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5;
  s.kmax = (g.C + gridDim.x - 1) / gridDim.x;
  s.wpc = s.kmax >= nw ? 1 : nw / (int)s.kmax;
  s.nslot = nw / s.wpc;
  s.slot = warp / s.wpc;
  s.first = (warp % s.wpc) * 32 + (threadIdx.x & 31);
  s.step = 32 * s.wpc;
  return s;
}
// Channel of slot `slot` in round `round` (>= C: none).
__device__ __forceinline__ int64_t param_channel(const ParamSplit& s, int64_t round) {
  return blockIdx.x + (round * s.nslot + s.slot) * (int64_t)gridDim.x;
}
constexpr int kParamBatch = 4;
struct ParamBatch {
  float2 v[kParamBatch];
  float r[kParamBatch];
};
// Requests records f0, f0 + step, ... (kParamBatch of them) of channel c.
__device__ __forceinline__ void param_load(const KParams& p, int64_t c, int64_t f0, int64_t step,
                                           ParamBatch& b) {
  const Geom& g = p.g;
  const int64_t total = g.N * g.Tp, gi = c / g.Cg;
  const float2* base = p.part + c * g.cstride;
#pragma unroll
  for (int k = 0; k < kParamBatch; ++k) {
    const int64_t f = f0 + k * step;
    const int64_t n = f / g.Tp, t1 = f - n * g.Tp;
    const bool in = c < g.C && f < total;
    b.v[k] = in ? __ldcg(base + n * g.C * g.Tp + t1 * g.tstride) : make_float2(0.f, 0.f);
    b.r[k] = in ? __ldg(p.rstd + n * g.G + gi) : 0.f;
  }
}
// This thread's share of channel c given its first batch b (further batches
// are loaded here), summed over the warp into wpart[warp] (lane 0).
__device__ __forceinline__ void param_warp_sum(const KParams& p, const ParamSplit& s, int64_t c,
                                               ParamBatch& b, float* wpart) {
  const int64_t total = p.g.N * p.g.Tp;
  float db = 0.f, dg = 0.f;
  for (int64_t f0 = s.first;; f0 += kParamBatch * s.step) {
#pragma unroll
    for (int k = 0; k < kParamBatch; ++k) {
      db += b.v[k].x;
      dg = fmaf(b.r[k], b.v[k].y, dg);
    }
    if (f0 + kParamBatch * s.step >= total || c >= p.g.C) break;
    param_load(p, c, f0 + kParamBatch * s.step, s.step, b);
  }
  db = warp_sum_lane0(db);
  dg = warp_sum_lane0(dg);
  if ((threadIdx.x & 31) == 0) {
    wpart[2 * (threadIdx.x >> 5)] = db;
    wpart[2 * (threadIdx.x >> 5) + 1] = dg;
  }
}
// Thread k < nslot adds its slot's warp sums in warp order and writes them
// (after a barrier that follows param_warp_sum).
__device__ __forceinline__ void param_write(const KParams& p, const ParamSplit& s, int64_t round,
                                            const float* wpart) {
  if ((int64_t)threadIdx.x >= s.nslot) return;
  ParamSplit t = s;
  t.slot = threadIdx.x;
  const int64_t c = param_channel(t, round);
  if (c >= p.g.C) return;
  float db = 0.f, dg = 0.f;
  for (int w = 0; w < s.wpc; ++w) {
    db += wpart[2 * (threadIdx.x * s.wpc + w)];
    dg += wpart[2 * (threadIdx.x * s.wpc + w) + 1];
  }
  if (p.dbeta) p.dbeta[c] = db;
  if (p.dgamma) p.dgamma[c] = dg;
}

// Second-kernel finalisation (NCHW plans) of channels [ca, cb) (whole
// groups, at most g.maxch2) of sample n.  Channel c's records are added in g.nsl2 fixed
// slices (slice s takes records s, s + nsl2, ...) and the slices in order, so
// every CTA that covers a group derives the same bits for it.  Returns, in
// shared memory, one float2 per group (index gi - ca/Cg): forward (mean,
// rstd), of which groups [wa, wb) are also written to p.mean / p.rstd;
// backward the dx coefficients (B, D), the backward also writing its share
// of dgamma/dbeta.  The records are staged in shared memory by 16-byte
// asynchronous copies, requested together with every other load the steps
// need (the channel's gamma or shift, the group's rstd, the first parameter
// batch), so the whole step costs about one round trip to L2.  `sm` is the
// 16-byte aligned base of fin2_smem(g).total floats.  Must be reached by all
// threads; ends with __syncthreads().
template <bool kBwd>
__device__ const float2* fin2_groups(const KParams& p, int64_t n, int64_t ca, int64_t cb,
                                     int64_t wa, int64_t wb, float* sm) {
  const Geom& g = p.g;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int64_t nch = cb - ca, ngr = nch / g.Cg, g0 = ca / g.Cg;
  const int nsl = g.nsl2;
  const Fin2Smem L = fin2_smem(g);
  float2* recs = reinterpret_cast<float2*>(sm + L.recs);
  float2* part = reinterpret_cast<float2*>(sm + L.part);
  float2* stage = reinterpret_cast<float2*>(sm + L.stage);
  float2* grp = reinterpret_cast<float2*>(sm + L.grp);
  float* wpart = sm + L.wpart;
  // the (c, t1) records of c in [ca, cb) are one contiguous run (NCHW record
  // index (n*C + c)*Tp + t1), staged from its even start: the run's record i
  // lands at recs[sh + i]
  const int64_t first = (n * g.C + ca) * g.Tp, rlen = nch * g.Tp;
  const int64_t a0 = first & ~int64_t(1), sh = first - a0;
  for (int64_t k = tid; 2 * k < sh + rlen; k += nt) cp_async16(recs + 2 * k, p.part + a0 + 2 * k);
  auto rec = [&](int64_t j, int64_t t1) { return recs[sh + j * g.Tp + t1]; };
  auto chan_in = [&](int64_t j) {
    if (kBwd) return p.gamma ? __ldg(p.gamma + ca + j) : 1.0f;
    return __ldcg(p.kst + n * g.C + ca + j);
  };
  const float cin = tid < nch ? chan_in(tid) : 0.f;
  const float rin = kBwd && tid < ngr ? __ldg(p.rstd + n * g.G + g0 + tid) : 0.f;
  ParamBatch pb;
  const bool params = kBwd && (p.dgamma || p.dbeta);
  if (params) {
    const ParamSplit ps = param_split(g);
    param_load(p, param_channel(ps, 0), ps.first, ps.step, pb);
  }
  cp_async_wait_all();
  if (params) {
    const ParamSplit ps = param_split(g);
    param_warp_sum(p, ps, param_channel(ps, 0), pb, wpart);
  }
  __syncthreads();
  for (int64_t pi = tid; pi < nch * nsl; pi += nt) {
    const int64_t j = pi % nch;
    const int s = (int)(pi / nch);
    float2 t = make_float2(0.f, 0.f);
    for (int64_t t1 = s; t1 < g.Tp; t1 += nsl) {
      const float2 v = rec(j, t1);
      t.x += v.x;
      t.y += v.y;
    }
    part[s * nch + j] = t;
  }
  __syncthreads();
  const float hw = (float)g.HW;
  for (int64_t j = tid; j < nch; j += nt) {
    float2 t = part[j];
    for (int s = 1; s < nsl; ++s) {
      t.x += part[s * nch + j].x;
      t.y += part[s * nch + j].y;
    }
    const float v = j == tid ? cin : chan_in(j);
    stage[j] = kBwd ? channel_terms(v, t) : channel_moments(v, t, hw);
  }
  if (params) param_write(p, param_split(g), 0, wpart);
  __syncthreads();
  for (int64_t q = tid; q < ngr; q += nt) {
    const int64_t gi = g0 + q;
    float2 v;
    if (kBwd) {
      v = group_coef(stage + q * g.Cg, g, q == tid ? rin : __ldg(p.rstd + n * g.G + gi));
    } else {
      v = group_moments(stage + q * g.Cg, g, p.eps);
      if (gi >= wa && gi < wb) {
        p.mean[n * g.G + gi] = v.x;
        p.rstd[n * g.G + gi] = v.y;
      }
    }
    grp[q] = v;
  }
  __syncthreads();
  if (params) {  // further rounds when a CTA has more channels than slots
    const ParamSplit ps = param_split(g);
    const int64_t rounds = (ps.kmax + ps.nslot - 1) / ps.nslot;
    for (int64_t round = 1; round < rounds; ++round) {
      param_load(p, param_channel(ps, round), ps.first, ps.step, pb);
      param_warp_sum(p, ps, param_channel(ps, round), pb, wpart);
      __syncthreads();
      param_write(p, ps, round, wpart);
      __syncthreads();
    }
  }
  return grp;
}

}  // namespace gn
