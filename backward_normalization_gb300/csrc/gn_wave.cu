// gn_wave.cu -- the wave regime: one persistent kernel per op that reads its
// input from HBM once and writes its output once, for problems whose
// reduction units fit in the shared memory of the CTAs that share them.
//
// Work.  A reduction unit is one (sample, group) span for NCHW -- Cg
// contiguous channel planes -- or one (sample, block of Cb channels made of
// whole groups) for NHWC -- HW rows of Cb channels, read as 2-D TMA tiles
// from the [N*HW, C] view.  A unit is cut into P pieces: for NCHW wm
// consecutive segments of each plane (P = Cg*wm), for NHWC blocks of wR
// rows.  Pieces are numbered unit-major, q = u*P + t, and CTA b of the NC
// co-resident CTAs takes pieces q = k*NC + b for k = 0, 1, ... (its steps).
// The plan makes P divide NC where it can, so that the pieces of a unit all
// belong to one step and arrive together.
//
// Per piece: bulk (TMA) copies bring it into one of S shared-memory slots,
// S-1 pieces ahead of the one in use; the CTA reduces it, writes one record
// per channel to the workspace and arrives on the unit's counter; it waits
// (bounded) until all P pieces of the unit have arrived, merges the unit's
// records in a fixed order into the group statistics (forward) or the dx
// coefficients (backward), and writes the piece's output from shared memory.
// x (and dy) are read from HBM once.
//
// A CTA waits for other CTAs' pieces, so all CTAs must be co-resident: the
// kernel is launched cooperatively.  Deadlock-freedom: a CTA publishes its
// piece of step k before it waits for that piece's unit.  Take the smallest
// unit u that some CTA waits for.  Every owner of a piece of u has published
// it, or is still in an earlier step, whose piece has a smaller index and so
// belongs to a unit smaller than u (an owner holds at most one piece of a
// unit, since P <= NC); by the minimality of u those steps complete, so every
// piece of u is published.
//
// The counters start from whatever the workspace holds: CTA 0 zero-fills the
// error word and the counters, and a grid-wide barrier, entered after each
// CTA has issued its first copies (whose latency hides it), orders that
// before any arrival.  Every wait is bounded in time; one that runs out sets
// a bit of the error word (gn_workspace_status reports it), after which every
// CTA skips its remaining work, waiting only for its own copies in flight.
//
// Statistics.  A forward record is, per (piece, channel), the mean and the
// sum of squared deviations M2 of the piece's values, accumulated about the
// piece's first value (a shift that keeps the sums small).  The records of a
// channel are merged in piece order with the pairwise update of Chan, Golub
// and LeVeque (counts na, nb: delta = mean_b - mean_a, mean = mean_a +
// delta*nb/(na+nb), M2 = M2_a + M2_b + delta^2*na*nb/(na+nb)), and the
// channels of a group by M2_g = sum M2_c + HW * sum (mean_c - mean_g)^2, the
// same identity for equal counts.  A backward record is, per (piece,
// channel), sum(dy) and sum(dy*(x - mean)), added per channel in piece order.
// Every CTA of a unit merges the same records in the same order, so all of
// them use identical statistics; results are bit-identical from run to run.
#include <cooperative_groups.h>

#include "gn_finalize.cuh"

namespace gn {
namespace {

constexpr uint64_t kWaveWaitNs = 500ull * 1000 * 1000;  // bound of every wait: 0.5 s

// Error word bits of this kernel.
constexpr unsigned kErrData = 1u;   // a piece's copy did not land in time
constexpr unsigned kErrUnit = 4u;   // a unit's pieces did not all arrive in time

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool aborted(const unsigned* err) {
  return *reinterpret_cast<const volatile unsigned*>(err) != 0u;
}

// Thread 0: waits for phase `parity` of `bar`, bounded in time.  Gives up at
// once when another CTA has already raised the error word.
__device__ bool wait_bar_t0(uint64_t* bar, uint32_t parity, unsigned* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  for (;;) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (now_ns() - t0 > kWaveWaitNs) {
      atomicOr(err, kErrData);
      return false;
    }
  }
}

// Thread 0: waits until the counter reaches `want` (acquire), bounded in time;
// gives up when the error word is raised.
__device__ bool wait_count_t0(const unsigned* ctr, unsigned want, unsigned* err) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v == want) return true;
    if ((i & 15) == 15) {
      if (aborted(err)) return false;
      const uint64_t t = now_ns();
      if (t0 == 0) {
        t0 = t;
      } else if (t - t0 > kWaveWaitNs) {
        atomicOr(err, kErrUnit);
        return false;
      }
    }
    __nanosleep(20);
  }
}

// Pairwise merge of (count, mean, M2) accumulators (Chan, Golub, LeVeque).
struct Moments {
  float n, mean, m2;
};
__device__ __forceinline__ void merge_into(Moments& a, float nb, float mb, float m2b) {
  const float n = a.n + nb;
  const float delta = mb - a.mean;
  const float f = nb / n;
  a.mean = fmaf(delta, f, a.mean);
  a.m2 = a.m2 + m2b + delta * delta * a.n * f;
  a.n = n;
}

// The piece that CTA `b` processes at step k, decoded.
struct Piece {
  int64_t q, u, t;
  int64_t n;       // sample
  int64_t gi;      // NCHW: the unit's group
  int64_t c;       // NCHW: the piece's channel
  int64_t e0;      // NCHW: first element (flat offset)
  int64_t len;     // NCHW: elements; NHWC: rows
  int64_t cb;      // NHWC: channel block of the unit
  int64_t cbase;   // NHWC: first channel of the unit
  int64_t r0;      // NHWC: first row (within the sample)
};

template <int LAYOUT>
__device__ __forceinline__ Piece piece_of(const Geom& g, int64_t q) {
  Piece pc;
  pc.q = q;
  pc.u = q / g.wP;
  pc.t = q - pc.u * g.wP;
  if (LAYOUT == kNCHW) {
    pc.n = pc.u / g.G;
    pc.gi = pc.u - pc.n * g.G;
    const int64_t plane = pc.t / g.wm, seg = pc.t - plane * g.wm;
    pc.c = pc.gi * g.Cg + plane;
    const int64_t h0 = seg * g.wR;
    pc.len = (h0 + g.wR < g.HW) ? g.wR : g.HW - h0;
    pc.e0 = (pc.n * g.C + pc.c) * g.HW + h0;
    pc.cb = pc.cbase = pc.r0 = 0;
  } else {
    pc.n = pc.u / g.ncbu;
    pc.cb = pc.u - pc.n * g.ncbu;
    pc.cbase = pc.cb * g.Cb;
    pc.r0 = pc.t * g.wR;
    pc.len = (pc.r0 + g.wR < g.HW) ? g.wR : g.HW - pc.r0;
    pc.gi = pc.c = pc.e0 = 0;
  }
  return pc;
}

// Number of values of piece t of a unit (rows for NHWC, elements for NCHW).
__device__ __forceinline__ float piece_count(const Geom& g, int64_t t) {
  const int64_t seg = g.layout == kNCHW ? t % g.wm : t;
  const int64_t a = seg * g.wR;
  return (float)((a + g.wR < g.HW) ? g.wR : g.HW - a);
}

template <typename T, int VW, int LAYOUT, bool BWD>
__global__ void __launch_bounds__(kWaveThreads, 1) wave_kernel(const __grid_constant__ KParams p) {
  extern __shared__ __align__(128) char smem_raw[];
  char* smem =
      reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const Geom& g = p.g;
  constexpr int NTEN = BWD ? 2 : 1;
  const int tid = threadIdx.x;
  const int nt = blockDim.x;
  char* ring = smem + g.off_ring;
  float* red = reinterpret_cast<float*>(smem + g.off_red);    // CTA sums, then the unit's records
  float2* chs = reinterpret_cast<float2*>(smem + g.off_tot);  // per-channel results of the unit
  float2* grp = reinterpret_cast<float2*>(smem + g.off_grp);  // per-group results of the unit
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + g.off_bar);
  __shared__ int s_ok;
  __shared__ int s_last;

  const int64_t NC = gridDim.x;
  const int64_t total = g.units * g.wP;
  const int64_t K = blockIdx.x < total ? (total - 1 - blockIdx.x) / NC + 1 : 0;
  const int S = g.S;
  const size_t slot_bytes = (size_t)g.ten_stride * NTEN;
  const int64_t P = g.wP;
  const T* x = static_cast<const T*>(p.x);
  const T* dy = static_cast<const T*>(p.dy);
  T* out = static_cast<T*>(p.out);

  if (tid == 0) {
    for (int i = 0; i < S; ++i) mbar_init(full + i, 1);
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_wait();  // earlier work on the stream (the inputs, the workspace) is done
  grid_launch_dependents();

  // ---- copies: piece k of this CTA into slot k % S (thread 0)
  const uint64_t pol_in = policy_evict_first();
  auto issue = [&](int64_t k) {
    const Piece pc = piece_of<LAYOUT>(g, k * NC + blockIdx.x);
    char* dst = ring + (k % S) * slot_bytes;
    uint64_t* bar = full + (k % S);
    if (LAYOUT == kNCHW) {
      const uint32_t bytes = (uint32_t)(pc.len * (int64_t)sizeof(T));
      mbar_arrive_expect_tx(bar, bytes * NTEN);
      tma_load_1d(dst, x + pc.e0, bytes, bar, pol_in);
      if (BWD) tma_load_1d(dst + g.ten_stride, dy + pc.e0, bytes, bar, pol_in);
    } else {
      const uint32_t box = (uint32_t)(g.chunk * g.Cb * (int64_t)sizeof(T));
      mbar_arrive_expect_tx(bar, box * (uint32_t)g.wnb * NTEN);
      for (int64_t b = 0; b < g.wnb; ++b) {
        const int32_t row = (int32_t)(pc.n * g.HW + pc.r0 + b * g.chunk);
        tma_load_2d(dst + b * box, &p.tmx, (int32_t)pc.cbase, row, bar, pol_in);
        if (BWD) tma_load_2d(dst + g.ten_stride + b * box, &p.tmdy, (int32_t)pc.cbase, row, bar, pol_in);
      }
    }
  };
  int64_t issued = 0;  // thread 0: pieces whose copies were issued
  if (tid == 0)
    for (; issued < K && issued < S - 1; ++issued) issue(issued);

  // ---- the counters start from whatever the workspace held: clear them
  // once, then a grid barrier before any arrival
  if (blockIdx.x == 0)
    for (int i = tid; i < p.clear_words; i += nt) p.err[i] = 0u;
  cooperative_groups::this_grid().sync();

  // NHWC thread layout: column j (VW channels of the block) of rows rl,
  // rl + rpi, ...; NCHW: the piece's 16-byte vectors tid, tid + nt, ...
  const int Wv = LAYOUT == kNHWC ? (int)(g.Cb / VW) : 1;
  const int rpi = LAYOUT == kNHWC ? nt / Wv : nt;
  const int j = LAYOUT == kNHWC ? tid % Wv : 0;
  const int rl = LAYOUT == kNHWC ? tid / Wv : tid;
  const bool lane_ok = LAYOUT == kNHWC ? rl < rpi : true;
  const int64_t rowb = g.Cb * (int64_t)sizeof(T);  // NHWC: bytes per row in a slot
  const uint64_t pol_out = policy_evict_first();
  const int64_t nch = LAYOUT == kNHWC ? g.Cb : 1;  // channels of a piece
  const int64_t rec_per_unit = P * nch;

  int64_t k = 0;
  bool ok = true;
  for (; k < K; ++k) {
    if (tid == 0 && issued < K && issued == k + S - 1) {
      fence_proxy_async_smem();  // the slot's previous reads precede the new copy
      issue(issued);
      ++issued;
    }
    const Piece pc = piece_of<LAYOUT>(g, k * NC + blockIdx.x);
    const char* slot = ring + (k % S) * slot_bytes;
    const uint32_t parity = (uint32_t)((k / S) & 1);
    if (tid == 0) s_ok = aborted(p.err) ? 0 : (wait_bar_t0(full + (k % S), parity, p.err) ? 1 : 0);
    __syncthreads();
    if (!s_ok) {
      ok = false;
      break;
    }
    mbar_try_wait(full + (k % S), parity);  // completed: orders this thread's reads after the copy

    // ---- reduce the piece: one record per channel
    const int64_t rbase = pc.u * rec_per_unit + pc.t * nch;  // first record of the piece
    float2* rec_g = p.part + rbase;
    float2* rec_s = reinterpret_cast<float2*>(red) + pc.t * nch;  // P == 1: kept in smem
    if (LAYOUT == kNCHW) {
      const float mu = BWD ? __ldg(p.mean + pc.u) : 0.f;
      const float K0 = BWD ? 0.f : Elem<T>::to_f(reinterpret_cast<const T*>(slot)[0]);
      float a = 0.f, b = 0.f;
      const int64_t nv = pc.len / VW;
      for (int64_t v = tid; v < nv; v += nt) {
        float xv[VW];
        Access<T, VW>::unpack(lds16(slot + v * 16), xv);
        if (BWD) {
          float dv[VW];
          Access<T, VW>::unpack(lds16(slot + g.ten_stride + v * 16), dv);
#pragma unroll
          for (int e = 0; e < VW; ++e) {
            a += dv[e];
            b = fmaf(dv[e], xv[e] - mu, b);
          }
        } else {
#pragma unroll
          for (int e = 0; e < VW; ++e) {
            const float d = xv[e] - K0;
            a += d;
            b = fmaf(d, d, b);
          }
        }
      }
      const float2 s2 = block_sum2_t0(a, b, red + 2 * rec_per_unit);
      if (tid == 0) {
        float2 r;
        if (BWD) {
          r = s2;
        } else {
          const float n = (float)pc.len;
          const float q = s2.x / n;
          r = make_float2(K0 + q, fmaxf(fmaf(-s2.x, q, s2.y), 0.f));
        }
        if (P > 1) rec_g[0] = r;
        else rec_s[0] = r;
      }
    } else {
      float acc[2 * VW], Ks[VW];
#pragma unroll
      for (int q = 0; q < 2 * VW; ++q) acc[q] = 0.f;
      {
        float mu[VW];
#pragma unroll
        for (int e = 0; e < VW; ++e) mu[e] = 0.f;
        if (lane_ok) {
          if (BWD) {
#pragma unroll
            for (int e = 0; e < VW; ++e)
              mu[e] = __ldg(p.mean + pc.n * g.G + (pc.cbase + j * VW + e) / g.Cg);
          } else {
            Access<T, VW>::unpack(lds16(slot + j * 16), Ks);  // the piece's first row
          }
          for (int64_t r = rl; r < pc.len; r += rpi) {
            float xv[VW];
            Access<T, VW>::unpack(lds16(slot + r * rowb + j * 16), xv);
            if (BWD) {
              float dv[VW];
              Access<T, VW>::unpack(lds16(slot + g.ten_stride + r * rowb + j * 16), dv);
#pragma unroll
              for (int e = 0; e < VW; ++e) {
                acc[2 * e] += dv[e];
                acc[2 * e + 1] = fmaf(dv[e], xv[e] - mu[e], acc[2 * e + 1]);
              }
            } else {
#pragma unroll
              for (int e = 0; e < VW; ++e) {
                const float d = xv[e] - Ks[e];
                acc[2 * e] += d;
                acc[2 * e + 1] = fmaf(d, d, acc[2 * e + 1]);
              }
            }
          }
        }
      }
      // CTA sums: every (column, value) adds its rpi row lanes in lane order
      float* cred = red + 2 * rec_per_unit;  // after the records kept in smem
#pragma unroll
      for (int q = 0; q < 2 * VW; ++q) cred[q * nt + tid] = acc[q];
      if (!BWD && rl == 0 && lane_ok) {
        float* ksh = cred + 2 * VW * nt;
#pragma unroll
        for (int e = 0; e < VW; ++e) ksh[j * VW + e] = Ks[e];
      }
      __syncthreads();
      const float n = (float)pc.len;
      for (int64_t c = tid; c < g.Cb; c += nt) {
        const int jj = (int)(c / VW), e = (int)(c % VW);
        float sa = 0.f, sb = 0.f;
        for (int r = 0; r < rpi; ++r) {
          sa += cred[(2 * e) * nt + r * Wv + jj];
          sb += cred[(2 * e + 1) * nt + r * Wv + jj];
        }
        float2 rr;
        if (BWD) {
          rr = make_float2(sa, sb);
        } else {
          const float Kc = cred[2 * VW * nt + c];
          const float q = sa / n;
          rr = make_float2(Kc + q, fmaxf(fmaf(-sa, q, sb), 0.f));
        }
        if (P > 1) rec_g[c] = rr;
        else rec_s[c] = rr;
      }
    }

    // ---- publish the piece's records, wait for the unit
    __syncthreads();
    if (P > 1) {
      if (tid == 0) {
        if (!(p.stall_unit == pc.u && pc.t == 0))
          asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.tickets + pc.u) : "memory");
        s_ok = wait_count_t0(p.tickets + pc.u, (unsigned)P, p.err) ? 1 : 0;
      }
      __syncthreads();
      if (!s_ok) {
        ok = false;
        ++k;  // this piece's data was consumed
        break;
      }
      // the unit's records into shared memory (one round trip)
      const float2* src = p.part + pc.u * rec_per_unit;
      float2* dst = reinterpret_cast<float2*>(red);
      for (int64_t i = tid; i < rec_per_unit; i += nt) dst[i] = __ldcg(src + i);
      __syncthreads();
    }

    // ---- merge: per channel over the pieces (piece order), then per group
    const float2* recs = reinterpret_cast<const float2*>(red);
    if (LAYOUT == kNCHW) {
      // channel cl of the group: pieces cl*wm .. cl*wm + wm - 1
      for (int64_t cl = tid; cl < g.Cg; cl += nt) {
        if (BWD) {
          float sa = 0.f, sb = 0.f;
          for (int64_t s = 0; s < g.wm; ++s) {
            const float2 v = recs[cl * g.wm + s];
            sa += v.x;
            sb += v.y;
          }
          chs[cl] = make_float2(sa, sb);
        } else {
          Moments m = {0.f, 0.f, 0.f};
          for (int64_t s = 0; s < g.wm; ++s) {
            const float2 v = recs[cl * g.wm + s];
            merge_into(m, piece_count(g, s), v.x, v.y);
          }
          chs[cl] = make_float2(m.mean, m.m2);
        }
      }
      __syncthreads();
      if (tid == 0) {
        const int64_t c0 = pc.gi * g.Cg;
        if (BWD) {
          float c1 = 0.f, c2 = 0.f;
          for (int64_t cl = 0; cl < g.Cg; ++cl) {
            const float2 t2 = channel_terms(p.gamma ? __ldg(p.gamma + c0 + cl) : 1.0f, chs[cl]);
            c1 += t2.x;
            c2 += t2.y;
          }
          grp[0] = coef_from(c1, c2, g, __ldg(p.rstd + pc.u));
        } else {
          grp[0] = group_moments(chs, g, p.eps);
        }
      }
    } else {
      for (int64_t c = tid; c < g.Cb; c += nt) {
        if (BWD) {
          float sa = 0.f, sb = 0.f;
          for (int64_t t = 0; t < P; ++t) {
            const float2 v = recs[t * g.Cb + c];
            sa += v.x;
            sb += v.y;
          }
          chs[c] = make_float2(sa, sb);
        } else {
          Moments m = {0.f, 0.f, 0.f};
          for (int64_t t = 0; t < P; ++t) {
            const float2 v = recs[t * g.Cb + c];
            merge_into(m, piece_count(g, t), v.x, v.y);
          }
          chs[c] = make_float2(m.mean, m.m2);
        }
      }
      __syncthreads();
      const int64_t gb = g.Cb / g.Cg, g0 = pc.n * g.G + pc.cbase / g.Cg;
      for (int64_t q = tid; q < gb; q += nt) {
        if (BWD) {
          float c1 = 0.f, c2 = 0.f;
          for (int64_t cl = 0; cl < g.Cg; ++cl) {
            const int64_t c = pc.cbase + q * g.Cg + cl;
            const float2 t2 = channel_terms(p.gamma ? __ldg(p.gamma + c) : 1.0f, chs[q * g.Cg + cl]);
            c1 += t2.x;
            c2 += t2.y;
          }
          grp[q] = coef_from(c1, c2, g, __ldg(p.rstd + g0 + q));
        } else {
          grp[q] = group_moments(chs + q * g.Cg, g, p.eps);
        }
      }
    }
    __syncthreads();

    // ---- the unit's outputs that the first piece writes: mean / rstd, or
    // the per-channel sums for dgamma / dbeta
    if (pc.t == 0) {
      if (LAYOUT == kNCHW) {
        if (BWD) {
          for (int64_t cl = tid; cl < g.Cg; cl += nt) p.chst[pc.n * g.C + pc.gi * g.Cg + cl] = chs[cl];
        } else if (tid == 0) {
          p.mean[pc.u] = grp[0].x;
          p.rstd[pc.u] = grp[0].y;
        }
      } else {
        if (BWD) {
          for (int64_t c = tid; c < g.Cb; c += nt) p.chst[pc.n * g.C + pc.cbase + c] = chs[c];
        } else {
          const int64_t g0 = pc.n * g.G + pc.cbase / g.Cg;
          for (int64_t q = tid; q < g.Cb / g.Cg; q += nt) {
            p.mean[g0 + q] = grp[q].x;
            p.rstd[g0 + q] = grp[q].y;
          }
        }
      }
    }

    // ---- output of the piece, from shared memory
    if (LAYOUT == kNCHW) {
      float ca, cb, cm, cd;
      if (BWD) {
        const float r = __ldg(p.rstd + pc.u);
        ca = r * (p.gamma ? __ldg(p.gamma + pc.c) : 1.0f);
        cm = __ldg(p.mean + pc.u);
        cb = grp[0].x;
        cd = grp[0].y;
      } else {
        cm = grp[0].x;
        ca = grp[0].y * (p.gamma ? __ldg(p.gamma + pc.c) : 1.0f);
        cb = p.beta ? __ldg(p.beta + pc.c) : 0.f;
        cd = 0.f;
      }
      const int64_t nv = pc.len / VW;
      T* o = out + pc.e0;
      for (int64_t v = tid; v < nv; v += nt) {
        float xv[VW];
        Access<T, VW>::unpack(lds16(slot + v * 16), xv);
        if (BWD) {
          float dv[VW];
          Access<T, VW>::unpack(lds16(slot + g.ten_stride + v * 16), dv);
#pragma unroll
          for (int e = 0; e < VW; ++e) xv[e] = fmaf(ca, dv[e], fmaf(cb, xv[e] - cm, cd));
        } else {
#pragma unroll
          for (int e = 0; e < VW; ++e) xv[e] = fmaf(xv[e] - cm, ca, cb);
        }
        Access<T, VW>::store(o + v * VW, xv, pol_out);
      }
    } else if (lane_ok) {
      float ca[VW], cb[VW], cm[VW], cd[VW];
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        const int64_t cl = (int64_t)j * VW + e;
        const int64_t c = pc.cbase + cl;
        const int64_t q = cl / g.Cg;
        const float gm = p.gamma ? __ldg(p.gamma + c) : 1.0f;
        if (BWD) {
          const int64_t gidx = pc.n * g.G + c / g.Cg;
          ca[e] = __ldg(p.rstd + gidx) * gm;
          cm[e] = __ldg(p.mean + gidx);
          cb[e] = grp[q].x;
          cd[e] = grp[q].y;
        } else {
          cm[e] = grp[q].x;
          ca[e] = grp[q].y * gm;
          cb[e] = p.beta ? __ldg(p.beta + c) : 0.f;
          cd[e] = 0.f;
        }
      }
      T* o = out + (pc.n * g.HW + pc.r0) * g.C + pc.cbase + (int64_t)j * VW;
      for (int64_t r = rl; r < pc.len; r += rpi) {
        float xv[VW];
        Access<T, VW>::unpack(lds16(slot + r * rowb + j * 16), xv);
        if (BWD) {
          float dv[VW];
          Access<T, VW>::unpack(lds16(slot + g.ten_stride + r * rowb + j * 16), dv);
#pragma unroll
          for (int e = 0; e < VW; ++e) xv[e] = fmaf(ca[e], dv[e], fmaf(cb[e], xv[e] - cm[e], cd[e]));
        } else {
#pragma unroll
          for (int e = 0; e < VW; ++e) xv[e] = fmaf(xv[e] - cm[e], ca[e], cb[e]);
        }
        Access<T, VW>::store(o + r * g.C, xv, pol_out);
      }
    }

    // ---- backward: the column's dgamma / dbeta once its N units are done
    if (BWD && pc.t == 0 && (p.dgamma || p.dbeta)) {
      __syncthreads();  // this unit's chst stores, before thread 0's arrival
      const int64_t col = LAYOUT == kNCHW ? pc.gi : pc.cb;
      if (tid == 0) s_last = publish_and_arrive(p.cnt1 + col, (unsigned)g.N);
      __syncthreads();
      if (s_last) {
        // channels [ca, cb) of the column, samples in fixed slices
        const int64_t ca = LAYOUT == kNCHW ? pc.gi * g.Cg : pc.cbase;
        const int64_t cw = LAYOUT == kNCHW ? g.Cg : g.Cb;
        float* sm = red;
        const SliceLayout L = slice_layout(cw, g.N);
        for (int64_t c0 = 0; c0 < cw; c0 += L.cpb) {
          const int64_t c = ca + c0 + L.cl;
          float db = 0.f, dg = 0.f;
          if (L.sl < L.nsl && c0 + L.cl < cw) {
            const int64_t gi = c / g.Cg;
            for (int64_t n = L.sl; n < g.N; n += 8 * L.nsl) {
              float2 v[8];
              float r[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int64_t jn = n + u * L.nsl;
                v[u] = jn < g.N ? __ldcg(p.chst + jn * g.C + c) : make_float2(0.f, 0.f);
                r[u] = jn < g.N ? __ldg(p.rstd + jn * g.G + gi) : 0.f;
              }
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                db += v[u].x;
                dg = fmaf(r[u], v[u].y, dg);
              }
            }
          }
          if (L.sl < L.nsl) {
            sm[2 * (L.sl * L.cpb + L.cl)] = db;
            sm[2 * (L.sl * L.cpb + L.cl) + 1] = dg;
          }
          __syncthreads();
          if (L.sl == 0 && c0 + L.cl < cw) {
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
    }
    __syncthreads();  // the slot and the shared scratch are free again
  }

  // ---- after a wait ran out: this CTA's copies still in flight land before it exits
  if (!ok && tid == 0) {
    for (int64_t i = k; i < issued; ++i) wait_bar_t0(full + (i % S), (uint32_t)((i / S) & 1), p.err);
  }
}

template <typename T, int VW, int LAYOUT, bool BWD>
const void* kernel_ptr() {
  return (const void*)wave_kernel<T, VW, LAYOUT, BWD>;
}

template <typename T>
const void* pick(int layout, bool bwd) {
  constexpr int V = Elem<T>::VEC;
  if (layout == kNCHW)
    return bwd ? kernel_ptr<T, V, kNCHW, true>() : kernel_ptr<T, V, kNCHW, false>();
  return bwd ? kernel_ptr<T, V, kNHWC, true>() : kernel_ptr<T, V, kNHWC, false>();
}

}  // namespace

const void* wave_kernel_ptr(const Geom& g, bool bwd) {
  switch (g.dtype) {
    case kF32: return pick<float>(g.layout, bwd);
    case kF16: return pick<__half>(g.layout, bwd);
    default: return pick<__nv_bfloat16>(g.layout, bwd);
  }
}

cudaError_t launch_wave(const KParams& p_in, cudaStream_t s, bool bwd) {
  KParams p = p_in;
  const Geom& g = p.g;
  cudaError_t e;
  if (g.layout == kNHWC) {
    e = encode_nhwc_map(&p.tmx, p.x, g);
    if (e == cudaSuccess && bwd) e = encode_nhwc_map(&p.tmdy, p.dy, g);
    if (e != cudaSuccess) return e;
  }
  const void* fn = wave_kernel_ptr(g, bwd);
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)g.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)g.grid, 1, 1);
  cfg.blockDim = dim3((unsigned)g.tpb, 1, 1);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&p};
  e = cudaLaunchKernelExC(&cfg, fn, args);
  const TimingEvents& ev = timing_events();
  if (ev.mid) cudaEventRecord(ev.mid, s);
  if (ev.end) cudaEventRecord(ev.end, s);
  return e;
}

}  // namespace gn
