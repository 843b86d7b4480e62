// gn_flat.cu -- the flat regime: one cooperative kernel per op for
// channels-last problems small enough for the whole grid to hold (forward)
// or for L2 to keep between the passes (backward).
//
// Work.  The [N*HW, C] row matrix of a dense channels-last tensor is cut into
// `grid` runs of consecutive rows of (almost) equal length, one CTA per SM:
// CTA b takes rows [b*R/grid, (b+1)*R/grid), R = N*HW.  A run is one
// contiguous span of bytes; it arrives by bulk (TMA) copies of `chunk` rows
// into S shared-memory slots.  A run may cross sample boundaries: the part of
// it inside one sample is a segment, and sums are kept per segment.
//
//   pass 1   every thread owns one 16-byte column (vw channels) and one row
//            lane, and folds the rows of its lane into per-channel sums as the
//            chunks land.  At the end of a segment the CTA adds its lanes in a
//            fixed order and writes one record per group (forward: the mean
//            and M2 of the segment's values of the group) or per channel
//            (backward: sum dy and sum dy*(x - mean)) to the workspace.
//   barrier  a grid-wide barrier (the launch is cooperative, so every CTA is
//            resident at once).
//   merge    every (sample, group) -- backward: every (sample, channel) -- is
//            merged by one CTA, its owner (an equal share of them per CTA), so
//            that each record is read once: forward, one warp per pair, lane l
//            taking the records of CTAs l, l + 32, ... and a fixed xor tree
//            adding the lanes, writes the pair's mean and rstd (the op's
//            outputs); backward, the records of an item are added in a fixed
//            order into the channel totals (sum dy, sum dy*(x - mean)) in the
//            workspace.  A second grid barrier; then every CTA reads what its
//            segments need (forward: mean and rstd; backward: the channel
//            totals, from which it forms the dx coefficients), and the backward
//            adds dgamma / dbeta of its share of the channels over the samples.
//   pass 2   the output is written chunk by chunk in reverse order: the chunks
//            still in their slots first, then the others copied in again (from
//            L2, where pass 1 left them with the evict_last policy).  When a
//            run fits in shared memory (the forward of the problems this
//            regime is chosen for) every chunk stays in its slot, so x is read
//            once; the backward keeps what fits and reads the rest again.
//
// Statistics.  A CTA folds a segment's values of a group about its first one
// (K, the value at the segment's first row and the group's first channel):
// S = sum(x - K), Q = sum((x - K)^2) over its m_i values, and records
// mean_i = K + S/m_i, M2_i = Q - S^2/m_i.  The records of a group merge by
// the parallel-axis identity (Chan, Golub and LeVeque) about the first
// record's mean K0: with d_i = mean_i - K0, A = sum m_i d_i and
// B = sum (M2_i + m_i d_i^2), mean = K0 + A/M and M2 = B - A^2/M, M = Cg*HW;
// var = M2/M (biased).  The backward coefficients follow the two-kernel
// path's (gn_finalize.cuh).
//
// Waits.  Only a slot's copies are waited for: thread 0 polls (the other
// warps wait at a barrier, so the polling takes no issue slots from work),
// bounded at 0.5 s, and the outcome reaches the CTA through shared memory, so
// every thread takes the same branch.  Every CTA reaches the grid barrier whatever
// happened before it; a CTA whose wait ran out skips the rest of its work,
// raises the workspace's error word after the barrier (CTA 0 clears the word
// before it) and waits, bounded, for its copies in flight before returning.
#include <cooperative_groups.h>

#include <type_traits>

#include "gn_finalize.cuh"

namespace gn {
namespace {

constexpr uint64_t kFlatWaitNs = 500ull * 1000 * 1000;  // bound of every wait: 0.5 s
constexpr unsigned kFlatErrData = 1u;                     // a chunk's copy did not land in time

__device__ __forceinline__ uint64_t flat_now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bookkeeping at the end of the CTA's shared memory (kFlatBookBytes).
struct FlatBook {
  uint64_t bar[kFlatMaxSlots];      // one mbarrier per slot
  unsigned issued[kFlatMaxSlots];   // fills of the slot so far (thread 0)
  unsigned pend[kFlatMaxSlots];     // 1: a copy into the slot is in flight (thread 0)
  int flag[2];                      // outcome of the last two waits, for the CTA
  int pad[2];
};
static_assert(sizeof(FlatBook) <= kFlatBookBytes, "flat bookkeeping outgrew its reservation");

// First row of CTA b's run, and the CTA whose run holds row r.
__device__ __forceinline__ int64_t run_start(int64_t b, int64_t R, int64_t nb) { return b * R / nb; }
__device__ __forceinline__ int64_t run_of_row(int64_t r, int64_t R, int64_t nb) {
  return ((r + 1) * nb - 1) / R;
}

// Thread 0: requests chunk k of the run (x, and dy for the backward) into slot
// k % S, completing on the slot's mbarrier.  `withhold` (fault injection)
// arms the barrier for the bytes but issues no copy, so its wait runs out.
template <typename T, bool BWD>
__device__ void flat_issue(const KParams& p, FlatBook* bk, unsigned char* ring, int64_t r0,
                           int64_t nrows, int k, uint64_t pol, bool withhold) {
  const Geom& g = p.g;
  const int q = k % g.S;
  const int64_t k0 = (int64_t)k * g.chunk;
  const int64_t rows = nrows - k0 < g.chunk ? nrows - k0 : g.chunk;
  const uint32_t bytes = (uint32_t)(rows * g.C * (int64_t)sizeof(T));
  unsigned char* dst = ring + (size_t)q * (size_t)g.ten_stride * (BWD ? 2 : 1);
  mbar_arrive_expect_tx(&bk->bar[q], bytes * (BWD ? 2u : 1u));
  bk->issued[q] += 1u;
  if (withhold) return;
  bk->pend[q] = 1u;
  const size_t off = (size_t)(r0 + k0) * (size_t)g.C;
  tma_load_1d(dst, static_cast<const T*>(p.x) + off, bytes, &bk->bar[q], pol);
  if (BWD) tma_load_1d(dst + g.ten_stride, static_cast<const T*>(p.dy) + off, bytes, &bk->bar[q], pol);
}

// Every thread: waits for the fill of slot q requested last.  Thread 0 polls
// (bounded in time); the outcome reaches the CTA
// through flag[w & 1] (w counts the CTA's waits, so a fast thread 0 never
// overwrites a flag that another thread has still to read).  Returns the same
// value in every thread; on success every thread has made its own acquiring
// test of the barrier, which orders its reads of the slot after the copy.
__device__ bool flat_wait(FlatBook* bk, int q, int w) {
  if (threadIdx.x == 0) {
    const uint32_t par = (bk->issued[q] - 1u) & 1u;
    int ok = 1;
    if (!mbar_try_wait(&bk->bar[q], par)) {
      const uint64_t t0 = flat_now_ns();
      for (unsigned i = 1;; ++i) {
        if (mbar_try_wait(&bk->bar[q], par)) break;
        if ((i & 63u) == 0u && flat_now_ns() - t0 > kFlatWaitNs) {
          ok = 0;
          break;
        }
      }
    }
    if (ok) bk->pend[q] = 0u;
    bk->flag[w & 1] = ok ? (int)(2u + par) : 0;
  }
  __syncthreads();
  const int f = bk->flag[w & 1];
  if (f == 0) return false;
  mbar_try_wait(&bk->bar[q], (uint32_t)(f - 2));
  return true;
}

// Thread 0, on the way out of a CTA that gave up: waits (bounded) for every
// copy it issued that is still in flight, so that none lands after the CTA's
// shared memory is released.
__device__ void flat_drain(FlatBook* bk, int S) {
  for (int q = 0; q < S; ++q) {
    if (!bk->pend[q]) continue;
    const uint32_t par = (bk->issued[q] - 1u) & 1u;
    const uint64_t t0 = flat_now_ns();
    while (!mbar_try_wait_hint(&bk->bar[q], par, 1000u))
      if (flat_now_ns() - t0 > kFlatWaitNs) break;
  }
}

template <typename T, int VW, bool BWD>
__global__ void __launch_bounds__(kFlatThreads, 1) flat_kernel(const __grid_constant__ KParams p) {
  using A = Access<T, VW>;
  static_assert(std::is_same<typename A::Raw, uint4>::value, "16-byte vectors");
  const Geom& g = p.g;
  extern __shared__ unsigned char flat_smem[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)flat_smem + 127) & ~(uintptr_t)127);
  unsigned char* ring = sm + g.off_ring;
  float* red = reinterpret_cast<float*>(sm + g.off_red);
  float* tab = reinterpret_cast<float*>(sm + g.off_grp);
  FlatBook* bk = reinterpret_cast<FlatBook*>(sm + g.off_bar);
  // every CTA's run: its first row, and the first and last sample it touches
  // (so that the merge computes no 64-bit quotients)
  int64_t* rs = reinterpret_cast<int64_t*>(sm + g.off_tot);
  int2* rn = reinterpret_cast<int2*>(sm + g.off_tot + (((size_t)gridDim.x + 1) * 8 + 127) / 128 * 128);
  const int tid = threadIdx.x, tpb = blockDim.x;
  const int64_t NB = gridDim.x, b = blockIdx.x;
  const int64_t HW = g.HW, C = g.C, G = g.G, Cg = g.Cg, R = g.N * HW;
  const int64_t rA = run_start(b, R, NB), rB = run_start(b + 1, R, NB), nrows = rB - rA;
  const int S = g.S;
  const int nk = (int)((nrows + g.chunk - 1) / g.chunk);
  const int64_t nA = rA / HW;
  const int nseg = nrows > 0 ? (int)((rB - 1) / HW - nA + 1) : 0;
  const int64_t segmax = g.fSeg, sgn = segmax * G;
  const int Wv = g.Wv, rpi = g.rpi;
  const int j = tid % Wv, lr = tid / Wv;  // this thread's column and row lane
  const int64_t rowb = C * (int64_t)sizeof(T);
  const size_t slotb = (size_t)g.ten_stride * (BWD ? 2 : 1);
  const uint64_t pkeep = policy_evict_last(), pfirst = policy_evict_first();
  // chunks that pass 2 copies in again (k < nk - S) are kept in L2
  auto pol_of = [&](int k) { return k < nk - S ? pkeep : pfirst; };
  if (tid == 0) {
    if (b == 0) *p.err = 0u;
    for (int q = 0; q < S; ++q) {
      mbar_init(&bk->bar[q], 1);
      bk->issued[q] = 0u;
      bk->pend[q] = 0u;
    }
    fence_mbar_init();
    const int n0 = nk < S ? nk : S;
    for (int k = 0; k < n0; ++k)
      flat_issue<T, BWD>(p, bk, ring, rA, nrows, k, pol_of(k), p.stall_unit >= 0 && b == 0 && k == 0);
  }
  // Tables per (segment, group).  Forward: (mean, rstd), then the current
  // segment's shift per group.  Backward: (mean, rstd) (loaded here by the
  // warps other than thread 0's, while it issues the copies), then the dx
  // coefficients (B, D), then one segment's channel terms.
  float2* st = reinterpret_cast<float2*>(tab);
  float* ksh = tab + 2 * sgn;
  float2* mr = reinterpret_cast<float2*>(tab);
  float2* cf = mr + sgn;
  float2* terms = cf + sgn;
  for (int64_t t = tid; t <= NB; t += tpb) {
    rs[t] = run_start(t, R, NB);
    if (t < NB) rn[t] = make_int2((int)(run_start(t, R, NB) / HW), (int)((run_start(t + 1, R, NB) - 1) / HW));
  }
  if (BWD) {
    const int t0 = tpb > 32 ? 32 : 0, nt = tpb - t0;
    for (int64_t t = tid - t0; tid >= t0 && t < (int64_t)nseg * G; t += nt) {
      const int64_t n = nA + t / G, gi = t % G;
      mr[t] = make_float2(__ldg(p.mean + n * G + gi), __ldg(p.rstd + n * G + gi));
    }
  }
  __syncthreads();

  const int64_t cj = (int64_t)j * VW;  // first channel of the column
  int gof[VW];                         // group of each channel of the column
#pragma unroll
  for (int e = 0; e < VW; ++e) gof[e] = (int)((cj + e) / Cg);
  auto seg_begin = [&](int s) -> int64_t {
    const int64_t v = (nA + s) * HW - rA;
    return v > 0 ? v : 0;
  };
  auto seg_end = [&](int s) -> int64_t {
    const int64_t v = (nA + s + 1) * HW - rA;
    return v < nrows ? v : nrows;
  };

  // ---------------------------------------------------------------- pass 1
  float acc[2 * VW];
#pragma unroll
  for (int e = 0; e < 2 * VW; ++e) acc[e] = 0.f;
  float sh[VW];  // the segment's shift (forward) or mean (backward) per channel
  // at the segment's first row (its chunk at `base`, row i0 of the run)
  auto seg_consts = [&](int s, const unsigned char* slot, int64_t k0, int64_t i0) {
    if (BWD) {
#pragma unroll
      for (int e = 0; e < VW; ++e) sh[e] = mr[s * G + gof[e]].x;
    } else {
      const T* row = reinterpret_cast<const T*>(slot + (i0 - k0) * rowb);
#pragma unroll
      for (int e = 0; e < VW; ++e) sh[e] = Elem<T>::to_f(row[(int64_t)gof[e] * Cg]);
      for (int64_t gi = tid; gi < G; gi += tpb) ksh[gi] = Elem<T>::to_f(row[gi * Cg]);
    }
  };
  auto fold = [&](const uint4& vx, const uint4& vd) {
    float xv[VW];
    A::unpack(vx, xv);
    if (BWD) {
      float dv[VW];
      A::unpack(vd, dv);
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        acc[2 * e] += dv[e];
        acc[2 * e + 1] = fmaf(dv[e], xv[e] - sh[e], acc[2 * e + 1]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        const float d = xv[e] - sh[e];
        acc[2 * e] += d;
        acc[2 * e + 1] = fmaf(d, d, acc[2 * e + 1]);
      }
    }
  };
  // rows [i0, i1) of the chunk starting at row k0 (its slot column at `base`)
  auto rows1 = [&](const unsigned char* base, int64_t k0, int64_t i0, int64_t i1) {
    int64_t i = i0 + lr;
    for (; i + 3 * rpi < i1; i += 4 * rpi) {
      uint4 vx[4], vd[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const unsigned char* px = base + (i + u * rpi - k0) * rowb;
        vx[u] = lds16(px);
        vd[u] = BWD ? lds16(px + g.ten_stride) : vx[u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) fold(vx[u], vd[u]);
    }
    for (; i < i1; i += rpi) {
      const unsigned char* px = base + (i - k0) * rowb;
      const uint4 vx = lds16(px);
      const uint4 vd = BWD ? lds16(px + g.ten_stride) : vx;
      fold(vx, vd);
    }
  };
  // End of segment s: the CTA's sums in a fixed order, one record per group
  // (forward) or channel (backward) in the workspace.
  auto flush = [&](int s) {
    if (!BWD) {
      float2* r2 = reinterpret_cast<float2*>(red);
      const int g0 = gof[0];
      for (int kk = 0; kk < g.fNgv; ++kk) {
        float a = 0.f, q2 = 0.f;
#pragma unroll
        for (int e = 0; e < VW; ++e)
          if (gof[e] - g0 == kk) {
            a += acc[2 * e];
            q2 += acc[2 * e + 1];
          }
        r2[kk * tpb + tid] = make_float2(a, q2);
      }
      __syncthreads();
      for (int64_t gi = tid; gi < G; gi += tpb) {
        const int64_t ja = gi * Cg / VW, jb = ((gi + 1) * Cg - 1) / VW;
        float a = 0.f, q2 = 0.f;
        for (int64_t jj = ja; jj <= jb; ++jj) {
          const int kk = (int)(gi - jj * VW / Cg);
          for (int rr = 0; rr < rpi; ++rr) {
            const float2 v = r2[kk * tpb + rr * Wv + jj];
            a += v.x;
            q2 += v.y;
          }
        }
        const float m = (float)((seg_end(s) - seg_begin(s)) * Cg);
        const float sm1 = a / m;
        p.part[(b * segmax + s) * G + gi] = make_float2(ksh[gi] + sm1, fmaxf(fmaf(-a, sm1, q2), 0.f));
      }
    } else {
      const int ld = tpb + 1;  // padded: the column sums below read without bank conflicts
#pragma unroll
      for (int q2 = 0; q2 < 2 * VW; ++q2) red[q2 * ld + tid] = acc[q2];
      __syncthreads();
      for (int64_t c = tid; c < C; c += tpb) {
        const int64_t jj = c / VW;
        const int e = (int)(c - jj * VW);
        float s1 = 0.f, s2 = 0.f;
        for (int rr = 0; rr < rpi; ++rr) {
          s1 += red[(2 * e) * ld + rr * Wv + jj];
          s2 += red[(2 * e + 1) * ld + rr * Wv + jj];
        }
        p.part[(b * segmax + s) * C + c] = make_float2(s1, s2);
      }
    }
#pragma unroll
    for (int e = 0; e < 2 * VW; ++e) acc[e] = 0.f;
    __syncthreads();
  };

  bool ok = true;
  int w = 0;  // the CTA's waits so far
  {
    int s = 0;
    int64_t send = nseg > 0 ? seg_end(0) : 0;
    for (int k = 0; k < nk; ++k) {
      const int q = k % S;
      if (!flat_wait(bk, q, w++)) {
        ok = false;
        break;
      }
      const int64_t k0 = (int64_t)k * g.chunk;
      const int64_t k1 = k0 + g.chunk < nrows ? k0 + g.chunk : nrows;
      const unsigned char* base = ring + (size_t)q * slotb + (size_t)j * 16;
      int64_t i0 = k0;
      while (i0 < k1) {
        const int64_t i1 = send < k1 ? send : k1;
        if (i0 == seg_begin(s)) seg_consts(s, ring + (size_t)q * slotb, k0, i0);
        rows1(base, k0, i0, i1);
        if (i1 == send) {
          flush(s);
          ++s;
          if (s < nseg) send = seg_end(s);
        }
        i0 = i1;
      }
      if (k + S < nk) {
        __syncthreads();  // every thread is done with slot q
        if (tid == 0) {
          fence_proxy_async_smem();
          flat_issue<T, BWD>(p, bk, ring, rA, nrows, k + S, pol_of(k + S), false);
        }
      }
    }
  }

  cooperative_groups::this_grid().sync();

  // ----------------------------------------------------------------- merge
  // Each (sample, group) pair P = n*G + g is merged by one CTA, its owner
  // (CTA b owns P in [b*NG/NB, (b+1)*NG/NB)), so that every record is read
  // once; the owner writes the result (forward: mean and rstd, the op's
  // outputs; backward: the dx coefficients, to the workspace), and after a
  // second grid barrier every CTA reads those of its segments.
  const int lane = tid & 31, warp = tid >> 5, nw = tpb >> 5;  // whole warps (see below)
  const int64_t NG = g.N * G;
  const int64_t P0 = run_start(b, NG, NB), P1 = run_start(b + 1, NG, NB);
  if (ok && !BWD) {
    // one warp per owned pair (a CTA of rpi * Wv threads may end in a partial
    // warp, which takes no part): lane l takes records l, l + 32, ... and
    // a fixed xor tree adds the lanes; a warp has up to kPairs pairs' loads
    // in flight at once
    const float M = (float)(HW * Cg);
    constexpr int kPairs = 3;
    for (int64_t t0 = P0 + warp; warp < nw && t0 < P1; t0 += kPairs * nw) {
      int n4[kPairs], blo[kPairs], bhi[kPairs], gi4[kPairs];  // sample, CTAs, group
      float K0[kPairs];
      float2 v[kPairs][4];
      float mi[kPairs][4];
      auto rec = [&](int pp, int bb) { return p.part + ((int64_t)bb * segmax + (n4[pp] - rn[bb].x)) * G + gi4[pp]; };
      auto cnt = [&](int pp, int bb) {
        const int64_t lo = (int64_t)n4[pp] * HW, hi = lo + HW, ra = rs[bb], rz = rs[bb + 1];
        return (float)(((rz < hi ? rz : hi) - (ra > lo ? ra : lo)) * Cg);
      };
#pragma unroll
      for (int pp = 0; pp < kPairs; ++pp) {
        const int64_t t = t0 + pp * nw;
        const bool live = t < P1;
        n4[pp] = live ? (int)(t / G) : 0;
        gi4[pp] = live ? (int)(t - (int64_t)n4[pp] * G) : 0;
        blo[pp] = (int)run_of_row((int64_t)n4[pp] * HW, R, NB);
        bhi[pp] = live ? (int)run_of_row(((int64_t)n4[pp] + 1) * HW - 1, R, NB) : blo[pp] - 1;
        K0[pp] = live ? __ldcg(rec(pp, blo[pp])).x : 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int bb = blo[pp] + lane + 32 * u;
          const bool in = bb <= bhi[pp];
          v[pp][u] = in ? __ldcg(rec(pp, bb)) : make_float2(0.f, 0.f);
          mi[pp][u] = in ? cnt(pp, bb) : 0.f;
        }
      }
      float A[kPairs], B[kPairs];
#pragma unroll
      for (int pp = 0; pp < kPairs; ++pp) {
        A[pp] = 0.f;
        B[pp] = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float d = v[pp][u].x - K0[pp];
          A[pp] = fmaf(mi[pp][u], d, A[pp]);
          B[pp] += fmaf(mi[pp][u] * d, d, v[pp][u].y);
        }
        for (int bb = blo[pp] + 128 + lane; bb <= bhi[pp]; bb += 32) {
          const float2 w2 = __ldcg(rec(pp, bb));
          const float m = cnt(pp, bb), d = w2.x - K0[pp];
          A[pp] = fmaf(m, d, A[pp]);
          B[pp] += fmaf(m * d, d, w2.y);
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
        for (int pp = 0; pp < kPairs; ++pp) {
          A[pp] += __shfl_xor_sync(0xffffffffu, A[pp], off);
          B[pp] += __shfl_xor_sync(0xffffffffu, B[pp], off);
        }
      }
#pragma unroll
      for (int pp = 0; pp < kPairs; ++pp) {
        const int64_t t = t0 + pp * nw;
        if (lane == 0 && t < P1) {
          const float am = A[pp] / M;
          const float var = fmaxf(fmaf(-A[pp], am, B[pp]), 0.f) / M;
          p.mean[t] = K0[pp] + am;
          p.rstd[t] = 1.0f / sqrtf(var + p.eps);
        }
      }
    }
  } else if (ok) {
    // backward owners take (sample, channel) items I = n*C + c in
    // [b*NC/NB, (b+1)*NC/NB): an item's records are split into `sl` slices of
    // stride sl, a thread per (item, slice) adds its records in order (eight
    // loads in flight), and the slices are added in order into the item's
    // channel totals (sum dy, sum dy*(x - mean)) in the workspace
    const int64_t NC = g.N * C;
    const int64_t I0 = run_start(b, NC, NB), I1 = run_start(b + 1, NC, NB), items = I1 - I0;
    const int sl = items > 0 && tpb / items > 1 ? (int)(tpb / items > 32 ? 32 : tpb / items) : 1;
    const int per = tpb / sl;  // items per round
    float2* part2 = reinterpret_cast<float2*>(red);
    for (int64_t it0 = 0; it0 < items; it0 += per) {
      const int k = tid / sl, slc = tid % sl;
      if (k < per && it0 + k < items) {
        const int64_t I = I0 + it0 + k;
        const int n = (int)(I / C);
        const int64_t c = I - (int64_t)n * C;
        const int blo = (int)run_of_row((int64_t)n * HW, R, NB);
        const int bhi = (int)run_of_row(((int64_t)n + 1) * HW - 1, R, NB);
        float2 t2 = make_float2(0.f, 0.f);
        for (int base = blo + slc; base <= bhi; base += 8 * sl) {
          float2 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int bb = base + u * sl;
            v[u] = bb <= bhi ? __ldcg(p.part + ((int64_t)bb * segmax + (n - rn[bb].x)) * C + c)
                             : make_float2(0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            t2.x += v[u].x;
            t2.y += v[u].y;
          }
        }
        part2[k * sl + slc] = t2;
      }
      __syncthreads();
      for (int k2 = tid; k2 < per && it0 + k2 < items; k2 += tpb) {
        float2 a2 = make_float2(0.f, 0.f);
        for (int q = 0; q < sl; ++q) {
          a2.x += part2[k2 * sl + q].x;
          a2.y += part2[k2 * sl + q].y;
        }
        p.chst[I0 + it0 + k2] = a2;
      }
      __syncthreads();
    }
  }

  cooperative_groups::this_grid().sync();
  if (!ok) {
    if (tid == 0) {
      atomicOr(p.err, kFlatErrData);
      flat_drain(bk, S);
    }
    return;
  }

  if (!BWD) {
    for (int64_t t = tid; t < (int64_t)nseg * G; t += tpb) {
      const int64_t P = nA * G + t;  // segment t / G is sample nA + t / G
      st[t] = make_float2(__ldcg(p.mean + P), __ldcg(p.rstd + P));
    }
    __syncthreads();
  } else {
    // the dx coefficients of this CTA's segments, from the channel totals
    for (int s = 0; s < nseg; ++s) {
      const int64_t n = nA + s;
      for (int64_t c = tid; c < C; c += tpb)
        terms[c] = channel_terms(p.gamma ? __ldg(p.gamma + c) : 1.0f, __ldcg(p.chst + n * C + c));
      __syncthreads();
      for (int64_t gi = tid; gi < G; gi += tpb) cf[s * G + gi] = group_coef(terms + gi * Cg, g, mr[s * G + gi].y);
      __syncthreads();
    }
    // dgamma / dbeta of this CTA's share of the channels, one warp per
    // channel: lane l adds the totals of samples l, l + 32, ... in order
    // (four loads, and their rstd, in flight at once), then a fixed xor tree
    if ((p.dgamma || p.dbeta) && warp < nw) {
      const int64_t ca = run_start(b, C, NB), cb = run_start(b + 1, C, NB);
      const int N = (int)g.N;
      for (int64_t c = ca + warp; c < cb; c += nw) {
        const int64_t gi = c / Cg;
        float db = 0.f, dg = 0.f;
        for (int n0 = lane; n0 < N; n0 += 32 * 4) {
          float2 v[4];
          float r4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int n = n0 + 32 * u;
            v[u] = n < N ? __ldcg(p.chst + (int64_t)n * C + c) : make_float2(0.f, 0.f);
            r4[u] = n < N ? __ldg(p.rstd + (int64_t)n * G + gi) : 0.f;
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            db += v[u].x;
            dg = fmaf(r4[u], v[u].y, dg);
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          db += __shfl_xor_sync(0xffffffffu, db, off);
          dg += __shfl_xor_sync(0xffffffffu, dg, off);
        }
        if (lane == 0) {
          if (p.dbeta) p.dbeta[c] = db;
          if (p.dgamma) p.dgamma[c] = dg;
        }
      }
    }
  }

  // ---------------------------------------------------------------- pass 2
  T* out = static_cast<T*>(p.out) + (size_t)rA * (size_t)C + (size_t)cj;
  // forward: y = (x - m) * a + bb; backward: dx = a * dy + bb * (x - m) + dd
  float ca_[VW], cm_[VW], cb_[VW], cd_[VW];
  auto out_consts = [&](int s) {
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      const int64_t c = cj + e;
      const int gi = gof[e];
      const float gm = p.gamma ? __ldg(p.gamma + c) : 1.0f;
      if (!BWD) {
        const float2 v = st[s * G + gi];
        cm_[e] = v.x;
        ca_[e] = v.y * gm;
        cb_[e] = p.beta ? __ldg(p.beta + c) : 0.0f;
        cd_[e] = 0.f;
      } else {
        const float2 v = mr[s * G + gi], k = cf[s * G + gi];
        cm_[e] = v.x;
        ca_[e] = v.y * gm;
        cb_[e] = k.x;
        cd_[e] = k.y;
      }
    }
  };
  auto apply = [&](const uint4& vx, const uint4& vd, T* dst) {
    float xv[VW];
    A::unpack(vx, xv);
    if (BWD) {
      float dv[VW];
      A::unpack(vd, dv);
#pragma unroll
      for (int e = 0; e < VW; ++e) xv[e] = fmaf(ca_[e], dv[e], fmaf(cb_[e], xv[e] - cm_[e], cd_[e]));
    } else {
#pragma unroll
      for (int e = 0; e < VW; ++e) xv[e] = fmaf(xv[e] - cm_[e], ca_[e], cb_[e]);
    }
    A::store(dst, xv, pfirst);
  };
  auto rows2 = [&](const unsigned char* base, int64_t k0, int64_t i0, int64_t i1) {
    int64_t i = i0 + lr;
    for (; i + 3 * rpi < i1; i += 4 * rpi) {
      uint4 vx[4], vd[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const unsigned char* px = base + (i + u * rpi - k0) * rowb;
        vx[u] = lds16(px);
        vd[u] = BWD ? lds16(px + g.ten_stride) : vx[u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) apply(vx[u], vd[u], out + (i + u * rpi) * C);
    }
    for (; i < i1; i += rpi) {
      const unsigned char* px = base + (i - k0) * rowb;
      const uint4 vx = lds16(px);
      const uint4 vd = BWD ? lds16(px + g.ten_stride) : vx;
      apply(vx, vd, out + i * C);
    }
  };
  if (nk > 0) {
    int s = nseg - 1;
    int64_t sbeg = seg_begin(s);
    out_consts(s);
    for (int k = nk - 1; k >= 0; --k) {
      const int q = k % S;
      if (k < nk - S && !flat_wait(bk, q, w++)) {
        ok = false;
        break;
      }
      const int64_t k0 = (int64_t)k * g.chunk;
      const int64_t k1 = k0 + g.chunk < nrows ? k0 + g.chunk : nrows;
      const unsigned char* base = ring + (size_t)q * slotb + (size_t)j * 16;
      int64_t i1 = k1;
      for (;;) {
        const int64_t i0 = sbeg > k0 ? sbeg : k0;
        rows2(base, k0, i0, i1);
        if (i0 == k0) break;
        --s;
        sbeg = seg_begin(s);
        out_consts(s);
        i1 = i0;
      }
      if (k - S >= 0) {  // chunk k - S left slot q in pass 1: copy it in again
        __syncthreads();
        if (tid == 0) {
          fence_proxy_async_smem();
          flat_issue<T, BWD>(p, bk, ring, rA, nrows, k - S, pfirst, false);
        }
      }
    }
  }
  if (!ok && tid == 0) {
    atomicOr(p.err, kFlatErrData);
    flat_drain(bk, S);
  }
}

template <typename T>
const void* pick_flat(bool bwd) {
  constexpr int V = Elem<T>::VEC;
  return bwd ? (const void*)flat_kernel<T, V, true> : (const void*)flat_kernel<T, V, false>;
}

}  // namespace

const void* flat_kernel_ptr(const Geom& g, bool bwd) {
  switch (g.dtype) {
    case kF32: return pick_flat<float>(bwd);
    case kF16: return pick_flat<__half>(bwd);
    default: return pick_flat<__nv_bfloat16>(bwd);
  }
}

cudaError_t launch_flat(const KParams& p_in, cudaStream_t s, bool bwd) {
  KParams p = p_in;
  const Geom& g = p.g;
  const void* fn = flat_kernel_ptr(g, bwd);
  cudaError_t e = prepare_smem(fn, g.smem);
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
