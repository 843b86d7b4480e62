// gn_resident.cu -- the cluster-resident regime: one kernel per op.
//
// A thread-block cluster of K CTAs owns one reduction unit made of whole
// groups: for NCHW one (n, g) span (Cg channel planes, contiguous), for NHWC
// one (sample n, block of Cb channels) -- HW rows of Cb channels, read as 2-D
// TMA tiles from a [N*HW, C] view.  Each CTA owns a contiguous slice of the
// unit (NCHW: 1/m of one channel plane, K = Cg*m; NHWC: HW/K rows).
//
//   pass 1  TMA copies bring the slice into shared memory in chunks: the
//           first nres chunks into slots of their own (all issued at once),
//           the rest through an S-slot ring.  Each chunk is folded into the
//           per-channel (NHWC) or per-slice (NCHW) sums as it lands.
//   reduce  CTA tree, then every CTA adds the K partials of the cluster in
//           rank order through DSMEM, so all CTAs hold identical statistics.
//   pass 2  the output (y, or dx) is computed from shared memory; the
//           streamed chunks are copied in again, newest first, so they come
//           from L2 rather than HBM.
//
// HBM traffic is the minimum (read x [, dy], write y or dx) whenever the
// streamed part of the units in flight stays in L2.  No grid-wide
// synchronisation is used: clusters are independent, and the backward's
// dgamma/dbeta step runs in the cluster whose arrival completes the last unit.
//
// Every mbarrier wait is bounded.  A wait that runs out raises the workspace
// error word; the CTA then stops computing, still takes part in every cluster
// barrier, and before exiting waits (bounded) for the copies it issued.
#include <cudaTypedefs.h>

#include "gn_finalize.cuh"

namespace gn {
namespace {

__device__ __forceinline__ bool res_wait(int* abort_flag, uint64_t* bar, uint32_t parity,
                                         unsigned* err) {
  if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
  if (mbar_wait(bar, parity, err)) return true;
  *reinterpret_cast<volatile int*>(abort_flag) = 1;
  return false;
}

// Sum of a float2 held at `local + 2*idx` in every CTA of the cluster, in
// rank order (at most 16 ranks; the remote loads are all issued first).
__device__ __forceinline__ float2 cluster_sum_at(cg::cluster_group& cluster, float* local,
                                                 int64_t idx, int K) {
  float2 v[16];
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    if (r < K) {
      const float* rem = cluster.map_shared_rank(local, r);
      v[r] = *reinterpret_cast<const float2*>(rem + 2 * idx);
    } else {
      v[r] = make_float2(0.f, 0.f);
    }
  }
  float2 s = make_float2(0.f, 0.f);
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    s.x += v[r].x;
    s.y += v[r].y;
  }
  return s;
}

// Consumer-only barrier (hardware barrier 1): the producer warp does not take
// part.
__device__ __forceinline__ void csync(int ncpad) { named_sync(1, ncpad); }

// Block sum of two values over the consumer threads (fixed order); the
// totals are returned in thread 0.  `scratch` holds 64 floats.
__device__ __forceinline__ float2 consumer_sum2_t0(float a, float b, float* scratch, int ncpad) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = warp_sum_lane0(a);
  b = warp_sum_lane0(b);
  if (lane == 0) {
    scratch[2 * warp] = a;
    scratch[2 * warp + 1] = b;
  }
  csync(ncpad);
  float2 r = make_float2(0.f, 0.f);
  if (threadIdx.x == 0)
    for (int w = 0; w < ncpad / 32; ++w) {
      r.x += scratch[2 * w];
      r.y += scratch[2 * w + 1];
    }
  csync(ncpad);
  return r;
}

template <typename T, int VW, int LAYOUT, bool BWD>
__global__ void __launch_bounds__(544, 1) resident_kernel(const __grid_constant__ KParams p) {
  extern __shared__ __align__(128) char smem_raw[];
  // TMA tile destinations need 128-byte alignment: align the base here (the
  // plan reserves 128 bytes of slack)
  char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const Geom& g = p.g;
  constexpr int ESZ = sizeof(T);
  constexpr int NTEN = BWD ? 2 : 1;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int64_t unit = blockIdx.x / g.K;
  const int tid = threadIdx.x;
  const int nc = g.tpb;                   // consumer threads doing work
  const int ncpad = (nc + 31) / 32 * 32;  // consumer threads (whole warps)
  const int ncw = ncpad / 32;             // consumer warps
  const bool producer = tid >= ncpad;     // the last warp issues the TMA copies
  __shared__ int s_abort;

  char* res = smem;
  char* ring = smem + g.off_ring;
  float* red = reinterpret_cast<float*>(smem + g.off_red);
  float* xch = reinterpret_cast<float*>(smem + g.off_xch);
  float* tot = reinterpret_cast<float*>(smem + g.off_tot);
  float* grp = reinterpret_cast<float*>(smem + g.off_grp);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + g.off_bar);
  uint64_t* empty = full + g.nres + g.S;
  const T* x = static_cast<const T*>(p.x);
  const T* dy = static_cast<const T*>(p.dy);
  T* out = static_cast<T*>(p.out);

  // ---- this CTA's slice
  // NCHW: elements [e0, e1) of one channel plane.  NHWC: rows [r0, r1) of
  // sample n, channels [cbase, cbase + Cb).
  int64_t n, e0 = 0, e1 = 0, chan = 0, r0 = 0, r1 = 0, cbase = 0, ngrp0;
  int nch;
  if (LAYOUT == kNCHW) {
    n = unit / g.G;
    const int64_t gi = unit % g.G;
    chan = gi * g.Cg + rank / g.m;
    const int64_t h0 = (int64_t)(rank % g.m) * g.slice;
    const int64_t h1 = (h0 + g.slice < g.HW) ? h0 + g.slice : g.HW;
    e0 = (n * g.C + chan) * g.HW + h0;
    e1 = (n * g.C + chan) * g.HW + (h1 > h0 ? h1 : h0);
    nch = (int)((e1 - e0 + g.chunk - 1) / g.chunk);
    ngrp0 = unit;  // index of the unit's (only) group in mean/rstd
  } else {
    n = unit / g.ncbu;
    cbase = (unit % g.ncbu) * g.Cb;
    r0 = (int64_t)rank * g.slice;
    r1 = (r0 + g.slice < g.HW) ? r0 + g.slice : g.HW;
    if (r1 < r0) r1 = r0;
    nch = (int)((r1 - r0 + g.chunk - 1) / g.chunk);
    ngrp0 = n * g.G + cbase / g.Cg;
  }
  const int nres = nch < g.nres ? nch : g.nres;
  const int nstr = nch - nres;
  const int S = g.S;
  const size_t slot_bytes = (size_t)g.ten_stride * NTEN;  // slots stay 128-byte aligned

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < g.nres + S; ++i) mbar_init(full + i, 1);
    for (int i = 0; i < S; ++i) mbar_init(empty + i, (uint32_t)ncw);
    fence_mbar_init();
  }
  __syncthreads();

  const uint64_t pol_once = policy_evict_first();  // resident chunks: read once from HBM
  const uint64_t pol_again = policy_evict_last();  // streamed chunks: read again in pass 2
  // chunk i of the slice into `dst`, completing on `b`
  auto issue = [&](int i, char* dst, uint64_t* b, uint64_t pol) {
    if (LAYOUT == kNCHW) {
      const int64_t a = e0 + (int64_t)i * g.chunk;
      const int64_t e = (a + g.chunk < e1) ? a + g.chunk : e1;
      const uint32_t bytes = (uint32_t)((e - a) * ESZ);
      mbar_arrive_expect_tx(b, bytes * NTEN);
      tma_load_1d(dst, x + a, bytes, b, pol);
      if (BWD) tma_load_1d(dst + g.ten_stride, dy + a, bytes, b, pol);
    } else {
      // a full box is always transferred; rows past the slice are ignored
      const int32_t row = (int32_t)(n * g.HW + r0 + (int64_t)i * g.chunk);
      mbar_arrive_expect_tx(b, (uint32_t)g.chunk_bytes * NTEN);
      tma_load_2d(dst, &p.tmx, (int32_t)cbase, row, b, pol);
      if (BWD) tma_load_2d(dst + g.ten_stride, &p.tmdy, (int32_t)cbase, row, b, pol);
    }
  };
  // Ring loads are numbered seq = 0 .. 2*nstr-1: pass-1 streamed chunks in
  // order, then the pass-2 reloads newest first.  Load seq uses slot seq % S;
  // it is issued once every consumer warp has released the slot's previous
  // load (phase seq/S - 1 of that slot's empty barrier).
  auto seq_chunk = [&](int seq) { return seq < nstr ? nres + seq : nch - 1 - (seq - nstr); };
  int issued = 0;  // producer lane 0: ring loads issued
  auto produce_until = [&](int upto) {
    for (; issued < upto; ++issued) {
      const int slot = issued % S;
      if (issued >= S) {
        if (!res_wait(&s_abort, empty + slot, ((issued / S) - 1) & 1, p.err)) return;
        fence_proxy_async_smem();  // the consumers' reads of the slot precede the new copy
      }
      issue(seq_chunk(issued), ring + slot * slot_bytes, full + g.nres + slot,
            issued < nstr ? pol_again : pol_once);
    }
  };
  const bool lead = producer && (tid & 31) == 0;
  if (lead) {
    for (int i = 0; i < nres; ++i) issue(i, res + i * slot_bytes, full + i, pol_once);
    // every pass-1 load, plus the first pass-2 reloads (they land during the reduction)
    produce_until(nstr + S < 2 * nstr ? nstr + S : 2 * nstr);
  }

  // ---- per-thread layout inside a chunk (consumers)
  // NHWC: thread (rl, j) owns column j (VW channels of the block) and rows
  // rl, rl + rpi, ...; NCHW: threads stride the chunk's 16-byte vectors.
  const bool worker = tid < nc;
  const int j = LAYOUT == kNHWC ? tid % g.Wv : 0;
  const int rl = LAYOUT == kNHWC ? tid / g.Wv : 0;
  const bool col_ok = worker && (LAYOUT == kNHWC ? rl < g.rpi : true);
  // Everything the constants need is loaded now; the latency hides under pass 1.
  float K[VW], mu[VW], gmv[VW], btv[VW], rsv[VW];
#pragma unroll
  for (int k = 0; k < VW; ++k) {
    const int64_t c = LAYOUT == kNHWC ? cbase + (int64_t)j * VW + k : chan;
    const int64_t gidx = LAYOUT == kNHWC ? n * g.G + c / g.Cg : unit;
    const bool ok = col_ok && (LAYOUT == kNHWC || k == 0);
    K[k] = 0.f;
    if (!BWD && ok)
      K[k] = LAYOUT == kNHWC ? Elem<T>::to_f(x[n * g.HW * g.C + c])
                             : Elem<T>::to_f(x[(n * g.C + (unit % g.G) * g.Cg) * g.HW]);
    mu[k] = (BWD && ok) ? __ldg(p.mean + gidx) : 0.f;
    rsv[k] = (BWD && ok) ? __ldg(p.rstd + gidx) : 0.f;
    gmv[k] = (ok && p.gamma) ? __ldg(p.gamma + c) : 1.f;
    btv[k] = (!BWD && ok && p.beta) ? __ldg(p.beta + c) : 0.f;
  }
  if (LAYOUT == kNCHW) {
#pragma unroll
    for (int k = 1; k < VW; ++k) {
      K[k] = K[0];
      mu[k] = mu[0];
      rsv[k] = rsv[0];
      gmv[k] = gmv[0];
      btv[k] = btv[0];
    }
  }
  float acc[2 * VW];
#pragma unroll
  for (int q = 0; q < 2 * VW; ++q) acc[q] = 0.f;

  const int64_t rowp = g.Cb * ESZ;  // NHWC: bytes per row in shared memory
  // Folds chunk i (at `slot`) into acc.
  auto consume = [&](const char* slot, int i) {
    if (LAYOUT == kNCHW) {
      if (!worker) return;
      const int64_t a = e0 + (int64_t)i * g.chunk;
      const int64_t nv = (((a + g.chunk < e1) ? a + g.chunk : e1) - a) / VW;
      for (int64_t v = tid; v < nv; v += nc) {
        float xv[VW];
        Access<T, VW>::unpack(lds16(slot + v * 16), xv);
        if (BWD) {
          float dv[VW];
          Access<T, VW>::unpack(lds16(slot + g.ten_stride + v * 16), dv);
#pragma unroll
          for (int k = 0; k < VW; ++k) {
            acc[0] += dv[k];
            acc[1] = fmaf(dv[k], xv[k] - mu[0], acc[1]);
          }
        } else {
#pragma unroll
          for (int k = 0; k < VW; ++k) {
            const float d = xv[k] - K[0];
            acc[0] += d;
            acc[1] = fmaf(d, d, acc[1]);
          }
        }
      }
    } else if (col_ok) {
      const int64_t rs = r0 + (int64_t)i * g.chunk;
      const int64_t rows = ((rs + g.chunk < r1) ? rs + g.chunk : r1) - rs;
      for (int64_t r = rl; r < rows; r += g.rpi) {
        const int64_t off = r * rowp + (int64_t)j * 16;
        float xv[VW];
        Access<T, VW>::unpack(lds16(slot + off), xv);
        if (BWD) {
          float dv[VW];
          Access<T, VW>::unpack(lds16(slot + g.ten_stride + off), dv);
#pragma unroll
          for (int k = 0; k < VW; ++k) {
            acc[2 * k] += dv[k];
            acc[2 * k + 1] = fmaf(dv[k], xv[k] - mu[k], acc[2 * k + 1]);
          }
        } else {
#pragma unroll
          for (int k = 0; k < VW; ++k) {
            const float d = xv[k] - K[k];
            acc[2 * k] += d;
            acc[2 * k + 1] = fmaf(d, d, acc[2 * k + 1]);
          }
        }
      }
    }
  };
  // A consumer warp is done with ring load seq: release its slot.
  auto release = [&](int seq) {
    __syncwarp();
    if ((tid & 31) == 0) mbar_arrive(empty + seq % S);
  };

  float ca[VW], cb[VW], cm[VW], cd[VW];  // output constants (see below)
  if (!producer) {
    // ---- pass 1
    for (int i = 0; i < nres; ++i)
      if (res_wait(&s_abort, full + i, 0, p.err)) consume(res + i * slot_bytes, i);
    for (int seq = 0; seq < nstr; ++seq) {
      if (res_wait(&s_abort, full + g.nres + seq % S, (seq / S) & 1, p.err))
        consume(ring + (seq % S) * slot_bytes, seq_chunk(seq));
      release(seq);
    }
    // ---- reduce within the CTA
    if (LAYOUT == kNCHW) {
      const float2 t = consumer_sum2_t0(acc[0], acc[1], red, ncpad);
      if (tid == 0) {
        xch[0] = t.x;
        xch[1] = t.y;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 2 * VW; ++q) red[q * ncpad + tid] = acc[q];
      csync(ncpad);
      for (int s = 1; s < g.rpi; s <<= 1) {
        if (col_ok && (rl % (2 * s)) == 0 && rl + s < g.rpi) {
#pragma unroll
          for (int q = 0; q < 2 * VW; ++q) red[q * ncpad + tid] += red[q * ncpad + tid + s * g.Wv];
        }
        csync(ncpad);
      }
      if (col_ok && rl == 0) {
#pragma unroll
        for (int k = 0; k < VW; ++k) {
          xch[2 * (j * VW + k)] = red[(2 * k) * ncpad + tid];
          xch[2 * (j * VW + k) + 1] = red[(2 * k + 1) * ncpad + tid];
          if (!BWD) tot[2 * (j * VW + k)] = K[k];  // the channel's shift, for the totals
        }
      }
    }
  }
  cluster.sync();  // every CTA of the cluster has published its partials

  // ---- statistics / coefficients (consumers); the producer keeps loading
  // Output constants: y = (x - cm)*ca + cb, or dx = ca*dy + cb*(x - cm) + cd.
  const float hwf = (float)g.HW;
  const float mf = (float)(g.Cg * g.HW);
  if (producer) {
    if (lead) produce_until(2 * nstr);
  } else if (LAYOUT == kNCHW) {
    if (tid == 0) {
      if (!BWD) {
        const float2 t = cluster_sum_at(cluster, xch, 0, g.K);
        const float sm = t.x / mf;
        const float var = fmaxf(fmaf(-t.x, sm, t.y), 0.f) / mf;
        grp[0] = K[0] + sm;                  // mean
        grp[1] = 1.0f / sqrtf(var + p.eps);  // rstd
        if (rank == 0) {
          p.mean[unit] = grp[0];
          p.rstd[unit] = grp[1];
        }
      } else {
        // per channel of the group: the m pieces in order, then the group sums
        float c1 = 0.f, c2 = 0.f;
        for (int64_t cl = 0; cl < g.Cg; ++cl) {
          float s1 = 0.f, s2 = 0.f;
          for (int64_t q = 0; q < g.m; ++q) {
            const float* rem = cluster.map_shared_rank(xch, (int)(cl * g.m + q));
            s1 += rem[0];
            s2 += rem[1];
          }
          const int64_t c = (unit % g.G) * g.Cg + cl;
          if (rank == 0) p.chst[n * g.C + c] = make_float2(s1, s2);
          const float gm = p.gamma ? __ldg(p.gamma + c) : 1.0f;
          c1 = fmaf(gm, s1, c1);
          c2 = fmaf(gm, s2, c2);
        }
        const float r = rsv[0];
        grp[0] = -(r * r * r) * c2 / mf;  // B
        grp[1] = -r * c1 / mf;            // D
      }
    }
    csync(ncpad);
    const float r = BWD ? rsv[0] : grp[1];
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      cm[k] = BWD ? mu[0] : grp[0];
      ca[k] = r * gmv[0];
      cb[k] = BWD ? grp[0] : btv[0];
      cd[k] = BWD ? grp[1] : 0.f;
    }
  } else {
    // channel totals of the block (rank order), then per group of the block
    for (int64_t c = tid; c < g.Cb; c += ncpad) {
      const float2 t = cluster_sum_at(cluster, xch, c, g.K);
      if (!BWD) {
        const float sm = t.x / hwf;
        tot[2 * c] += sm;                                  // mean_c = shift + S/HW
        tot[2 * c + 1] = fmaxf(fmaf(-t.x, sm, t.y), 0.f);  // M2_c
      } else {
        tot[2 * c] = t.x;
        tot[2 * c + 1] = t.y;
        if (rank == 0) p.chst[n * g.C + cbase + c] = t;
      }
    }
    csync(ncpad);
    const int64_t gb = g.Cb / g.Cg;
    for (int64_t gi = tid; gi < gb; gi += ncpad) {
      const float* ts = tot + 2 * gi * g.Cg;
      if (!BWD) {
        float s = 0.f;
        for (int64_t k = 0; k < g.Cg; ++k) s += ts[2 * k];
        const float mg = s / (float)g.Cg;
        float m2 = 0.f;
        for (int64_t k = 0; k < g.Cg; ++k) {
          const float d = ts[2 * k] - mg;
          m2 += fmaf(hwf * d, d, ts[2 * k + 1]);
        }
        const float r = 1.0f / sqrtf(m2 / mf + p.eps);
        grp[2 * gi] = mg;
        grp[2 * gi + 1] = r;
        if (rank == 0) {
          p.mean[ngrp0 + gi] = mg;
          p.rstd[ngrp0 + gi] = r;
        }
      } else {
        float c1 = 0.f, c2 = 0.f;
        for (int64_t k = 0; k < g.Cg; ++k) {
          const float gm = p.gamma ? __ldg(p.gamma + cbase + gi * g.Cg + k) : 1.0f;
          c1 = fmaf(gm, ts[2 * k], c1);
          c2 = fmaf(gm, ts[2 * k + 1], c2);
        }
        const float r = __ldg(p.rstd + ngrp0 + gi);
        grp[2 * gi] = -(r * r * r) * c2 / mf;  // B
        grp[2 * gi + 1] = -r * c1 / mf;        // D
      }
    }
    csync(ncpad);
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      const int64_t gi = ((int64_t)j * VW + k) / g.Cg;
      if (!col_ok) {
        cm[k] = ca[k] = cb[k] = cd[k] = 0.f;
        continue;
      }
      if (!BWD) {
        const float r = grp[2 * gi + 1];
        cm[k] = grp[2 * gi];
        ca[k] = r * gmv[k];
        cb[k] = btv[k];
        cd[k] = 0.f;
      } else {
        cm[k] = mu[k];
        ca[k] = rsv[k] * gmv[k];
        cb[k] = grp[2 * gi];
        cd[k] = grp[2 * gi + 1];
      }
    }
  }

  // ---- pass 2: outputs (consumers)
  if (!producer) {
    const uint64_t pol_out = policy_evict_first();
    auto emit = [&](const char* slot, int i) {
      if (LAYOUT == kNCHW) {
        if (!worker) return;
        const int64_t a = e0 + (int64_t)i * g.chunk;
        const int64_t nv = (((a + g.chunk < e1) ? a + g.chunk : e1) - a) / VW;
        for (int64_t v = tid; v < nv; v += nc) {
          float xv[VW];
          Access<T, VW>::unpack(lds16(slot + v * 16), xv);
          if (BWD) {
            float dv[VW];
            Access<T, VW>::unpack(lds16(slot + g.ten_stride + v * 16), dv);
#pragma unroll
            for (int k = 0; k < VW; ++k) xv[k] = fmaf(ca[k], dv[k], fmaf(cb[k], xv[k] - cm[k], cd[k]));
          } else {
#pragma unroll
            for (int k = 0; k < VW; ++k) xv[k] = fmaf(xv[k] - cm[k], ca[k], cb[k]);
          }
          Access<T, VW>::store(out + a + v * VW, xv, pol_out);
        }
      } else if (col_ok) {
        const int64_t rs = r0 + (int64_t)i * g.chunk;
        const int64_t rows = ((rs + g.chunk < r1) ? rs + g.chunk : r1) - rs;
        for (int64_t r = rl; r < rows; r += g.rpi) {
          const int64_t off = r * rowp + (int64_t)j * 16;
          float xv[VW];
          Access<T, VW>::unpack(lds16(slot + off), xv);
          if (BWD) {
            float dv[VW];
            Access<T, VW>::unpack(lds16(slot + g.ten_stride + off), dv);
#pragma unroll
            for (int k = 0; k < VW; ++k) xv[k] = fmaf(ca[k], dv[k], fmaf(cb[k], xv[k] - cm[k], cd[k]));
          } else {
#pragma unroll
            for (int k = 0; k < VW; ++k) xv[k] = fmaf(xv[k] - cm[k], ca[k], cb[k]);
          }
          Access<T, VW>::store(out + (n * g.HW + rs + r) * g.C + cbase + (int64_t)j * VW, xv, pol_out);
        }
      }
    };
    for (int seq = nstr; seq < 2 * nstr; ++seq) {
      if (res_wait(&s_abort, full + g.nres + seq % S, (seq / S) & 1, p.err))
        emit(ring + (seq % S) * slot_bytes, seq_chunk(seq));
      release(seq);
    }
    if (!*reinterpret_cast<volatile int*>(&s_abort))
      for (int i = nres - 1; i >= 0; --i) emit(res + i * slot_bytes, i);
  }

  // ---- after an abandoned wait: drain this CTA's own copies (bounded)
  __syncthreads();
  if (s_abort && lead) {
    for (int i = 0; i < nres; ++i) mbar_wait(full + i, 0, p.err);
    for (int seq = 0; seq < issued; ++seq) mbar_wait(full + g.nres + seq % S, (seq / S) & 1, p.err);
  }
  // no CTA leaves while a peer may still read its partials
  cluster.sync();

  // ---- backward: dgamma/dbeta once every unit is done
  if (BWD && rank == 0) {
    __shared__ int s_last;
    __syncthreads();
    if (tid == 0) s_last = publish_and_arrive(p.tickets + g.N, (unsigned)g.units);
    __syncthreads();
    if (s_last) {
      finalize_params(p, red);
      if (tid == 0) atomicExch(p.tickets + g.N, 0u);
    }
  }
}

template <typename T, int VW, int LAYOUT, bool BWD>
const void* kernel_ptr() {
  return (const void*)resident_kernel<T, VW, LAYOUT, BWD>;
}

template <typename T>
const void* pick(int layout, bool bwd) {
  constexpr int V = Elem<T>::VEC;
  if (layout == kNCHW)
    return bwd ? kernel_ptr<T, V, kNCHW, true>() : kernel_ptr<T, V, kNCHW, false>();
  return bwd ? kernel_ptr<T, V, kNHWC, true>() : kernel_ptr<T, V, kNHWC, false>();
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda needed).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      f = nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

}  // namespace

// [N*HW, C] view of an NHWC tensor, boxes of [chunk rows, Cb channels].
cudaError_t encode_nhwc_map(CUtensorMap* map, const void* base, const Geom& g) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const CUtensorMapDataType dt = g.dtype == kF32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : g.dtype == kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int esz = g.dtype == kF32 ? 4 : 2;
  const cuuint64_t dims[2] = {(cuuint64_t)g.C, (cuuint64_t)(g.N * g.HW)};
  const cuuint64_t strides[1] = {(cuuint64_t)(g.C * esz)};
  const cuuint32_t box[2] = {(cuuint32_t)g.Cb, (cuuint32_t)g.chunk};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

const void* resident_kernel_ptr(const Geom& g, bool bwd) {
  switch (g.dtype) {
    case kF32: return pick<float>(g.layout, bwd);
    case kF16: return pick<__half>(g.layout, bwd);
    default: return pick<__nv_bfloat16>(g.layout, bwd);
  }
}

cudaError_t launch_resident(const KParams& p_in, cudaStream_t s, bool bwd) {
  KParams p = p_in;
  const Geom& g = p.g;
  cudaError_t e;
  if (g.layout == kNHWC) {
    e = encode_nhwc_map(&p.tmx, p.x, g);
    if (e == cudaSuccess && bwd) e = encode_nhwc_map(&p.tmdy, p.dy, g);
    if (e != cudaSuccess) return e;
  }
  const void* fn = resident_kernel_ptr(g, bwd);
  e = prepare_resident_kernel(fn, g);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(g.units * g.K), 1, 1);
  cfg.blockDim = dim3((unsigned)resident_threads(g), 1, 1);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)g.K;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&p};
  const TimingEvents& ev = timing_events();
  e = cudaLaunchKernelExC(&cfg, fn, args);
  if (ev.mid) cudaEventRecord(ev.mid, s);
  if (ev.end) cudaEventRecord(ev.end, s);
  return e;
}

}  // namespace gn
