// gn_resident.cu -- the cluster-resident regime: one kernel per op.
//
// A thread-block cluster of K CTAs owns one reduction unit -- one (n, g)
// span for NCHW (Cg channel planes, contiguous), one sample n for NHWC (HW
// rows of C channels, contiguous) -- and each CTA owns one contiguous slice of
// it (NCHW: 1/m of one channel plane, K = Cg*m; NHWC: HW/K rows).
//
//   pass 1  TMA bulk copies bring the slice into shared memory in chunks: the
//           first nres chunks into slots of their own (all issued at once),
//           the rest through an S-slot ring.  Every chunk is folded into the
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
#include "gn_finalize.cuh"

namespace gn {
namespace {

struct ResCtx {
  const Geom& g;
  char* res;
  char* ring;
  float* red;
  float* xch;
  float* tot;
  float* grp;
  uint64_t* bar;
  int* abort_flag;
};

__device__ __forceinline__ bool res_wait(const ResCtx& c, uint64_t* bar, uint32_t parity,
                                         unsigned* err) {
  if (*reinterpret_cast<volatile int*>(c.abort_flag)) return false;
  if (mbar_wait(bar, parity, err)) return true;
  *reinterpret_cast<volatile int*>(c.abort_flag) = 1;
  return false;
}

template <typename T, int VW, int LAYOUT, bool BWD>
__global__ void __launch_bounds__(512, 1) resident_kernel(const __grid_constant__ KParams p) {
  extern __shared__ __align__(128) char smem[];
  const Geom& g = p.g;
  constexpr int ESZ = sizeof(T);
  constexpr int NT_TENS = BWD ? 2 : 1;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int64_t unit = blockIdx.x / g.K;
  const int tid = threadIdx.x, nt = blockDim.x;
  __shared__ int s_abort;

  ResCtx cx{g,
            smem,
            smem + g.off_ring,
            reinterpret_cast<float*>(smem + g.off_red),
            reinterpret_cast<float*>(smem + g.off_xch),
            reinterpret_cast<float*>(smem + g.off_tot),
            reinterpret_cast<float*>(smem + g.off_grp),
            reinterpret_cast<uint64_t*>(smem + g.off_bar),
            &s_abort};
  const T* x = static_cast<const T*>(p.x);
  const T* dy = static_cast<const T*>(p.dy);
  T* out = static_cast<T*>(p.out);

  // ---- this CTA's slice [e0, e1) of the flat tensor
  int64_t n, e0, e1, chan = 0;
  if (LAYOUT == kNCHW) {
    n = unit / g.G;
    const int64_t gi = unit % g.G;
    chan = gi * g.Cg + rank / g.m;
    const int64_t h0 = (int64_t)(rank % g.m) * g.slice;
    const int64_t h1 = (h0 + g.slice < g.HW) ? h0 + g.slice : g.HW;
    e0 = (n * g.C + chan) * g.HW + h0;
    e1 = (n * g.C + chan) * g.HW + (h1 > h0 ? h1 : h0);
  } else {
    n = unit;
    const int64_t r0 = (int64_t)rank * g.slice;
    const int64_t r1 = (r0 + g.slice < g.HW) ? r0 + g.slice : g.HW;
    e0 = (n * g.HW + r0) * g.C;
    e1 = (n * g.HW + (r1 > r0 ? r1 : r0)) * g.C;
  }
  const int64_t ce = LAYOUT == kNCHW ? g.chunk : g.chunk * g.C;  // elements per chunk
  const int nch = (int)((e1 - e0 + ce - 1) / ce);
  const int nres = nch < g.nres ? nch : g.nres;
  const int nstr = nch - nres;
  const int S = g.S;
  const size_t slot_bytes = (size_t)g.chunk_bytes * NT_TENS;

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < g.nres + S; ++i) mbar_init(cx.bar + i, 1);
    fence_mbar_init();
  }
  __syncthreads();

  const uint64_t pol_once = policy_evict_first();  // resident chunks: read once from HBM
  const uint64_t pol_again = policy_evict_last();  // streamed chunks: read again in pass 2
  // Producer (thread 0): chunk i of the slice into `dst`, completing on `bar`.
  auto issue = [&](int i, char* dst, uint64_t* bar, uint64_t pol) {
    const int64_t a = e0 + (int64_t)i * ce;
    const int64_t b = (a + ce < e1) ? a + ce : e1;
    const uint32_t bytes = (uint32_t)((b - a) * ESZ);
    mbar_arrive_expect_tx(bar, bytes * NT_TENS);
    tma_load_1d(dst, x + a, bytes, bar, pol);
    if (BWD) tma_load_1d(dst + g.chunk_bytes, dy + a, bytes, bar, pol);
  };
  // Ring loads are numbered seq = 0 .. 2*nstr-1: pass-1 streamed chunks in
  // order, then the pass-2 reloads newest first.
  auto seq_chunk = [&](int seq) { return seq < nstr ? nres + seq : nch - 1 - (seq - nstr); };
  auto seq_issue = [&](int seq) {
    const int slot = seq % S;
    issue(seq_chunk(seq), cx.ring + slot * slot_bytes, cx.bar + g.nres + slot,
          seq < nstr ? pol_again : pol_once);
  };
  int issued = 0;  // ring loads issued (thread 0's view)
  if (tid == 0) {
    for (int i = 0; i < nres; ++i) issue(i, cx.res + i * slot_bytes, cx.bar + i, pol_once);
    for (; issued < S && issued < 2 * nstr; ++issued) seq_issue(issued);
  }

  // ---- per-thread layout inside a chunk
  // NHWC: thread (r, j) owns column j (VW channels) and rows r, r+rpi, ...
  const int j = LAYOUT == kNHWC ? tid % g.Wv : 0;
  const int rl = LAYOUT == kNHWC ? tid / g.Wv : 0;
  const bool col_ok = LAYOUT == kNHWC ? rl < g.rpi : true;
  float K[VW];  // forward shift: x(n, c, hw = 0) (NHWC per channel, NCHW per group)
  if (!BWD) {
    if (LAYOUT == kNHWC) {
      if (col_ok) Access<T, VW>::load(x + n * g.HW * g.C + j * VW, K, pol_once);
    } else {
      const float k0 = Elem<T>::to_f(x[(n * g.C + (unit % g.G) * g.Cg) * g.HW]);
#pragma unroll
      for (int k = 0; k < VW; ++k) K[k] = k0;
    }
  }
  float mu[VW];  // backward: the group mean of each owned channel
  if (BWD) {
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      const int64_t c = LAYOUT == kNHWC ? (int64_t)j * VW + k : chan;
      mu[k] = (LAYOUT == kNCHW || col_ok) ? __ldg(p.mean + n * g.G + c / g.Cg) : 0.f;
    }
  }
  float acc[2 * VW];
#pragma unroll
  for (int q = 0; q < 2 * VW; ++q) acc[q] = 0.f;

  using Raw = typename Access<T, VW>::Raw;
  // Folds one chunk (at `slot`, chunk index i) into acc.
  auto consume = [&](const char* slot, int i) {
    const int64_t a = e0 + (int64_t)i * ce;
    const int64_t cnt = ((a + ce < e1) ? a + ce : e1) - a;  // elements
    if (LAYOUT == kNCHW) {
      const int64_t nv = cnt / VW;
      for (int64_t v = tid; v < nv; v += nt) {
        float xv[VW];
        Access<T, VW>::unpack(*reinterpret_cast<const Raw*>(slot + v * 16), xv);
        if (BWD) {
          float dv[VW];
          Access<T, VW>::unpack(*reinterpret_cast<const Raw*>(slot + g.chunk_bytes + v * 16), dv);
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
      const int64_t rows = cnt / g.C;
      for (int64_t r = rl; r < rows; r += g.rpi) {
        const int64_t off = (r * g.C + (int64_t)j * VW) * ESZ;
        float xv[VW];
        Access<T, VW>::unpack(*reinterpret_cast<const Raw*>(slot + off), xv);
        if (BWD) {
          float dv[VW];
          Access<T, VW>::unpack(*reinterpret_cast<const Raw*>(slot + g.chunk_bytes + off), dv);
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

  // ---- pass 1
  for (int i = 0; i < nres; ++i)
    if (res_wait(cx, cx.bar + i, 0, p.err)) consume(cx.res + i * slot_bytes, i);
  for (int seq = 0; seq < nstr; ++seq) {
    const int slot = seq % S;
    if (res_wait(cx, cx.bar + g.nres + slot, (seq / S) & 1, p.err))
      consume(cx.ring + slot * slot_bytes, seq_chunk(seq));
    __syncthreads();  // the slot is free again
    if (tid == 0 && issued < 2 * nstr && !s_abort) {
      fence_proxy_async_smem();
      seq_issue(issued++);
    }
  }

  // ---- reduce: CTA, then cluster (every CTA sums the K partials in rank order)
  if (LAYOUT == kNCHW) {
    const float2 t = block_sum2_t0(acc[0], acc[1], cx.red);
    if (tid == 0) {
      cx.xch[0] = t.x;
      cx.xch[1] = t.y;
    }
  } else {
    const int tpb = nt;
#pragma unroll
    for (int q = 0; q < 2 * VW; ++q) cx.red[q * tpb + tid] = acc[q];
    __syncthreads();
    for (int s = 1; s < g.rpi; s <<= 1) {
      if (col_ok && (rl % (2 * s)) == 0 && rl + s < g.rpi) {
#pragma unroll
        for (int q = 0; q < 2 * VW; ++q) cx.red[q * tpb + tid] += cx.red[q * tpb + tid + s * g.Wv];
      }
      __syncthreads();
    }
    if (rl == 0) {
#pragma unroll
      for (int k = 0; k < VW; ++k) {
        cx.xch[2 * (j * VW + k)] = cx.red[(2 * k) * tpb + tid];
        cx.xch[2 * (j * VW + k) + 1] = cx.red[(2 * k + 1) * tpb + tid];
      }
    }
  }
  cluster.sync();

  // Per-thread output constants: y = (x - mu)*a + b, or
  // dx = A*dy + B*(x - mu) + D.
  float ca[VW], cb[VW], cm[VW], cd[VW];
  const float hwf = (float)g.HW;
  const float mf = (float)(g.Cg * g.HW);
  if (LAYOUT == kNCHW) {
    if (tid == 0) {
      if (!BWD) {
        float s = 0.f, q = 0.f;
        for (int r = 0; r < g.K; ++r) {
          const float* rem = cluster.map_shared_rank(cx.xch, r);
          s += rem[0];
          q += rem[1];
        }
        const float sm = s / mf;
        const float var = fmaxf(fmaf(-s, sm, q), 0.f) / mf;
        cx.grp[0] = K[0] + sm;                  // mean
        cx.grp[1] = 1.0f / sqrtf(var + p.eps);  // rstd
      } else {
        // per channel of the group: sum of the m pieces, then the group sums
        float c1 = 0.f, c2 = 0.f;
        for (int64_t cl = 0; cl < g.Cg; ++cl) {
          float s1 = 0.f, s2 = 0.f;
          for (int q = 0; q < g.m; ++q) {
            const float* rem = cluster.map_shared_rank(cx.xch, (int)(cl * g.m + q));
            s1 += rem[0];
            s2 += rem[1];
          }
          const int64_t c = (unit % g.G) * g.Cg + cl;
          if (rank == 0) p.chst[n * g.C + c] = make_float2(s1, s2);
          const float gm = p.gamma ? __ldg(p.gamma + c) : 1.0f;
          c1 = fmaf(gm, s1, c1);
          c2 = fmaf(gm, s2, c2);
        }
        const float r = __ldg(p.rstd + unit);
        cx.grp[0] = -(r * r * r) * c2 / mf;  // B
        cx.grp[1] = -r * c1 / mf;            // D
      }
    }
    __syncthreads();
    if (!BWD) {
      const float m_ = cx.grp[0], r = cx.grp[1];
      if (rank == 0 && tid == 0) {
        p.mean[unit] = m_;
        p.rstd[unit] = r;
      }
      cm[0] = m_;
      ca[0] = p.gamma ? r * __ldg(p.gamma + chan) : r;
      cb[0] = p.beta ? __ldg(p.beta + chan) : 0.f;
    } else {
      const float r = __ldg(p.rstd + unit);
      cm[0] = mu[0];
      ca[0] = p.gamma ? r * __ldg(p.gamma + chan) : r;
      cb[0] = cx.grp[0];
      cd[0] = cx.grp[1];
    }
  } else {
    // channel totals (rank order), then per group
    for (int64_t c = tid; c < g.C; c += nt) {
      float s = 0.f, q = 0.f;
      for (int r = 0; r < g.K; ++r) {
        const float* rem = cluster.map_shared_rank(cx.xch, r);
        s += rem[2 * c];
        q += rem[2 * c + 1];
      }
      if (!BWD) {
        const float K0 = Elem<T>::to_f(x[n * g.HW * g.C + c]);
        const float sm = s / hwf;
        cx.tot[2 * c] = K0 + sm;                          // mean_c
        cx.tot[2 * c + 1] = fmaxf(fmaf(-s, sm, q), 0.f);  // M2_c
      } else {
        cx.tot[2 * c] = s;
        cx.tot[2 * c + 1] = q;
        if (rank == 0) p.chst[n * g.C + c] = make_float2(s, q);
      }
    }
    __syncthreads();
    for (int64_t gi = tid; gi < g.G; gi += nt) {
      const float* ts = cx.tot + 2 * gi * g.Cg;
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
        cx.grp[2 * gi] = mg;
        cx.grp[2 * gi + 1] = r;
        if (rank == 0) {
          p.mean[n * g.G + gi] = mg;
          p.rstd[n * g.G + gi] = r;
        }
      } else {
        float c1 = 0.f, c2 = 0.f;
        for (int64_t k = 0; k < g.Cg; ++k) {
          const float gm = p.gamma ? __ldg(p.gamma + gi * g.Cg + k) : 1.0f;
          c1 = fmaf(gm, ts[2 * k], c1);
          c2 = fmaf(gm, ts[2 * k + 1], c2);
        }
        const float r = __ldg(p.rstd + n * g.G + gi);
        cx.grp[2 * gi] = -(r * r * r) * c2 / mf;  // B
        cx.grp[2 * gi + 1] = -r * c1 / mf;        // D
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      const int64_t c = (int64_t)j * VW + k;
      const int64_t gi = c / g.Cg;
      if (!col_ok) {
        cm[k] = ca[k] = cb[k] = cd[k] = 0.f;
        continue;
      }
      if (!BWD) {
        const float r = cx.grp[2 * gi + 1];
        cm[k] = cx.grp[2 * gi];
        ca[k] = p.gamma ? r * __ldg(p.gamma + c) : r;
        cb[k] = p.beta ? __ldg(p.beta + c) : 0.f;
      } else {
        const float r = __ldg(p.rstd + n * g.G + gi);
        cm[k] = mu[k];
        ca[k] = p.gamma ? r * __ldg(p.gamma + c) : r;
        cb[k] = cx.grp[2 * gi];
        cd[k] = cx.grp[2 * gi + 1];
      }
    }
  }

  // ---- pass 2: outputs
  const uint64_t pol_out = policy_evict_first();
  auto produce = [&](const char* slot, int i) {
    const int64_t a = e0 + (int64_t)i * ce;
    const int64_t cnt = ((a + ce < e1) ? a + ce : e1) - a;
    if (LAYOUT == kNCHW) {
      const int64_t nv = cnt / VW;
      for (int64_t v = tid; v < nv; v += nt) {
        float xv[VW];
        Access<T, VW>::unpack(*reinterpret_cast<const Raw*>(slot + v * 16), xv);
        if (BWD) {
          float dv[VW];
          Access<T, VW>::unpack(*reinterpret_cast<const Raw*>(slot + g.chunk_bytes + v * 16), dv);
#pragma unroll
          for (int k = 0; k < VW; ++k) xv[k] = fmaf(ca[0], dv[k], fmaf(cb[0], xv[k] - cm[0], cd[0]));
        } else {
#pragma unroll
          for (int k = 0; k < VW; ++k) xv[k] = fmaf(xv[k] - cm[0], ca[0], cb[0]);
        }
        Access<T, VW>::store(out + a + v * VW, xv, pol_out);
      }
    } else if (col_ok) {
      const int64_t rows = cnt / g.C;
      for (int64_t r = rl; r < rows; r += g.rpi) {
        const int64_t eoff = r * g.C + (int64_t)j * VW;
        float xv[VW];
        Access<T, VW>::unpack(*reinterpret_cast<const Raw*>(slot + eoff * ESZ), xv);
        if (BWD) {
          float dv[VW];
          Access<T, VW>::unpack(*reinterpret_cast<const Raw*>(slot + g.chunk_bytes + eoff * ESZ), dv);
#pragma unroll
          for (int k = 0; k < VW; ++k) xv[k] = fmaf(ca[k], dv[k], fmaf(cb[k], xv[k] - cm[k], cd[k]));
        } else {
#pragma unroll
          for (int k = 0; k < VW; ++k) xv[k] = fmaf(xv[k] - cm[k], ca[k], cb[k]);
        }
        Access<T, VW>::store(out + a + eoff, xv, pol_out);
      }
    }
  };
  for (int seq = nstr; seq < 2 * nstr; ++seq) {
    const int slot = seq % S;
    if (res_wait(cx, cx.bar + g.nres + slot, (seq / S) & 1, p.err))
      produce(cx.ring + slot * slot_bytes, seq_chunk(seq));
    __syncthreads();
    if (tid == 0 && issued < 2 * nstr && !s_abort) {
      fence_proxy_async_smem();
      seq_issue(issued++);
    }
  }
  if (!s_abort)
    for (int i = nres - 1; i >= 0; --i) produce(cx.res + i * slot_bytes, i);

  // ---- after an abandoned wait: drain this CTA's own copies (bounded)
  __syncthreads();
  if (s_abort && tid == 0) {
    for (int i = 0; i < nres; ++i) mbar_wait(cx.bar + i, 0, p.err);
    for (int seq = 0; seq < issued; ++seq)
      mbar_wait(cx.bar + g.nres + seq % S, (seq / S) & 1, p.err);
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
      finalize_params(p, cx.red);
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

}  // namespace

const void* resident_kernel_ptr(const Geom& g, bool bwd) {
  switch (g.dtype) {
    case kF32: return pick<float>(g.layout, bwd);
    case kF16: return pick<__half>(g.layout, bwd);
    default: return pick<__nv_bfloat16>(g.layout, bwd);
  }
}

cudaError_t launch_resident(const KParams& p, cudaStream_t s, bool bwd) {
  const Geom& g = p.g;
  const void* fn = resident_kernel_ptr(g, bwd);
  cudaError_t e = prepare_resident_kernel(fn, g);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(g.units * g.K), 1, 1);
  cfg.blockDim = dim3((unsigned)g.tpb, 1, 1);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)g.K;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<KParams*>(&p)};
  const TimingEvents& ev = timing_events();
  if (ev.begin) cudaEventRecord(ev.begin, s);
  e = cudaLaunchKernelExC(&cfg, fn, args);
  if (ev.mid) cudaEventRecord(ev.mid, s);
  if (ev.end) cudaEventRecord(ev.end, s);
  return e;
}

}  // namespace gn
