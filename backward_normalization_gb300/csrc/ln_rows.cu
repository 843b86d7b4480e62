// ln_rows.cu -- LayerNorm and RMSNorm over the last dimension of a row-major
// [M, N] array, forward and backward (include/ln.h), after "Optimize AMD
// normalization backward kernel by using tiled and two pass" (ROCm/pytorch PR
// #3564: layer_norm / rms_norm backward with their gamma/beta gradients).
//
// A row is held in registers by a team of TW threads (a power of two, at most
// the CTA's 256): thread `lane` of the team owns the row's 16-byte vectors
// lane, lane + TW, ..., VPT of them, so its columns are the same for every row
// it visits.  Team sums are xor butterflies (every lane ends with the same
// bits: each pairwise add is commutative) or, for teams wider than a warp,
// per-warp butterflies added in warp order through shared memory.
//
//   forward:  load the row, shifted sums of x and x^2 (one team reduction),
//             mean and biased variance, rstd, then y; one read of x, one
//             write of y.
//   backward: load x and dy rows, xhat and g = gamma*dy, the two row sums,
//             dx; dgamma/dbeta partials stay in registers across the CTA's
//             rows.  The CTA then adds its teams' partials in team order into
//             one record per feature, and a second kernel adds the CTAs'
//             records in CTA order: the two-level deterministic reduction of
//             the GroupNorm path, applied to rows.
// Rows are assigned to CTAs in a fixed grid-stride order (the grid depends
// only on the problem and the device), so results are bit-identical from run
// to run.
#include <cuda_runtime.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/ln.h"
#include "gn_device.cuh"

namespace gn {
namespace {

constexpr int kRowThreads = 256;
// Dynamic shared memory above which a launch must opt in (the 48 KB default,
// less room for the kernels' static shared memory).
constexpr size_t kSmemNoOptIn = 44 * 1024;

struct RowParams {
  const void* x;
  const void* dy;
  void* out;  // y or dx
  const float* gamma;
  const float* beta;
  float* mean;   // forward: written (LayerNorm); backward: read
  float* rstd;   // forward: written; backward: read
  float* dgamma;
  float* dbeta;
  float2* part;  // backward: [grid][N] (dgamma, dbeta) partials
  int64_t M, N, V;  // V: vectors per row
  int64_t ldx, ldd, ldo;  // row strides (elements) of x, dy and the output
  int tw;           // team width
  float eps;
  int want_part;    // backward: 1 if any parameter gradient is wanted
};

// Sum over the team of the pair (a, b) (TW a power of two), one exchange for
// both; `red` holds blockDim/16 floats.  Every thread of the CTA calls it the
// same number of times (the row loops run uniformly over the CTA).  With
// kTeamBar the warps of a team meet on a barrier of their own (hardware
// barrier 1 + team; at most four teams span warps), so teams never wait for
// one another; otherwise the whole CTA meets.  Measured on GB300: team
// barriers speed the forward up (LayerNorm bf16 131072x4096: 477 -> 455 us)
// and slow the backward down (625 -> 638 us), so each kernel takes its own.
template <bool kTeamBar>
__device__ __forceinline__ float2 team_sum2(float a, float b, int tw, float* red) {
  const int w = tw < 32 ? tw : 32;
  for (int o = w >> 1; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  if (tw <= 32) return make_float2(a, b);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red[2 * warp] = a;
    red[2 * warp + 1] = b;
  }
  const int bar = 1 + (int)threadIdx.x / tw;
  if (kTeamBar)
    named_sync(bar, tw);
  else
    __syncthreads();
  const int first = (threadIdx.x / tw) * (tw >> 5);
  float sa = 0.f, sb = 0.f;
  for (int k = 0; k < (tw >> 5); ++k) {
    sa += red[2 * (first + k)];
    sb += red[2 * (first + k) + 1];
  }
  if (kTeamBar)
    named_sync(bar, tw);
  else
    __syncthreads();
  return make_float2(sa, sb);
}

// VW consecutive fp32 values from shared memory (16-byte aligned when VW >= 4).
template <int VW>
__device__ __forceinline__ void load_smem(const float* s, int64_t c0, float (&out)[VW]) {
  if (VW == 8 || VW == 4) {
#pragma unroll
    for (int e = 0; e < VW; e += 4) {
      const float4 f = *reinterpret_cast<const float4*>(s + c0 + e);
      out[e] = f.x;
      out[e + 1] = f.y;
      out[e + 2] = f.z;
      out[e + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < VW; ++e) out[e] = s[c0 + e];
  }
}

// gamma / beta for one vector of features (fp32, VW wide).
template <int VW>
__device__ __forceinline__ void load_param(const float* p, int64_t c0, float dflt,
                                           float (&out)[VW]) {
  if (!p) {
#pragma unroll
    for (int e = 0; e < VW; ++e) out[e] = dflt;
    return;
  }
  if (VW == 8 || VW == 4) {
#pragma unroll
    for (int e = 0; e < VW; e += 4) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(p + c0 + e));
      out[e] = f.x;
      out[e + 1] = f.y;
      out[e + 2] = f.z;
      out[e + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < VW; ++e) out[e] = __ldg(p + c0 + e);
  }
}

// ------------------------------------------------------------------ forward
// Three CTAs per SM (at most 85 registers) while a thread holds at most 64
// bytes of its row: measured on GB300 the large forwards gain (LayerNorm
// bf16 131072x4096 454 -> 443 us, RMSNorm 361 -> 350 us); fp32 threads
// holding 32 values (and the backward, with its dgamma/dbeta registers)
// would spill under that bound.
template <typename T, int VW, int VPT, bool kRms>
__global__ void __launch_bounds__(kRowThreads, (VPT * VW * (int)sizeof(T) > 64 ? 2 : 3))
    row_fwd(const __grid_constant__ RowParams p) {
  __shared__ float red[kRowThreads / 16];
  const int tw = p.tw, team = threadIdx.x / tw, lane = threadIdx.x % tw;
  const int nteams = blockDim.x / tw;
  const float inv_n = 1.0f / (float)p.N;
  const T* x = static_cast<const T*>(p.x);
  T* y = static_cast<T*>(p.out);
  const uint64_t pol = policy_evict_first();
  // rows are software-pipelined: the next row's vectors are requested before
  // the current row's reductions, so two rows per team are in flight
  using Raw = typename Access<T, VW>::Raw;
  Raw cur[VPT], nxt[VPT];
  T kcur{}, knxt{};  // LayerNorm: the row's first element (the shift), fetched with the row
  const int64_t step = (int64_t)gridDim.x * nteams;
  auto fetch = [&](int64_t r0, Raw (&buf)[VPT], T& kb) {
    const int64_t row = r0 + team;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int64_t vi = lane + (int64_t)k * tw;
      buf[k] = (row < p.M && vi < p.V) ? Access<T, VW>::load_raw(x + row * p.ldx + vi * VW, pol) : Raw{};
    }
    if (!kRms && row < p.M) kb = __ldg(x + row * p.ldx);
  };
  int64_t r0 = (int64_t)blockIdx.x * nteams;
  if (r0 < p.M) fetch(r0, cur, kcur);
  // gamma / beta: a thread's columns are the same in every row.  Up to 16
  // values per thread they are loaded once into registers; LayerNorm rows of
  // more are staged once per CTA in shared memory (beta doubles the
  // parameter loads per row).  Measured on GB300: LayerNorm bf16
  // 131072x4096 443 -> 413 us staged; RMSNorm, with gamma alone, was slower
  // staged (350 -> 391 us) and keeps its loads through L1.
  constexpr bool kHoist = VPT * VW <= 16;
  constexpr bool kStage = !kRms && !kHoist;
  constexpr int HV = kHoist ? VPT : 1, HE = kHoist ? VW : 1;
  float gmr[HV][HE], btr[HV][HE];
  if constexpr (kHoist) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int64_t vi = lane + (int64_t)k * tw;
      load_param<VW>(vi < p.V ? p.gamma : nullptr, vi * VW, 1.f, gmr[k]);
      load_param<VW>(kRms || vi >= p.V ? nullptr : p.beta, vi * VW, 0.f, btr[k]);
    }
  }
  extern __shared__ __align__(16) float prm[];  // kStage: gamma [0, N), beta [N, 2N)
  if constexpr (kStage) {
    for (int64_t i = threadIdx.x; i < p.N; i += blockDim.x) {
      prm[i] = p.gamma ? __ldg(p.gamma + i) : 1.f;
      prm[p.N + i] = p.beta ? __ldg(p.beta + i) : 0.f;
    }
    __syncthreads();
  }
  for (; r0 < p.M; r0 += step) {
    if (r0 + step < p.M) fetch(r0 + step, nxt, knxt);
    const int64_t row = r0 + team;
    const bool act = row < p.M;
    float v[VPT][VW];
#pragma unroll
    for (int k = 0; k < VPT; ++k) Access<T, VW>::unpack(cur[k], v[k]);
    // LayerNorm: shifted sums S = sum(x - K), Q = sum((x - K)^2) with K the
    // row's first element, one team reduction for both; mean = K + S/N and
    // var = Q/N - (S/N)^2 (exact in real arithmetic; the shift keeps the
    // subtraction well conditioned, as for the GroupNorm statistics).
    // RMSNorm: Q = sum(x^2).
    const float K = kRms ? 0.f : Elem<T>::to_f(kcur);
    float sx = 0.f, q = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const bool in = act && lane + (int64_t)k * tw < p.V;
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        const float d = in ? v[k][e] - K : 0.f;
        sx += d;
        q = fmaf(d, d, q);
      }
    }
    const float2 t = team_sum2<true>(sx, q, tw, red);
    float mean = 0.f, var;
    if (kRms) {
      var = t.y * inv_n;
    } else {
      const float sm = t.x * inv_n;
      mean = K + sm;
      var = fmaxf(fmaf(-sm, sm, t.y * inv_n), 0.f);
    }
    const float rstd = 1.0f / sqrtf(var + p.eps);
    if (act) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int64_t vi = lane + (int64_t)k * tw;
        if (vi >= p.V) continue;
        float gm[VW], bt[VW];
        if constexpr (kHoist) {
#pragma unroll
          for (int e = 0; e < VW; ++e) {
            gm[e] = gmr[k % HV][e % HE];
            bt[e] = btr[k % HV][e % HE];
          }
        } else if constexpr (kStage) {
          load_smem<VW>(prm, vi * VW, gm);
          load_smem<VW>(prm + p.N, vi * VW, bt);
        } else {
          load_param<VW>(p.gamma, vi * VW, 1.f, gm);
          load_param<VW>(kRms ? nullptr : p.beta, vi * VW, 0.f, bt);
        }
#pragma unroll
        for (int e = 0; e < VW; ++e) v[k][e] = fmaf(v[k][e] - mean, rstd * gm[e], bt[e]);
        Access<T, VW>::store(y + row * p.ldo + vi * VW, v[k], pol);
      }
      if (lane == 0) {
        if (!kRms) p.mean[row] = mean;
        p.rstd[row] = rstd;
      }
    }
#pragma unroll
    for (int k = 0; k < VPT; ++k) cur[k] = nxt[k];
    kcur = knxt;
  }
}

// ----------------------------------------------------------------- backward
// Dynamic shared memory: nteams * N floats for dgamma partials, the same for
// dbeta (teams' per-feature partials before the CTA adds them in team order).
template <typename T, int VW, int VPT, bool kRms>
__global__ void __launch_bounds__(kRowThreads) row_bwd(const __grid_constant__ RowParams p) {
  extern __shared__ __align__(16) float colsum[];
  __shared__ float red[kRowThreads / 16];
  const int tw = p.tw, team = threadIdx.x / tw, lane = threadIdx.x % tw;
  const int nteams = blockDim.x / tw;
  float* gs = colsum + (int64_t)2 * nteams * p.N;  // gamma, staged below
  const float inv_n = 1.0f / (float)p.N;
  const T* x = static_cast<const T*>(p.x);
  const T* dy = static_cast<const T*>(p.dy);
  T* dx = static_cast<T*>(p.out);
  const uint64_t pol = policy_evict_first();
  float pg[VPT][VW], pb[VPT][VW];  // this thread's dgamma / dbeta partials
#pragma unroll
  for (int k = 0; k < VPT; ++k)
#pragma unroll
    for (int e = 0; e < VW; ++e) pg[k][e] = pb[k][e] = 0.f;
  // rows are software-pipelined: x, dy, mean and rstd of the next row are
  // requested before the current row's reductions
  using Raw = typename Access<T, VW>::Raw;
  Raw cx[VPT], cd[VPT], nx[VPT], nd[VPT];
  float cm = 0.f, cr = 0.f, nm = 0.f, nr = 0.f;  // mean, rstd of the current / next row
  const int64_t step = (int64_t)gridDim.x * nteams;
  auto fetch = [&](int64_t r0, Raw (&bx)[VPT], Raw (&bd)[VPT], float& m, float& r) {
    const int64_t row = r0 + team;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int64_t vi = lane + (int64_t)k * tw;
      const bool in = row < p.M && vi < p.V;
      bx[k] = in ? Access<T, VW>::load_raw(x + row * p.ldx + vi * VW, pol) : Raw{};
      bd[k] = in ? Access<T, VW>::load_raw(dy + row * p.ldd + vi * VW, pol) : Raw{};
    }
    m = (!kRms && row < p.M) ? __ldg(p.mean + row) : 0.f;
    r = row < p.M ? __ldg(p.rstd + row) : 0.f;
  };
  int64_t r0 = (int64_t)blockIdx.x * nteams;
  if (r0 < p.M) fetch(r0, cx, cd, cm, cr);
  // gamma (1 without one) staged once per CTA after the partials' area, while
  // the first row is in flight: the rows read it from shared memory instead of
  // reloading it through L1
  for (int64_t c = threadIdx.x; c < p.N; c += blockDim.x) gs[c] = p.gamma ? __ldg(p.gamma + c) : 1.f;
  __syncthreads();
  for (; r0 < p.M; r0 += step) {
    if (r0 + step < p.M) fetch(r0 + step, nx, nd, nm, nr);
    const int64_t row = r0 + team;
    const bool act = row < p.M;
    const float mean = cm, rstd = cr;
    float xv[VPT][VW], dv[VPT][VW];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      Access<T, VW>::unpack(cx[k], xv[k]);
      Access<T, VW>::unpack(cd[k], dv[k]);
    }
    // xhat in xv, g = gamma*dy kept apart from dy (both are needed)
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int64_t vi = lane + (int64_t)k * tw;
      float gm[VW];
      load_smem<VW>(gs, (vi < p.V ? vi : 0) * VW, gm);
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        xv[k][e] = (xv[k][e] - mean) * rstd;
        const float g = gm[e] * dv[k][e];
        s1 += g;
        s2 = fmaf(g, xv[k][e], s2);
      }
    }
    const float2 cs = team_sum2<false>(s1, s2, tw, red);
    const float c1 = kRms ? 0.f : cs.x * inv_n;
    const float c2 = cs.y * inv_n;
    if (act) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int64_t vi = lane + (int64_t)k * tw;
        if (vi >= p.V) continue;
        float gm[VW], o[VW];
        load_smem<VW>(gs, vi * VW, gm);
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          const float g = gm[e] * dv[k][e];
          o[e] = rstd * (g - c1 - xv[k][e] * c2);
          pg[k][e] = fmaf(dv[k][e], xv[k][e], pg[k][e]);
          pb[k][e] += dv[k][e];
        }
        Access<T, VW>::store(dx + row * p.ldo + vi * VW, o, pol);
      }
    }
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      cx[k] = nx[k];
      cd[k] = nd[k];
    }
    cm = nm;
    cr = nr;
  }
  if (!p.want_part) return;
  // the teams' partials -> shared memory -> one record per feature, in team order
  float* sg = colsum;
  float* sb = colsum + (int64_t)nteams * p.N;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int64_t vi = lane + (int64_t)k * tw;
    if (vi >= p.V) continue;
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      sg[team * p.N + vi * VW + e] = pg[k][e];
      sb[team * p.N + vi * VW + e] = pb[k][e];
    }
  }
  __syncthreads();
  for (int64_t c = threadIdx.x; c < p.N; c += blockDim.x) {
    float a = 0.f, b = 0.f;
    for (int t = 0; t < nteams; ++t) {
      a += sg[t * p.N + c];
      b += sb[t * p.N + c];
    }
    p.part[(int64_t)blockIdx.x * p.N + c] = make_float2(a, b);
  }
  grid_launch_dependents();  // the column kernel may start launching
}

// dgamma[c] = sum over the P CTA records of feature c, dbeta likewise.  A CTA
// takes kColF features with kColS slices each: slice s adds records s,
// s + kColS, ... in order (eight loads in flight at a time, so up to
// 8*kColS records cost one round trip to L2), then the slices are added by a
// fixed pairwise tree.  kColF * kColS threads.
constexpr int kColF = 16, kColS = 64;
__global__ void __launch_bounds__(kColF * kColS) row_col_reduce(const __grid_constant__ RowParams p,
                                                               int64_t P) {
  __shared__ float2 acc[kColS][kColF];
  grid_dependency_wait();  // the records of the row kernel are complete
  const int j = threadIdx.x % kColF, sl = threadIdx.x / kColF;
  const int64_t c = (int64_t)blockIdx.x * kColF + j;
  float a = 0.f, b = 0.f;
  if (c < p.N) {
    for (int64_t r = sl; r < P; r += 8 * kColS) {
      float2 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int64_t rr = r + (int64_t)kColS * k;
        v[k] = rr < P ? __ldcg(p.part + rr * p.N + c) : make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        a += v[k].x;
        b += v[k].y;
      }
    }
  }
  acc[sl][j] = make_float2(a, b);
  __syncthreads();
#pragma unroll
  for (int h = kColS / 2; h > 0; h >>= 1) {
    if (sl < h) {
      const float2 o = acc[sl + h][j];
      acc[sl][j].x += o.x;
      acc[sl][j].y += o.y;
    }
    __syncthreads();
  }
  if (sl == 0 && c < p.N) {
    if (p.dgamma) p.dgamma[c] = acc[0][j].x;
    if (p.dbeta) p.dbeta[c] = acc[0][j].y;
  }
}

// -------------------------------------------------------------------- host
int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }
int pow2ceil(int64_t v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

// The shape of one call: vector width, vectors per thread, team width, grid.
struct RowPlan {
  int vw = 0, vpt = 0, tw = 0, nteams = 0;
  int64_t V = 0, grid = 0;
  size_t smem = 0;  // backward: dynamic shared memory
  bool ok = false;
};

// Only the combinations the plan can choose are instantiated (backward at
// most 16 values per thread, forward at most 32).
template <typename T, int VW, int VPT, bool kRms>
const void* row_kernel(bool bwd) {
  if (bwd) {
    if constexpr (VPT * VW <= 16) return (const void*)row_bwd<T, VW, VPT, kRms>;
    return nullptr;
  }
  if constexpr (VPT * VW <= 32) return (const void*)row_fwd<T, VW, VPT, kRms>;
  return nullptr;
}

template <typename T, int VW, bool kRms>
const void* row_kernel_vpt(int vpt, bool bwd) {
  switch (vpt) {
    case 1: return row_kernel<T, VW, 1, kRms>(bwd);
    case 2: return row_kernel<T, VW, 2, kRms>(bwd);
    case 4: return row_kernel<T, VW, 4, kRms>(bwd);
    default: return row_kernel<T, VW, 8, kRms>(bwd);
  }
}

template <typename T, bool kRms>
const void* row_kernel_for(const RowPlan& pl, bool bwd) {
  constexpr int V = Elem<T>::VEC;
  return pl.vw == 1 ? row_kernel_vpt<T, 1, kRms>(pl.vpt, bwd)
                    : row_kernel_vpt<T, V, kRms>(pl.vpt, bwd);
}

const void* kernel_of(const RowPlan& pl, int dtype, bool rms, bool bwd) {
  switch (dtype) {
    case kF32: return rms ? row_kernel_for<float, true>(pl, bwd) : row_kernel_for<float, false>(pl, bwd);
    case kF16: return rms ? row_kernel_for<__half, true>(pl, bwd) : row_kernel_for<__half, false>(pl, bwd);
    default:
      return rms ? row_kernel_for<__nv_bfloat16, true>(pl, bwd)
                 : row_kernel_for<__nv_bfloat16, false>(pl, bwd);
  }
}

// Co-resident CTAs of a kernel on the current device (cached), or an estimate
// of 4 per SM with no device.
int64_t resident(const void* fn, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, size_t>, int64_t> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 152 * 4;
  }
  const auto key = std::make_tuple(dev, fn, smem);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int sms = 0, nb = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (smem > kSmemNoOptIn)
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, kRowThreads, smem) != cudaSuccess)
    nb = 0;
  cudaGetLastError();
  const int64_t r = (int64_t)nb * (sms > 0 ? sms : 152);
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = r;
  return r;
}

// vw: 16-byte vectors when rows and parameters allow, else 1.  vpt: as many
// vectors per thread as registers allow (forward 32 values, backward 16, as
// the backward also holds dy and two partials per value); team width the
// power of two that covers the row.
RowPlan row_plan(int64_t M, int64_t N, int dtype, bool rms, bool bwd, bool aligned) {
  RowPlan pl;
  const int esz = dtype == kF32 ? 4 : 2;
  pl.vw = (aligned && (N * esz) % 16 == 0) ? 16 / esz : 1;  // aligned: bases and strides
  pl.V = N / pl.vw;
  // forward: 32 values per thread for large problems (more bytes in flight);
  // small ones, whose rows are latency-bound, take two 16-byte vectors per
  // thread (16 values at 16 bits, 8 in fp32).  Measured on GB300 on the
  // benchmark table's small shapes: one vector per thread is slower, and four
  // too (RMSNorm fp16 4096x1024 10.7 us at four vectors, 8.2 us at two;
  // LayerNorm fp32 4096x1024 14.3 us at eight, 12.3 at four, 10.2 at two).
  // Rows too long for a team of kRowThreads at the small-problem cap take
  // more values per thread, up to the large one (the row limit stays 256 x 32
  // values in the forward).
  // The backward keeps 16 values per thread at every size.
  const bool small = (double)M * (double)N <= 16.0 * (1 << 20);
  const int cap_max = bwd ? 16 : 32;
  const int cap = !small || bwd ? cap_max : (pl.vw > 1 ? 2 * pl.vw : 16);
  auto clampv = [](int v) { return v > 8 ? 8 : (v < 1 ? 1 : v); };
  const int vmax = clampv(cap / pl.vw), vmax_hi = clampv(cap_max / pl.vw);
  int vpt = 1;
  while (vpt < vmax && vpt < pl.V) vpt <<= 1;
  while (pow2ceil(cdiv64(pl.V, vpt)) > kRowThreads && vpt < vmax_hi) vpt <<= 1;
  pl.vpt = vpt;
  pl.tw = pow2ceil(cdiv64(pl.V, vpt));
  if (pl.tw > kRowThreads) return pl;  // rows too long to hold in one CTA's registers
  pl.nteams = kRowThreads / pl.tw;
  // backward: the teams' partials, then gamma; forward LayerNorm above 16
  // values per thread: gamma and beta (row_fwd's kStage)
  const bool stage = !bwd && !rms && pl.vpt * pl.vw > 16;
  pl.smem = bwd ? sizeof(float) * (2 * (size_t)pl.nteams + 1) * (size_t)N
                : (stage ? sizeof(float) * 2 * (size_t)N : 0);
  if (pl.smem > 200 * 1024) return pl;
  const int64_t res = resident(kernel_of(pl, dtype, rms, bwd), pl.smem);
  pl.grid = std::min<int64_t>(cdiv64(M, pl.nteams), res > 0 ? res : 1);
  if (pl.grid < 1) pl.grid = 1;
  pl.ok = true;
  return pl;
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b) return false;
  const char* pa = static_cast<const char*>(a);
  const char* pb = static_cast<const char*>(b);
  return pa < pb + nb && pb < pa + na;
}

int fail(cudaError_t e) {
  return e == cudaSuccess ? GN_OK : GN_ERR_CUDA;
}

// Bytes spanned by M rows of N elements, `ld` elements apart.
size_t span(int64_t M, int64_t N, int64_t ld, int esz) {
  return ((size_t)(M - 1) * (size_t)ld + (size_t)N) * (size_t)esz;
}

bool stride_ok(int64_t ld, int esz) { return (ld * esz) % 16 == 0; }

int run_fwd(const void* x, int64_t ldx, int64_t M, int64_t N, int dtype, const float* gamma,
            const float* beta, float eps, void* y, int64_t ldy, float* mean, float* rstd,
            void* stream, bool rms) {
  if (dtype != kF32 && dtype != kF16 && dtype != kBF16) return GN_ERR_UNSUPPORTED;
  if (M < 0 || N <= 0 || !(eps >= 0.f) || ldx < N || ldy < N) return GN_ERR_INVALID;
  if (M == 0) return GN_OK;
  if (!x || !y || !rstd || (!rms && !mean)) return GN_ERR_INVALID;
  const int esz = dtype == kF32 ? 4 : 2;
  const size_t bx = span(M, N, ldx, esz), by = span(M, N, ldy, esz);
  if (y == x ? ldy != ldx : overlaps(y, by, x, bx)) return GN_ERR_INVALID;
  if (overlaps(rstd, sizeof(float) * M, y, by) || overlaps(mean, sizeof(float) * M, y, by) ||
      overlaps(mean, sizeof(float) * M, rstd, sizeof(float) * M))
    return GN_ERR_INVALID;
  const bool aligned = a16(x) && a16(y) && (!gamma || a16(gamma)) && (!beta || a16(beta)) &&
                       stride_ok(ldx, esz) && stride_ok(ldy, esz);
  const RowPlan pl = row_plan(M, N, dtype, rms, false, aligned);
  if (!pl.ok) return GN_ERR_UNSUPPORTED;
  RowParams p{};
  p.x = x;
  p.out = y;
  p.gamma = gamma;
  p.beta = rms ? nullptr : beta;
  p.mean = mean;
  p.rstd = rstd;
  p.M = M;
  p.N = N;
  p.V = pl.V;
  p.ldx = ldx;
  p.ldo = ldy;
  p.tw = pl.tw;
  p.eps = eps;
  const void* fn = kernel_of(pl, dtype, rms, false);
  void* args[] = {&p};
  // (row_plan's occupancy query has raised the kernel's shared memory limit
  // for pl.smem where it exceeds the default)
  return fail(cudaLaunchKernel(fn, dim3((unsigned)pl.grid), dim3(kRowThreads), args, pl.smem,
                               static_cast<cudaStream_t>(stream)));
}

int run_bwd(const void* dy, int64_t ldd, const void* x, int64_t ldx, const float* mean,
            const float* rstd, const float* gamma, int64_t M, int64_t N, int dtype, void* dx,
            int64_t ldo, float* dgamma, float* dbeta, void* workspace, size_t workspace_bytes,
            void* stream, bool rms) {
  if (dtype != kF32 && dtype != kF16 && dtype != kBF16) return GN_ERR_UNSUPPORTED;
  if (M < 0 || N <= 0 || ldd < N || ldx < N || ldo < N) return GN_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (rms) dbeta = nullptr;
  if (M == 0) {  // empty sums
    if (dgamma && cudaMemsetAsync(dgamma, 0, sizeof(float) * N, s) != cudaSuccess) return GN_ERR_CUDA;
    if (dbeta && cudaMemsetAsync(dbeta, 0, sizeof(float) * N, s) != cudaSuccess) return GN_ERR_CUDA;
    return GN_OK;
  }
  if (!dy || !x || !rstd || !dx || (!rms && !mean)) return GN_ERR_INVALID;
  const int esz = dtype == kF32 ? 4 : 2;
  const size_t bd = span(M, N, ldd, esz), bx = span(M, N, ldx, esz), bo = span(M, N, ldo, esz);
  if (dx == dy ? ldo != ldd : overlaps(dx, bo, dy, bd)) return GN_ERR_INVALID;
  if (overlaps(dx, bo, x, bx)) return GN_ERR_INVALID;
  const size_t nb = sizeof(float) * (size_t)N;
  if (overlaps(dgamma, nb, dx, bo) || overlaps(dbeta, nb, dx, bo) ||
      overlaps(dgamma, nb, dbeta, nb))
    return GN_ERR_INVALID;
  const bool aligned = a16(x) && a16(dy) && a16(dx) && (!gamma || a16(gamma)) &&
                       stride_ok(ldd, esz) && stride_ok(ldx, esz) && stride_ok(ldo, esz);
  const RowPlan pl = row_plan(M, N, dtype, rms, true, aligned);
  if (!pl.ok) return GN_ERR_UNSUPPORTED;
  const bool want = dgamma || dbeta;
  const size_t need = want ? sizeof(float2) * (size_t)pl.grid * (size_t)N : 0;
  if (want && (!workspace || workspace_bytes < need || !a16(workspace))) return GN_ERR_WORKSPACE;
  RowParams p{};
  p.x = x;
  p.dy = dy;
  p.out = dx;
  p.gamma = gamma;
  p.mean = const_cast<float*>(mean);
  p.rstd = const_cast<float*>(rstd);
  p.dgamma = dgamma;
  p.dbeta = dbeta;
  p.part = static_cast<float2*>(workspace);
  p.M = M;
  p.N = N;
  p.V = pl.V;
  p.ldx = ldx;
  p.ldd = ldd;
  p.ldo = ldo;
  p.tw = pl.tw;
  p.want_part = want ? 1 : 0;
  const void* fn = kernel_of(pl, dtype, rms, true);
  if (pl.smem > kSmemNoOptIn) {
    const cudaError_t e =
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
    if (e != cudaSuccess) return GN_ERR_CUDA;
  }
  void* args[] = {&p};
  cudaError_t e = cudaLaunchKernel(fn, dim3((unsigned)pl.grid), dim3(kRowThreads), args,
                                   pl.smem, s);
  if (e != cudaSuccess || !want) return fail(e);
  // the column kernel, launched early (programmatic dependent launch): it
  // waits for the row kernel's records before reading them
  int64_t P = pl.grid;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cdiv64(N, kColF), 1, 1);
  cfg.blockDim = dim3(kColF * kColS, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return fail(cudaLaunchKernelEx(&cfg, row_col_reduce, p, P));
}

}  // namespace
}  // namespace gn

extern "C" {

size_t ln_workspace_size(int64_t M, int64_t N, int dtype) {
  if (M <= 0 || N <= 0 || (dtype != gn::kF32 && dtype != gn::kF16 && dtype != gn::kBF16)) return 0;
  size_t best = 0;
  for (int rms = 0; rms < 2; ++rms)
    for (int a = 0; a < 2; ++a) {
      const gn::RowPlan pl = gn::row_plan(M, N, dtype, rms != 0, true, a != 0);
      if (pl.ok) best = std::max(best, sizeof(float2) * (size_t)pl.grid * (size_t)N);
    }
  return best;
}

int ln_fwd_ex(const void* x, int64_t ldx, int64_t M, int64_t N, int dtype, const float* gamma,
              const float* beta, float eps, void* y, int64_t ldy, float* mean, float* rstd,
              void* stream) {
  return gn::run_fwd(x, ldx, M, N, dtype, gamma, beta, eps, y, ldy, mean, rstd, stream, false);
}

int ln_bwd_ex(const void* dy, int64_t lddy, const void* x, int64_t ldx, const float* mean,
              const float* rstd, const float* gamma, int64_t M, int64_t N, int dtype, void* dx,
              int64_t lddx, float* dgamma, float* dbeta, void* workspace,
              size_t workspace_bytes, void* stream) {
  return gn::run_bwd(dy, lddy, x, ldx, mean, rstd, gamma, M, N, dtype, dx, lddx, dgamma, dbeta,
                     workspace, workspace_bytes, stream, false);
}

int rms_fwd_ex(const void* x, int64_t ldx, int64_t M, int64_t N, int dtype, const float* gamma,
               float eps, void* y, int64_t ldy, float* rstd, void* stream) {
  return gn::run_fwd(x, ldx, M, N, dtype, gamma, nullptr, eps, y, ldy, nullptr, rstd, stream,
                     true);
}

int rms_bwd_ex(const void* dy, int64_t lddy, const void* x, int64_t ldx, const float* rstd,
               const float* gamma, int64_t M, int64_t N, int dtype, void* dx, int64_t lddx,
               float* dgamma, void* workspace, size_t workspace_bytes, void* stream) {
  return gn::run_bwd(dy, lddy, x, ldx, nullptr, rstd, gamma, M, N, dtype, dx, lddx, dgamma,
                     nullptr, workspace, workspace_bytes, stream, true);
}

int ln_fwd(const void* x, int64_t M, int64_t N, int dtype, const float* gamma, const float* beta,
           float eps, void* y, float* mean, float* rstd, void* stream) {
  return ln_fwd_ex(x, N, M, N, dtype, gamma, beta, eps, y, N, mean, rstd, stream);
}

int ln_bwd(const void* dy, const void* x, const float* mean, const float* rstd,
           const float* gamma, int64_t M, int64_t N, int dtype, void* dx, float* dgamma,
           float* dbeta, void* workspace, size_t workspace_bytes, void* stream) {
  return ln_bwd_ex(dy, N, x, N, mean, rstd, gamma, M, N, dtype, dx, N, dgamma, dbeta, workspace,
                   workspace_bytes, stream);
}

int rms_fwd(const void* x, int64_t M, int64_t N, int dtype, const float* gamma, float eps,
            void* y, float* rstd, void* stream) {
  return rms_fwd_ex(x, N, M, N, dtype, gamma, eps, y, N, rstd, stream);
}

int rms_bwd(const void* dy, const void* x, const float* rstd, const float* gamma, int64_t M,
            int64_t N, int dtype, void* dx, float* dgamma, void* workspace,
            size_t workspace_bytes, void* stream) {
  return rms_bwd_ex(dy, N, x, N, rstd, gamma, M, N, dtype, dx, N, dgamma, workspace,
                    workspace_bytes, stream);
}

}  // extern "C"
