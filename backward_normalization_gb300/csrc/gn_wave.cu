// gn_wave.cu -- the wave regime: one persistent kernel per op that reads its
// input from HBM once and writes its output once, for problems whose
// reduction units fit on chip (shared and tensor memory) across the CTAs
// that share them.
//
// Work.  A reduction unit is one (sample, group) span for NCHW -- Cg
// contiguous channel planes -- or one (sample, block of Cb channels made of
// whole groups) for NHWC -- HW rows of Cb channels, read as 2-D TMA tiles
// from the [N*HW, C] view.  A unit is cut into P pieces: for NCHW wm
// consecutive segments of each plane (P = Cg*wm), for NHWC blocks of wR
// rows.  Pieces are numbered unit-major, q = u*P + t, and CTA b of the NC
// co-resident CTAs takes pieces q = k*NC + b for k = 0, 1, ... (its steps).
// The plan picks P by a cost model fitted to measurements; a unit whose P
// does not divide NC straddles two steps.
//
// Per piece: bulk (TMA) copies bring it into one of S shared-memory slots
// (all slots are kept loading); stage A reduces the piece and writes one
// record per channel to the workspace; stage B reads every record of the
// piece's unit (polling until all are written, bounded), merges them in a
// fixed order into the group statistics (forward) or the dx coefficients
// (backward), and writes the piece's output.  x (and dy) are read from HBM
// once.
//
// Where the plan allows (wH > 0), a reduced piece waits for its unit's
// statistics in tensor memory rather than in its slot: in stage A every
// thread also stores the 16-byte vectors it reduces into its own lane of one
// of wH hold buffers (tcgen05.st), and stage B reads them back (tcgen05.ld),
// so the slot takes its next copy as soon as stage A is done with it.  Stage
// A then runs on warps 0-3 and stage B on warps 4-7 at the same time (warp
// specialisation; thread t of either stage owns lane 32*(warp % 4) + t % 32):
// the reduce of one piece (shared-memory reads, tensor-memory writes)
// overlaps the output of an earlier one (tensor-memory reads, global
// stores).  Per hold buffer an mbarrier `tm_full` tells stage B that a piece
// is in, and `tm_empty` tells stage A that it has been written out.  For
// NCHW a ninth warp gathers and merges each unit's records into a result per
// hold buffer (`mg_done`), so that stage B only writes.  Waiting threads are
// suspended by the hardware (mbarrier try_wait with a time hint) rather than
// spinning, which leaves issue slots to the working stage.  Without
// hold buffers the CTA runs the stages in turn, stage A one piece ahead of
// stage B when a third slot is free, and the piece waits in its slot.
//
// Records are self-validating 64-bit words (a cleared word is zero, a written
// one never is), written and polled with single relaxed accesses: no
// release/acquire pair orders them, so publishing a record never waits for
// the CTA's earlier output stores to drain.
//
// A CTA waits for other CTAs' pieces, so all CTAs must be co-resident: the
// kernel is launched cooperatively.  Deadlock-freedom: a CTA publishes its
// piece of step k before it waits for that piece's unit, and stage A of step
// k waits only for copies and for the stage B of an earlier step of its own
// CTA.  Take the smallest unit u that some CTA waits for.  Every owner of a
// piece of u has published it, or is still in an earlier step, whose piece
// has a smaller index and so belongs to a unit smaller than u (an owner holds
// at most one piece of a unit, since P <= NC); by the minimality of u those
// steps complete, so every piece of u is published.
//
// The workspace holds anything when the call starts: CTA 0 zero-fills the
// error word, every CTA the record slots of its own pieces, and a grid-wide
// barrier (entered after each CTA has issued its first copies, whose latency
// hides it) orders that before any record is written.  Every wait is bounded
// in time; one that runs out sets a bit of the error word (gn_workspace_status
// reports it), after which every CTA skips its remaining work, waiting only
// for its own copies in flight.  The backward's dgamma / dbeta follow a second
// grid barrier, spread over the CTAs by channel.
//
// Statistics.  A forward record is, per (piece, channel), the mean and the
// sum of squared deviations M2 of the piece's n_i values, accumulated about
// the piece's first value (a shift that keeps the sums small).  A group's
// records merge by the parallel-axis identity (Chan, Golub and LeVeque),
// taken over all of them at once: mean = sum(n_i * mean_i) / M and M2 =
// sum(M2_i + n_i * (mean_i - mean)^2), M = Cg*HW.  A backward record is, per
// (piece, channel), sum(dy) and sum(dy*(x - mean)); a group's coefficients
// come from sum gamma_c * S1 and sum gamma_c * S2 over its records.  Every
// CTA of a unit merges the same records in the same order (lane i of a warp
// takes records i, i + 32, ..., then a fixed xor tree), so all of them use
// identical statistics; results are bit-identical from run to run.
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

// A piece's record in the workspace: two floats in one 64-bit word, each
// XORed with kWaveKey (a NaN bit pattern that arithmetic never produces), so
// that a written record is never zero while a cleared slot is.  Written and
// read as single 64-bit accesses: a reader that sees a non-zero word has the
// record itself, and no release / acquire ordering is needed -- in
// particular a CTA's records never wait for its earlier output stores.
constexpr uint32_t kWaveKey = 0x7fbadbadu;

__device__ __forceinline__ void put_rec(float2* slot, float2 v) {
  const unsigned long long w =
      ((unsigned long long)(__float_as_uint(v.y) ^ kWaveKey) << 32) | (__float_as_uint(v.x) ^ kWaveKey);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(slot), "l"(w) : "memory");
}

__device__ __forceinline__ bool get_rec(const float2* slot, float2* v) {
  unsigned long long w;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(slot) : "memory");
  if (w == 0ull) return false;
  v->x = __uint_as_float((unsigned)w ^ kWaveKey);
  v->y = __uint_as_float((unsigned)(w >> 32) ^ kWaveKey);
  return true;
}

// A record's raw word, loaded without waiting for it (the caller decodes it
// later, so the load's latency overlaps other work).
__device__ __forceinline__ unsigned long long ld_rec_raw(const float2* slot) {
  unsigned long long w;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(slot) : "memory");
  return w;
}
__device__ __forceinline__ float2 rec_decode(unsigned long long w) {
  return make_float2(__uint_as_float((unsigned)w ^ kWaveKey),
                     __uint_as_float((unsigned)(w >> 32) ^ kWaveKey));
}

// The threads that run one stage of the kernel: the whole CTA (barrier 0,
// __syncthreads), or with warp specialisation one half of it on its own
// named barrier.  t is this thread's index in the group, n the group's size.
struct Group {
  int id, n, t;
  __device__ __forceinline__ void sync() const {
    if (id == 0) __syncthreads();
    else named_sync(id, n);
  }
  __device__ __forceinline__ bool sync_or(bool c) const {
    if (id == 0) return __syncthreads_or(c) != 0;
    return named_sync_or(id, n, c);
  }
};

// This thread's share of a unit's n records: records t + i*gr.n, bit i of
// the mask for each (a thread holds at most 32: n <= 32*gr.n).
__device__ __forceinline__ unsigned record_mask(int n, const Group& gr) {
  unsigned todo = 0;
  for (int i = 0; i < 32 && gr.t + i * gr.n < n; ++i) todo |= 1u << i;
  return todo;
}

// Sums of two values over a group with a fixed tree (shuffles within warps,
// then the warp results in warp order); the totals land in the group's
// thread 0.  `scratch` holds 2 floats per warp of the group.
__device__ __forceinline__ float2 group_sum2_t0(float a, float b, float* scratch, const Group& gr) {
  const int lane = gr.t & 31, w = gr.t >> 5;
  a = warp_sum_lane0(a);
  b = warp_sum_lane0(b);
  if (lane == 0) {
    scratch[2 * w] = a;
    scratch[2 * w + 1] = b;
  }
  gr.sync();
  float2 r = make_float2(0.f, 0.f);
  if (gr.t == 0)
    for (int i = 0; i < (gr.n >> 5); ++i) {
      r.x += scratch[2 * i];
      r.y += scratch[2 * i + 1];
    }
  gr.sync();
  return r;
}

// Every thread of a group: waits until phase `parity` of `bar` has completed.
// The group's thread 0 polls, bounded in time and giving up once the error
// word is raised; the outcome reaches the group through *flag.  Returns true
// (after an acquiring test of the barrier by every thread) or false, uniformly.
__device__ bool group_wait(uint64_t* bar, uint32_t parity, unsigned* err, int* flag, const Group& gr) {
  if (gr.t == 0) {
    int go = 1;
    if (!mbar_try_wait(bar, parity)) {
      const uint64_t t0 = now_ns();
      for (unsigned i = 1;; ++i) {
        // suspended for up to 2 us a test: the waiting warp leaves its issue
        // slots to the other stage (c3 backward 4.20 -> 3.98 ms)
        if (mbar_try_wait_hint(bar, parity, 2000u)) break;
        if ((i & 15u) == 0u) {
          if (aborted(err)) {
            go = 0;
            break;
          }
          if (now_ns() - t0 > kWaveWaitNs) {
            atomicOr(err, kErrData);
            go = 0;
            break;
          }
        }
      }
    }
    *flag = go;
  }
  gr.sync();
  if (!*flag) return false;
  mbar_try_wait(bar, parity);  // completed: orders this thread's later reads after it
  return true;
}

// Every thread of a group: reads the records at src still marked in `todo`
// into dst (shared memory), polling until all of them are written.  Bounded
// in time (the group's thread 0 keeps the clock); returns false, uniformly,
// when the bound runs out or the error word is raised.
__device__ bool gather_records(const float2* src, float2* dst, unsigned todo, unsigned* err,
                               int* s_flag, const Group& gr) {
  const int tid = gr.t, nt = gr.n;
  uint64_t t0 = 0;
  for (unsigned round = 0;; ++round) {
    for (int i = 0; i < 32 && (todo >> i) != 0u; ++i) {
      if (!((todo >> i) & 1u)) continue;
      float2 v;
      if (get_rec(src + tid + i * nt, &v)) {
        dst[tid + i * nt] = v;
        todo &= ~(1u << i);
      }
    }
    if (!gr.sync_or(todo != 0u)) return true;
    if (tid == 0) {
      int go = 1;
      if ((round & 7u) == 7u && aborted(err)) {
        go = 0;
      } else {
        const uint64_t t = now_ns();
        if (t0 == 0) {
          t0 = t;
        } else if (t - t0 > kWaveWaitNs) {
          atomicOr(err, kErrUnit);
          go = 0;
        }
      }
      *s_flag = go;
    }
    gr.sync();
    if (!*s_flag) return false;
    __nanosleep(64);
  }
}

// Vector u (4 words) of a 16-register tensor-memory transfer.
__device__ __forceinline__ void put4(uint32_t (&w)[16], int u, const uint4& r) {
  w[4 * u] = r.x;
  w[4 * u + 1] = r.y;
  w[4 * u + 2] = r.z;
  w[4 * u + 3] = r.w;
}
__device__ __forceinline__ uint4 get4(const uint32_t (&w)[16], int u) {
  return make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
}

// Sum over the 32 lanes of a warp with a fixed xor tree; every lane gets it.
__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// The piece that CTA b processes at step k, decoded (32-bit index arithmetic:
// the plan keeps units * pieces below 2^31).
struct Piece {
  int u, t;       // unit, piece within the unit
  int n;          // sample
  int gi;         // NCHW: the unit's group
  int c;          // NCHW: the piece's channel
  int cb;         // NHWC: channel block of the unit
  int len;        // NCHW: elements; NHWC: rows
  int64_t e0;     // NCHW: first element (flat offset)
  int64_t row0;   // NHWC: first row in the [N*HW, C] view
  int cbase;      // NHWC: first channel of the unit
};

template <int LAYOUT>
__device__ __forceinline__ Piece piece_of(const Geom& g, int q) {
  Piece pc;
  const int P = (int)g.wP;
  pc.u = q / P;
  pc.t = q - pc.u * P;
  const int HW32 = (int)(g.HW < 0x7fffffff ? g.HW : 0x7fffffff);
  const int R = (int)g.wR;
  if (LAYOUT == kNCHW) {
    const int G = (int)g.G, wm = (int)g.wm;
    pc.n = pc.u / G;
    pc.gi = pc.u - pc.n * G;
    const int plane = pc.t / wm, seg = pc.t - plane * wm;
    pc.c = pc.gi * (int)g.Cg + plane;
    const int64_t h0 = (int64_t)seg * R;
    pc.len = (int)((h0 + R < g.HW) ? R : g.HW - h0);
    pc.e0 = ((int64_t)pc.n * g.C + pc.c) * g.HW + h0;
    pc.cb = pc.cbase = 0;
    pc.row0 = 0;
  } else {
    const int ncbu = (int)g.ncbu;
    pc.n = pc.u / ncbu;
    pc.cb = pc.u - pc.n * ncbu;
    pc.cbase = pc.cb * (int)g.Cb;
    const int r0 = pc.t * R;
    pc.len = (r0 + R < HW32) ? R : HW32 - r0;
    pc.row0 = (int64_t)pc.n * g.HW + r0;
    pc.gi = pc.c = 0;
    pc.e0 = 0;
  }
  return pc;
}

// Values in piece t of a unit (rows for NHWC, elements of a plane for NCHW).
__device__ __forceinline__ float piece_count(const Geom& g, int t) {
  const int seg = g.layout == kNCHW ? t % (int)g.wm : t;
  const int64_t a = (int64_t)seg * g.wR;
  return (float)((a + g.wR < g.HW) ? g.wR : g.HW - a);
}

// MODE 0: a piece waits for its unit's statistics in its slot, and the CTA
// runs stage A and stage B in turn; MODE 1: it waits in tensor memory;
// MODE 2: it waits in tensor memory, and stage A (warps 0-3) and stage B
// (warps 4-7) run concurrently, handing pieces over through mbarriers.
template <typename T, int VW, int LAYOUT, bool BWD, int MODE>
__global__ void __launch_bounds__(LAYOUT == kNCHW && MODE == 2 ? kWaveThreads + 32 : kWaveThreads, kWaveCtasPerSm)
    wave_kernel(const __grid_constant__ KParams p) {
  constexpr bool HOLD = MODE >= 1;
  constexpr bool WS = MODE == 2;
  // WS, NCHW: a ninth warp (threads 256-287) gathers and merges each unit's
  // records, so that stage B only writes
  constexpr bool MW = WS && LAYOUT == kNCHW;
  extern __shared__ __align__(128) char smem_raw[];
  char* smem =
      reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const Geom& g = p.g;
  constexpr int NTEN = BWD ? 2 : 1;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nt >> 5;
  // the stages' threads: the whole CTA, or (WS) warps 0-3 for stage A and
  // warps 4-7 for stage B; tg is this thread's index in its stage
  const int ng = WS ? kWaveThreads / 2 : nt;
  const bool is_a = !WS || tid < ng;
  const bool is_m = MW && tid >= 2 * ng;
  const int tg = !WS || is_a ? tid : is_m ? tid - 2 * ng : tid - ng;
  const Group ga{WS ? 1 : 0, ng, tg};
  const Group gb{WS ? 2 : 0, ng, tg};
  const Group gq{3, 32, tg};  // the merge warp
  char* ring = smem + g.off_ring;
  float* red = reinterpret_cast<float*>(smem + g.off_red);
  float2* grp = reinterpret_cast<float2*>(smem + g.off_grp);  // per-group results of the unit
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + g.off_bar);
  // outcomes of the waits, one flag per waiting site: a flag is written
  // again only after every thread of its stage has passed another barrier
  __shared__ int s_ok, s_ok_b, s_ok_e, s_ok_f, s_ok_m, s_ok_q, s_ok_r;
  __shared__ uint32_t s_tmem;  // HOLD: base address of the CTA's tensor memory

  const int NC = gridDim.x, b = blockIdx.x;
  const int P = (int)g.wP;
  const int total = (int)(g.units * g.wP);
  const int K = b < total ? (total - 1 - b) / NC + 1 : 0;  // this CTA's pieces
  const int S = g.S;
  const int nch = LAYOUT == kNHWC ? (int)g.Cb : 1;  // channels of a piece
  const int Cg = (int)g.Cg;
  const int rec_unit = P * nch;  // records of a unit
  const int H = HOLD ? (int)g.wH : 0;  // tensor-memory buffers
  // stage A runs `ahead` pieces before stage B: with tensor-memory buffers
  // one less than their number, else one when a third slot is free to land
  const int ahead = HOLD ? H - 1 : (S >= 3 ? 1 : 0);
  const int NCB = (int)g.wB;            // buffers of per-piece constants
  const int NRB = HOLD && H > 2 ? H : 2;  // P == 1: buffers of the CTA's own records
  // WS: tm_full[h] completes when stage A has put a piece into hold buffer
  // h, tm_empty[h] when stage B has written that piece out
  uint64_t* tm_full = full + S;
  uint64_t* tm_empty = tm_full + H;
  uint64_t* mg_done = tm_empty + H;  // MW: the merge warp has piece k's unit statistics in grp[k % H]
  // shared scratch: the unit's records (P > 1: gathered; P == 1: the CTA's
  // own, NRB pieces' worth), then the CTA sums
  float2* recs = reinterpret_cast<float2*>(red);
  float* cred = red + 2 * (P > 1 ? rec_unit : NRB * nch);
  const size_t slot_bytes = (size_t)g.ten_stride * NTEN;
  const T* x = static_cast<const T*>(p.x);
  const T* dy = static_cast<const T*>(p.dy);
  T* out = static_cast<T*>(p.out);

  if (tid == 0) {
    for (int i = 0; i < S; ++i) mbar_init(full + i, 1);
    if (WS)
      for (int h = 0; h < H; ++h) {
        mbar_init(tm_full + h, 1);
        mbar_init(tm_empty + h, 1);
        if (MW) mbar_init(mg_done + h, 1);
      }
    fence_mbar_init();
  }
  if (HOLD) {
    __syncwarp();
    if (warp == 0) tmem_alloc(&s_tmem, kWaveTmemCols);
    tmem_fence_before();
  }
  __syncthreads();
  if (HOLD) tmem_fence_after();
  grid_dependency_wait();  // earlier work on the stream (the inputs, the workspace) is done
  grid_launch_dependents();

  // ---- copies: piece k of this CTA into slot k % S (thread 0)
  const uint64_t pol_in = policy_evict_first();
  auto issue = [&](int k) {
    const Piece pc = piece_of<LAYOUT>(g, k * NC + b);
    char* dst = ring + (size_t)(k % S) * slot_bytes;
    uint64_t* bar = full + (k % S);
    if (LAYOUT == kNCHW) {
      const uint32_t bytes = (uint32_t)pc.len * (uint32_t)sizeof(T);
      mbar_arrive_expect_tx(bar, bytes * NTEN);
      tma_load_1d(dst, x + pc.e0, bytes, bar, pol_in);
      if (BWD) tma_load_1d(dst + g.ten_stride, dy + pc.e0, bytes, bar, pol_in);
    } else {
      const uint32_t box = (uint32_t)(g.chunk * g.Cb * (int64_t)sizeof(T));
      mbar_arrive_expect_tx(bar, box * (uint32_t)g.wnb * NTEN);
      for (int bx = 0; bx < (int)g.wnb; ++bx) {
        const int32_t row = (int32_t)(pc.row0 + (int64_t)bx * g.chunk);
        tma_load_2d(dst + (size_t)bx * box, &p.tmx, pc.cbase, row, bar, pol_in);
        if (BWD) tma_load_2d(dst + g.ten_stride + (size_t)bx * box, &p.tmdy, pc.cbase, row, bar, pol_in);
      }
    }
  };
  int issued = 0;  // thread 0: pieces whose copies were issued
  if (tid == 0)
    for (; issued < K && issued < S; ++issued) issue(issued);

  // ---- the workspace holds anything when the call starts: CTA 0 clears the
  // error word, every CTA the record slots of its own pieces, and a grid
  // barrier orders those stores before any record is written or polled
  if (b == 0)
    for (int i = tid; i < p.clear_words; i += nt) p.err[i] = 0u;
  // a unit's piece counts (and, NCHW, each piece's plane), for the merges
  float* cnt = reinterpret_cast<float*>(smem + g.off_tot);
  int* plane_of = reinterpret_cast<int*>(cnt + P);
  for (int t = tid; t < P; t += nt) {
    cnt[t] = piece_count(g, t);
    plane_of[t] = LAYOUT == kNCHW ? t / (int)g.wm : 0;
  }
  if (P > 1) {
    unsigned long long* slots = reinterpret_cast<unsigned long long*>(p.part);
    for (int i = tid; i < K * nch; i += nt) {
      const int kk = i / nch, c = i - kk * nch;
      const int q = kk * NC + b;
      slots[(int64_t)(q / P) * rec_unit + (q % P) * nch + c] = 0ull;
    }
  }
  cooperative_groups::this_grid().sync();

  // ---- per-thread layout.  NHWC: column j (VW channels of the block) of rows
  // rl, rl + rpi, ...; qe[e] is the group (within the block) of its channel
  // e.  NCHW: the piece's 16-byte vectors tid, tid + nt, ...
  const int Wv = LAYOUT == kNHWC ? nch / VW : 1;
  const int rpi = LAYOUT == kNHWC ? ng / Wv : ng;
  const int j = LAYOUT == kNHWC ? tg % Wv : 0;
  const int rl = LAYOUT == kNHWC ? tg / Wv : tg;
  const bool lane_ok = LAYOUT == kNHWC ? rl < rpi : true;
  int qe[VW];
#pragma unroll
  for (int e = 0; e < VW; ++e) qe[e] = LAYOUT == kNHWC ? (j * VW + e) / Cg : 0;
  const int rowb = nch * (int)sizeof(T);  // NHWC: bytes per row in a slot
  const uint64_t pol_out = policy_evict_first();
  const float Mg = (float)(g.Cg * g.HW);  // values per group
  const int ngrp = LAYOUT == kNHWC ? nch / Cg : 1;  // groups of a unit

  // ---- per-slot constants of a piece, fetched one step ahead with 4-byte
  // asynchronous copies (every thread commits one cp.async group per call)
  const int CST = wave_cst_floats(g);
  float* cstb = reinterpret_cast<float*>(smem + g.off_xch);
  auto fetch_constants = [&](int k) {
    if (k < K) {
      const Piece pc = piece_of<LAYOUT>(g, k * NC + b);
      float* cs = cstb + (k % NCB) * CST;
      if (LAYOUT == kNHWC) {
        for (int c = tg; c < nch; c += ng) {
          if (p.gamma) cp_async4(cs + c, p.gamma + pc.cbase + c);
          else cs[c] = 1.0f;
          if (!BWD) {
            if (p.beta) cp_async4(cs + nch + c, p.beta + pc.cbase + c);
            else cs[nch + c] = 0.f;
          }
        }
        if (BWD) {
          const int64_t g0 = (int64_t)pc.n * g.G + pc.cbase / Cg;
          for (int q = tg; q < ngrp; q += ng) {
            cp_async4(cs + nch + q, p.mean + g0 + q);
            cp_async4(cs + nch + ngrp + q, p.rstd + g0 + q);
          }
        }
      } else {
        for (int cl = tg; cl < Cg; cl += ng) {
          if (p.gamma) cp_async4(cs + cl, p.gamma + (int64_t)pc.gi * Cg + cl);
          else cs[cl] = 1.0f;
        }
        if (tg == ng - 1) {
          if (BWD) {
            cp_async4(cs + Cg, p.mean + pc.u);
            cp_async4(cs + Cg + 1, p.rstd + pc.u);
          } else if (p.beta) {
            cp_async4(cs + Cg, p.beta + pc.c);
          } else {
            cs[Cg] = 0.f;
          }
        }
      }
    }
    cp_async_commit();
  };
  if (is_a) fetch_constants(0);

  // ---- a unit's records are read ahead: during the stage A before their
  // stage B (when stage A runs ahead), or (WS) by stage B during the output
  // of its previous piece.  Raw words land in registers while the stage
  // works, and are decoded into shared memory at its end.
  constexpr int kPre = 8;  // records per thread read ahead (at most)
  const bool read_ahead = P > 1 && (WS || ahead >= 1) && rec_unit <= kPre * (MW ? 32 : ng);
  unsigned long long pre[kPre];
  int pre_unit = -1;       // the unit whose records sit in `recs`, or -1
  unsigned pre_todo = 0;   // of those, the ones not yet written

  // ---- HOLD: thread t of a stage keeps the vectors it reduces in stage A
  // (and writes in stage B) in tensor-memory lane 32*(warp % 4) + t % 32, T4
  // vectors of x then T4 of dy from column 0 (WS) or (warp / 4) * tcols of
  // the piece's buffer
  const int T4 = HOLD ? (int)g.wT : 0;
  const uint32_t tcols = 4u * NTEN * (uint32_t)T4;
  const uint32_t bcols = WS ? tcols : tcols * (uint32_t)(nt / 128);
  const uint32_t tthr =
      HOLD ? s_tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (WS ? 0u : (uint32_t)(warp >> 2) * tcols) : 0u;

  // ---- stage A of piece k: wait for its copy, reduce it, publish its records
  auto stage_a = [&](int k) -> bool {
    const Piece pc = piece_of<LAYOUT>(g, k * NC + b);
    const int si = k % S;
    const char* slot = ring + (size_t)si * slot_bytes;
    const float* cs = cstb + (k % NCB) * CST;
    const uint32_t parity = (uint32_t)((k / S) & 1);
    cp_async_wait_all();    // this piece's constants (fetched one step ago)
    fetch_constants(k + 1);  // and the next piece's, for the next step
    // the records of the unit of the stage B that follows (piece k - ahead)
    const int pre_k = k - ahead;
    const int pre_u = !WS && read_ahead && pre_k >= 0 ? piece_of<LAYOUT>(g, pre_k * NC + b).u : -1;
    if (pre_u >= 0) {
      const float2* src = p.part + (int64_t)pre_u * rec_unit;
#pragma unroll
      for (int i = 0; i < kPre; ++i)
        pre[i] = tg + i * ng < rec_unit ? ld_rec_raw(src + tg + i * ng) : 0ull;
    }
    // the piece's copy (the group barrier also publishes the constants)
    if (!group_wait(full + si, parity, p.err, &s_ok, ga)) return false;
    float2* rec_g = p.part + (int64_t)pc.u * rec_unit + pc.t * nch;
    float2* rec_s = recs + (k % NRB) * nch;  // P == 1: kept in shared memory
    const bool publish = !(p.stall_unit == pc.u && pc.t == 0);  // fault injection
    if (LAYOUT == kNCHW) {
      const float mu = BWD ? cs[Cg] : 0.f;
      const float K0 = BWD ? 0.f : Elem<T>::to_f(reinterpret_cast<const T*>(slot)[0]);
      float a = 0.f, c = 0.f;
      const int nv = pc.len / VW;
      auto add = [&](const uint4& rx, const uint4& rd) {
        float xv[VW];
        Access<T, VW>::unpack(rx, xv);
        if (BWD) {
          float dv[VW];
          Access<T, VW>::unpack(rd, dv);
#pragma unroll
          for (int e = 0; e < VW; ++e) {
            a += dv[e];
            c = fmaf(dv[e], xv[e] - mu, c);
          }
        } else {
#pragma unroll
          for (int e = 0; e < VW; ++e) {
            const float d = xv[e] - K0;
            a += d;
            c = fmaf(d, d, c);
          }
        }
      };
      if constexpr (HOLD) {
        // vectors tg + i*ng, i < T4, also go to tensor memory (zeros past the
        // piece).  Ordinary shared-memory loads (the compiler may run them
        // ahead), and one partial sum per vector element, so that the
        // dependency chains stay short; the partial sums meet in element
        // order at the end.
        float ae[VW], ce[VW];
#pragma unroll
        for (int e = 0; e < VW; ++e) ae[e] = ce[e] = 0.f;
        const uint32_t tb = tthr + (uint32_t)(k % H) * bcols;
        for (int i0 = 0; i0 < T4; i0 += 4) {
          uint32_t wx[16], wd[16];
          uint4 rx[4], rd[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int v = tg + (i0 + u) * ng;
            rx[u] = rd[u] = make_uint4(0u, 0u, 0u, 0u);
            if (v < nv) {
              rx[u] = *reinterpret_cast<const uint4*>(slot + (size_t)v * 16);
              if (BWD) rd[u] = *reinterpret_cast<const uint4*>(slot + g.ten_stride + (size_t)v * 16);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (tg + (i0 + u) * ng < nv) {
              float xv[VW];
              Access<T, VW>::unpack(rx[u], xv);
              if (BWD) {
                float dv[VW];
                Access<T, VW>::unpack(rd[u], dv);
#pragma unroll
                for (int e = 0; e < VW; ++e) {
                  ae[e] += dv[e];
                  ce[e] = fmaf(dv[e], xv[e] - mu, ce[e]);
                }
              } else {
#pragma unroll
                for (int e = 0; e < VW; ++e) {
                  const float d = xv[e] - K0;
                  ae[e] += d;
                  ce[e] = fmaf(d, d, ce[e]);
                }
              }
            }
            put4(wx, u, rx[u]);
            if (BWD) put4(wd, u, rd[u]);
          }
          tmem_st16(tb + 4u * (uint32_t)i0, wx);
          if (BWD) tmem_st16(tb + 4u * (uint32_t)(T4 + i0), wd);
        }
        tmem_wait_st();
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          a += ae[e];
          c += ce[e];
        }
      } else {
#pragma unroll 4
        for (int v = tg; v < nv; v += ng)
          add(lds16(slot + (size_t)v * 16),
              BWD ? lds16(slot + g.ten_stride + (size_t)v * 16) : make_uint4(0u, 0u, 0u, 0u));
      }
      const float2 s2 = group_sum2_t0(a, c, cred, ga);
      if (tg == 0) {
        float2 r;
        if (BWD) {
          r = s2;
        } else {
          const float q = s2.x / (float)pc.len;
          r = make_float2(K0 + q, fmaxf(fmaf(-s2.x, q, s2.y), 0.f));
        }
        if (P == 1) rec_s[0] = r;
        else if (publish) put_rec(rec_g, r);
      }
    } else {
      float acc[2 * VW], Ks[VW], mu[VW];
#pragma unroll
      for (int q = 0; q < 2 * VW; ++q) acc[q] = 0.f;
#pragma unroll
      for (int e = 0; e < VW; ++e) Ks[e] = mu[e] = 0.f;
      if (lane_ok) {
        if (BWD) {
#pragma unroll
          for (int e = 0; e < VW; ++e) mu[e] = cs[nch + qe[e]];
        } else {
          Access<T, VW>::unpack(lds16(slot + j * 16), Ks);  // the piece's first row: the shift
        }
      }
      const char* col = slot + j * 16;
      auto add = [&](const uint4& rx, const uint4& rd) {
        float xv[VW];
        Access<T, VW>::unpack(rx, xv);
        if (BWD) {
          float dv[VW];
          Access<T, VW>::unpack(rd, dv);
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
      };
      if constexpr (HOLD) {
        // rows rl + i*rpi, i < T4, of column j also go to tensor memory
        // (zeros past the piece, and for threads without a column)
        // (ordinary shared-memory loads, which the compiler may run ahead)
        const uint32_t tb = tthr + (uint32_t)(k % H) * bcols;
        for (int i0 = 0; i0 < T4; i0 += 4) {
          uint32_t wx[16], wd[16];
          uint4 rx[4], rd[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int r = rl + (i0 + u) * rpi;
            rx[u] = rd[u] = make_uint4(0u, 0u, 0u, 0u);
            if (lane_ok && r < pc.len) {
              rx[u] = *reinterpret_cast<const uint4*>(col + (size_t)r * rowb);
              if (BWD) rd[u] = *reinterpret_cast<const uint4*>(col + g.ten_stride + (size_t)r * rowb);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (lane_ok && rl + (i0 + u) * rpi < pc.len) add(rx[u], rd[u]);
            put4(wx, u, rx[u]);
            if (BWD) put4(wd, u, rd[u]);
          }
          tmem_st16(tb + 4u * (uint32_t)i0, wx);
          if (BWD) tmem_st16(tb + 4u * (uint32_t)(T4 + i0), wd);
        }
        tmem_wait_st();
      } else if (lane_ok) {
#pragma unroll 2
        for (int r = rl; r < pc.len; r += rpi)
          add(lds16(col + (size_t)r * rowb),
              BWD ? lds16(col + g.ten_stride + (size_t)r * rowb) : make_uint4(0u, 0u, 0u, 0u));
      }
      // CTA sums: each of the 2*nch sums (value q of column jj) is taken by
      // tps lanes of one warp; lane l adds row lanes l, l + tps, ... into four
      // accumulators in a fixed rotation, then the lanes meet in a fixed xor
      // tree
#pragma unroll
      for (int q = 0; q < 2 * VW; ++q) cred[q * ng + tg] = acc[q];
      float* ksh = cred + 2 * VW * ng;
      float* sums = ksh + nch;
      if (!BWD && rl == 0 && lane_ok) {
#pragma unroll
        for (int e = 0; e < VW; ++e) ksh[j * VW + e] = Ks[e];
      }
      ga.sync();
      {
        const int nsum = 2 * VW * Wv;
        int tps = 1;
        while (tps < 32 && 2 * tps * nsum <= ng) tps *= 2;
        const int l = tg % tps;
        // with more sums than the stage has threads (tps = 1), each thread
        // takes several; the trip count is the same for every thread
        for (int base = 0; base < nsum * tps; base += ng) {
          const int sidx = (base + tg) / tps;
          const bool mine = sidx < nsum;
          const int q = mine ? sidx / Wv : 0, jj = mine ? sidx % Wv : 0;
          float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
          if (mine) {
            const float* src = cred + q * ng + jj;
            int r = l;
            for (; r + 3 * tps < rpi; r += 4 * tps) {
              a0 += src[r * Wv];
              a1 += src[(r + tps) * Wv];
              a2 += src[(r + 2 * tps) * Wv];
              a3 += src[(r + 3 * tps) * Wv];
            }
            for (; r < rpi; r += tps) a0 += src[r * Wv];
          }
          float a = (a0 + a1) + (a2 + a3);
          for (int off = tps / 2; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
          if (mine && l == 0) sums[sidx] = a;
        }
      }
      ga.sync();
      const float n = (float)pc.len;
      for (int c = tg; c < nch; c += ng) {
        const int jj = c / VW, e = c - jj * VW;
        const float sa = sums[(2 * e) * Wv + jj];
        const float sb = sums[(2 * e + 1) * Wv + jj];
        float2 rr;
        if (BWD) {
          rr = make_float2(sa, sb);
        } else {
          const float q = sa / n;
          rr = make_float2(ksh[c] + q, fmaxf(fmaf(-sa, q, sb), 0.f));
        }
        if (P == 1) rec_s[c] = rr;
        else if (publish) put_rec(rec_g + c, rr);
      }
    }
    if (HOLD) tmem_fence_before();  // the piece's tensor-memory stores (waited for) precede the barrier
    ga.sync();  // the records are out; the scratch and the slot are free
    if (pre_u >= 0) {
      unsigned todo = 0;
#pragma unroll
      for (int i = 0; i < kPre; ++i) {
        if (tg + i * ng >= rec_unit) continue;
        if (pre[i]) recs[tg + i * ng] = rec_decode(pre[i]);
        else todo |= 1u << i;
      }
      pre_todo = todo;
      pre_unit = pre_u;
    }
    return true;
  };

  // ---- the statistics of piece k's unit, by the threads of `gr`: its
  // records (all published by now, or polled until they are), merged into
  // the unit's per-group results at gout; the unit's first piece also writes
  // the forward's mean and rstd or the backward's per-channel sums
  auto merge_unit = [&](int k, const Group& gr, int* flag, float2* gout) -> bool {
    const Piece pc = piece_of<LAYOUT>(g, k * NC + b);
    const float* cs = cstb + (k % NCB) * CST;
    const float2* R = recs + (k % NRB) * nch;
    const int lane = gr.t & 31, wg = gr.t >> 5, nwg = gr.n >> 5;
    if (P > 1) {
      const unsigned todo = pre_unit == pc.u ? pre_todo : record_mask(rec_unit, gr);
      pre_unit = -1;
      if (!gather_records(p.part + (int64_t)pc.u * rec_unit, recs, todo, p.err, flag, gr)) return false;
      R = recs;
    }
    // one warp per group of the unit, over the group's records (lane l takes
    // records l, l + 32, ... in piece-major order), then a fixed xor tree.  Forward: mean =
    // sum(n_i*mean_i) / M and M2 = sum(M2_i + n_i*(mean_i - mean)^2), the
    // parallel-axis identity over all of a group's records at once; backward:
    // c1 = sum gamma_c*S1 and c2 = sum gamma_c*S2.
    const int64_t gbase = LAYOUT == kNHWC ? (int64_t)pc.n * g.G + pc.cbase / Cg : pc.u;
    for (int q = wg; q < ngrp; q += nwg) {
      const int nrow = LAYOUT == kNHWC ? Cg : 1;  // records of a piece in the group
      const float2* Rq = R + (LAYOUT == kNHWC ? q * Cg : 0);
      const int rstride = LAYOUT == kNHWC ? nch : 1;
      // record f of the group (f < P * nrow): piece f / nrow, channel f % nrow
      const int nrec = P * nrow;
      if (!BWD) {
        float s = 0.f;
        for (int f = lane; f < nrec; f += 32) {
          const int t = f / nrow, i = f - t * nrow;
          s = fmaf(cnt[t], Rq[t * rstride + i].x, s);
        }
        const float mean = warp_allsum(s) / Mg;
        float m2 = 0.f;
        for (int f = lane; f < nrec; f += 32) {
          const int t = f / nrow, i = f - t * nrow;
          const float2 v = Rq[t * rstride + i];
          const float d = v.x - mean;
          m2 += fmaf(cnt[t] * d, d, v.y);
        }
        m2 = warp_allsum(m2);
        if (lane == 0) gout[q] = make_float2(mean, 1.0f / sqrtf(m2 / Mg + p.eps));
      } else {
        float c1 = 0.f, c2 = 0.f;
        for (int f = lane; f < nrec; f += 32) {
          const int t = f / nrow, i = f - t * nrow;
          const float gm = LAYOUT == kNHWC ? cs[q * Cg + i] : cs[plane_of[t]];
          const float2 tm = channel_terms(gm, Rq[t * rstride + i]);
          c1 += tm.x;
          c2 += tm.y;
        }
        c1 = warp_allsum(c1);
        c2 = warp_allsum(c2);
        const float r = LAYOUT == kNHWC ? cs[nch + ngrp + q] : cs[Cg + 1];
        if (lane == 0) gout[q] = coef_from(c1, c2, g, r);
      }
    }
    // the unit's first piece also writes its per-channel sums (backward, for
    // dgamma / dbeta) -- channel c's pieces in piece order
    if (BWD && pc.t == 0 && (p.dgamma || p.dbeta)) {
      const int nchan = LAYOUT == kNHWC ? nch : Cg;
      const int64_t c0 = LAYOUT == kNHWC ? pc.cbase : (int64_t)pc.gi * Cg;
      for (int c = gr.t; c < nchan; c += gr.n) {
        float sa = 0.f, sb = 0.f;
        const int cnt_c = LAYOUT == kNHWC ? P : (int)g.wm;
        for (int t = 0; t < cnt_c; ++t) {
          const float2 v = LAYOUT == kNHWC ? R[t * nch + c] : R[c * (int)g.wm + t];
          sa += v.x;
          sb += v.y;
        }
        p.chst[(int64_t)pc.n * g.C + c0 + c] = make_float2(sa, sb);
      }
    }
    gr.sync();  // the groups' values; the gathered records are read
    if (!BWD && pc.t == 0)
      for (int q = gr.t; q < ngrp; q += gr.n) {
        p.mean[gbase + q] = gout[q].x;
        p.rstd[gbase + q] = gout[q].y;
      }
    return true;
  };

  // ---- stage B of piece k: the unit's statistics (merged here, or by the
  // merge warp), the piece's output
  auto stage_b = [&](int k) -> bool {
    const Piece pc = piece_of<LAYOUT>(g, k * NC + b);
    const char* slot = ring + (size_t)(k % S) * slot_bytes;  // without HOLD the piece is still there
    const float* cs = cstb + (k % NCB) * CST;
    if (!MW && !merge_unit(k, gb, &s_ok_b, grp)) return false;
    const float2* gres = MW ? grp + k % H : grp;  // the unit's per-group results
    // WS: the records of the next piece's unit, read while this one is written
    int nxt_u = -1;
    if (WS && !MW && read_ahead && k + 1 < K) {
      nxt_u = piece_of<LAYOUT>(g, (k + 1) * NC + b).u;
      const float2* src = p.part + (int64_t)nxt_u * rec_unit;
#pragma unroll
      for (int i = 0; i < kPre; ++i)
        pre[i] = tg + i * ng < rec_unit ? ld_rec_raw(src + tg + i * ng) : 0ull;
    }

    // ---- the piece's output, from tensor memory (HOLD) or its slot
    if (LAYOUT == kNCHW) {
      float ca, cb, cm, cd;
      const float gm = cs[pc.c - pc.gi * Cg];
      if (BWD) {
        ca = cs[Cg + 1] * gm;
        cm = cs[Cg];
        cb = gres[0].x;
        cd = gres[0].y;
      } else {
        cm = gres[0].x;
        ca = gres[0].y * gm;
        cb = cs[Cg];
        cd = 0.f;
      }
      const int nv = pc.len / VW;
      T* o = out + pc.e0;
      auto put = [&](int v, const uint4& rx, const uint4& rd) {
        float xv[VW];
        Access<T, VW>::unpack(rx, xv);
        if (BWD) {
          float dv[VW];
          Access<T, VW>::unpack(rd, dv);
#pragma unroll
          for (int e = 0; e < VW; ++e) xv[e] = fmaf(ca, dv[e], fmaf(cb, xv[e] - cm, cd));
        } else {
#pragma unroll
          for (int e = 0; e < VW; ++e) xv[e] = fmaf(xv[e] - cm, ca, cb);
        }
        Access<T, VW>::store(o + (int64_t)v * VW, xv, pol_out);
      };
      if constexpr (HOLD) {
        // the tensor-memory loads run one batch ahead: batch i0 + 4 is in
        // flight while batch i0 is written (two register sets, a and b)
        const uint32_t tb = tthr + (uint32_t)(k % H) * bcols;
        uint32_t xa[16], da[16], xb[16], db[16];
        auto load = [&](int i0, uint32_t (&xr)[16], uint32_t (&dr)[16]) {
          tmem_ld16(tb + 4u * (uint32_t)i0, xr);
          if constexpr (BWD) tmem_ld16(tb + 4u * (uint32_t)(T4 + i0), dr);
        };
        auto write = [&](int i0, const uint32_t (&xr)[16], const uint32_t (&dr)[16]) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int v = tg + (i0 + u) * ng;
            if (v < nv) {
              if constexpr (BWD) put(v, get4(xr, u), get4(dr, u));
              else put(v, get4(xr, u), get4(xr, u));
            }
          }
        };
        load(0, xa, da);
        tmem_wait_ld();
        for (int i0 = 0; i0 < T4; i0 += 8) {
          const bool nb = i0 + 4 < T4;
          if (nb) load(i0 + 4, xb, db);
          write(i0, xa, da);
          tmem_wait_ld();
          if (!nb) break;
          const bool na = i0 + 8 < T4;
          if (na) load(i0 + 8, xa, da);
          write(i0 + 4, xb, db);
          tmem_wait_ld();
        }
      } else {
#pragma unroll 4
        for (int v = tg; v < nv; v += ng)
          put(v, lds16(slot + (size_t)v * 16),
              BWD ? lds16(slot + g.ten_stride + (size_t)v * 16) : make_uint4(0u, 0u, 0u, 0u));
      }
    } else {
      float ca[VW], cb[VW], cm[VW], cd[VW];
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        const int cl = j * VW + e;
        const float gm = cs[cl];
        const float2 gv = gres[qe[e]];
        if (BWD) {
          ca[e] = cs[nch + ngrp + qe[e]] * gm;
          cm[e] = cs[nch + qe[e]];
          cb[e] = gv.x;
          cd[e] = gv.y;
        } else {
          cm[e] = gv.x;
          ca[e] = gv.y * gm;
          cb[e] = cs[nch + cl];
          cd[e] = 0.f;
        }
      }
      T* o = out + pc.row0 * g.C + pc.cbase + j * VW;
      const char* col = slot + j * 16;
      auto put = [&](int r, const uint4& rx, const uint4& rd) {
        float xv[VW];
        Access<T, VW>::unpack(rx, xv);
        if (BWD) {
          float dv[VW];
          Access<T, VW>::unpack(rd, dv);
#pragma unroll
          for (int e = 0; e < VW; ++e) xv[e] = fmaf(ca[e], dv[e], fmaf(cb[e], xv[e] - cm[e], cd[e]));
        } else {
#pragma unroll
          for (int e = 0; e < VW; ++e) xv[e] = fmaf(xv[e] - cm[e], ca[e], cb[e]);
        }
        Access<T, VW>::store(o + (int64_t)r * g.C, xv, pol_out);
      };
      if constexpr (HOLD) {
        // the tensor-memory loads run one batch ahead, as for NCHW
        const uint32_t tb = tthr + (uint32_t)(k % H) * bcols;
        uint32_t xa[16], da[16], xb[16], db[16];
        auto load = [&](int i0, uint32_t (&xr)[16], uint32_t (&dr)[16]) {
          tmem_ld16(tb + 4u * (uint32_t)i0, xr);
          if constexpr (BWD) tmem_ld16(tb + 4u * (uint32_t)(T4 + i0), dr);
        };
        auto write = [&](int i0, const uint32_t (&xr)[16], const uint32_t (&dr)[16]) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int r = rl + (i0 + u) * rpi;
            if (lane_ok && r < pc.len) {
              if constexpr (BWD) put(r, get4(xr, u), get4(dr, u));
              else put(r, get4(xr, u), get4(xr, u));
            }
          }
        };
        load(0, xa, da);
        tmem_wait_ld();
        for (int i0 = 0; i0 < T4; i0 += 8) {
          const bool nb = i0 + 4 < T4;
          if (nb) load(i0 + 4, xb, db);
          write(i0, xa, da);
          tmem_wait_ld();
          if (!nb) break;
          const bool na = i0 + 8 < T4;
          if (na) load(i0 + 8, xa, da);
          write(i0 + 4, xb, db);
          tmem_wait_ld();
        }
      } else if (lane_ok) {
#pragma unroll 2
        for (int r = rl; r < pc.len; r += rpi)
          put(r, lds16(col + (size_t)r * rowb),
              BWD ? lds16(col + g.ten_stride + (size_t)r * rowb) : make_uint4(0u, 0u, 0u, 0u));
      }
    }
    if (nxt_u >= 0) {
      unsigned todo = 0;
#pragma unroll
      for (int i = 0; i < kPre; ++i) {
        if (tg + i * ng >= rec_unit) continue;
        if (pre[i]) recs[tg + i * ng] = rec_decode(pre[i]);
        else todo |= 1u << i;
      }
      pre_todo = todo;
      pre_unit = nxt_u;
    }
    if (HOLD) tmem_fence_before();  // the piece's tensor-memory loads (waited for) precede the barrier
    gb.sync();  // the slot's (or buffer's) reads are done; the scratch is free
    return true;
  };

  // ---- the pipeline.  A slot takes its next copy (piece k + S) once piece k
  // is done with it: after stage A with HOLD (the piece waits in tensor
  // memory), after stage B without.
  auto issue_next = [&]() {
    if (tid == 0 && issued < K) {
      fence_proxy_async_smem();  // the slot's generic reads precede the new copy
      issue(issued);
      ++issued;
    }
  };
  int ka = 0;  // pieces through stage A
  if constexpr (WS) {
    // Stage A puts piece k into hold buffer k % H once stage B has written
    // piece k - H out of it; stage B takes piece k once stage A has put it
    // there.  Either side gives up when the other has raised the error word.
    if (is_a) {
      for (int k = 0; k < K; ++k) {
        const int h = k % H;
        if (k >= H && !group_wait(tm_empty + h, (uint32_t)((k / H - 1) & 1), p.err, &s_ok_e, ga)) break;
        tmem_fence_after();
        if (!stage_a(k)) break;
        if (tg == 0) mbar_arrive(tm_full + h);
        issue_next();
        ka = k + 1;
      }
    } else if (!is_m) {
      for (int k = 0; k < K; ++k) {
        const int h = k % H;
        if (!group_wait(tm_full + h, (uint32_t)((k / H) & 1), p.err, &s_ok_f, gb)) break;
        if (MW && !group_wait(mg_done + h, (uint32_t)((k / H) & 1), p.err, &s_ok_m, gb)) break;
        tmem_fence_after();
        if (!stage_b(k)) break;
        if (tg == 0) mbar_arrive(tm_empty + h);
      }
    } else {
      // the merge warp: once stage A has piece k in (and so its constants),
      // the statistics of its unit into grp[k % H]; the records of the next
      // piece's unit are read while it merges
      for (int k = 0; k < K; ++k) {
        const int h = k % H;
        if (!group_wait(tm_full + h, (uint32_t)((k / H) & 1), p.err, &s_ok_q, gq)) break;
        int nxt_u = -1;
        if (read_ahead && k + 1 < K) {
          nxt_u = piece_of<LAYOUT>(g, (k + 1) * NC + b).u;
          const float2* src = p.part + (int64_t)nxt_u * rec_unit;
#pragma unroll
          for (int i = 0; i < kPre; ++i) pre[i] = tg + i * 32 < rec_unit ? ld_rec_raw(src + tg + i * 32) : 0ull;
        }
        if (!merge_unit(k, gq, &s_ok_r, grp + h)) break;
        gq.sync();  // the merge has read the gathered records
        if (tg == 0) mbar_arrive(mg_done + h);
        if (nxt_u >= 0) {
          unsigned todo = 0;
#pragma unroll
          for (int i = 0; i < kPre; ++i) {
            if (tg + i * 32 >= rec_unit) continue;
            if (pre[i]) recs[tg + i * 32] = rec_decode(pre[i]);
            else todo |= 1u << i;
          }
          pre_todo = todo;
          pre_unit = nxt_u;
        }
      }
    }
  } else {
    // Stage A runs `ahead` pieces before stage B: by the time a CTA needs a
    // unit's records, every CTA has had `ahead` steps to publish them.
    bool ok = true;
    for (; ok && ka <= ahead && ka < K; ++ka) {
      ok = stage_a(ka);
      if (ok && HOLD) issue_next();
    }
    if (!ok) --ka;  // that piece's copy may still be in flight
    for (int k = 0; ok && k < K; ++k) {
      if (!stage_b(k)) {
        ok = false;
        break;
      }
      if (!HOLD) issue_next();
      if (ka < K) {
        if (!stage_a(ka)) {
          ok = false;
          break;
        }
        if (HOLD) issue_next();
        ++ka;
      }
    }
  }

  // ---- after a wait ran out: this CTA's copies still in flight land first
  if (tid == 0)
    for (int i = ka; i < issued; ++i) wait_bar_t0(full + (i % S), (uint32_t)((i / S) & 1), p.err);
  cp_async_wait_all();  // no asynchronous copy into shared memory outlives the CTA
  if (HOLD) {  // every thread's tensor-memory accesses have completed (waited for)
    tmem_fence_before();
    __syncthreads();
    if (warp == 0) {
      tmem_fence_after();
      tmem_dealloc(s_tmem, kWaveTmemCols);
    }
  }

  // ---- backward: dgamma / dbeta once every unit's per-channel sums are in
  // the workspace (a grid barrier, which every CTA reaches), spread over the
  // CTAs by channel:  dbeta_c = sum_n S1[n, c],  dgamma_c = sum_n rstd[n, g(c)] *
  // S2[n, c]; thread t adds samples t, t + nt, ... in order, then the warps
  // meet in a fixed tree and in warp order.
  if (BWD && (p.dgamma || p.dbeta)) {
    cooperative_groups::this_grid().sync();
    if (!aborted(p.err)) {
      float* wsum = red;
      for (int64_t c = b; c < g.C; c += NC) {
        const int64_t gi = c / g.Cg;
        float db = 0.f, dg = 0.f;
        for (int64_t n = tid; n < g.N; n += nt) {
          const float2 v = __ldcg(p.chst + n * g.C + c);
          db += v.x;
          dg = fmaf(__ldg(p.rstd + n * g.G + gi), v.y, dg);
        }
        db = warp_sum_lane0(db);
        dg = warp_sum_lane0(dg);
        if (lane == 0) {
          wsum[2 * warp] = db;
          wsum[2 * warp + 1] = dg;
        }
        __syncthreads();
        if (tid == 0) {
          float tb = 0.f, tg = 0.f;
          for (int w = 0; w < nwarps; ++w) {
            tb += wsum[2 * w];
            tg += wsum[2 * w + 1];
          }
          if (p.dbeta) p.dbeta[c] = tb;
          if (p.dgamma) p.dgamma[c] = tg;
        }
        __syncthreads();
      }
    }
  }
}

template <typename T, int VW, int LAYOUT, bool BWD>
const void* kernel_ptr(int mode) {
  if (mode == 2) return (const void*)wave_kernel<T, VW, LAYOUT, BWD, 2>;
  if (mode == 1) return (const void*)wave_kernel<T, VW, LAYOUT, BWD, 1>;
  return (const void*)wave_kernel<T, VW, LAYOUT, BWD, 0>;
}

template <typename T>
const void* pick(int layout, bool bwd, int mode) {
  constexpr int V = Elem<T>::VEC;
  if (layout == kNCHW)
    return bwd ? kernel_ptr<T, V, kNCHW, true>(mode) : kernel_ptr<T, V, kNCHW, false>(mode);
  return bwd ? kernel_ptr<T, V, kNHWC, true>(mode) : kernel_ptr<T, V, kNHWC, false>(mode);
}

}  // namespace

const void* wave_kernel_ptr(const Geom& g, bool bwd) {
  const int mode = g.wH > 0 ? (g.wWs ? 2 : 1) : 0;
  switch (g.dtype) {
    case kF32: return pick<float>(g.layout, bwd, mode);
    case kF16: return pick<__half>(g.layout, bwd, mode);
    default: return pick<__nv_bfloat16>(g.layout, bwd, mode);
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
  e = prepare_smem(fn, g.smem);
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
