// gn_tasks.cuh -- the pipelined regime: a lockstep schedule of the reduction
// units, fed by a ring of bulk copies.
//
// One persistent kernel, cooperatively launched so that all its CTAs are
// co-resident.  A unit (one (sample, group)) is cut into P pieces; piece i of
// every unit belongs to CTA i.  Every CTA runs the same steps s = 0, 1, ...,
// U + D - 1:
//   pass 1 of unit s (s < U):     stream the piece, add it up, write its record
//                                 and arrive on the unit's counter -- without
//                                 waiting for the counter's old value;
//   pass 2 of unit s - D (s >= D): wait for that unit's ready record, stream
//                                 the piece again (it is still in L2: only D
//                                 units were read since) and write the output.
// Unit u is finalised (statistics, then its ready record) by CTA u mod P at
// the start of its step u + 1, once all pieces of u have arrived; arrivals are
// fire-and-forget.  Deadlock-free: take the smallest unit w that some CTA
// waits for, either for w's record or, as w's finaliser, for w's arrivals.
// Every CTA's waits before its pass 1 of w (steps <= w) are on units < w, so
// by minimality each CTA gets past its pass 1 of w; then w's finaliser, whose
// waits before step w + 1 are also on smaller units, finalises w.  Every wait is also
// bounded: after kReadyWaitLimit polls the CTA raises bit 1 of the workspace
// error word and skips that piece's output.  Results do not depend on timing:
// records have fixed slots and every sum has a fixed order.
#pragma once

#include "gn_finalize.cuh"

namespace gn {

constexpr uint32_t kReadyWaitLimit = 1u << 22;  // polls, about 100 ns apart

struct Task {
  int pass;
  int64_t unit, piece, step;
};

// A unit's ready record: two floats (the forward's mean and rstd, or the
// backward's coefficients B and D) in one 64-bit word, each XORed with
// kRecKey, so that the zero-filled workspace reads "not ready" and a written
// record never does (kRecKey is a NaN bit pattern that no arithmetic
// produces).  Written once with release semantics, read with acquire.
constexpr uint32_t kRecKey = 0x7fbadbadu;

__device__ __forceinline__ void put_record(unsigned long long* rec, float lo, float hi) {
  const unsigned long long v =
      ((unsigned long long)(__float_as_uint(hi) ^ kRecKey) << 32) | (__float_as_uint(lo) ^ kRecKey);
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(rec), "l"(v) : "memory");
}

// Thread 0 polls the record with acquire loads, at most kReadyWaitLimit
// times; the whole CTA then learns whether it was seen and its two floats.
// On timeout bit 1 of the error word is raised.
__device__ __forceinline__ bool wait_record(const unsigned long long* rec, unsigned* err,
                                            float* lo, float* hi) {
  __shared__ int s_ok;
  __shared__ float s_v[2];
  if (threadIdx.x == 0) {
    int ok = 0;
    for (uint32_t i = 0; i < kReadyWaitLimit; ++i) {
      unsigned long long v;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(rec) : "memory");
      if (v) {
        ok = 1;
        s_v[0] = __uint_as_float((unsigned)v ^ kRecKey);
        s_v[1] = __uint_as_float((unsigned)(v >> 32) ^ kRecKey);
        break;
      }
      __nanosleep(64);
    }
    if (!ok) atomicOr(err, 2u);
    s_ok = ok;
  }
  __syncthreads();
  *lo = s_v[0];
  *hi = s_v[1];
  return s_ok != 0;
}

// Thread 0 arrives on unit u's counter; the record stores before it are
// ordered by the release.  Nothing waits for the counter's value here.
__device__ __forceinline__ void arrive_release(const KParams& p, int64_t u) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.tickets + u) : "memory");
}

// At the first task of step `step`: if this CTA is the finaliser of unit
// step - 1 (CTA u mod P for unit u), thread 0 waits (bounded) until all P
// pieces of that unit have arrived, then the whole CTA runs fin(u).  The
// finalisation work rotates over the CTAs, so no CTA falls behind by doing
// all of it.  Called by every thread.
template <typename Fin>
__device__ __forceinline__ void finalize_due(const KParams& p, int64_t step, Fin fin) {
  const int64_t u = step - 1;
  if (u < 0 || u >= p.g.units_fin || u % p.g.pieces != (int64_t)blockIdx.x) return;
  __shared__ int s_go;
  if (threadIdx.x == 0) {
    int ok = 0;
    const unsigned want = (unsigned)p.g.arrivals_per_n;
    for (uint32_t i = 0; i < kReadyWaitLimit; ++i) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p.tickets + u) : "memory");
      if (v == want) {
        ok = 1;
        break;
      }
      __nanosleep(32);
    }
    if (!ok) atomicOr(p.err, 2u);
    s_go = ok;
  }
  __syncthreads();
  if (s_go) fin(u);
}

// ------------------------------------------------------------ the ring
// Thread 0 streams the chunks of the CTA's tasks, in step order, into a ring
// of S shared-memory slots with 1-D bulk copies (TMA), each slot completing on
// its own mbarrier; S - 1 chunks stay in flight while the whole CTA consumes
// the current one.  A slot holds one chunk of x (and, in the backward, the
// matching chunk of dy at offset ten_stride) and a header naming its task and
// chunk; a header with k = kStopTask ends the loop.

constexpr int64_t kStopTask = -1;

// A slot's header: the task and chunk it holds, decoded once by thread 0 so
// that consumers do no index arithmetic of their own.  a..e describe the
// piece in the layout's terms (set by the kernel's describe function).
struct SlotHdr {
  int64_t k;     // task sequence number in this CTA, or kStopTask
  int64_t unit;  // reduction unit
  int64_t step;  // the step the task belongs to
  int64_t a, b, c, d, e;
  int32_t pass, chunk, nchunks, bytes;  // bytes: of each tensor's chunk
  int64_t aux_off;                      // byte address of the 16-byte aux copy, or 0
  int64_t pad_;
  uint4 aux;  // 16 bytes copied with the first chunk of a task (see run_ring)
};

static_assert(sizeof(SlotHdr) <= kSlotHdrBytes, "slot header larger than the plan reserves");

struct RingSmem {
  char* ring;       // S slots, slot s at ring + s * slot_stride
  SlotHdr* hdr;     // S headers
  uint64_t* full;   // S mbarriers
  int S;
  int64_t slot_stride, ten_stride;
};

__device__ __forceinline__ RingSmem ring_smem(const Geom& g, char* smem) {
  RingSmem r;
  r.ring = smem + g.off_ring;
  r.hdr = reinterpret_cast<SlotHdr*>(smem + g.off_tot);  // kSlotHdrBytes apart
  r.full = reinterpret_cast<uint64_t*>(smem + g.off_bar);
  r.S = g.S;
  r.ten_stride = g.ten_stride;
  r.slot_stride = g.ten_stride * (g.dy_in_ring ? 2 : 1);
  return r;
}

__device__ __forceinline__ SlotHdr* hdr_at(const RingSmem& R, int s) {
  return reinterpret_cast<SlotHdr*>(reinterpret_cast<char*>(R.hdr) + s * kSlotHdrBytes);
}

// Runs the CTA's tasks through the ring.  Thread 0 only:
// `describe(task, hdr)` fills hdr.a..e, hdr.nchunks and hdr.aux_off (the
// 16-byte aligned global address of 16 bytes the task's first chunk brings
// along into hdr.aux, or 0 for none) for a task, and
// `chunk_off(hdr, c, &bytes)` gives the element offset in x (and dy) of chunk
// c and its bytes.  `consume(hdr, slot_x, slot_dy)` is called by every thread
// of the CTA for each chunk in order and may use __syncthreads; it returns
// (the same in every thread) whether it left an output chunk in place of x in
// the slot, which thread 0 then sends to `out_at(hdr)` with a bulk store (one
// bulk group per chunk, empty if there is none).  A slot is refilled one chunk
// later, once its store has read it, so the CTA's threads make no global
// stores of their own for the output and a fence waits for none.  Every wait is
// bounded: a copy that does not land in time raises bit 0 of the error word,
// the CTA stops consuming, waits (bounded) for the copies it issued and
// leaves.  The last CTA to leave clears the ready records and its counter.
template <bool kDy, typename Describe, typename ChunkOff, typename Consume, typename OutAt>
__device__ __forceinline__ void run_ring(const KParams& p, const RingSmem& R, Describe describe,
                                         ChunkOff chunk_off, Consume consume, OutAt out_at) {
  const Geom& g = p.g;
  const int64_t U = g.units_fin, D = g.lag, piece = blockIdx.x;
  const char* xb = static_cast<const char*>(p.x);
  const char* db = static_cast<const char*>(p.dy);
  const int esz = dtype_size(g.dtype);
  __shared__ int s_ok;
  if (threadIdx.x == 0) {
    for (int i = 0; i < R.S; ++i) mbar_init(R.full + i, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // thread 0's issue state: the step and half-step (pass) of the next task
  int64_t st = 0, seq = 0;
  int half = 0;
  SlotHdr cur{};
  bool idone = piece >= g.pieces;  // CTAs beyond the pieces have no tasks
  int issued = 0;                  // slots issued and not yet consumed
  cur.nchunks = 0;
  cur.chunk = 0;
  const uint64_t pol1 = policy_evict_last(), pol2 = policy_evict_first();
  auto next_task = [&](Task& t) {
    while (st < U + D) {
      if (half == 0) {
        half = 1;
        if (st < U) {
          t.pass = 1;
          t.unit = st;
          t.piece = piece;
          t.step = st;
          return true;
        }
      } else {
        half = 0;
        const int64_t u = st - D, s0 = st++;
        if (u >= 0) {
          t.pass = 2;
          t.unit = u;
          t.piece = piece;
          t.step = s0;
          return true;
        }
      }
    }
    return false;
  };
  auto stop = [&](int s) {  // the stop marker: completes the phase, no bytes expected
    hdr_at(R, s)->k = kStopTask;
    mbar_arrive(R.full + s);
    idone = true;
    ++issued;
  };
  auto issue = [&](int s) {
    if (idone) return;
    if (cur.chunk == cur.nchunks) {
      Task t;
      if (!next_task(t)) {
        stop(s);
        return;
      }
      cur.k = seq++;
      cur.pass = t.pass;
      cur.unit = t.unit;
      cur.step = t.step;
      describe(t, cur);
      cur.chunk = 0;
    }
    int32_t bytes = 0;
    const int64_t off = chunk_off(cur, cur.chunk, &bytes);
    cur.bytes = bytes;
    SlotHdr* hd = hdr_at(R, s);
    *hd = cur;
    const bool aux = cur.chunk == 0 && cur.aux_off != 0;
    if (aux) fence_proxy_async_smem();  // the header store before the copy into hd->aux
    const uint64_t pol = cur.pass == 1 ? pol1 : pol2;  // pass 1 keeps its input in L2 for pass 2
    char* slot = R.ring + s * R.slot_stride;
    mbar_arrive_expect_tx(R.full + s, (uint32_t)bytes * (kDy ? 2u : 1u) + (aux ? 16u : 0u));
    if (aux)
      tma_load_1d(&hd->aux, reinterpret_cast<const void*>(cur.aux_off), 16u, R.full + s, pol1);
    tma_load_1d(slot, xb + off * esz, (uint32_t)bytes, R.full + s, pol);
    if (kDy) tma_load_1d(slot + R.ten_stride, db + off * esz, (uint32_t)bytes, R.full + s, pol);
    ++cur.chunk;
    ++issued;
  };
  if (threadIdx.x == 0) {
    if (idone)
      stop(0);
    else
      for (int i = 0; i < R.S && !idone; ++i) issue(i);
  }
  int s = 0, refill = -1;  // refill: the slot consumed one chunk ago
  uint32_t ph = 0;
  const uint64_t pfirst = pol2;
  while (true) {
    if (threadIdx.x == 0) s_ok = mbar_wait(R.full + s, ph, p.err) ? 1 : 0;
    __syncthreads();
    if (!s_ok) break;  // the same decision in every thread
    mbar_wait(R.full + s, ph, p.err);  // completed: returns at once (acquire for this thread)
    const SlotHdr& h = *hdr_at(R, s);
    if (h.k == kStopTask) {
      if (threadIdx.x == 0) --issued;
      break;
    }
    char* slot = R.ring + s * R.slot_stride;
    const bool out = consume(h, slot, slot + R.ten_stride);
    __syncthreads();  // every thread is done with slot s
    if (threadIdx.x == 0) {
      --issued;
      fence_proxy_async_smem();  // the slot's generic accesses before async-proxy ones
      if (out) tma_store_1d(out_at(h), slot, (uint32_t)h.bytes, pfirst);
      bulk_commit();
      if (refill >= 0) {
        bulk_wait_read<1>();  // the refilled slot's store (if any) has read it
        issue(refill);
      }
      refill = s;
    }
    if (++s == R.S) {
      s = 0;
      ph ^= 1u;
    }
  }
  unsigned* q = p.queue;
  if (threadIdx.x == 0) {
    bulk_wait_all<0>();  // the output stores are complete
    // after an abort: wait (bounded) for the copies still in flight
    for (int i = 0; i < issued; ++i) {
      const int si = (s + i) % R.S;
      const uint32_t pi = ph ^ (uint32_t)(((s + i) / R.S) & 1);
      mbar_wait(R.full + si, pi, p.err);
    }
    __threadfence();
    s_ok = atomicAdd(q, 1u) == gridDim.x - 1 ? 1 : 0;
  }
  __syncthreads();
  if (s_ok) {
    // every CTA has left its steps: no record is read any more in this call
    unsigned long long* rec = reinterpret_cast<unsigned long long*>(p.ready);
    for (int64_t u = threadIdx.x; u < U; u += blockDim.x) rec[u] = 0ull;
    if (threadIdx.x == 0) atomicExch(q, 0u);
  }
}

// Host: one cooperative launch (all CTAs co-resident) of `kernel` on g.grid
// CTAs of g.tpb threads, between the timing events when they are set.
inline cudaError_t launch_cooperative(const void* kernel, const KParams& p, size_t smem,
                                      cudaStream_t s) {
  if (smem > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const TimingEvents& ev = timing_events();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.g.grid, 1, 1);
  cfg.blockDim = dim3((unsigned)p.g.tpb, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<KParams*>(&p)};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, kernel, args);
  if (ev.end) cudaEventRecord(ev.end, s);
  return e;
}

}  // namespace gn
