// gn_tasks.cuh -- the task queue of the pipelined regime.
//
// One persistent, cooperatively launched kernel (all CTAs co-resident) runs
// two kinds of task per unit (a sample, or one (sample, group)):
//   pass 1, piece q: stream the piece, write its partial record to a fixed
//           slot, arrive on the unit's counter; the last arrival finalises
//           the unit and raises its ready flag;
//   pass 2, piece q: wait for the unit's ready flag, then the elementwise
//           output of the piece, reading its input again (from L2).
// Tasks are handed out in one global order in which every pass-1 task of a
// unit precedes all pass-2 tasks of that unit, and the pass-2 tasks of unit u
// follow the pass-1 tasks of unit u + lag.  A CTA waiting on a flag holds at
// most one later task (its prefetched next index); following the waits from
// any waiting CTA leads to strictly earlier pass-2 tasks, so the earliest
// waiting task's unit only needs tasks that are running or done, and every
// wait ends.  Each wait is also bounded: after kReadyWaitLimit polls the CTA
// raises bit 1 of the workspace error word and skips that piece's output.
// Results do not depend on which CTA runs which task: records have fixed
// slots and every sum has a fixed order.
#pragma once

#include "gn_finalize.cuh"

namespace gn {

constexpr uint32_t kReadyWaitLimit = 1u << 22;  // polls, about 100 ns apart

struct Task {
  int pass;
  int64_t unit, piece;
};

// Queue index k -> task, for U units of P pieces and a lag of D units:
//   P1(0) .. P1(D-1) | P1(D) P2(0) | P1(D+1) P2(1) | ... | P2(U-D) .. P2(U-1)
// where P1(u) / P2(u) stand for the P pass-1 / pass-2 tasks of unit u.
__device__ __forceinline__ Task decode_task(int64_t k, int64_t U, int64_t P, int64_t D) {
  Task t;
  const int64_t a = D * P, b = (U - D) * 2 * P;
  if (k < a) {
    t.pass = 1;
    t.unit = k / P;
    t.piece = k % P;
  } else if (k < a + b) {
    const int64_t j = k - a, s = D + j / (2 * P), r = j % (2 * P);
    t.pass = r < P ? 1 : 2;
    t.unit = r < P ? s : s - D;
    t.piece = r < P ? r : r - P;
  } else {
    const int64_t j = k - a - b;
    t.pass = 2;
    t.unit = U - D + j / P;
    t.piece = j % P;
  }
  return t;
}

// Thread 0 polls the flag with acquire semantics, at most kReadyWaitLimit
// times; every thread then learns whether it was seen.  On timeout bit 1 of
// the error word is raised.
__device__ __forceinline__ bool wait_ready(const unsigned* flag, unsigned* err) {
  __shared__ int s_ok;
  if (threadIdx.x == 0) {
    int ok = 0;
    for (uint32_t i = 0; i < kReadyWaitLimit; ++i) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
      if (v) {
        ok = 1;
        break;
      }
      __nanosleep(64);
    }
    if (!ok) atomicOr(err, 2u);
    s_ok = ok;
  }
  __syncthreads();
  __threadfence();
  return s_ok != 0;
}

// Runs f(task) on the tasks this CTA takes from the queue; the next index is
// fetched while the current task runs.  The last CTA to leave resets the
// queue, so every call starts from task 0.
template <typename F>
__device__ __forceinline__ void run_tasks(const KParams& p, F f) {
  const Geom& g = p.g;
  const int64_t total = 2 * g.units_fin * g.pieces;
  __shared__ unsigned s_k[2];
  unsigned* q = p.queue;
  if (threadIdx.x == 0) s_k[0] = atomicAdd(q, 1u);
  __syncthreads();
  int b = 0;
  unsigned k = s_k[0];
  while ((int64_t)k < total) {
    if (threadIdx.x == 0) s_k[b ^ 1] = atomicAdd(q, 1u);
    f(decode_task((int64_t)k, g.units_fin, g.pieces, g.lag));
    __syncthreads();
    b ^= 1;
    k = s_k[b];
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(q + 1, 1u) == gridDim.x - 1) {
      atomicExch(q, 0u);
      atomicExch(q + 1, 0u);
    }
  }
}

// After a pass-2 task of unit u: the unit's last pass-2 task clears the
// unit's ready flag and counter, so the workspace leaves the call as it came.
__device__ __forceinline__ void finish_pass2(const KParams& p, int64_t u) {
  __syncthreads();
  if (threadIdx.x == 0 && atomicAdd(p.p2cnt + u, 1u) == (unsigned)p.g.pieces - 1) {
    atomicExch(p.ready + u, 0u);
    atomicExch(p.p2cnt + u, 0u);
  }
}

// Host: one cooperative launch (all CTAs co-resident) of `kernel` on g.grid
// CTAs of g.tpb threads, between the timing events when they are set.
inline cudaError_t launch_cooperative(const void* kernel, const KParams& p, size_t smem,
                                      cudaStream_t s) {
  const TimingEvents& ev = timing_events();
  if (ev.begin) cudaEventRecord(ev.begin, s);
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
