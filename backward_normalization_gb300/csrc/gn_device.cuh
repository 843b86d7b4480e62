// gn_device.cuh -- device-side building blocks shared by the GroupNorm kernels:
// 16-byte vector loads/stores with L2 cache-policy hints, fp16/bf16/fp32
// conversion, deterministic block and cluster reductions and the per-unit
// arrival counter used by the "last CTA finalises" reductions.
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gn_internal.h"

namespace gn {

namespace cg = cooperative_groups;

// ------------------------------------------------------------ cache policies
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Read-only 16-byte load through the non-coherent path, not kept in L1, with
// an L2 eviction policy.  Inputs are never written while a kernel runs.
__device__ __forceinline__ uint4 ld16(const void* p, uint64_t pol) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p), "l"(pol));
  return r;
}
__device__ __forceinline__ void st16(void* p, const uint4& v, uint64_t pol) {
  asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;"
               :
               : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}

// ----------------------------------------------------------- element access
template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int VEC = 4;  // elements per 16 bytes
  __device__ static float to_f(float v) { return v; }
  __device__ static float from_f(float v) { return v; }
};
template <>
struct Elem<__half> {
  static constexpr int VEC = 8;
  __device__ static float to_f(__half v) { return __half2float(v); }
  __device__ static __half from_f(float v) { return __float2half_rn(v); }
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int VEC = 8;
  __device__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

template <>
struct Elem<double> {  // storage only: computed in fp32
  static constexpr int VEC = 2;
  __device__ static float to_f(double v) { return __double2float_rn(v); }
  __device__ static double from_f(float v) { return (double)v; }
};

__device__ __forceinline__ float2 h2f(uint32_t w) {
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = w;
  return __half22float2(h);
}
__device__ __forceinline__ float2 b2f(uint32_t w) {
  __nv_bfloat162 h;
  *reinterpret_cast<uint32_t*>(&h) = w;
  return __bfloat1622float2(h);
}
__device__ __forceinline__ uint32_t f2h(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t f2b(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Load VW consecutive elements starting at p as floats.  VW is either the
// 16-byte vector width of T (p 16-byte aligned) or 1 (scalar path).
template <typename T, int VW>
struct Access;

// Besides load/store, each access type exposes load_raw (the bits, kept packed
// while loads are in flight) and unpack (bits -> floats), so that deep unrolls
// hold 4 registers per 16-byte vector instead of VW floats.
template <typename T>
struct Access<T, 1> {
  using Raw = T;
  __device__ static Raw load_raw(const T* p, uint64_t) { return __ldg(p); }
  __device__ static void unpack(const Raw& r, float (&f)[1]) { f[0] = Elem<T>::to_f(r); }
  __device__ static void load(const T* p, float (&f)[1], uint64_t) {
    f[0] = Elem<T>::to_f(__ldg(p));
  }
  __device__ static void store(T* p, const float (&f)[1], uint64_t) {
    *p = Elem<T>::from_f(f[0]);
  }
};
template <>
struct Access<float, 4> {
  using Raw = uint4;
  __device__ static Raw load_raw(const float* p, uint64_t pol) { return ld16(p, pol); }
  __device__ static void unpack(const Raw& u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  __device__ static void load(const float* p, float (&f)[4], uint64_t pol) {
    const uint4 u = ld16(p, pol);
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  __device__ static Raw pack(const float (&f)[4]) {
    uint4 u;
    u.x = __float_as_uint(f[0]);
    u.y = __float_as_uint(f[1]);
    u.z = __float_as_uint(f[2]);
    u.w = __float_as_uint(f[3]);
    return u;
  }
  __device__ static void store(float* p, const float (&f)[4], uint64_t pol) { st16(p, pack(f), pol); }
};
template <>
struct Access<double, 2> {  // two doubles per 16 bytes, rounded to fp32 on load
  using Raw = uint4;
  __device__ static Raw load_raw(const double* p, uint64_t pol) { return ld16(p, pol); }
  __device__ static void unpack(const Raw& u, float (&f)[2]) {
    f[0] = __double2float_rn(__hiloint2double((int)u.y, (int)u.x));
    f[1] = __double2float_rn(__hiloint2double((int)u.w, (int)u.z));
  }
  __device__ static void load(const double* p, float (&f)[2], uint64_t pol) {
    unpack(ld16(p, pol), f);
  }
  __device__ static Raw pack(const float (&f)[2]) {
    const double a = f[0], b = f[1];
    uint4 u;
    u.x = (uint32_t)__double2loint(a);
    u.y = (uint32_t)__double2hiint(a);
    u.z = (uint32_t)__double2loint(b);
    u.w = (uint32_t)__double2hiint(b);
    return u;
  }
  __device__ static void store(double* p, const float (&f)[2], uint64_t pol) { st16(p, pack(f), pol); }
};
template <>
struct Access<__half, 8> {
  using Raw = uint4;
  __device__ static Raw load_raw(const __half* p, uint64_t pol) { return ld16(p, pol); }
  __device__ static void unpack(const Raw& u, float (&f)[8]) {
    float2 a = h2f(u.x), b = h2f(u.y), c = h2f(u.z), d = h2f(u.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
  }
  __device__ static void load(const __half* p, float (&f)[8], uint64_t pol) {
    const uint4 u = ld16(p, pol);
    float2 a = h2f(u.x), b = h2f(u.y), c = h2f(u.z), d = h2f(u.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
  }
  __device__ static Raw pack(const float (&f)[8]) {
    uint4 u;
    u.x = f2h(f[0], f[1]);
    u.y = f2h(f[2], f[3]);
    u.z = f2h(f[4], f[5]);
    u.w = f2h(f[6], f[7]);
    return u;
  }
  __device__ static void store(__half* p, const float (&f)[8], uint64_t pol) { st16(p, pack(f), pol); }
};
template <>
struct Access<__nv_bfloat16, 8> {
  using Raw = uint4;
  __device__ static Raw load_raw(const __nv_bfloat16* p, uint64_t pol) { return ld16(p, pol); }
  __device__ static void unpack(const Raw& u, float (&f)[8]) {
    float2 a = b2f(u.x), b = b2f(u.y), c = b2f(u.z), d = b2f(u.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
  }
  __device__ static void load(const __nv_bfloat16* p, float (&f)[8], uint64_t pol) {
    const uint4 u = ld16(p, pol);
    float2 a = b2f(u.x), b = b2f(u.y), c = b2f(u.z), d = b2f(u.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
  }
  __device__ static Raw pack(const float (&f)[8]) {
    uint4 u;
    u.x = f2b(f[0], f[1]);
    u.y = f2b(f[2], f[3]);
    u.z = f2b(f[4], f[5]);
    u.w = f2b(f[6], f[7]);
    return u;
  }
  __device__ static void store(__nv_bfloat16* p, const float (&f)[8], uint64_t pol) {
    st16(p, pack(f), pol);
  }
};

// ------------------------------------------------------------- reductions
// Warp sum with a fixed association; the result is meaningful in lane 0 only.
__device__ __forceinline__ float warp_sum_lane0(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_down_sync(0xffffffffu, v, off);
  return v;
}

// Block sum of two values with a fixed tree (shuffle within warps, then the
// warp results in warp order).  Returns the totals in thread 0.
// `scratch` holds at least 2 * 32 floats.
__device__ __forceinline__ float2 block_sum2_t0(float a, float b, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  a = warp_sum_lane0(a);
  b = warp_sum_lane0(b);
  if (lane == 0) {
    scratch[2 * warp] = a;
    scratch[2 * warp + 1] = b;
  }
  __syncthreads();
  float2 r = make_float2(0.f, 0.f);
  if (threadIdx.x == 0) {
    for (int w = 0; w < nw; ++w) {
      r.x += scratch[2 * w];
      r.y += scratch[2 * w + 1];
    }
  }
  __syncthreads();
  return r;
}


// ------------------------------------------------- TMA bulk copies, mbarriers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
// Makes initialised mbarriers visible to the async (TMA) proxy and the cluster.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Orders this thread's earlier generic-proxy shared-memory accesses (and those
// of the CTA, after a barrier) before later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
// One contiguous global -> shared copy of `bytes` (16-byte aligned, multiple of
// 16) that completes on `bar`, with an L2 eviction policy for the source.
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes,
                                            uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}
// One contiguous shared -> global copy of `bytes` (16-byte aligned, multiple
// of 16) in the current bulk async-group, with an L2 eviction policy for the
// destination.
__device__ __forceinline__ void tma_store_1d(void* dst, const void* src, uint32_t bytes,
                                             uint64_t pol) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::
                   "l"(dst), "r"(smem_addr(src)), "r"(bytes), "l"(pol)
               : "memory");
}
// Closes the current bulk async-group (an empty one if it holds no copy).
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most N bulk async-groups are still reading their shared
// memory sources (.read), or are still in flight at all.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// One 2-D tile [rows x cols] at (col c0, row r0) of the tensor map -> shared
// memory (rows packed, no swizzle), completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t c0,
                                            int32_t r0, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(r0), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same test, letting the hardware suspend the thread for up to `hint_ns`
// nanoseconds while the phase is incomplete (fewer polls, more issue slots
// for the other warps of the SM).
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Waits for phase `parity` of `bar` to complete.  The wait is bounded: after
// kMbarWaitLimit polls (far longer than any copy takes) it raises the error
// word and returns false instead of hanging.
constexpr int kMbarWaitLimit = 1 << 22;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* err) {
  for (int i = 0; i < kMbarWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  atomicOr(err, 1u);
  return false;
}
// One arrival on `bar` (count-based phase completion).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Barrier among the first `nthreads` threads of the CTA (a multiple of 32),
// using hardware barrier `id` (1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// The same barrier, returning whether `c` holds in any of those threads.
__device__ __forceinline__ bool named_sync_or(int id, int nthreads, bool c) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)c), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0u;
}
__device__ __forceinline__ uint4 lds16(const void* p) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(smem_addr(p)));
  return r;
}

// --------------------------------------------------------------- tickets
// An arrival counter per reduction unit.  Every CTA that publishes a partial
// result increments it once; the CTA that brings it to `total` is the last one
// and finalises the unit, then sets the counter back to 0, so every completed
// call leaves its counters at 0 for the next call.  (The workspace therefore
// has to be zero-filled once, before its first use.)  atomicAdd never retries,
// so arrivals cost one atomic each however many CTAs arrive together.
//
// Called by one thread after the CTA's partial stores and a __syncthreads().
// One acquire-release atomic at GPU scope: its release half publishes every
// store the barrier ordered before it (the whole CTA's partials) ahead of the
// arrival, and its acquire half orders the last CTA's reads of the other
// CTAs' partials after it (that CTA's other threads read after a following
// barrier).  Returns whether this arrival completed the count.
__device__ __forceinline__ bool publish_and_arrive(unsigned* t, unsigned total) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(t) : "memory");
  return old == total - 1u;
}

// 16-byte asynchronous copy from global to shared memory that bypasses L1
// (the data may have been written by the previous kernel).  Both addresses
// must be 16-byte aligned; the copy is complete after cp_async_wait_all() in
// the issuing thread (then a barrier publishes it to the CTA).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)),
               "l"(__cvta_generic_to_global(src))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
// 4-byte asynchronous copy from global to shared memory (both 4-byte
// aligned), in the issuing thread's current cp.async group.
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)),
               "l"(__cvta_generic_to_global(src))
               : "memory");
}
// Closes this thread's current cp.async group (an empty one if it holds no copy).
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// ------------------------------------------------------------ tensor memory
// Tensor memory (TMEM): 128 lanes x 512 columns of 32-bit cells per SM.  An
// address is (lane << 16) | column.  Warp w of a CTA reaches lanes
// 32*(w % 4) .. 32*(w % 4) + 31; in the 32x32b shapes thread i of the warp
// owns lane 32*(w % 4) + i and register r holds column (address column + r).
// Allocation, release and every load / store below are warp-wide
// (.sync.aligned): all 32 threads execute them with the same address.

// Warp-wide: allocates `ncols` columns (a power of two, 32..512) and writes
// the base address to *dst (shared memory).  Blocks until the columns are free.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
// Warp-wide: frees the columns of tmem_alloc.
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols) : "memory");
}
// Order tensor-memory operations across a thread barrier: `before` ahead of
// the barrier, `after` behind it.
__device__ __forceinline__ void tmem_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Warp-wide: 16 consecutive columns of this thread's lane from / to registers.
// A load's registers are valid only after tmem_wait_ld; a store has finished
// (its cells readable, its columns reusable) after tmem_wait_st.  Neither
// touches memory the compiler sees, so ordinary loads and stores may move
// across them; the waits, fences and barriers keep their order (volatile).
__device__ __forceinline__ void tmem_st16(uint32_t a, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(a),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]));
}
__device__ __forceinline__ void tmem_ld16(uint32_t a, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(a));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------ cluster reduction
// Adds, for every q < NQ, red[q*stride + slot] of all CTAs of the cluster into
// the copy of cluster rank 0, in rank order.  Every thread of every CTA of the
// cluster must call it.  The second cluster barrier keeps each CTA's shared
// memory alive until rank 0 has read it.
template <int NQ>
__device__ __forceinline__ void cluster_sum_to_rank0(float* red, int stride, int slot, bool active) {
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  if (cluster.block_rank() == 0 && active) {
    float acc[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) acc[q] = red[q * stride + slot];
    const unsigned nb = cluster.num_blocks();
    for (unsigned r = 1; r < nb; ++r) {
      const float* rem = cluster.map_shared_rank(red, r);
#pragma unroll
      for (int q = 0; q < NQ; ++q) acc[q] += rem[q * stride + slot];
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) red[q * stride + slot] = acc[q];
  }
  cluster.sync();
}

__device__ __forceinline__ unsigned cluster_rank() {
  return cg::this_cluster().block_rank();
}

// ------------------------------------------- programmatic dependent launch
// The two-kernel path launches every kernel with programmatic stream
// serialisation: a kernel may be scheduled while the previous kernel on the
// stream is still running, and waits (grid_dependency_wait) for that kernel to
// complete and its writes to be visible before it touches global memory that
// earlier work produced or will read.  Each kernel lets its successor launch
// as soon as all of its own CTAs are running (grid_launch_dependents), so the
// successor's CTAs take the SMs as this kernel's CTAs exit instead of after a
// launch gap.  Without the launch attribute both instructions are no-ops.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Host: launches kernel(p) on `grid` CTAs with the programmatic-serialisation
// attribute (see above).
template <typename Kernel>
inline cudaError_t launch_pdl(Kernel kernel, int64_t grid, int block, size_t smem,
                              cudaStream_t s, const KParams& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3((unsigned)block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace gn
