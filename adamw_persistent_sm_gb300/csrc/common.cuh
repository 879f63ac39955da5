// common.cuh - device helpers shared by every phase of the megakernel:
// conversions, the status word, bounded waits and the grid-wide barrier.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include "plan.h"
#include "../../include/moe_train.h"

#define MT_THREADS 256
#define MT_WARPS 8

// error sites recorded with the status word
enum ErrSite {
  SITE_BARRIER = 1,
  SITE_TOKEN_RANGE = 2,
  SITE_ROUTE_RANGE = 3,
  SITE_TC_FULL = 10,
  SITE_TC_EMPTY = 11,
  SITE_TC_ACC_FULL = 12,
  SITE_TC_ACC_EMPTY = 13,
  SITE_TC_DRAIN = 14,
  SITE_TC_ALIGN = 15,
  SITE_DEP = 16,
  SITE_TC_EPI = 17,
  SITE_TC_QUEUE = 18,
  SITE_TEST_STALL = 20
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <class T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_volatile(const int* p) { return *(const volatile int*)p; }

// First error wins; later ones keep the first site.
__device__ __forceinline__ void set_error(ArenaHdr* h, int status, int site) {
  if (atomicCAS(&h->status, 0, status) == 0) h->error_site = site;
  __threadfence();
}

// Packed pairs of fp32 (the two-wide fp32 instructions of this architecture;
// each lane rounds as the scalar instruction does).
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ uint64_t u2(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Bounded wait until a dependency counter reaches `target` (acquire, so the
// producers' stores before their release are visible afterwards).  Returns
// false at once when the status word holds an error, or after recording a
// timeout; callers then carry on without the data (the results are void and
// every CTA leaves at the next grid barrier).
static __device__ __noinline__ bool dep_wait(ArenaHdr* h, const unsigned* c, unsigned target, long long timeout_ns) {
  if (ld_acquire_gpu(c) >= target) return true;
  const unsigned long long t0 = globaltimer();
  unsigned ns = 32;
  while (ld_acquire_gpu(c) < target) {
    if (ld_volatile(&h->status) != 0) return false;
    if ((long long)(globaltimer() - t0) > timeout_ns) {
      set_error(h, MT_ERR_DEVICE_TIMEOUT, SITE_DEP);
      return false;
    }
    __nanosleep(ns);
    if (ns < 256) ns <<= 1;
  }
  return true;
}
// Publish a producer part: every store the calling thread has observed
// (after a CTA or named barrier over the writers) is released with the add.
__device__ __forceinline__ void dep_signal(unsigned* c) {
  __threadfence();
  atomicAdd(c, 1u);
}
// Next item of a dynamically scheduled job: thread 0 draws a ticket and the
// CTA reads it after a CTA barrier.
__device__ __forceinline__ int draw_ticket(unsigned* ticket) {
  __shared__ int s_ticket;
  __syncthreads();
  if (threadIdx.x == 0) s_ticket = (int)atomicAdd(ticket, 1u);
  __syncthreads();
  return s_ticket;
}

// Work distribution inside a phase: item i of the current job runs on CTA
// (i + base) % G.  Rotating `base` from job to job spreads small jobs over
// different SMs.
struct Sched {
  int bid, G, base;
  __device__ __forceinline__ int first() const {
    int f = bid - base;
    f %= G;
    return f < 0 ? f + G : f;
  }
  __device__ __forceinline__ void next(int n) { base = (base + n) % G; }
};

// Grid-wide barrier for a cooperative launch (all CTAs co-resident).  The
// count returns to zero after every barrier and the generation only grows,
// so no host-side fill is needed between launches.  Returns false when the
// status word holds an error (then every CTA leaves the kernel).
static __device__ __noinline__ bool grid_barrier(ArenaHdr* h, unsigned G, long long timeout_ns,
                                          long long* trace, bool stall) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    if (trace) trace[0] = (long long)globaltimer();
    if (stall) {
      ok = 0;                       // test hook: never arrive; the others time out
    } else {
      unsigned gen = ld_acquire_gpu(&h->bar_gen);
      __threadfence();
      unsigned arrived = atomicAdd(&h->bar_count, 1u);
      if (arrived == G - 1) {
        h->bar_count = 0;
        __threadfence();
        st_release_gpu(&h->bar_gen, gen + 1);
      } else {
        unsigned long long t0 = globaltimer();
        unsigned ns = 32;
        while (ld_acquire_gpu(&h->bar_gen) == gen) {
          if (ld_volatile(&h->status) != 0) { ok = 0; break; }
          if ((long long)(globaltimer() - t0) > timeout_ns) {
            set_error(h, MT_ERR_DEVICE_TIMEOUT, SITE_BARRIER);
            ok = 0;
            break;
          }
          __nanosleep(ns);
          if (ns < 256) ns <<= 1;
        }
      }
      if (ld_volatile(&h->status) != 0) ok = 0;
    }
    if (trace) trace[1] = (long long)globaltimer();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}
