// rowpipe.cuh - asynchronous row staging for the per-token row jobs.
//
// A row job works on one token per warp at a time and needs a few whole
// rows of d values per token (the residual stream, expert outputs, their
// gradients).  Loading them with ordinary loads leaves a chain of dependent
// round trips per token (index, row, reduction, next row), so a warp has
// little in flight and the job runs far below the HBM bandwidth.  Here each
// warp owns a ring of NS stages in shared memory: lane 0 copies the rows of
// token j + NS with cp.async.bulk (completion counted in bytes on the
// stage's mbarrier) while the warp computes on token j from shared memory.
//
// Stage layout: a 128-byte header (scalars lane 0 read while issuing: row
// indices, router weights) followed by the rows, each 16-byte aligned.
// Every wait is bounded; on expiry the status word records the site.
#pragma once
#include "common.cuh"
#include "gemm_tc.cuh"
#include "rows.cuh"

#define RP_MAX_STAGES 8
#define RP_WIN_OFF 1024          // rings start here (the low kilobyte is left to the product jobs)
#define RP_HDR 128               // stage header bytes
#define RP_TBL 32                // tokens of a warp whose indices are read up front
#define SITE_ROWPIPE 40           // + job: 0 router, 1 route, 2 combine, 3/4 combine bwd 1/2, 5 attention-norm bwd

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// bulk store shared -> global in the thread's bulk async-group
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}
// every committed group has finished reading its shared-memory source
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// all but the most recent committed group have finished reading their source
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// every committed group has completed its writes
__device__ __forceinline__ void bulk_wait_all0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ float4 lds4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ int lds_i32(uint32_t a) {
  int v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts_i32(uint32_t a, int v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void sts_f32(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
__device__ __forceinline__ void sts4(uint32_t a, float4 v) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}
__device__ __forceinline__ void sts_u2(uint32_t a, uint32_t x, uint32_t y) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(a), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}

// A d-wide fp32 row staged in shared memory at byte address `a`.
template <int NC>
__device__ __forceinline__ void row_lds(Row<NC>& r, uint32_t a, int n4) {
  const int l = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const int c = l + 32 * i;
    r.v[i] = (c < n4) ? lds4(a + 16u * (uint32_t)c) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// The ring mbarriers live in a static shared array of their own.  The
// tensor-core jobs place their mbarriers at the bottom of the dynamic window
// and re-initialise them job after job; a ring barrier initialised over one
// of those locations was seen never to complete its phase although its bytes
// had landed, so the rings keep their barriers apart, initialise them at the
// start of a job and invalidate them at its end.
static __shared__ __align__(8) unsigned long long rp_bars[MT_WARPS * RP_MAX_STAGES];

// r += the staged row at shared address `a` (one float4 at a time)
template <int NC>
__device__ __forceinline__ void row_add_lds(Row<NC>& r, uint32_t a, int n4) {
  const int l = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const int c = l + 32 * i;
    if (c < n4) {
      const float4 v = lds4(a + 16u * (uint32_t)c);
      r.v[i] = join2(add2(lo2(r.v[i]), lo2(v)), add2(hi2(r.v[i]), hi2(v)));
    }
  }
}

struct RowPipe {
  uint32_t ring;     // shared address of this warp's stage 0
  uint32_t bar;      // shared address of this warp's first mbarrier
  uint32_t tbl;      // shared address of this warp's index table (after its stages)
  uint32_t sbytes;   // bytes per stage
  int ns;            // stages; 0 when two stages do not fit (callers then take their register path)
  __device__ __forceinline__ uint32_t stage(int j) const { return ring + (uint32_t)(j % ns) * sbytes; }
  __device__ __forceinline__ uint32_t sbar(int j) const { return bar + 8u * (uint32_t)(j % ns); }
  __device__ __forceinline__ uint32_t parity(int j) const { return (uint32_t)(j / ns) & 1u; }
};

// Carve this warp's ring out of the shared-memory window [win_off, win_end)
// for stages of `rows_bytes` bytes of rows, plus `tbl_bytes` of index table
// after the stages.  Grid-uniform: every warp gets the same number of stages.
__device__ __forceinline__ RowPipe rp_make(char* smem, uint32_t win_off, uint32_t win_end, uint32_t rows_bytes,
                                          uint32_t tbl_bytes = 0) {
  RowPipe p;
  const int warp = threadIdx.x >> 5;
  const uint32_t per = win_end > win_off ? ((win_end - win_off) / MT_WARPS) & ~127u : 0u;
  p.sbytes = (RP_HDR + rows_bytes + 127u) & ~127u;
  const uint32_t tb = (tbl_bytes + 127u) & ~127u;
  int ns = per > tb ? (int)((per - tb) / p.sbytes) : 0;
  if (ns > RP_MAX_STAGES) ns = RP_MAX_STAGES;
  p.ns = ns >= 2 ? ns : 0;
  p.ring = smem_u32(smem) + win_off + (uint32_t)warp * per;
  p.tbl = p.ring + (uint32_t)p.ns * p.sbytes;
  p.bar = smem_u32(&rp_bars[warp * RP_MAX_STAGES]);
  return p;
}

// Start of a pipelined job (all threads): the previous job's use of shared
// memory is over, barriers are initialised, and the rows stored by earlier
// phases (generic proxy) are ordered before the bulk copies (async proxy).
__device__ __forceinline__ void rp_begin(const RowPipe& p) {
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    for (int s = 0; s < p.ns; ++s) mbar_init(p.bar + 8u * s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async;" ::: "memory");
  }
  __syncwarp();
}
// End of a pipelined job (all threads): every issued stage has been waited
// for; the barriers are invalidated before the memory is used for anything else.
__device__ __forceinline__ void rp_end(const RowPipe& p, bool drained) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0 && drained)
    for (int s = 0; s < p.ns; ++s) asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(p.bar + 8u * s) : "memory");
  __syncthreads();
}

// Drive one warp's token list through the ring.
//   n            : tokens of this warp (uniform within the warp)
//   issue(j, st, bar) : lane 0 only - write the stage header at `st`, then
//                  mbar_expect_tx + bulk copies of token j's rows to
//                  st + RP_HDR ...; or a plain arrive when j has no rows
//   compute(j, st): all lanes, after the stage landed
//   after(j)     : all lanes, after compute (also when a wait failed, so
//                  that CTA-wide barriers inside it stay paired)
// Returns false when a wait timed out (the status word holds the error).
template <class Issue, class Compute, class After>
__device__ __forceinline__ bool rp_run(const RowPipe& p, int n, ArenaHdr* hdr, long long tmo, int site, Issue&& issue,
                                       Compute&& compute, After&& after) {
  const int lane = threadIdx.x & 31;
  const int pro = n < p.ns ? n : p.ns;
  if (lane == 0)
    for (int j = 0; j < pro; ++j) issue(j, p.stage(j), p.sbar(j));
  __syncwarp();
  bool ok = true;
  for (int j = 0; j < n; ++j) {
    if (ok && !mbar_wait(p.sbar(j), p.parity(j), tmo)) {
      if (lane == 0) set_error(hdr, MT_ERR_DEVICE_TIMEOUT, site);
      ok = false;
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok) compute(j, p.stage(j));
    after(j);
    __syncwarp();
    if (ok && j + p.ns < n && lane == 0) {
      // the warp's reads of this stage come before the next copy into it
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(j + p.ns, p.stage(j), p.sbar(j));
    }
    __syncwarp();
  }
  return ok;
}
