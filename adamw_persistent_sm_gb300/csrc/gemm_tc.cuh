// gemm_tc.cuh - tensor-core matrix products (tcgen05 + TMEM + TMA) inside
// the persistent kernel, for the bf16-product policy.
//
// Tile 128 x 256 x 64.  Per GEMM job:
//   warp 0 (one lane)  - TMA producer: two 64x64 boxes of A and four of B per
//                        stage into a 4-stage ring of 128B-swizzled tiles;
//   warp 1 (one lane)  - MMA issuer: 4 x tcgen05.mma (128 x 256 x 16) per
//                        stage into one of two TMEM accumulators (128 lanes x
//                        256 fp32 columns each), tcgen05.commit frees the stage;
//   warps 4..7         - epilogue: tcgen05.ld of the accumulator rows (warp
//                        w reads TMEM lanes 32*(w-4)..), fused epilogue, store.
// A and B may each be K-major or MN-major in memory (forward, dgrad and
// wgrad products read the same buffers without transposed copies); the
// shared-memory descriptors describe either layout.  Every mbarrier wait is
// bounded: on expiry the status word records the site and the job drains.
#pragma once
#include "common.cuh"
#include "gemm.cuh"

#define TC_BM 128
#define TC_BN 256
#define TC_BK 64
#define TC_STAGES 4
#define TC_BOX_BYTES (64 * 64 * 2)
#define TC_STAGE_BYTES ((TC_BM + TC_BN) / 64 * TC_BOX_BYTES)
#define TC_RING_OFF 1024
#define TC_STAGE_OFF (TC_RING_OFF + TC_STAGES * TC_STAGE_BYTES)   // epilogue windows
#define TC_EPI_WARP_BYTES 8192                                    // one window per epilogue warp
#define TC_EPI_SLOT 2048                                          // one 32x32 bf16 box
#define TC_EPI_MBAR 512                                           // aux-load mbarriers (2 per warp)
#define TC_Q_SLOTS 4                                              // drawn-tile queue: producer -> MMA, epilogue
#define TC_Q_IDX 160                                              // tile indices (int per slot)
#define TC_Q_FULL 576                                             // mbarriers: index written
#define TC_Q_EMPTY 608                                            // mbarriers: index read by MMA + 4 epilogue warps
#define TC_XPOSE_BYTES (32 * 33 * 4)                              // 32x32 fp32 transpose tile
#define MT_TC_SMEM (TC_STAGE_OFF + 4 * TC_EPI_WARP_BYTES)
static_assert(TC_XPOSE_BYTES <= TC_EPI_WARP_BYTES, "transpose tile exceeds the epilogue window");
static_assert(MT_TC_SMEM <= 232448, "tensor-core shared memory exceeds 227 KB");
#define TC_TMEM_COLS 512
#define MT_TC_AVAILABLE 1

struct TcState {
  uint32_t tmem_base;
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase of parity `parity` to complete; false after timeout_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if ((long long)(globaltimer() - t0) > timeout_ns) return false;
  }
  return true;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"((unsigned long long)map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Bulk tensor store of a shared-memory box (one bulk group per commit).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   (unsigned long long)map),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
// L2 policy for data streamed once (evicted before other lines)
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, uint32_t src, int x, int y, uint64_t pol) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
                   (unsigned long long)map),
               "r"(src), "r"(x), "r"(y), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], "
      "[%4], %5;" ::"r"(dst),
      "l"((unsigned long long)map), "r"(x), "r"(y), "r"(bar), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// at most N of this thread's latest bulk groups still read shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// every bulk group of this thread has written global memory; later generic
// accesses (after a release by any thread of the CTA) observe the writes
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// shared-memory writes of this thread become visible to bulk copies
__device__ __forceinline__ void fence_smem_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// The same two instructions for a whole converged warp: every lane walks
// the issue loop (so the operands are warp-uniform values) and one elected
// lane - always the same one while all 32 are active - issues.  The commit
// tracks the products of the lane that issued them, so both go through the
// same election.
__device__ __forceinline__ void mma_bf16_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\t"
      "elect.sync l|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit_warp(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 l;\n\t"
      "elect.sync l|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive fp32 columns of this thread's TMEM lane (one round trip).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, "
      "%36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, "
      "%57, %58, %59, %60, %61, %62, %63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor, 128-byte swizzle.
//   K-major : rows of 128 B, 8-row groups 1024 B apart (SBO); LBO unused.
//   MN-major: 64-element MN chunks LBO apart, 8-row K groups 1024 B apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo & 0x3FFFFu) >> 4) << 16) |
         ((uint64_t)((sbo & 0x3FFFFu) >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// A descriptor advanced by `bytes` (a multiple of 16): the start-address
// field holds addr >> 4 in its low bits and shared addresses stay below
// 256 KB, so the advance is a plain add (no per-step rebuild).
__device__ __forceinline__ uint64_t sdesc_add(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }
// Instruction descriptor of kind::f16: bf16 A and B, fp32 accumulator.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// setup / teardown (once per kernel)
// ---------------------------------------------------------------------------
template <class OP>
__device__ __forceinline__ void tc_setup(const KArgs& a, char* smem, TcState& tc) {
  tc.tmem_base = 0;
  if constexpr (sizeof(OP) == 2) {
    if (!a.use_tc) return;
    uint32_t slot = smem_u32(smem + 256);
    if ((threadIdx.x >> 5) == 0) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                   "r"(TC_TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    tc.tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + 256);
    __syncthreads();
  }
}

template <class OP>
__device__ __forceinline__ void tc_teardown(const KArgs& a, char* smem, TcState& tc) {
  if constexpr (sizeof(OP) == 2) {
    if (!a.use_tc) return;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if ((threadIdx.x >> 5) == 0)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tc.tmem_base), "r"(TC_TMEM_COLS)
                   : "memory");
  }
}

// ---------------------------------------------------------------------------
// tiles
// ---------------------------------------------------------------------------
struct TcTile {
  int m0, n0, seg, kbeg, nk;
};

// Loop-invariant shape of a product, copied into registers by each role.
struct TcShape {
  int rag, M, K, nseg, nt, ksplit;
  const int* offs;
};
__device__ __forceinline__ TcShape tc_shape(const GemmDesc& g) {
  TcShape sh;
  sh.rag = g.rag; sh.M = g.M; sh.K = g.K; sh.nseg = g.nseg; sh.nt = g.N / TC_BN; sh.offs = g.offs;
  sh.ksplit = (g.rag == RAG_NONE && g.ksplit > 1) ? g.ksplit : 1;
  return sh;
}

__device__ __forceinline__ TcTile tc_tile(const TcShape& g, int t) {
  TcTile ti;
  const int nt = g.nt;
  if (g.rag == RAG_K) {
    const int mt = g.M / TC_BM;
    ti.seg = t / (mt * nt);
    const int rem = t % (mt * nt);
    ti.m0 = (rem / nt) * TC_BM;
    ti.n0 = (rem % nt) * TC_BN;
    ti.kbeg = g.offs[ti.seg];
    ti.nk = (g.offs[ti.seg + 1] - ti.kbeg) / TC_BK;
  } else if (g.ksplit > 1) {
    // slice s of the reduction; the output of slice s is redirected by seg
    const int mt = g.M / TC_BM;
    ti.seg = t / (mt * nt);
    const int rem = t % (mt * nt);
    ti.m0 = (rem / nt) * TC_BM;
    ti.n0 = (rem % nt) * TC_BN;
    const int kc = g.K / g.ksplit;
    ti.kbeg = ti.seg * kc;
    ti.nk = kc / TC_BK;
  } else {
    ti.m0 = (t / nt) * TC_BM;
    ti.n0 = (t % nt) * TC_BN;
    ti.seg = (g.rag == RAG_M) ? seg_of_row(g.offs, g.nseg, ti.m0) : 0;
    ti.kbeg = 0;
    ti.nk = g.K / TC_BK;
  }
  return ti;
}

// Loop-invariant TMA state of one operand.
struct TmaOp {
  const CUtensorMap* m0;
  const CUtensorMap* m1;
  int mn, two, split, y0, yseg, rpb;
};
__device__ __forceinline__ TmaOp tma_op(const KArgs& a, const GOperand& o) {
  TmaOp t;
  t.m0 = &a.maps[o.map0];
  t.m1 = (o.map1 >= 0) ? &a.maps[o.map1] : t.m0;
  t.mn = o.mn; t.two = o.two; t.split = o.split; t.y0 = o.y0; t.yseg = o.yseg;
  t.rpb = (!o.mn && o.two != 1) ? o.rows_per_box : 64;
  return t;
}

// Load the A (rows m0..m0+127) or B (rows n0..n0+255) operand slice of one
// 64-wide K block as NBOX 64 x 64 boxes.
template <int NBOX>
__device__ __forceinline__ void tc_load_operand(const TmaOp& o, int r0, int k0, int yseg_off, uint32_t dst,
                                                uint32_t bar) {
  if (o.rpb > 64) {
    // K-major, one source: taller boxes of the same 128-byte-swizzled rows
    // (a 128-row box lands exactly where two 64-row boxes would)
    for (int rr = 0; rr < NBOX * 64; rr += o.rpb)
      tma_load_2d(dst + (uint32_t)rr * 128u, o.m0, k0, o.y0 + yseg_off + r0 + rr, bar);
    return;
  }
#pragma unroll
  for (int i = 0; i < NBOX; ++i) {
    const CUtensorMap* map = o.m0;
    int x, y;
    if (!o.mn) {
      // element (r, k) at row y0 + r, column k
      int rr = r0 + 64 * i;
      if (o.two == 1) {
        // columns interleaved by 64 between two sources: box i is block
        // r0/64 + i, even blocks from m0, odd from m1, row (block/2)*64
        map = (i & 1) ? o.m1 : o.m0;
        rr = (r0 >> 1) + (i >> 1) * 64;
      }
      x = k0;
      y = o.y0 + yseg_off + rr;
    } else {
      // element (r, k) at row y0 + k, column r
      int kk = k0;
      if (o.two == 2 && k0 >= o.split) {
        map = o.m1;
        kk = k0 - o.split;
      }
      x = r0 + 64 * i;
      y = o.y0 + yseg_off + kk;
    }
    tma_load_2d(dst + i * TC_BOX_BYTES, map, x, y, bar);
  }
}

// ---------------------------------------------------------------------------
// epilogue helpers: one thread owns one output row of the tile
// ---------------------------------------------------------------------------
template <int N>
__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const float* v) {
#pragma unroll
  for (int i = 0; i < N; i += 8) {
    uint4 u;
    __nv_bfloat162 h0 = __floats2bfloat162_rn(v[i], v[i + 1]);
    __nv_bfloat162 h1 = __floats2bfloat162_rn(v[i + 2], v[i + 3]);
    __nv_bfloat162 h2 = __floats2bfloat162_rn(v[i + 4], v[i + 5]);
    __nv_bfloat162 h3 = __floats2bfloat162_rn(v[i + 6], v[i + 7]);
    u.x = *reinterpret_cast<uint32_t*>(&h0);
    u.y = *reinterpret_cast<uint32_t*>(&h1);
    u.z = *reinterpret_cast<uint32_t*>(&h2);
    u.w = *reinterpret_cast<uint32_t*>(&h3);
    *reinterpret_cast<uint4*>(dst + i) = u;
  }
}
template <int N>
__device__ __forceinline__ void store_row_f32(float* dst, const float* v) {
#pragma unroll
  for (int i = 0; i < N; i += 4) *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
}
template <int N>
__device__ __forceinline__ void load_row_bf16(const __nv_bfloat16* src, float* v) {
#pragma unroll
  for (int i = 0; i < N; i += 8) {
    uint4 u = *reinterpret_cast<const uint4*>(src + i);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 f = __bfloat1622float2(h[j]);
      v[i + 2 * j] = f.x;
      v[i + 2 * j + 1] = f.y;
    }
  }
}

// Coalesced fp32 epilogue stores.  A warp owns 32 rows of the tile (one per
// lane); a 32-column chunk is staged through a padded 32x33 shared tile so
// that each store instruction writes a whole 128-byte row segment: lane l
// then owns column l.  (bf16 outputs keep one 16-byte store per thread and
// row: for them the extra shared-memory traffic costs more than it saves.)
__device__ __forceinline__ void xpose_put(float* st, const float* v) {
  const int l = threadIdx.x & 31;
  __syncwarp();
#pragma unroll
  for (int c = 0; c < 32; ++c) st[l * 33 + c] = v[c];
  __syncwarp();
}
// rows row0..row0+31, columns col..col+31 of an fp32 matrix
__device__ __forceinline__ void xpose_store_f32(float* st, const float* v, float* out, long long ld, long long row0,
                                                int col) {
  const int l = threadIdx.x & 31;
  xpose_put(st, v);
  float* p = out + row0 * ld + col + l;
#pragma unroll 8
  for (int r = 0; r < 32; ++r) p[(long long)r * ld] = st[r * 33 + l];
}
// same, out = aux + v (aux fp32, same shape and stride)
__device__ __forceinline__ void xpose_store_f32_add(float* st, const float* v, float* out, const float* aux,
                                                    long long ld, long long ld_aux, long long row0, int col) {
  const int l = threadIdx.x & 31;
  xpose_put(st, v);
  float* p = out + row0 * ld + col + l;
  const float* q = aux + row0 * ld_aux + col + l;
  float a[32];                      // every load is issued before the first store
#pragma unroll
  for (int r = 0; r < 32; ++r) a[r] = q[(long long)r * ld_aux];
#pragma unroll
  for (int r = 0; r < 32; ++r) p[(long long)r * ld] = a[r] + st[r * 33 + l];
}
// ---------------------------------------------------------------------------
// Bulk-copy epilogue.  Each epilogue warp owns an 8 KB shared-memory window
// of four 2 KB slots.  A 32-row x 32-column output box (one row per lane)
// is staged there with the swizzle of its tensor map - the 16-byte chunk j
// of row r sits at chunk j ^ ((r >> 1) & 3) of the row (bf16, 64-byte rows)
// or j ^ (r & 7) (fp32, 128-byte rows), so the eight lanes of every
// 128-byte shared-memory wavefront hit distinct banks - and lane 0 writes it
// to global memory with one bulk tensor store.  The warp goes on with the
// next box while the copy engine drains the slot.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t sw64(int r, int j) { return r * 64 + ((j ^ ((r >> 1) & 3)) << 4); }
__device__ __forceinline__ uint32_t sw128(int r, int j) { return r * 128 + ((j ^ (r & 7)) << 4); }
__device__ __forceinline__ uint32_t bf2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ void box_put_bf16(uint32_t box, int r, const float* v) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    sts128(box + sw64(r, j), bf2(v[8 * j], v[8 * j + 1]), bf2(v[8 * j + 2], v[8 * j + 3]),
           bf2(v[8 * j + 4], v[8 * j + 5]), bf2(v[8 * j + 6], v[8 * j + 7]));
}
__device__ __forceinline__ void box_get_bf16(uint32_t box, int r, float* v) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 u = lds128(box + sw64(r, j));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[8 * j + 2 * i] = __uint_as_float(w[i] << 16);
      v[8 * j + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}
__device__ __forceinline__ void box_put_f32(uint32_t box, int r, const float* v) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    sts128(box + sw128(r, j), __float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
           __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
}
__device__ __forceinline__ void box_get_f32(uint32_t box, int r, float* v) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 u = lds128(box + sw128(r, j));
    v[4 * j] = __uint_as_float(u.x); v[4 * j + 1] = __uint_as_float(u.y);
    v[4 * j + 2] = __uint_as_float(u.z); v[4 * j + 3] = __uint_as_float(u.w);
  }
}

// Epilogue arithmetic for bf16 outputs: 2^x by the special-function unit and
// the logistic function with an approximate reciprocal (relative error a few
// 1e-7, far below the bf16 rounding of the stored values).
__device__ __forceinline__ float epi_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
#define EPI_LOG2E 1.4426950408889634f
__device__ __forceinline__ float epi_sigmoid(float x) { return __fdividef(1.0f, 1.0f + epi_ex2(-x * EPI_LOG2E)); }

// 32 columns at each of two TMEM addresses of this thread's lane, one wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, float* va, float* vb) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(ta));
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(tb));
  // the wait takes the loaded registers as operands, so no use of them is
  // scheduled before it
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
  asm volatile(""
               : "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]),
                 "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]),
                 "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]),
                 "+r"(r[53]), "+r"(r[54]), "+r"(r[55]), "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]),
                 "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63])
               :
               : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    va[i] = __uint_as_float(r[i]);
    vb[i] = __uint_as_float(r[32 + i]);
  }
}

// Per-warp state of the bulk-copy epilogue (warp-uniform).
struct EpiSt {
  uint32_t win;       // the warp's 8 KB window
  uint32_t mbar;      // two aux-load mbarriers, 8 bytes apart
  uint32_t nbox;      // boxes stored by the store-only epilogues
  uint32_t use[2];    // completed phases of the two mbarriers
  bool dead;          // an aux load timed out: skip the remaining work
};

// Store-only epilogues: stage box k in slot k & 3 (bf16) or half k & 1
// (fp32) once the store four (two) boxes back has read it.
__device__ __forceinline__ void epi_store_bf16(EpiSt& e, const CUtensorMap* map, int x, int y, const float* v) {
  const int lane = threadIdx.x & 31;
  const uint32_t box = e.win + (e.nbox & 3) * TC_EPI_SLOT;
  if (lane == 0) bulk_wait_read<3>();
  __syncwarp();
  box_put_bf16(box, lane, v);
  fence_smem_async();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, box, x, y);
    bulk_commit();
  }
  ++e.nbox;
}
// 64 bf16 columns per row: a 32 x 64 box (128-byte rows, chunk j of row r at
// j ^ (r & 7)) in half k & 1 of the window
__device__ __forceinline__ void epi_store_bf16_64(EpiSt& e, const CUtensorMap* map, int x, int y, const float* v) {
  const int lane = threadIdx.x & 31;
  const uint32_t box = e.win + (e.nbox & 1) * 2 * TC_EPI_SLOT;
  if (lane == 0) bulk_wait_read<1>();
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 8; ++j)
    sts128(box + sw128(lane, j), bf2(v[8 * j], v[8 * j + 1]), bf2(v[8 * j + 2], v[8 * j + 3]),
           bf2(v[8 * j + 4], v[8 * j + 5]), bf2(v[8 * j + 6], v[8 * j + 7]));
  fence_smem_async();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, box, x, y);
    bulk_commit();
  }
  ++e.nbox;
}
__device__ __forceinline__ void epi_store_f32(EpiSt& e, const CUtensorMap* map, int x, int y, const float* v) {
  const int lane = threadIdx.x & 31;
  const uint32_t box = e.win + (e.nbox & 1) * 2 * TC_EPI_SLOT;
  if (lane == 0) bulk_wait_read<1>();
  __syncwarp();
  box_put_f32(box, lane, v);
  fence_smem_async();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, box, x, y);
    bulk_commit();
  }
  ++e.nbox;
}

// Epilogues with an input box per output box: chunk c of the tile uses half
// c & 1 of the window.  Lane 0 loads the chunk's input boxes by TMA (two
// chunks ahead), every lane replaces its row of them by the output rows, and
// lane 0 stores them from the same slots.  issue(c, half, bar) and
// store(c, half) run on lane 0; work(c, half) on every lane.
template <class Issue, class Work, class Store>
__device__ __forceinline__ void epi_aux_tile(EpiSt& e, int nch, long long tmo, ArenaHdr* hdr, Issue issue,
                                             Work work, Store store) {
  const int lane = threadIdx.x & 31;
  if (e.dead) return;
  if (lane == 0) {
    bulk_wait_read<0>();
    issue(0, e.win, e.mbar);
    if (nch > 1) issue(1, e.win + 2 * TC_EPI_SLOT, e.mbar + 8);
  }
  __syncwarp();
  for (int c = 0; c < nch; ++c) {
    const int h = c & 1;
    const uint32_t half = e.win + h * 2 * TC_EPI_SLOT, bar = e.mbar + 8 * h;
    const uint32_t par = e.use[h] & 1;
    ++e.use[h];
    const bool late = !mbar_wait(bar, par, tmo);
    if (__any_sync(0xffffffffu, late)) {
      if (lane == 0) set_error(hdr, MT_ERR_DEVICE_TIMEOUT, SITE_TC_EPI);
      e.dead = true;
      return;
    }
    work(c, half);
    fence_smem_async();
    __syncwarp();
    if (lane == 0) {
      store(c, half);
      bulk_commit();
      if (c + 2 < nch) {
        bulk_wait_read<0>();
        issue(c + 2, half, bar);
      }
    }
    __syncwarp();
  }
}

// Epilogue parameters copied into registers once per job: stores through
// the output pointers can then not force re-reads of the descriptor.
struct EpiRegs {
  int epi, S, hq, F, accumulate, osplit, ceparts, N;
  long long ldo, ldo2, ldaux, oseg;
  void* out;
  void* out1;
  void* out2;
  const void* aux;
  const float* rope;
  const int* tok;
  float* cepart;
  float* cetgt;
  const CUtensorMap* om;     // bulk-store map of out (null: plain stores)
  const CUtensorMap* om2;    // of out2
  const CUtensorMap* am;     // bulk-load map of aux
  int oy0, oy02, ay0;
};
__device__ __forceinline__ EpiRegs epi_regs(const KArgs& a, const GemmDesc& g) {
  EpiRegs e;
  e.epi = g.epi; e.S = g.S; e.hq = g.hq; e.F = g.F; e.accumulate = g.accumulate; e.osplit = g.osplit;
  e.ceparts = g.ceparts; e.N = g.N; e.ldo = g.ldo; e.ldo2 = g.ldo2; e.ldaux = g.ldaux; e.oseg = g.oseg;
  e.out = g.out; e.out1 = g.out1; e.out2 = g.out2; e.aux = g.aux; e.rope = g.rope; e.tok = g.tok;
  e.cepart = g.cepart; e.cetgt = g.cetgt;
  e.om = g.omap >= 0 ? &a.maps[g.omap] : nullptr;
  e.om2 = g.omap2 >= 0 ? &a.maps[g.omap2] : nullptr;
  e.am = g.amap >= 0 ? &a.maps[g.amap] : nullptr;
  e.oy0 = g.oy0; e.oy02 = g.oy02; e.ay0 = g.ay0;
  // every tensor-map path of an epilogue needs all of its maps
  if ((g.epi == EPI_SWIGLU && !e.om2) || ((g.epi == EPI_SWIGLU_BWD || g.epi == EPI_RESID ||
                                            g.epi == EPI_STORE_OP_D) && !e.am))
    e.om = nullptr;
  return e;
}

// The tensor-map paths of the epilogue (g.om set).  row0: first row of the
// warp's 32 rows in the product; m = row0 + lane.
__device__ __forceinline__ void tc_epilogue_tma(const EpiRegs& g, const TcTile& ti, uint32_t trow, int m,
                                                int row0, EpiSt& es, long long tmo, ArenaHdr* hdr) {
  constexpr int NCH = TC_BN / 32;
  const int lane = threadIdx.x & 31;
  const int y = g.oy0 + row0;
  switch (g.epi) {
    case EPI_ROPE: {
      // hd == 64: columns [64h, 64h+32) pair with [64h+32, 64h+64)
      const float4* tab4 = reinterpret_cast<const float4*>(g.rope + (long long)(m % g.S) * 64);
      for (int h2 = 0; h2 < TC_BN / 64; ++h2) {
        float x[64];
        tmem_ld64(trow + h2 * 64, x);
        const int n = ti.n0 + h2 * 64;
        if (n < 2 * g.hq) {
#pragma unroll
          for (int i2 = 0; i2 < 16; ++i2) {
            const float4 cs = tab4[i2];     // (cos, sin) of pairs 2*i2, 2*i2+1
            const int i = 2 * i2;
            float x1 = x[i], x2 = x[i + 32];
            x[i] = x1 * cs.x - x2 * cs.y;
            x[i + 32] = x2 * cs.x + x1 * cs.y;
            x1 = x[i + 1];
            x2 = x[i + 33];
            x[i + 1] = x1 * cs.z - x2 * cs.w;
            x[i + 33] = x2 * cs.z + x1 * cs.w;
          }
        }
        epi_store_bf16_64(es, g.om, n, y, x);
      }
      break;
    }
    case EPI_SWIGLU: {
      // each 128-column half = [64 gate | 64 up] of expert rows f0..f0+63
      const int y2 = g.oy02 + row0;
      for (int half = 0; half < TC_BN / 128; ++half) {
        const int f0 = ((ti.n0 >> 7) + half) * 64;
        for (int c = 0; c < 2; ++c) {
          float gg[32], uu[32];
          tmem_ld32x2(trow + half * 128 + c * 32, trow + half * 128 + 64 + c * 32, gg, uu);
          const int f = f0 + c * 32;
          epi_store_bf16(es, g.om, f, y, gg);
          epi_store_bf16(es, g.om, g.F + f, y, uu);
          const uint64_t nl2 = f2(-EPI_LOG2E, -EPI_LOG2E), one2 = f2(1.f, 1.f);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            // silu(g) u = g u / (1 + 2^(-g log2 e)), two columns per step
            const uint64_t g2 = f2(gg[i], gg[i + 1]);
            float e0, e1;
            unf2(mul2(g2, nl2), e0, e1);
            float d0, d1;
            unf2(add2(one2, f2(epi_ex2(e0), epi_ex2(e1))), d0, d1);
            unf2(mul2(mul2(g2, f2(uu[i], uu[i + 1])), f2(__fdividef(1.0f, d0), __fdividef(1.0f, d1))), gg[i], gg[i + 1]);
          }
          epi_store_bf16(es, g.om2, f, y2, gg);
        }
      }
      break;
    }
    case EPI_SWIGLU_BWD: {
      // aux = [g | u] boxes at columns n and F + n; out = [dg | du] in their slots
      const int ya = g.ay0 + row0;
      const CUtensorMap* am = g.am;
      const CUtensorMap* om = g.om;
      const int F = g.F, n0 = ti.n0;
      epi_aux_tile(
          es, NCH, tmo, hdr,
          [&](int c, uint32_t half, uint32_t bar) {
            mbar_expect_tx(bar, 2 * TC_EPI_SLOT);
            tma_load_2d(half, am, n0 + 32 * c, ya, bar);
            tma_load_2d(half + TC_EPI_SLOT, am, F + n0 + 32 * c, ya, bar);
          },
          [&](int c, uint32_t half) {
            float da[32], gg[32], uu[32];
            tmem_ld32(trow + c * 32, da);
            box_get_bf16(half, lane, gg);
            box_get_bf16(half + TC_EPI_SLOT, lane, uu);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float sg = epi_sigmoid(gg[i]);
              const float du = da[i] * gg[i] * sg;
              gg[i] = da[i] * uu[i] * sg * (1.0f + gg[i] * (1.0f - sg));
              uu[i] = du;
            }
            box_put_bf16(half, lane, gg);
            box_put_bf16(half + TC_EPI_SLOT, lane, uu);
          },
          [&](int c, uint32_t half) {
            tma_store_2d(om, half, n0 + 32 * c, y);
            tma_store_2d(om, half + TC_EPI_SLOT, F + n0 + 32 * c, y);
          });
      break;
    }
    case EPI_STORE_OP_D: {
      // 64-column heads: out = dO (bf16); D = rowsum(bf16(dO) * O), O from aux
      const int ya = g.ay0 + row0;
      const CUtensorMap* am = g.am;
      const CUtensorMap* om = g.om;
      const int n0 = ti.n0;
      float* dsum = (float*)g.out2 + (long long)(m / g.S) * g.ldo2 * g.S + (m % g.S);
      epi_aux_tile(
          es, TC_BN / 64, tmo, hdr,
          [&](int c, uint32_t half, uint32_t bar) {
            mbar_expect_tx(bar, 2 * TC_EPI_SLOT);
            tma_load_2d(half, am, n0 + 64 * c, ya, bar);
            tma_load_2d(half + TC_EPI_SLOT, am, n0 + 64 * c + 32, ya, bar);
          },
          [&](int c, uint32_t half) {
            float x[32], oo[32];
            float dot = 0.f;
#pragma unroll
            for (int p = 0; p < 2; ++p) {
              tmem_ld32(trow + c * 64 + p * 32, x);
              box_get_bf16(half + p * TC_EPI_SLOT, lane, oo);
#pragma unroll
              for (int i = 0; i < 32; ++i) dot = fmaf(__bfloat162float(__float2bfloat16_rn(x[i])), oo[i], dot);
              box_put_bf16(half + p * TC_EPI_SLOT, lane, x);
            }
            dsum[(long long)((n0 + 64 * c) / 64) * g.S] = dot;
          },
          [&](int c, uint32_t half) {
            tma_store_2d(om, half, n0 + 64 * c, y);
            tma_store_2d(om, half + TC_EPI_SLOT, n0 + 64 * c + 32, y);
          });
      break;
    }
    case EPI_LOGITS: {
      int tgt = -1;
      if (m % g.S != g.S - 1) {
        tgt = g.tok[m + 1];
        if (tgt < 0 || tgt >= g.N) tgt = 0;   // out-of-range ids are reported by the embedding job
      }
      // running (max, sum of exp(l - max)) over the tile's columns, in base 2
      // internally: sum_i 2^((l_i - max) log2 e) = sum_i exp(l_i - max)
      float mx = -INFINITY, sm = 0.f, tv = 0.f;
      bool has_t = false;
      for (int c = 0; c < NCH; c += 2) {
        float v[64];
        tmem_ld64(trow + c * 32, v);
        const int n = ti.n0 + c * 32;
        epi_store_bf16_64(es, g.om, n, y, v);
        const int off = tgt - n;
        if ((unsigned)off < 64u) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i == off) tv = v[i];
          has_t = true;
        }
        float m8[8], s8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = v[k];
#pragma unroll
        for (int i = 8; i < 64; ++i) m8[i & 7] = fmaxf(m8[i & 7], v[i]);
        const float bm = fmaxf(fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                     fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))), mx);
        const float bml = bm * EPI_LOG2E;
        const uint64_t l2 = f2(EPI_LOG2E, EPI_LOG2E), nb2 = f2(-bml, -bml);
        uint64_t s2[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) s2[k] = f2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          float t0, t1;
          unf2(fma2(f2(v[i], v[i + 1]), l2, nb2), t0, t1);
          s2[(i >> 1) & 3] = add2(s2[(i >> 1) & 3], f2(epi_ex2(t0), epi_ex2(t1)));
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) unf2(s2[k], s8[2 * k], s8[2 * k + 1]);
        const float bs = ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
        sm = sm * epi_ex2((mx - bm) * EPI_LOG2E) + bs;
        mx = bm;
      }
      if (has_t) g.cetgt[m] = tv;
      float* pp = g.cepart + ((long long)m * g.ceparts + ti.n0 / TC_BN) * 2;
      pp[0] = mx;
      pp[1] = sm;
      break;
    }
    case EPI_STORE_F32: {
      for (int c = 0; c < NCH; c += 2) {
        float v[64];
        tmem_ld64(trow + c * 32, v);
        epi_store_f32(es, g.om, ti.n0 + c * 32, y, v);
        epi_store_f32(es, g.om, ti.n0 + c * 32 + 32, y, v + 32);
      }
      break;
    }
    case EPI_STORE_OP: {
      for (int c = 0; c < NCH; c += 2) {
        float v[64];
        tmem_ld64(trow + c * 32, v);
        epi_store_bf16(es, g.om, ti.n0 + c * 32, y, v);
        epi_store_bf16(es, g.om, ti.n0 + c * 32 + 32, y, v + 32);
      }
      break;
    }
    case EPI_RESID: {
      // out = aux + accumulator, fp32 boxes (one per half of the window)
      const int ya = g.ay0 + row0;
      const CUtensorMap* am = g.am;
      const CUtensorMap* om = g.om;
      const int n0 = ti.n0;
      epi_aux_tile(
          es, NCH, tmo, hdr,
          [&](int c, uint32_t half, uint32_t bar) {
            mbar_expect_tx(bar, 2 * TC_EPI_SLOT);
            tma_load_2d(half, am, n0 + 32 * c, ya, bar);
          },
          [&](int c, uint32_t half) {
            float v[32], x[32];
            tmem_ld32(trow + c * 32, v);
            box_get_f32(half, lane, x);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] += x[i];
            box_put_f32(half, lane, v);
          },
          [&](int c, uint32_t half) { tma_store_2d(om, half, n0 + 32 * c, y); });
      break;
    }
    default:
      break;
  }
}

__device__ __forceinline__ void tc_epilogue(const EpiRegs& g, const TcTile& ti, uint32_t trow, int m, float* st,
                                            long long row0) {
  typedef __nv_bfloat16 bf;
  constexpr int NCH = TC_BN / 32;     // 32-column chunks per row
  switch (g.epi) {
    case EPI_ROPE: {
      // hd == 64: columns [64h, 64h+32) pair with [64h+32, 64h+64)
      const float4* tab4 = reinterpret_cast<const float4*>(g.rope + (long long)(m % g.S) * 64);
      for (int h2 = 0; h2 < TC_BN / 64; ++h2) {
        float x[64];
        tmem_ld32(trow + h2 * 64, x);
        tmem_ld32(trow + h2 * 64 + 32, x + 32);
        const int n = ti.n0 + h2 * 64;
        if (n < 2 * g.hq) {
#pragma unroll
          for (int i2 = 0; i2 < 16; ++i2) {
            const float4 cs = tab4[i2];     // (cos, sin) of pairs 2*i2, 2*i2+1
            const int i = 2 * i2;
            float x1 = x[i], x2 = x[i + 32];
            x[i] = x1 * cs.x - x2 * cs.y;
            x[i + 32] = x2 * cs.x + x1 * cs.y;
            x1 = x[i + 1];
            x2 = x[i + 33];
            x[i + 1] = x1 * cs.z - x2 * cs.w;
            x[i + 33] = x2 * cs.z + x1 * cs.w;
          }
        }
        store_row_bf16<64>((bf*)g.out + (long long)m * g.ldo + n, x);
      }
      break;
    }
    case EPI_SWIGLU: {
      // each 128-column half = [64 gate | 64 up] of expert rows f0..f0+63
      for (int half = 0; half < TC_BN / 128; ++half) {
        const int f0 = ((ti.n0 >> 7) + half) * 64;
        for (int c = 0; c < 2; ++c) {
          float gg[32], uu[32];
          tmem_ld32(trow + half * 128 + c * 32, gg);
          tmem_ld32(trow + half * 128 + 64 + c * 32, uu);
          const int f = f0 + c * 32;
          bf* gu = (bf*)g.out + (long long)m * g.ldo;
          store_row_bf16<32>(gu + f, gg);
          store_row_bf16<32>(gu + g.F + f, uu);
          float act[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) act[i] = silu_f(gg[i]) * uu[i];
          store_row_bf16<32>((bf*)g.out2 + (long long)m * g.ldo2 + f, act);
        }
      }
      break;
    }
    case EPI_SWIGLU_BWD: {
      const bf* gu = (const bf*)g.aux + (long long)m * g.ldaux;
      bf* dgu = (bf*)g.out + (long long)m * g.ldo;
      for (int c = 0; c < NCH; ++c) {
        float da[32], gg[32], uu[32], dg[32], du[32];
        tmem_ld32(trow + c * 32, da);
        const int n = ti.n0 + c * 32;
        load_row_bf16<32>(gu + n, gg);
        load_row_bf16<32>(gu + g.F + n, uu);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float sg = 1.0f / (1.0f + __expf(-gg[i]));
          du[i] = da[i] * gg[i] * sg;
          dg[i] = da[i] * uu[i] * sg * (1.0f + gg[i] * (1.0f - sg));
        }
        store_row_bf16<32>(dgu + n, dg);
        store_row_bf16<32>(dgu + g.F + n, du);
      }
      break;
    }
    case EPI_STORE_OP: {
      for (int c = 0; c < NCH; ++c) {
        float v[32];
        tmem_ld32(trow + c * 32, v);
        store_row_bf16<32>((bf*)g.out + (long long)m * g.ldo + ti.n0 + c * 32, v);
      }
      break;
    }
    case EPI_STORE_OP_D: {
      // 64-column heads
      bf* o = (bf*)g.out + (long long)m * g.ldo;
      const bf* ao = (const bf*)g.aux + (long long)m * g.ldaux;
      // D is stored [batch][head][position] (the log-sum-exp's layout); ldo2 = heads
      float* dsum = (float*)g.out2 + (long long)(m / g.S) * g.ldo2 * g.S + (m % g.S);
      for (int h2 = 0; h2 < TC_BN / 64; ++h2) {
        float x[64], oo[64];
        tmem_ld32(trow + h2 * 64, x);
        tmem_ld32(trow + h2 * 64 + 32, x + 32);
        const int n = ti.n0 + h2 * 64;
        store_row_bf16<64>(o + n, x);
        load_row_bf16<64>(ao + n, oo);
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i) dot = fmaf(__bfloat162float(__float2bfloat16_rn(x[i])), oo[i], dot);
        dsum[(long long)(n / 64) * g.S] = dot;
      }
      break;
    }
    case EPI_LOGITS: {
      int tgt = -1;
      if (m % g.S != g.S - 1) {
        tgt = g.tok[m + 1];
        if (tgt < 0 || tgt >= g.N) tgt = 0;   // out-of-range ids are reported by the embedding job
      }
      float mx = -INFINITY, sm = 0.f, tv = 0.f;
      bool has_t = false;
      for (int c = 0; c < NCH; ++c) {
        float v[32];
        tmem_ld32(trow + c * 32, v);
        const int n = ti.n0 + c * 32;
        store_row_bf16<32>((bf*)g.out + (long long)m * g.ldo + n, v);
        float bm = mx;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          bm = fmaxf(bm, v[i]);
          if (n + i == tgt) { tv = v[i]; has_t = true; }
        }
        float bs = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) bs += __expf(v[i] - bm);
        sm = sm * __expf(mx - bm) + bs;
        mx = bm;
      }
      if (has_t) g.cetgt[m] = tv;
      float* pp = g.cepart + ((long long)m * g.ceparts + ti.n0 / TC_BN) * 2;
      pp[0] = mx;
      pp[1] = sm;
      break;
    }
    case EPI_NONE: {
      float acc = 0.f;
      for (int c = 0; c < NCH; ++c) {
        float v[32];
        tmem_ld32(trow + c * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) acc += v[i];
      }
      if (acc == 12345.678f) ((float*)g.out)[m] = acc;    // keeps the loads alive
      break;
    }
    case EPI_STORE_F32: {
      for (int c = 0; c < NCH; ++c) {
        float v[32];
        tmem_ld32(trow + c * 32, v);
        xpose_store_f32(st, v, (float*)g.out, g.ldo, row0, ti.n0 + c * 32);
      }
      break;
    }
    case EPI_RESID: {
      for (int c = 0; c < NCH; ++c) {
        float v[32];
        tmem_ld32(trow + c * 32, v);
        xpose_store_f32_add(st, v, (float*)g.out, (const float*)g.aux, g.ldo, g.ldaux, row0, ti.n0 + c * 32);
      }
      break;
    }
    case EPI_GRAD: {
      // rows of one tile never straddle osplit (multiples of 128)
      float* out = (float*)g.out;
      long long r0 = row0;
      if (g.osplit > 0 && row0 >= g.osplit) { out = (float*)g.out1; r0 = row0 - g.osplit; }
      out += (long long)ti.seg * g.oseg;
      for (int c = 0; c < NCH; ++c) {
        float v[32];
        tmem_ld32(trow + c * 32, v);
        if (g.accumulate)
          xpose_store_f32_add(st, v, out, out, g.ldo, g.ldo, r0, ti.n0 + c * 32);
        else
          xpose_store_f32(st, v, out, g.ldo, r0, ti.n0 + c * 32);
      }
      break;
    }
  }
}

// A weight-gradient tile whose expert received no rows: zero (or keep) the output.
__device__ __forceinline__ void tc_epilogue_empty(const EpiRegs& g, const TcTile& ti, int m) {
  if (g.epi != EPI_GRAD || g.accumulate) return;
  float* out = (float*)g.out;
  int mm = m;
  if (g.osplit > 0 && m >= g.osplit) { out = (float*)g.out1; mm = m - g.osplit; }
  out += (long long)ti.seg * g.oseg + (long long)mm * g.ldo + ti.n0;
  for (int i = 0; i < TC_BN; i += 4) *reinterpret_cast<float4*>(out + i) = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ---------------------------------------------------------------------------
// the job
// ---------------------------------------------------------------------------
// All four epilogue warps have stored their rows of the tile: publish it.
__device__ __forceinline__ void epi_signal(unsigned* c) {
  asm volatile("bar.sync 1, 128;" ::: "memory");
  if (threadIdx.x == 128) dep_signal(c);
}

// The tiles a role of this CTA works on, in order.  Static: first, first+G,
// ...  Drawn: the producer takes the next ticket for every tile and passes
// it through a TC_Q_SLOTS-entry shared-memory queue (mbarrier hand-off); the
// MMA issuer and the epilogue warps read the same sequence.  -1 ends it.
struct TileSeq {
  unsigned* ticket;
  uint32_t sbase;
  int items, G, t, k;
  bool producer;
  // next tile; false at the end of the sequence or after a timed-out wait
  __device__ __forceinline__ bool next(int& tile, ArenaHdr* hdr, long long tmo, int lane) {
    if (!ticket) {
      if (k++ > 0) t += G;
      tile = t;
      return t < items;
    }
    const uint32_t slot = (uint32_t)(k % TC_Q_SLOTS), par = (uint32_t)(k / TC_Q_SLOTS) & 1u;
    const uint32_t idx = sbase + TC_Q_IDX + 4u * slot;
    ++k;
    int v = -1;
    bool ok = true;
    if (producer) {
      // lane 0 alone
      if (!mbar_wait(sbase + TC_Q_EMPTY + 8u * slot, par ^ 1u, tmo)) {
        set_error(hdr, MT_ERR_DEVICE_TIMEOUT, SITE_TC_QUEUE);
        ok = false;
      } else {
        v = (int)atomicAdd(ticket, 1u);
        if (v >= items) v = -1;
      }
      asm volatile("st.shared.b32 [%0], %1;" ::"r"(idx), "r"(v) : "memory");
      mbar_arrive(sbase + TC_Q_FULL + 8u * slot);
    } else {
      if (!mbar_wait(sbase + TC_Q_FULL + 8u * slot, par, tmo)) {
        set_error(hdr, MT_ERR_DEVICE_TIMEOUT, SITE_TC_QUEUE);
        ok = false;
      } else {
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(idx) : "memory");
      }
      if (lane == 0) mbar_arrive(sbase + TC_Q_EMPTY + 8u * slot);
    }
    tile = v;
    return ok && v >= 0;
  }
};

static __device__ __noinline__ void gemm_tc_job(const KArgs& a, const GemmDesc& g, Sched& s, char* smem, TcState& tc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t full = sbase, empty = sbase + 64, accf = sbase + 128, acce = sbase + 144;
  const uint32_t ring = sbase + TC_RING_OFF;
  ArenaHdr* hdr = reinterpret_cast<ArenaHdr*>(a.arena + a.aoff[A_HDR]);
  const long long tmo = a.timeout_ns;
  if (sbase & 1023u) {
    // 128-byte swizzled tiles need 1024-byte aligned shared memory
    if (threadIdx.x == 0) set_error(hdr, MT_ERR_DEVICE_BOUNDS, SITE_TC_ALIGN);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < TC_STAGES; ++i) {
      mbar_init(full + 8 * i, 1);
      mbar_init(empty + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(accf + 8 * i, 1);
      mbar_init(acce + 8 * i, 4);
    }
    for (int i = 0; i < 8; ++i) mbar_init(sbase + TC_EPI_MBAR + 8 * i, 1);
    for (int i = 0; i < TC_Q_SLOTS; ++i) {
      mbar_init(sbase + TC_Q_FULL + 8 * i, 1);
      mbar_init(sbase + TC_Q_EMPTY + 8 * i, 5);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  const TcShape sh = tc_shape(g);
  const int items = gemm_items(g, TC_BM, TC_BN) * sh.ksplit;
  const int first = s.first(), G = s.G;
  TileSeq seq{g.ticket, sbase, items, G, first, 0, warp == 0};

  if (warp == 0) {
    if (lane == 0) {
      // make the generic-proxy writes of earlier phases visible to TMA reads
      asm volatile("fence.proxy.async;" ::: "memory");
      const TmaOp oa = tma_op(a, g.A), ob = tma_op(a, g.B);
      const unsigned* dw = g.dwait;
      const unsigned dtarget = g.dtarget;
      uint32_t it = 0;
      bool ok = true;
      int t;
      while (ok && seq.next(t, hdr, tmo, lane)) {
        const TcTile ti = tc_tile(sh, t);
        const int bseg = (sh.rag == RAG_M) ? ti.seg * ob.yseg : 0;
        if (dw) {
          // the A rows of this tile come from another CTA's stores (generic
          // proxy): acquire them, then order the TMA reads after the acquire
          dep_wait(hdr, dw + (ti.m0 >> 7), dtarget, tmo);
          asm volatile("fence.proxy.async;" ::: "memory");
        }
        for (int kb = 0; kb < ti.nk; ++kb, ++it) {
          const int st = it % TC_STAGES;
          const uint32_t ph = (it / TC_STAGES) & 1;
          if (!mbar_wait(empty + 8 * st, ph ^ 1, tmo)) {
            set_error(hdr, MT_ERR_DEVICE_TIMEOUT, SITE_TC_EMPTY);
            ok = false;
            break;
          }
          const uint32_t fb = full + 8 * st;
          const uint32_t sa = ring + st * TC_STAGE_BYTES, sb = sa + 2 * TC_BOX_BYTES;
          const int k0 = ti.kbeg + kb * TC_BK;
          mbar_expect_tx(fb, TC_STAGE_BYTES);
          tc_load_operand<TC_BM / 64>(oa, ti.m0, k0, 0, sa, fb);
          tc_load_operand<TC_BN / 64>(ob, ti.n0, k0, bseg, sb, fb);
        }
      }
      // drain: every issued stage must have landed before smem is reused
      const uint32_t lo = it > TC_STAGES ? it - TC_STAGES : 0;
      for (uint32_t j = lo; j < it; ++j)
        if (!mbar_wait(full + 8 * (j % TC_STAGES), (j / TC_STAGES) & 1, tmo)) {
          set_error(hdr, MT_ERR_DEVICE_TIMEOUT, SITE_TC_DRAIN);
          break;
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    // the whole warp walks the tile sequence (warp-uniform operands); one
    // elected lane issues the products and their commits
    {
      const uint32_t idesc = idesc_bf16(TC_BM, TC_BN, g.A.mn, g.B.mn);
      const uint32_t a_lbo = g.A.mn ? TC_BOX_BYTES : 16, b_lbo = g.B.mn ? TC_BOX_BYTES : 16;
      const uint32_t a_kstep = g.A.mn ? 16 * 128 : 32, b_kstep = g.B.mn ? 16 * 128 : 32;
      // descriptors of stage 0; a stage and a K step are plain address advances
      const uint64_t ad0 = sdesc(ring, a_lbo, 1024), bd0 = sdesc(ring + 2 * TC_BOX_BYTES, b_lbo, 1024);
      uint32_t it = 0, tcount = 0;
      bool ok = true;
      uint32_t last_bar = 0, last_par = 0;
      // every lane waits; the outcome is made warp-uniform
      auto wait = [&](uint32_t bar, uint32_t par, int site) {
        const bool w = __all_sync(0xffffffffu, mbar_wait(bar, par, tmo));
        if (!w && lane == 0) set_error(hdr, MT_ERR_DEVICE_TIMEOUT, site);
        return w;
      };
      while (ok) {
        // a drawn sequence is read by lane 0 and shared with the warp
        int t = -1;
        bool more = false;
        if (lane == 0) more = seq.next(t, hdr, tmo, 0);
        else if (!seq.ticket) more = seq.next(t, hdr, tmo, lane);
        if (seq.ticket) {
          more = __shfl_sync(0xffffffffu, more, 0);
          t = __shfl_sync(0xffffffffu, t, 0);
        }
        if (!more) break;
        const TcTile ti = tc_tile(sh, t);
        if (ti.nk == 0) continue;
        const int ab = tcount & 1;
        const uint32_t aph = (tcount >> 1) & 1;
        if (!wait(acce + 8 * ab, aph ^ 1, SITE_TC_ACC_EMPTY)) break;
        tc_fence_after();
        const uint32_t dt = tc.tmem_base + ab * TC_BN;
        for (int kb = 0; kb < ti.nk; ++kb, ++it) {
          const int st = it % TC_STAGES;
          const uint32_t ph = (it / TC_STAGES) & 1;
          if (!wait(full + 8 * st, ph, SITE_TC_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t soff = st * TC_STAGE_BYTES;
#pragma unroll
          for (int j = 0; j < TC_BK / 16; ++j)
            mma_bf16_warp(dt, sdesc_add(ad0, soff + j * a_kstep), sdesc_add(bd0, soff + j * b_kstep), idesc,
                          (kb > 0 || j > 0) ? 1u : 0u);
          mma_commit_warp(empty + 8 * st);
          last_bar = empty + 8 * st;
          last_par = ph;
        }
        if (!ok) break;
        mma_commit_warp(accf + 8 * ab);
        ++tcount;
      }
      // the tensor core must be idle before the job returns
      if (last_bar) wait(last_bar, last_par, SITE_TC_DRAIN);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int q = warp - 4;
    const EpiRegs er = epi_regs(a, g);
    float* xst = reinterpret_cast<float*>(smem + TC_STAGE_OFF + q * TC_EPI_WARP_BYTES);
    EpiSt es;
    es.win = sbase + TC_STAGE_OFF + q * TC_EPI_WARP_BYTES;
    es.mbar = sbase + TC_EPI_MBAR + 16 * q;
    es.nbox = 0; es.use[0] = es.use[1] = 0; es.dead = false;
    const bool tma = er.om != nullptr;
    // aux rows were stored by generic writes before this job: order the bulk
    // loads after them
    if (tma && lane == 0) asm volatile("fence.proxy.async;" ::: "memory");
    unsigned* const dsig = g.dsig;
    const unsigned* const dwa = g.dwait_aux;
    const unsigned dta = g.dtarget_aux;
    uint32_t tcount = 0;
    bool dead = false;     // after a timed-out wait: skip the work, keep the named barriers paired
    int t;
    while (true) {
      // a drawn sequence is read by lane 0 and shared with the warp
      int tt = -1;
      bool more = false;
      if (lane == 0) more = seq.next(tt, hdr, tmo, 0);
      else if (!seq.ticket) more = seq.next(tt, hdr, tmo, lane);
      if (seq.ticket) {
        more = __shfl_sync(0xffffffffu, more, 0);
        tt = __shfl_sync(0xffffffffu, tt, 0);
      }
      if (!more) break;
      t = tt;
      const TcTile ti = tc_tile(sh, t);
      const int m = ti.m0 + q * 32 + lane;
      if (dwa) {
        if (lane == 0) {
          dep_wait(hdr, dwa + (ti.m0 >> 7), dta, tmo);
          asm volatile("fence.proxy.async;" ::: "memory");
        }
        __syncwarp();
      }
      if (ti.nk == 0) {
        tc_epilogue_empty(er, ti, m);
        if (dsig) epi_signal(dsig + (ti.m0 >> 7));
        continue;
      }
      const int ab = tcount & 1;
      const uint32_t aph = (tcount >> 1) & 1;
      if (!dead && !mbar_wait(accf + 8 * ab, aph, tmo)) {
        set_error(hdr, MT_ERR_DEVICE_TIMEOUT, SITE_TC_ACC_FULL);
        dead = true;
      }
      if (!dead) {
        __syncwarp();
        tc_fence_after();
        const uint32_t trow = tc.tmem_base + ab * TC_BN + ((uint32_t)(q * 32) << 16);
        if (tma)
          tc_epilogue_tma(er, ti, trow, m, ti.m0 + q * 32, es, tmo, hdr);
        else
          tc_epilogue(er, ti, trow, m, xst, (long long)(ti.m0 + q * 32));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce + 8 * ab);
      }
      if (dsig) {
        // the tile's bulk stores have landed before its counter moves
        if (tma && lane == 0) bulk_wait_all();
        __syncwarp();
        epi_signal(dsig + (ti.m0 >> 7));
      }
      ++tcount;
    }
    // every bulk store of the job has landed before the job ends (the next
    // hand-off is a grid barrier or a later counter) and the window is free
    if (tma && lane == 0) bulk_wait_all();
    __syncwarp();
  }
  __syncthreads();
  s.next(items);
}
