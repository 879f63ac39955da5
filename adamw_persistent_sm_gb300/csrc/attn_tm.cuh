// attn_tm.cuh - causal attention forward on the 5th-generation tensor cores
// (tcgen05) for head_dim 64: the pages' bf16_sdpa.sdpa forward ("How a
// training megakernel works", section "1 - Describe the model and update").
//
// One item = 128 query rows of one (batch, head); keys in blocks of 128.
//   warp 0 (one thread): TMA loads of Q (once per item) and of K, V blocks
//                        into a two-stage ring (128-byte swizzled tiles);
//   warp 1 (one thread): S_j = Q K_j^T into one of two TMEM buffers
//                        (128 lanes x 128 fp32 columns), issued one block
//                        ahead, and PV_j = P_j V_j into one of two 64-column
//                        TMEM buffers;
//   warps 4-7          : one query row per thread.  The row of S_j is read
//                        from TMEM (tcgen05.ld), masked on the diagonal
//                        block, exponentiated against the running maximum
//                        (exp2 domain) and written as bf16 into a swizzled
//                        shared tile P_j (the A operand of PV_j); PV_{j-1} is
//                        read from TMEM and added into the row's output
//                        registers after rescaling to the new maximum.
// The output row is divided by the row sum and stored with the row
// log-sum-exp (natural log), the same formats as the other attention paths.
// P is rounded to bf16 before the PV product, as on the mma.sync path.
#pragma once
#include "common.cuh"
#include "gemm_tc.cuh"
#include <type_traits>

// Dependency counters of the attention forward (all null: phases fenced by
// grid barriers).
struct AttnDeps {
  const unsigned* wait;    // per 128-row block of q,k,v: stored column tiles
  unsigned wtarget;
  unsigned* sig;           // per 128-row block of the output: +1 per stored head
  ArenaHdr* hdr;
  long long timeout_ns;
};

namespace attn_tm {

// Item of round rnd for the CTA whose first item is `first`: the items are
// ordered longest first and dealt to the G CTAs in alternating directions
// (round 0: CTA c takes c, round 1: G - 1 - c, ...), so that no CTA takes the
// longest item of every round.  Every CTA's role loops walk the same sequence.
__device__ __forceinline__ int snake_item(int first, int G, int rnd) {
  return rnd * G + ((rnd & 1) ? (G - 1 - first) : first);
}

constexpr int BQ = 128, BKEY = 128, HD = 64;
constexpr float LOG2E = 1.4426950408889634f;

// shared memory (offsets from the 1024-aligned base)
constexpr int KST = 3;                           // K and V ring stages
constexpr uint32_t BAR_OFF = 0;                  // mbarriers
constexpr uint32_t Q_OFF = 1024;                 // 2 x Q: 128 rows x 128 B
constexpr uint32_t TILE = 16384;                 // one 128-row x 64-column bf16 tile
constexpr uint32_t K_OFF = Q_OFF + 2 * TILE;     // KST x K tile
constexpr uint32_t V_OFF = K_OFF + KST * TILE;   // KST x V tile
constexpr uint32_t P_OFF = V_OFF + KST * TILE;   // 2 x P (128 rows x 128 keys bf16: two 16 KB boxes)
constexpr uint32_t P_BUF = 2 * TILE;
constexpr uint32_t OUT_OFF = P_OFF + 2 * P_BUF;   // 4 x 4 KB: each softmax warp's output rows (bulk-store staging)
constexpr uint32_t SMEM_END = OUT_OFF + 4 * 4096;
static_assert(SMEM_END <= MT_TC_SMEM, "attention tiles exceed the shared-memory window");

// mbarrier slots (8 bytes each)
enum { B_QFULL = 0, B_QEMPTY = 2, B_KFULL = 4, B_KEMPTY = B_KFULL + KST, B_VFULL = B_KEMPTY + KST,
       B_VEMPTY = B_VFULL + KST, B_SFULL = B_VEMPTY + KST, B_SEMPTY = B_SFULL + 2, B_PFULL = B_SEMPTY + 2,
       B_OFULL = B_PFULL + 2, B_OEMPTY = B_OFULL + 2, B_COUNT = B_OEMPTY + 2 };
static_assert(B_COUNT * 8 <= 1024, "mbarriers exceed their slot");

// TMEM columns: S buffers at 0 and 128, PV buffers at 256 and 320
constexpr uint32_t TM_S = 0, TM_PV = 256;

struct Job {
  const CUtensorMap* map;    // q,k,v of all layers: rows l*T + t, columns [q | k | v]
  const CUtensorMap* map_o;  // o of all layers, 32-row x 64-column boxes (bulk stores)
  int y0;                    // row of token 0 of this layer
  __nv_bfloat16* o;          // [T][hq]
  float* lse;                // [B*H][S]
  int B, H, S, hq;
  float scale;
  // dependency counters (null: the phase is fenced by grid barriers)
  const unsigned* wait; unsigned wtarget;
  unsigned* sig;
  ArenaHdr* hdr;
  long long timeout_ns;
};

// Item k of this CTA: sequence-major (following the q,k,v product's row
// order), longest query blocks first within a sequence.
__device__ __forceinline__ void item_of(const Job& j, int it, int& b, int& h, int& qb) {
  const int nqb = j.S / BQ;
  b = it / (j.H * nqb);
  const int r = it % (j.H * nqb);
  qb = nqb - 1 - r / j.H;
  h = r % j.H;
}

// Byte offset of element (row r, key k) in a P buffer: two 64-key boxes of
// 128 rows x 128 B, 8-row groups of 1024 B, 16-byte chunks XOR-swizzled by
// the row's position in its group (the layout a 128-byte-swizzled TMA tile
// has, which the K-major operand descriptor expects).
__device__ __forceinline__ uint32_t p_chunk_off(int r, int k) {
  const int box = k >> 6, kk = k & 63;
  return (uint32_t)(box * 16384 + (r >> 3) * 1024 + (r & 7) * 128 + ((((kk >> 3) ^ r) & 7) << 4));
}

// 32 consecutive fp32 columns of this thread's TMEM lane, without waiting:
// several loads are issued back to back and completed by one tmem_wait_ld.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
// 2^x on the special-function unit (approximate, flush-to-zero)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

static __device__ __noinline__ void fwd_job(const Job& j, Sched& s, char* smem, const TcState& tc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar = sbase + BAR_OFF;
  auto B_ = [&](int i) { return bar + 8u * (uint32_t)i; };
  const long long tmo = j.timeout_ns;
  const int nqb = j.S / BQ;
  const int items = j.B * j.H * nqb;
  const int first = s.first(), G = s.G;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(B_(B_QFULL + i), 1);
      mbar_init(B_(B_QEMPTY + i), 1);
      mbar_init(B_(B_SFULL + i), 1);
      mbar_init(B_(B_SEMPTY + i), 4);
      mbar_init(B_(B_PFULL + i), 4);
      mbar_init(B_(B_OFULL + i), 1);
      mbar_init(B_(B_OEMPTY + i), 4);
    }
    for (int i = 0; i < KST; ++i) {
      mbar_init(B_(B_KFULL + i), 1);
      mbar_init(B_(B_KEMPTY + i), 1);
      mbar_init(B_(B_VFULL + i), 1);
      mbar_init(B_(B_VEMPTY + i), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      asm volatile("fence.proxy.async;" ::: "memory");
      uint32_t kvc = 0, ni = 0;
      bool dead = false;
      auto wait = [&](uint32_t b_, uint32_t par) {
        if (!dead && !mbar_wait(b_, par, tmo)) { set_error(j.hdr, MT_ERR_DEVICE_TIMEOUT, SITE_TC_EMPTY); dead = true; }
      };
      auto load_tile = [&](uint32_t dst, int x, int y, uint32_t fb) {
        mbar_expect_tx(fb, TILE);
        tma_load_2d(dst, j.map, x, y, fb);
        tma_load_2d(dst + 8192, j.map, x, y + 64, fb);
      };
      for (int rnd_ = 0, it = first; it < items; it = snake_item(first, G, ++rnd_), ++ni) {
        int b, h, qb;
        item_of(j, it, b, h, qb);
        if (j.wait) {
          for (int q = 0; q <= qb; ++q) dep_wait(j.hdr, j.wait + b * nqb + q, j.wtarget, tmo);
          asm volatile("fence.proxy.async;" ::: "memory");
        }
        const int row0 = j.y0 + b * j.S;
        const uint32_t qs = ni & 1;
        wait(B_(B_QEMPTY + qs), ((ni >> 1) & 1) ^ 1);
        load_tile(sbase + Q_OFF + qs * TILE, h * HD, row0 + qb * BQ, B_(B_QFULL + qs));
        for (int kb = 0; kb <= qb; ++kb, ++kvc) {
          const uint32_t st = kvc % KST, par = ((kvc / KST) & 1) ^ 1;
          wait(B_(B_KEMPTY + st), par);
          load_tile(sbase + K_OFF + st * TILE, j.hq + h * HD, row0 + kb * BKEY, B_(B_KFULL + st));
          wait(B_(B_VEMPTY + st), par);
          load_tile(sbase + V_OFF + st * TILE, 2 * j.hq + h * HD, row0 + kb * BKEY, B_(B_VFULL + st));
        }
      }
      // every load issued must land before the shared memory is reused
      if (!dead) {
        const uint32_t lo = kvc > KST ? kvc - KST : 0;
        for (uint32_t c = lo; c < kvc; ++c) {
          wait(B_(B_KFULL + c % KST), (c / KST) & 1);
          wait(B_(B_VFULL + c % KST), (c / KST) & 1);
        }
        for (uint32_t n = ni > 2 ? ni - 2 : 0; n < ni; ++n) wait(B_(B_QFULL + (n & 1)), (n >> 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(BQ, BKEY, 0, 0);    // Q (K-major) x K^T (K-major)
      const uint32_t id_pv = idesc_bf16(BQ, HD, 0, 1);     // P (K-major) x V (MN-major)
      uint32_t sc = 0, ni = 0;
      uint32_t last_bar = 0, last_par = 0;
      bool dead = false;
      auto wait = [&](uint32_t b_, uint32_t par, int site) {
        if (!dead && !mbar_wait(b_, par, tmo)) { set_error(j.hdr, MT_ERR_DEVICE_TIMEOUT, site); dead = true; }
      };
      // S of global block c = Q (buffer qs) K_c^T into S buffer c & 1
      auto issue_s = [&](uint32_t c, uint32_t qs) {
        const uint32_t ks = c % KST, sb = c & 1;
        wait(B_(B_KFULL + ks), (c / KST) & 1, SITE_TC_FULL);
        wait(B_(B_SEMPTY + sb), ((c >> 1) & 1) ^ 1, SITE_TC_ACC_EMPTY);
        tc_fence_after();
        const uint32_t sq = sbase + Q_OFF + qs * TILE, sk = sbase + K_OFF + ks * TILE;
        const uint64_t dq = sdesc(sq, 16, 1024), dk = sdesc(sk, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          mma_bf16(tc.tmem_base + TM_S + sb * BKEY, sdesc_add(dq, kk * 32), sdesc_add(dk, kk * 32), id_s,
                   kk > 0 ? 1u : 0u);
        mma_commit(B_(B_SFULL + sb));
        mma_commit(B_(B_KEMPTY + ks));                    // K_c is read
      };
      for (int rnd_ = 0, it = first; it < items; it = snake_item(first, G, ++rnd_), ++ni) {
        int b, h, qb;
        item_of(j, it, b, h, qb);
        const uint32_t qs = ni & 1;
        wait(B_(B_QFULL + qs), (ni >> 1) & 1, SITE_TC_FULL);
        issue_s(sc, qs);
        for (int kb = 0; kb <= qb; ++kb, ++sc) {
          if (kb < qb) issue_s(sc + 1, qs);
          else mma_commit(B_(B_QEMPTY + qs));             // Q is free once the item's last S is done
          const uint32_t pb = sc & 1, vs = sc % KST;
          wait(B_(B_VFULL + vs), (sc / KST) & 1, SITE_TC_FULL);
          wait(B_(B_PFULL + pb), (sc >> 1) & 1, SITE_TC_FULL);
          wait(B_(B_OEMPTY + pb), ((sc >> 1) & 1) ^ 1, SITE_TC_ACC_EMPTY);
          tc_fence_after();
          const uint32_t sp = sbase + P_OFF + pb * P_BUF, sv = sbase + V_OFF + vs * TILE;
          const uint64_t dp0 = sdesc(sp, 16, 1024), dv0 = sdesc(sv, 8192, 1024);
#pragma unroll
          for (int kk = 0; kk < BKEY / 16; ++kk)
            mma_bf16(tc.tmem_base + TM_PV + pb * HD, sdesc_add(dp0, (kk >> 2) * 16384 + (kk & 3) * 32),
                     sdesc_add(dv0, kk * 2048), id_pv, kk > 0 ? 1u : 0u);
          mma_commit(B_(B_OFULL + pb));
          mma_commit(B_(B_VEMPTY + vs));
          last_bar = B_(B_VEMPTY + vs);
          last_par = (sc / KST) & 1;
        }
      }
      // the tensor core must be idle before the job returns
      if (last_bar && !dead && !mbar_wait(last_bar, last_par, tmo)) set_error(j.hdr, MT_ERR_DEVICE_TIMEOUT, SITE_TC_DRAIN);
      if (ni > 0 && !dead && !mbar_wait(B_(B_QEMPTY + ((ni - 1) & 1)), ((ni - 1) >> 1) & 1, tmo))
        set_error(j.hdr, MT_ERR_DEVICE_TIMEOUT, SITE_TC_DRAIN);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------- softmax and output: one query row per thread ----------------
    const int q = warp - 4;
    const int r = q * 32 + lane;                           // row within the item, TMEM lane
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const float sc_l2 = j.scale * LOG2E;
    const uint64_t sc2 = f2(sc_l2, sc_l2);
    uint32_t sc = 0;
    bool dead = false;
    auto wait = [&](uint32_t b_, uint32_t par, int site) {
      if (!dead && !mbar_wait(b_, par, tmo)) { set_error(j.hdr, MT_ERR_DEVICE_TIMEOUT, site); dead = true; }
    };
    // add the PV block with counter c (relative to maximum mc) into o (relative to m_o)
    auto add_pv = [&](float* o, float& m_o, uint32_t c, float mc) {
      const uint32_t pb = c & 1;
      wait(B_(B_OFULL + pb), (c >> 1) & 1, SITE_TC_ACC_FULL);
      __syncwarp();
      tc_fence_after();
      const float alpha = (m_o == -INFINITY) ? 0.f : exp2f(m_o - mc);
      const uint32_t tp = tc.tmem_base + lane_off + TM_PV + pb * HD;
      uint32_t v[HD];
      tmem_ld32_async(tp, v);
      tmem_ld32_async(tp + 32, v + 32);
      tmem_wait_ld();
      const uint64_t al2 = f2(alpha, alpha);
#pragma unroll
      for (int i = 0; i < HD; i += 2) unf2(fma2(f2(o[i], o[i + 1]), al2, u2(v[i], v[i + 1])), o[i], o[i + 1]);
      m_o = mc;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(B_(B_OEMPTY + pb));
    };
    for (int rnd_ = 0, it = first; it < items; it = snake_item(first, G, ++rnd_)) {
      int b, h, qb;
      item_of(j, it, b, h, qb);
      float o[HD];
#pragma unroll
      for (int i = 0; i < HD; ++i) o[i] = 0.f;
      float m = -INFINITY, lsum = 0.f, m_o = -INFINITY;
      for (int kb = 0; kb <= qb; ++kb, ++sc) {
        const uint32_t sb = sc & 1;
        wait(B_(B_SFULL + sb), (sc >> 1) & 1, SITE_TC_ACC_FULL);
        __syncwarp();
        tc_fence_after();
        const uint32_t ts = tc.tmem_base + lane_off + TM_S + sb * BKEY;
        const bool diag = (kb == qb);
        // the whole row of S (128 fp32 columns) in four loads and one wait
        uint32_t sr[BKEY];
#pragma unroll
        for (int c = 0; c < BKEY / 32; ++c) tmem_ld32_async(ts + c * 32, sr + c * 32);
        tmem_wait_ld();
        // diagonal block: keys after the row's query are masked as -inf (their
        // probability is then exactly 0)
        if (diag) {
#pragma unroll
          for (int i = 0; i < BKEY; ++i)
            if (i > r) sr[i] = 0xff800000u;
        }
        // row maximum with eight independent partial maxima
        float mx8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mx8[u] = __uint_as_float(sr[u]);
#pragma unroll
        for (int i = 8; i < BKEY; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(sr[i]));
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        const float mn = fmaxf(m, mx * sc_l2);
        // probabilities against the new maximum (eight partial row sums) and
        // the bf16 P tile
        uint64_t rs2[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) rs2[u] = f2(0.f, 0.f);
        const uint64_t nmn2 = f2(-mn, -mn);
        const uint32_t pbase = sbase + P_OFF + sb * P_BUF;
#pragma unroll
        for (int c = 0; c < BKEY / 32; ++c) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const int k = c * 32 + i;
            float t0, t1;
            unf2(fma2(u2(sr[k], sr[k + 1]), sc2, nmn2), t0, t1);
            const float p0 = ex2(t0), p1 = ex2(t1);
            rs2[(k >> 1) & 3] = add2(rs2[(k >> 1) & 3], f2(p0, p1));
            w[i >> 1] = pack2(p0, p1);
          }
#pragma unroll
          for (int g = 0; g < 4; ++g)
            st_shared_v4(pbase + p_chunk_off(r, c * 32 + g * 8), w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
        }
        float rs8[8];
#pragma unroll
        for (int u = 0; u < 4; ++u) unf2(rs2[u], rs8[2 * u], rs8[2 * u + 1]);
        const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
        // the S buffer is read and the P tile written (generic proxy -> tensor core)
        tc_fence_before();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(B_(B_SEMPTY + sb));
          mbar_arrive(B_(B_PFULL + sb));
        }
        const float m_prev = m;                    // the maximum P_{kb-1} was taken against
        lsum = (m == -INFINITY ? 0.f : lsum * exp2f(m - mn)) + rs;
        m = mn;
        if (kb > 0) add_pv(o, m_o, sc - 1, m_prev);
      }
      add_pv(o, m_o, sc - 1, m);                   // the item's last block
      // normalise, store the output row and the log-sum-exp
      const float inv = 1.f / lsum;
#pragma unroll
      for (int i = 0; i < HD; ++i) o[i] *= inv;
      // the output rows go out by one bulk store per warp (the previous
      // item's store has read the staging rows first)
      const uint32_t ob = sbase + OUT_OFF + (uint32_t)q * 4096u;
      if (lane == 0) bulk_wait_read<0>();
      __syncwarp();
#pragma unroll
      for (int g = 0; g < HD / 8; ++g)
        st_shared_v4(ob + (uint32_t)lane * 128u + ((uint32_t)(g ^ (lane & 7)) << 4), pack2(o[8 * g], o[8 * g + 1]),
                     pack2(o[8 * g + 2], o[8 * g + 3]), pack2(o[8 * g + 4], o[8 * g + 5]), pack2(o[8 * g + 6], o[8 * g + 7]));
      fence_smem_async();
      __syncwarp();
      if (lane == 0 && !dead) {
        tma_store_2d(j.map_o, ob, h * HD, j.y0 + b * j.S + qb * BQ + q * 32);
        bulk_commit();
      }
      j.lse[((long long)b * j.H + h) * j.S + qb * BQ + r] = m + log2f(lsum);   // log2 units
      if (j.sig) {
        // every row of the block is stored: publish it
        if (lane == 0) bulk_wait_all();
        __syncwarp();
        asm volatile("bar.sync 2, 128;" ::: "memory");
        if (threadIdx.x == 128) dep_signal(j.sig + b * nqb + qb);
      }
    }
    // every output row has landed before the phase ends
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  __syncthreads();
  s.next(items);
}


// ===========================================================================
// Backward ("How a training megakernel works", section "1 - Describe the
// model and update": the backward of bf16_sdpa.sdpa).  P is recomputed from
// the saved log-sum-exp; D = rowsum(dO * O) comes from the dO product's
// epilogue.  Two item families, so that every output row is written once
// and without atomics:
//   dK/dV : 128 keys per item, 64-query steps.  S^T = K Q^T and
//           dP^T = V dO^T go to TMEM (two buffers each); the softmax warps
//           (one key row per thread) write P^T and dS^T = P^T (dP^T - D) as
//           bf16 tiles; dV += P^T dO and dK += dS^T Q accumulate in TMEM.
//   dQ    : 128 queries per item, 64-key steps.  S = Q K^T and dP = dO V^T
//           in TMEM; the softmax warps (one query row per thread) write
//           dS = P (dP - D); dQ += dS K accumulates in TMEM.
// dK and dQ are scaled by the softmax scale and the rotary embedding is
// undone on them before they are stored (bf16 rows of dqkv).
// ===========================================================================
struct BwdJob {
  const CUtensorMap* map_qkv;  // q,k,v of all layers
  const CUtensorMap* map_do;   // dO [T][hq]
  const CUtensorMap* map_dqkv; // dq,dk,dv [T][3hq], 32-row x 64-column boxes (bulk stores)
  const CUtensorMap* map_ds;   // dS^T [B*H*S keys][S queries]: 128-row x 64-column boxes (stores)
  const CUtensorMap* map_dsl;  // the same buffer, 64 x 64 boxes (loads of the dQ product)
  int dsg;                     // dK/dV stores dS^T and dQ is a product over it (else dQ recomputes dS)
  int y0;                      // row of token 0 of this layer in map_qkv
  const float* lse;            // [B*H][S] log2 of the row sum of exp2(scale log2(e) s) (this path's forward)
  const float* dsum;           // [B*H][S]
  __nv_bfloat16* dqkv;         // [T][3hq]
  const float* rope;           // [S][32][2] cos, sin
  int B, H, S, hq;
  float scale;
  ArenaHdr* hdr;
  long long timeout_ns;
};

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Undo the rotary embedding on a 64-wide gradient row (dims i and i + 32
// form a pair; cs = the position's 32 (cos, sin) pairs) and scale it.
__device__ __forceinline__ void rope_undo(float* g, const float4* cs, float scale) {
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int i = 2 * q;
    float d1 = g[i] * scale, d2 = g[i + 32] * scale;
    g[i] = d1 * cs[q].x + d2 * cs[q].y;
    g[i + 32] = d2 * cs[q].x - d1 * cs[q].y;
    d1 = g[i + 1] * scale;
    d2 = g[i + 33] * scale;
    g[i + 1] = d1 * cs[q].z + d2 * cs[q].w;
    g[i + 33] = d2 * cs[q].z - d1 * cs[q].w;
  }
}
// Row r of a 32-row x 64-column bf16 box with the 128-byte swizzle (16-byte
// chunk j at chunk j ^ (r & 7) of the row) <- v[0..63]
__device__ __forceinline__ void box_put_row64(uint32_t box, int r, const float* v) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    st_shared_v4(box + (uint32_t)r * 128u + ((uint32_t)(j ^ (r & 7)) << 4), pack2(v[8 * j], v[8 * j + 1]),
                 pack2(v[8 * j + 2], v[8 * j + 3]), pack2(v[8 * j + 4], v[8 * j + 5]), pack2(v[8 * j + 6], v[8 * j + 7]));
}

namespace kv {   // dK/dV layout
constexpr int NST = 4;                              // query-step ring stages
constexpr uint32_t KV_OFF = 1024;                    // 2 x (K 16 KB | V 16 KB): the next item's keys load early
constexpr uint32_t ST_OFF = KV_OFF + 4 * TILE;       // stage: Q 8 KB | dO 8 KB | lse 256 B | D 256 B
constexpr uint32_t ST_BYTES = 17408;
constexpr uint32_t P_OFF = ST_OFF + NST * ST_BYTES;   // 2 x P^T (128 keys x 64 queries)
constexpr uint32_t DS_OFF = P_OFF + 2 * TILE;         // 3 x dS^T (step c uses buffer c % 3)
constexpr int NDS = 3;
constexpr uint32_t END = DS_OFF + NDS * TILE;
static_assert(END <= MT_TC_SMEM, "dK/dV tiles exceed the shared-memory window");
static_assert(P_OFF % 1024 == 0 && ST_OFF % 1024 == 0 && ST_BYTES % 1024 == 0, "swizzled tiles need 1024-byte alignment");
enum { KVFULL = 0, KVEMPTY = 2, ACCFULL = 4, ACCEMPTY = 5, STFULL = 6, STEMPTY = STFULL + NST, SDFULL = STEMPTY + NST,
       SDEMPTY = SDFULL + 2, PDFULL = SDEMPTY + 2, PDEMPTY = PDFULL + 2, DSFREE = PDEMPTY + 2, COUNT = DSFREE + NDS };
// TMEM: S^T at 0/64, dP^T at 128/192, dV at 256, dK at 320
constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 320;
}

static __device__ __noinline__ void dkdv_job(const BwdJob& j, Sched& s, char* smem, const TcState& tc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  auto B_ = [&](int i) { return sbase + 8u * (uint32_t)i; };
  const long long tmo = j.timeout_ns;
  const int nkb = j.S / 128;
  const int items = j.B * j.H * nkb;
  const int first = s.first(), G = s.G;
  // item: longest (first key blocks) first
  auto item_of = [&](int it, int& b, int& h, int& kb) {
    kb = it / (j.B * j.H);
    const int bh = it % (j.B * j.H);
    b = bh / j.H; h = bh % j.H;
  };
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) { mbar_init(B_(kv::KVFULL + i), 1); mbar_init(B_(kv::KVEMPTY + i), 1); }
    mbar_init(B_(kv::ACCFULL), 1); mbar_init(B_(kv::ACCEMPTY), 4);
    for (int i = 0; i < kv::NST; ++i) { mbar_init(B_(kv::STFULL + i), 1); mbar_init(B_(kv::STEMPTY + i), 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(B_(kv::SDFULL + i), 1); mbar_init(B_(kv::SDEMPTY + i), 4);
      mbar_init(B_(kv::PDFULL + i), 4); mbar_init(B_(kv::PDEMPTY + i), 1);
    }
    for (int i = 0; i < kv::NDS; ++i) mbar_init(B_(kv::DSFREE + i), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  bool dead = false;
  auto wait = [&](uint32_t b_, uint32_t par, int site) {
    if (!dead && !mbar_wait(b_, par, tmo)) { set_error(j.hdr, MT_ERR_DEVICE_TIMEOUT, site); dead = true; }
  };
  if (warp == 0) {
    if (lane == 0) {
      // ---------------- loads ----------------
      uint32_t c = 0, ni = 0;
      for (int rnd_ = 0, it = first; it < items; it = snake_item(first, G, ++rnd_), ++ni) {
        int b, h, kb;
        item_of(it, b, h, kb);
        const int row0 = b * j.S;
        const uint32_t kbf = ni & 1, kva = sbase + kv::KV_OFF + kbf * 2 * TILE;
        wait(B_(kv::KVEMPTY + kbf), ((ni >> 1) & 1) ^ 1, SITE_TC_EMPTY);
        mbar_expect_tx(B_(kv::KVFULL + kbf), 2 * TILE);
        for (int half = 0; half < 2; ++half) {
          tma_load_2d(kva + half * 8192, j.map_qkv, j.hq + h * HD, j.y0 + row0 + kb * 128 + half * 64, B_(kv::KVFULL + kbf));
          tma_load_2d(kva + TILE + half * 8192, j.map_qkv, 2 * j.hq + h * HD, j.y0 + row0 + kb * 128 + half * 64,
                      B_(kv::KVFULL + kbf));
        }
        const int nst = (j.S - kb * 128) / 64;
        const float* lrow = j.lse + ((long long)b * j.H + h) * j.S;
        const float* drow = j.dsum + ((long long)b * j.H + h) * j.S;
        for (int i = 0; i < nst; ++i, ++c) {
          const int q0 = kb * 128 + i * 64;
          const uint32_t st = c % kv::NST, sa = sbase + kv::ST_OFF + st * kv::ST_BYTES;
          wait(B_(kv::STEMPTY + st), ((c / kv::NST) & 1) ^ 1, SITE_TC_EMPTY);
          mbar_expect_tx(B_(kv::STFULL + st), 2 * 8192 + 512);
          tma_load_2d(sa, j.map_qkv, h * HD, j.y0 + row0 + q0, B_(kv::STFULL + st));
          tma_load_2d(sa + 8192, j.map_do, h * HD, row0 + q0, B_(kv::STFULL + st));
          bulk_load(sa + 16384, lrow + q0, 256, B_(kv::STFULL + st));
          bulk_load(sa + 16640, drow + q0, 256, B_(kv::STFULL + st));
        }
      }
      if (!dead) {
        for (uint32_t x = c > kv::NST ? c - kv::NST : 0; x < c; ++x) wait(B_(kv::STFULL + x % kv::NST), (x / kv::NST) & 1, SITE_TC_DRAIN);
        for (uint32_t n = ni > 2 ? ni - 2 : 0; n < ni; ++n) wait(B_(kv::KVFULL + (n & 1)), (n >> 1) & 1, SITE_TC_DRAIN);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA ----------------
      const uint32_t id_sd = idesc_bf16(128, 64, 0, 0);     // K (or V) x Q^T (or dO^T)
      const uint32_t id_acc = idesc_bf16(128, 64, 0, 1);    // P^T (or dS^T) x dO (or Q), MN-major B
      uint32_t c = 0, ni = 0, last_bar = 0, last_par = 0;
      uint32_t kva = sbase + kv::KV_OFF;
      auto issue_sd = [&](uint32_t cc) {
        const uint32_t st = cc % kv::NST, sb = cc & 1, sa = sbase + kv::ST_OFF + st * kv::ST_BYTES;
        wait(B_(kv::STFULL + st), (cc / kv::NST) & 1, SITE_TC_FULL);
        wait(B_(kv::SDEMPTY + sb), ((cc >> 1) & 1) ^ 1, SITE_TC_ACC_EMPTY);
        tc_fence_after();
        const uint64_t dk = sdesc(kva, 16, 1024), dq = sdesc(sa, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          mma_bf16(tc.tmem_base + kv::TM_S + sb * 64, sdesc_add(dk, kk * 32), sdesc_add(dq, kk * 32), id_sd,
                   kk > 0 ? 1u : 0u);
          mma_bf16(tc.tmem_base + kv::TM_DP + sb * 64, sdesc_add(dk, TILE + kk * 32), sdesc_add(dq, 8192 + kk * 32),
                   id_sd, kk > 0 ? 1u : 0u);
        }
        mma_commit(B_(kv::SDFULL + sb));
      };
      for (int rnd_ = 0, it = first; it < items; it = snake_item(first, G, ++rnd_), ++ni) {
        int b, h, kb;
        item_of(it, b, h, kb);
        const int nst = (j.S - kb * 128) / 64;
        const uint32_t kbf = ni & 1;
        kva = sbase + kv::KV_OFF + kbf * 2 * TILE;
        wait(B_(kv::KVFULL + kbf), (ni >> 1) & 1, SITE_TC_FULL);
        issue_sd(c);
        for (int i = 0; i < nst; ++i, ++c) {
          if (i + 1 < nst) issue_sd(c + 1);
          const uint32_t st = c % kv::NST, sb = c & 1, sa = sbase + kv::ST_OFF + st * kv::ST_BYTES;
          wait(B_(kv::PDFULL + sb), (c >> 1) & 1, SITE_TC_FULL);
          if (i == 0) wait(B_(kv::ACCEMPTY), (ni & 1) ^ 1, SITE_TC_ACC_EMPTY);   // dK, dV of the last item are read
          tc_fence_after();
          const uint64_t dpt = sdesc(sbase + kv::P_OFF + sb * TILE, 16, 1024);
          const uint64_t dst = sdesc(sbase + kv::DS_OFF + (c % kv::NDS) * TILE, 16, 1024);
          const uint64_t dqm = sdesc(sa, 8192, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
            mma_bf16(tc.tmem_base + kv::TM_DV, sdesc_add(dpt, kk * 32), sdesc_add(dqm, 8192 + kk * 2048), id_acc, acc);
            mma_bf16(tc.tmem_base + kv::TM_DK, sdesc_add(dst, kk * 32), sdesc_add(dqm, kk * 2048), id_acc, acc);
          }
          mma_commit(B_(kv::PDEMPTY + sb));
          mma_commit(B_(kv::STEMPTY + st));
          last_bar = B_(kv::STEMPTY + st);
          last_par = (c / kv::NST) & 1;
        }
        mma_commit(B_(kv::ACCFULL));
        mma_commit(B_(kv::KVEMPTY + kbf));
      }
      if (last_bar && !dead && !mbar_wait(last_bar, last_par, tmo)) set_error(j.hdr, MT_ERR_DEVICE_TIMEOUT, SITE_TC_DRAIN);
      if (ni > 0) wait(B_(kv::KVEMPTY + ((ni - 1) & 1)), ((ni - 1) >> 1) & 1, SITE_TC_DRAIN);
    }
    __syncwarp();
  } else if (warp == 2) {
    if (lane == 0 && j.dsg) {
      // ---------------- dS^T stores ----------------
      // each step's dS^T tile (128 keys x 64 queries, swizzled) goes to HBM
      // for the dQ product with one bulk store; its buffer (one of three) is
      // released as soon as that store has read it
      const uint64_t pol = l2_evict_first();
      uint32_t c = 0;
      for (int rnd_ = 0, it = first; it < items; it = snake_item(first, G, ++rnd_)) {
        int b, h, kb;
        item_of(it, b, h, kb);
        const int nst = (j.S - kb * 128) / 64;
        for (int i = 0; i < nst; ++i, ++c) {
          const uint32_t sb = c & 1, dsb = c % kv::NDS;
          wait(B_(kv::PDFULL + sb), (c >> 1) & 1, SITE_TC_FULL);
          if (!dead) {
            tma_store_2d_hint(j.map_ds, sbase + kv::DS_OFF + dsb * TILE, kb * 128 + i * 64, (b * j.H + h) * j.S + kb * 128,
                              pol);
            bulk_commit();
          }
          bulk_wait_read<0>();
          mbar_arrive(B_(kv::DSFREE + dsb));
        }
      }
      bulk_wait_all();
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------- softmax and output: one key row per thread ----------------
    const int q = warp - 4, r = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const float sc_l2 = j.scale * LOG2E;
    const uint64_t sc2 = f2(sc_l2, sc_l2);
    uint32_t c = 0, ni = 0;
    for (int rnd_ = 0, it = first; it < items; it = snake_item(first, G, ++rnd_), ++ni) {
      int b, h, kb;
      item_of(it, b, h, kb);
      const int nst = (j.S - kb * 128) / 64;
      for (int i = 0; i < nst; ++i, ++c) {
        const uint32_t st = c % kv::NST, sb = c & 1, sa = sbase + kv::ST_OFF + st * kv::ST_BYTES;
        wait(B_(kv::SDFULL + sb), (c >> 1) & 1, SITE_TC_ACC_FULL);
        wait(B_(kv::STFULL + st), (c / kv::NST) & 1, SITE_TC_ACC_FULL);      // lse and D of the step
        __syncwarp();
        tc_fence_after();
        uint32_t sv[64], dp[64];
        tmem_ld32_async(tc.tmem_base + lane_off + kv::TM_S + sb * 64, sv);
        tmem_ld32_async(tc.tmem_base + lane_off + kv::TM_S + sb * 64 + 32, sv + 32);
        tmem_ld32_async(tc.tmem_base + lane_off + kv::TM_DP + sb * 64, dp);
        tmem_ld32_async(tc.tmem_base + lane_off + kv::TM_DP + sb * 64 + 32, dp + 32);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(B_(kv::SDEMPTY + sb));
        const float* sl = reinterpret_cast<const float*>(smem + kv::ST_OFF + st * kv::ST_BYTES + 16384);
        const float* sd = sl + 64;
        // queries q0 + x with q0 + x < key are masked (only the first two steps)
        const int lim = r - i * 64;            // x < lim is masked
        if (i == 0) {
          // the previous item's dK, dV bulk stores have read their staging rows
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
        }
        wait(B_(kv::PDEMPTY + sb), ((c >> 1) & 1) ^ 1, SITE_TC_EMPTY);
        // the dS^T store of three steps back has read this step's buffer
        const uint32_t dsb = c % kv::NDS;
        if (j.dsg) wait(B_(kv::DSFREE + dsb), ((c / kv::NDS) & 1) ^ 1, SITE_TC_EMPTY);
        const uint32_t pb = sbase + kv::P_OFF + sb * TILE, db = sbase + kv::DS_OFF + dsb * TILE;
        // P^T and dS^T of the step; the mask only touches the first two steps,
        // the others run without the compare and select
        auto soft = [&](auto MASKc) {
          constexpr bool MASK = decltype(MASKc)::value;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            uint32_t wp[4], wd[4];
            const float4 la = reinterpret_cast<const float4*>(sl)[2 * g], lb = reinterpret_cast<const float4*>(sl)[2 * g + 1];
            const float4 da = reinterpret_cast<const float4*>(sd)[2 * g], dbv = reinterpret_cast<const float4*>(sd)[2 * g + 1];
            const uint64_t z2 = f2(0.f, 0.f);
            const uint64_t nl[4] = {sub2(z2, f2(la.x, la.y)), sub2(z2, f2(la.z, la.w)), sub2(z2, f2(lb.x, lb.y)),
                                    sub2(z2, f2(lb.z, lb.w))};
            const uint64_t dv[4] = {f2(da.x, da.y), f2(da.z, da.w), f2(dbv.x, dbv.y), f2(dbv.z, dbv.w)};
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const int x = g * 8 + e;
              float t0, t1;
              unf2(fma2(u2(sv[x], sv[x + 1]), sc2, nl[e >> 1]), t0, t1);
              float p0 = ex2(t0), p1 = ex2(t1);
              if (MASK) {
                if (x < lim) p0 = 0.f;
                if (x + 1 < lim) p1 = 0.f;
              }
              float d0, d1;
              unf2(mul2(f2(p0, p1), sub2(u2(dp[x], dp[x + 1]), dv[e >> 1])), d0, d1);
              wp[e >> 1] = pack2(p0, p1);
              wd[e >> 1] = pack2(d0, d1);
            }
            st_shared_v4(pb + p_chunk_off(r, g * 8), wp[0], wp[1], wp[2], wp[3]);
            st_shared_v4(db + p_chunk_off(r, g * 8), wd[0], wd[1], wd[2], wd[3]);
          }
        };
        if (i < 2) soft(std::true_type());
        else soft(std::false_type());
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(B_(kv::PDFULL + sb));
      }
      // dK, dV of the item's 128 keys: the key's rotary table row is loaded
      // while the last products finish; the rows are staged in this warp's
      // rows of P^T buffer 0 (dK) and P^T buffer 1 (dV), free once every
      // product of the item has completed, and written by bulk stores
      const int key = kb * 128 + r;
      float4 cs[16];
      {
        const float4* tab = reinterpret_cast<const float4*>(j.rope + (long long)key * 64);
#pragma unroll
        for (int x = 0; x < 16; ++x) cs[x] = tab[x];
      }
      wait(B_(kv::ACCFULL), ni & 1, SITE_TC_ACC_FULL);
      __syncwarp();
      tc_fence_after();
      uint32_t vk[64], vv[64];
      tmem_ld32_async(tc.tmem_base + lane_off + kv::TM_DK, vk);
      tmem_ld32_async(tc.tmem_base + lane_off + kv::TM_DK + 32, vk + 32);
      tmem_ld32_async(tc.tmem_base + lane_off + kv::TM_DV, vv);
      tmem_ld32_async(tc.tmem_base + lane_off + kv::TM_DV + 32, vv + 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(B_(kv::ACCEMPTY));
      // dK rows in P^T buffer 0, dV rows in P^T buffer 1 (both free: every
      // product of the item has completed, and the next item's first step
      // waits for these stores to have read them before writing P^T)
      const uint32_t bk = sbase + kv::P_OFF + (uint32_t)q * 4096u, bv = sbase + kv::P_OFF + TILE + (uint32_t)q * 4096u;
      float g[64];
#pragma unroll
      for (int x = 0; x < 64; ++x) g[x] = __uint_as_float(vk[x]);
      rope_undo(g, cs, j.scale);
      box_put_row64(bk, lane, g);
#pragma unroll
      for (int x = 0; x < 64; ++x) g[x] = __uint_as_float(vv[x]);
      box_put_row64(bv, lane, g);
      fence_smem_async();
      __syncwarp();
      if (lane == 0 && !dead) {
        const int y = b * j.S + kb * 128 + q * 32;
        tma_store_2d(j.map_dqkv, bk, j.hq + h * HD, y);
        tma_store_2d(j.map_dqkv, bv, 2 * j.hq + h * HD, y);
        bulk_commit();
      }
      __syncwarp();
    }
    // every dK, dV row has landed before the phase ends
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  __syncthreads();
  s.next(items);
}

namespace qd {   // dQ layout
constexpr int NST = 4;                              // key-step ring stages: K 8 KB | V 8 KB
constexpr uint32_t QD_OFF = 1024;                    // 2 x (Q 16 KB | dO 16 KB): the next item's rows load early
constexpr uint32_t ST_OFF = QD_OFF + 4 * TILE;
constexpr uint32_t ST_BYTES = 16384;
constexpr uint32_t DS_OFF = ST_OFF + NST * ST_BYTES;  // 2 x dS (128 queries x 64 keys)
constexpr uint32_t OUT_OFF = DS_OFF + 2 * TILE;   // 4 x 4 KB: each epilogue warp's dQ rows (bulk-store staging)
constexpr uint32_t END = OUT_OFF + 4 * 4096;
static_assert(END <= MT_TC_SMEM, "dQ tiles exceed the shared-memory window");
static_assert(OUT_OFF % 1024 == 0, "swizzled staging needs 1024-byte alignment");
enum { QFULL = 0, QEMPTY = 2, ACCFULL = 4, ACCEMPTY = 5, STFULL = 6, STEMPTY = STFULL + NST, SDFULL = STEMPTY + NST,
       SDEMPTY = SDFULL + 2, DSFULL = SDEMPTY + 2, DSEMPTY = DSFULL + 2, COUNT = DSEMPTY + 2 };
constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DQ = 256;
}

static __device__ __noinline__ void dq_job(const BwdJob& j, Sched& s, char* smem, const TcState& tc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  auto B_ = [&](int i) { return sbase + 8u * (uint32_t)i; };
  const long long tmo = j.timeout_ns;
  const int nqb = j.S / 128;
  const int items = j.B * j.H * nqb;
  const int first = s.first(), G = s.G;
  // item: longest (last query blocks) first
  auto item_of = [&](int it, int& b, int& h, int& qb) {
    qb = nqb - 1 - it / (j.B * j.H);
    const int bh = it % (j.B * j.H);
    b = bh / j.H; h = bh % j.H;
  };
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) { mbar_init(B_(qd::QFULL + i), 1); mbar_init(B_(qd::QEMPTY + i), 1); }
    mbar_init(B_(qd::ACCFULL), 1); mbar_init(B_(qd::ACCEMPTY), 4);
    for (int i = 0; i < qd::NST; ++i) { mbar_init(B_(qd::STFULL + i), 1); mbar_init(B_(qd::STEMPTY + i), 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(B_(qd::SDFULL + i), 1); mbar_init(B_(qd::SDEMPTY + i), 4);
      mbar_init(B_(qd::DSFULL + i), 4); mbar_init(B_(qd::DSEMPTY + i), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  bool dead = false;
  auto wait = [&](uint32_t b_, uint32_t par, int site) {
    if (!dead && !mbar_wait(b_, par, tmo)) { set_error(j.hdr, MT_ERR_DEVICE_TIMEOUT, site); dead = true; }
  };
  if (warp == 0) {
    if (lane == 0) {
      uint32_t c = 0, ni = 0;
      for (int rnd_ = 0, it = first; it < items; it = snake_item(first, G, ++rnd_), ++ni) {
        int b, h, qb;
        item_of(it, b, h, qb);
        const int row0 = b * j.S;
        const uint32_t qbf = ni & 1, qa = sbase + qd::QD_OFF + qbf * 2 * TILE;
        wait(B_(qd::QEMPTY + qbf), ((ni >> 1) & 1) ^ 1, SITE_TC_EMPTY);
        mbar_expect_tx(B_(qd::QFULL + qbf), 2 * TILE);
        for (int half = 0; half < 2; ++half) {
          tma_load_2d(qa + half * 8192, j.map_qkv, h * HD, j.y0 + row0 + qb * 128 + half * 64, B_(qd::QFULL + qbf));
          tma_load_2d(qa + TILE + half * 8192, j.map_do, h * HD, row0 + qb * 128 + half * 64, B_(qd::QFULL + qbf));
        }
        const int nst = 2 * (qb + 1);
        for (int i = 0; i < nst; ++i, ++c) {
          const uint32_t st = c % qd::NST, sa = sbase + qd::ST_OFF + st * qd::ST_BYTES;
          wait(B_(qd::STEMPTY + st), ((c / qd::NST) & 1) ^ 1, SITE_TC_EMPTY);
          mbar_expect_tx(B_(qd::STFULL + st), 2 * 8192);
          tma_load_2d(sa, j.map_qkv, j.hq + h * HD, j.y0 + row0 + i * 64, B_(qd::STFULL + st));
          tma_load_2d(sa + 8192, j.map_qkv, 2 * j.hq + h * HD, j.y0 + row0 + i * 64, B_(qd::STFULL + st));
        }
      }
      if (!dead) {
        for (uint32_t x = c > qd::NST ? c - qd::NST : 0; x < c; ++x) wait(B_(qd::STFULL + x % qd::NST), (x / qd::NST) & 1, SITE_TC_DRAIN);
        for (uint32_t n = ni > 2 ? ni - 2 : 0; n < ni; ++n) wait(B_(qd::QFULL + (n & 1)), (n >> 1) & 1, SITE_TC_DRAIN);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_sd = idesc_bf16(128, 64, 0, 0);     // Q (or dO) x K^T (or V^T)
      const uint32_t id_acc = idesc_bf16(128, 64, 0, 1);    // dS x K, MN-major B
      uint32_t c = 0, ni = 0, last_bar = 0, last_par = 0;
      uint32_t qa = sbase + qd::QD_OFF;
      auto issue_sd = [&](uint32_t cc) {
        const uint32_t st = cc % qd::NST, sb = cc & 1, sa = sbase + qd::ST_OFF + st * qd::ST_BYTES;
        wait(B_(qd::STFULL + st), (cc / qd::NST) & 1, SITE_TC_FULL);
        wait(B_(qd::SDEMPTY + sb), ((cc >> 1) & 1) ^ 1, SITE_TC_ACC_EMPTY);
        tc_fence_after();
        const uint64_t dq = sdesc(qa, 16, 1024), dk = sdesc(sa, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          mma_bf16(tc.tmem_base + qd::TM_S + sb * 64, sdesc_add(dq, kk * 32), sdesc_add(dk, kk * 32), id_sd,
                   kk > 0 ? 1u : 0u);
          mma_bf16(tc.tmem_base + qd::TM_DP + sb * 64, sdesc_add(dq, TILE + kk * 32), sdesc_add(dk, 8192 + kk * 32),
                   id_sd, kk > 0 ? 1u : 0u);
        }
        mma_commit(B_(qd::SDFULL + sb));
      };
      for (int rnd_ = 0, it = first; it < items; it = snake_item(first, G, ++rnd_), ++ni) {
        int b, h, qb;
        item_of(it, b, h, qb);
        const int nst = 2 * (qb + 1);
        const uint32_t qbf = ni & 1;
        qa = sbase + qd::QD_OFF + qbf * 2 * TILE;
        wait(B_(qd::QFULL + qbf), (ni >> 1) & 1, SITE_TC_FULL);
        issue_sd(c);
        for (int i = 0; i < nst; ++i, ++c) {
          if (i + 1 < nst) issue_sd(c + 1);
          else mma_commit(B_(qd::QEMPTY + qbf));              // Q and dO are free after the last S, dP
          const uint32_t st = c % qd::NST, sb = c & 1, sa = sbase + qd::ST_OFF + st * qd::ST_BYTES;
          wait(B_(qd::DSFULL + sb), (c >> 1) & 1, SITE_TC_FULL);
          if (i == 0) wait(B_(qd::ACCEMPTY), (ni & 1) ^ 1, SITE_TC_ACC_EMPTY);
          tc_fence_after();
          const uint64_t dds = sdesc(sbase + qd::DS_OFF + sb * TILE, 16, 1024), dkm = sdesc(sa, 8192, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tc.tmem_base + qd::TM_DQ, sdesc_add(dds, kk * 32), sdesc_add(dkm, kk * 2048), id_acc,
                     (i > 0 || kk > 0) ? 1u : 0u);
          mma_commit(B_(qd::DSEMPTY + sb));
          mma_commit(B_(qd::STEMPTY + st));
          last_bar = B_(qd::STEMPTY + st);
          last_par = (c / qd::NST) & 1;
        }
        mma_commit(B_(qd::ACCFULL));
      }
      if (last_bar && !dead && !mbar_wait(last_bar, last_par, tmo)) set_error(j.hdr, MT_ERR_DEVICE_TIMEOUT, SITE_TC_DRAIN);
      if (ni > 0) wait(B_(qd::QEMPTY + ((ni - 1) & 1)), ((ni - 1) >> 1) & 1, SITE_TC_DRAIN);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------- softmax and output: one query row per thread ----------------
    const int q = warp - 4, r = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const float sc_l2 = j.scale * LOG2E;
    const uint64_t sc2 = f2(sc_l2, sc_l2);
    uint32_t c = 0, ni = 0;
    for (int rnd_ = 0, it = first; it < items; it = snake_item(first, G, ++rnd_), ++ni) {
      int b, h, qb;
      item_of(it, b, h, qb);
      const int nst = 2 * (qb + 1);
      const int query = qb * 128 + r;
      const long long lrow = ((long long)b * j.H + h) * j.S + query;
      const float lse2 = j.lse[lrow], dd = j.dsum[lrow];
      const uint64_t nl2 = f2(-lse2, -lse2), dd2 = f2(dd, dd);
      for (int i = 0; i < nst; ++i, ++c) {
        const uint32_t sb = c & 1;
        wait(B_(qd::SDFULL + sb), (c >> 1) & 1, SITE_TC_ACC_FULL);
        __syncwarp();
        tc_fence_after();
        uint32_t sv[64], dp[64];
        tmem_ld32_async(tc.tmem_base + lane_off + qd::TM_S + sb * 64, sv);
        tmem_ld32_async(tc.tmem_base + lane_off + qd::TM_S + sb * 64 + 32, sv + 32);
        tmem_ld32_async(tc.tmem_base + lane_off + qd::TM_DP + sb * 64, dp);
        tmem_ld32_async(tc.tmem_base + lane_off + qd::TM_DP + sb * 64 + 32, dp + 32);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(B_(qd::SDEMPTY + sb));
        // keys i*64 + x > query are masked
        const int lim = query - i * 64;        // x > lim is masked
        wait(B_(qd::DSEMPTY + sb), ((c >> 1) & 1) ^ 1, SITE_TC_EMPTY);
        const uint32_t db = sbase + qd::DS_OFF + sb * TILE;
        // dS of the step; the mask only touches the last two steps
        auto soft = [&](auto MASKc) {
          constexpr bool MASK = decltype(MASKc)::value;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            uint32_t wd[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const int x = g * 8 + e;
              float t0, t1;
              unf2(fma2(u2(sv[x], sv[x + 1]), sc2, nl2), t0, t1);
              float p0 = ex2(t0), p1 = ex2(t1);
              if (MASK) {
                if (x > lim) p0 = 0.f;
                if (x + 1 > lim) p1 = 0.f;
              }
              float d0, d1;
              unf2(mul2(f2(p0, p1), sub2(u2(dp[x], dp[x + 1]), dd2)), d0, d1);
              wd[e >> 1] = pack2(d0, d1);
            }
            st_shared_v4(db + p_chunk_off(r, g * 8), wd[0], wd[1], wd[2], wd[3]);
          }
        };
        if (i >= nst - 2) soft(std::true_type());
        else soft(std::false_type());
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(B_(qd::DSFULL + sb));
      }
      wait(B_(qd::ACCFULL), ni & 1, SITE_TC_ACC_FULL);
      __syncwarp();
      tc_fence_after();
      uint32_t vq[64];
      tmem_ld32_async(tc.tmem_base + lane_off + qd::TM_DQ, vq);
      tmem_ld32_async(tc.tmem_base + lane_off + qd::TM_DQ + 32, vq + 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(B_(qd::ACCEMPTY));
      float g[64];
#pragma unroll
      for (int x = 0; x < 64; ++x) g[x] = __uint_as_float(vq[x]);
      float4 cs[16];
      {
        const float4* tab = reinterpret_cast<const float4*>(j.rope + (long long)query * 64);
#pragma unroll
        for (int x = 0; x < 16; ++x) cs[x] = tab[x];
      }
      rope_undo(g, cs, j.scale);
      // the previous item's bulk store has read the staging rows
      const uint32_t bq = sbase + qd::OUT_OFF + (uint32_t)q * 4096u;
      if (lane == 0) bulk_wait_read<0>();
      __syncwarp();
      box_put_row64(bq, lane, g);
      fence_smem_async();
      __syncwarp();
      if (lane == 0 && !dead) {
        tma_store_2d(j.map_dqkv, bq, h * HD, b * j.S + qb * 128 + q * 32);
        bulk_commit();
      }
      __syncwarp();
    }
    // every dQ row has landed before the phase ends
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  __syncthreads();
  s.next(items);
}

// dQ as a product over the stored dS^T (the dK/dV job wrote every dS^T tile
// of the layer, a grid barrier before this job): dQ = dS K for 128 queries
// per item, 64-key steps.  dS is read MN-major in place (dS^T rows are keys),
// K MN-major from the q,k,v buffer; no exponential is recomputed.
namespace qs {
constexpr int NST = 6;                                // stages: dS 2 x 8 KB (64 keys x 2 x 64 queries) | K 8 KB
constexpr uint32_t ST_OFF = 1024;
constexpr uint32_t ST_BYTES = 24576;
constexpr uint32_t OUT_OFF = ST_OFF + NST * ST_BYTES; // 4 x 4 KB: each epilogue warp's dQ rows
constexpr uint32_t END = OUT_OFF + 4 * 4096;
static_assert(END <= MT_TC_SMEM, "dQ product tiles exceed the shared-memory window");
static_assert(OUT_OFF % 1024 == 0 && ST_BYTES % 1024 == 0, "swizzled tiles need 1024-byte alignment");
enum { STFULL = 0, STEMPTY = NST, ACCFULL = 2 * NST, ACCEMPTY = ACCFULL + 2, COUNT = ACCEMPTY + 2 };
}

static __device__ __noinline__ void dqs_job(const BwdJob& j, Sched& s, char* smem, const TcState& tc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  auto B_ = [&](int i) { return sbase + 8u * (uint32_t)i; };
  const long long tmo = j.timeout_ns;
  const int nqb = j.S / 128;
  const int items = j.B * j.H * nqb;
  const int first = s.first(), G = s.G;
  auto item_of = [&](int it, int& b, int& h, int& qb) {   // longest (last query blocks) first
    qb = nqb - 1 - it / (j.B * j.H);
    const int bh = it % (j.B * j.H);
    b = bh / j.H; h = bh % j.H;
  };
  if (threadIdx.x == 0) {
    for (int i = 0; i < qs::NST; ++i) { mbar_init(B_(qs::STFULL + i), 1); mbar_init(B_(qs::STEMPTY + i), 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(B_(qs::ACCFULL + i), 1); mbar_init(B_(qs::ACCEMPTY + i), 4); }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  bool dead = false;
  auto wait = [&](uint32_t b_, uint32_t par, int site) {
    if (!dead && !mbar_wait(b_, par, tmo)) { set_error(j.hdr, MT_ERR_DEVICE_TIMEOUT, site); dead = true; }
  };
  if (warp == 0) {
    if (lane == 0) {
      // the dS^T tiles were written by bulk stores of other CTAs before the barrier
      asm volatile("fence.proxy.async;" ::: "memory");
      const uint64_t pol = l2_evict_first();     // each dS^T tile is read once
      uint32_t c = 0;
      for (int rnd_ = 0, it = first; it < items; it = snake_item(first, G, ++rnd_)) {
        int b, h, qb;
        item_of(it, b, h, qb);
        const int nst = 2 * (qb + 1), bh = b * j.H + h;
        for (int i = 0; i < nst; ++i, ++c) {
          const uint32_t st = c % qs::NST, sa = sbase + qs::ST_OFF + st * qs::ST_BYTES;
          wait(B_(qs::STEMPTY + st), ((c / qs::NST) & 1) ^ 1, SITE_TC_EMPTY);
          mbar_expect_tx(B_(qs::STFULL + st), qs::ST_BYTES);
          tma_load_2d_hint(sa, j.map_dsl, qb * 128, bh * j.S + i * 64, B_(qs::STFULL + st), pol);
          tma_load_2d_hint(sa + 8192, j.map_dsl, qb * 128 + 64, bh * j.S + i * 64, B_(qs::STFULL + st), pol);
          tma_load_2d(sa + 16384, j.map_qkv, j.hq + h * HD, j.y0 + b * j.S + i * 64, B_(qs::STFULL + st));
        }
      }
      if (!dead)
        for (uint32_t x = c > qs::NST ? c - qs::NST : 0; x < c; ++x)
          wait(B_(qs::STFULL + x % qs::NST), (x / qs::NST) & 1, SITE_TC_DRAIN);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_q = idesc_bf16(128, 64, 1, 1);     // dS (MN-major) x K (MN-major)
      uint32_t c = 0, ni = 0, last_bar = 0, last_par = 0;
      for (int rnd_ = 0, it = first; it < items; it = snake_item(first, G, ++rnd_), ++ni) {
        int b, h, qb;
        item_of(it, b, h, qb);
        const int nst = 2 * (qb + 1);
        const uint32_t ab = ni & 1;
        wait(B_(qs::ACCEMPTY + ab), ((ni >> 1) & 1) ^ 1, SITE_TC_ACC_EMPTY);
        tc_fence_after();
        for (int i = 0; i < nst; ++i, ++c) {
          const uint32_t st = c % qs::NST, sa = sbase + qs::ST_OFF + st * qs::ST_BYTES;
          wait(B_(qs::STFULL + st), (c / qs::NST) & 1, SITE_TC_FULL);
          tc_fence_after();
          const uint64_t da = sdesc(sa, 8192, 1024), dk = sdesc(sa + 16384, 8192, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tc.tmem_base + ab * 64, sdesc_add(da, kk * 2048), sdesc_add(dk, kk * 2048), id_q,
                     (i > 0 || kk > 0) ? 1u : 0u);
          mma_commit(B_(qs::STEMPTY + st));
          last_bar = B_(qs::STEMPTY + st);
          last_par = (c / qs::NST) & 1;
        }
        mma_commit(B_(qs::ACCFULL + ab));
      }
      // the tensor core must be idle before the job returns
      if (last_bar && !dead && !mbar_wait(last_bar, last_par, tmo)) set_error(j.hdr, MT_ERR_DEVICE_TIMEOUT, SITE_TC_DRAIN);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------- output: one query row per thread ----------------
    const int q = warp - 4, r = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const uint32_t bq = sbase + qs::OUT_OFF + (uint32_t)q * 4096u;
    uint32_t ni = 0;
    for (int rnd_ = 0, it = first; it < items; it = snake_item(first, G, ++rnd_), ++ni) {
      int b, h, qb;
      item_of(it, b, h, qb);
      const int query = qb * 128 + r;
      float4 cs[16];
      {
        const float4* tab = reinterpret_cast<const float4*>(j.rope + (long long)query * 64);
#pragma unroll
        for (int x = 0; x < 16; ++x) cs[x] = tab[x];
      }
      const uint32_t ab = ni & 1;
      wait(B_(qs::ACCFULL + ab), (ni >> 1) & 1, SITE_TC_ACC_FULL);
      __syncwarp();
      tc_fence_after();
      uint32_t vq[64];
      tmem_ld32_async(tc.tmem_base + lane_off + ab * 64, vq);
      tmem_ld32_async(tc.tmem_base + lane_off + ab * 64 + 32, vq + 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(B_(qs::ACCEMPTY + ab));
      float g[64];
#pragma unroll
      for (int x = 0; x < 64; ++x) g[x] = __uint_as_float(vq[x]);
      rope_undo(g, cs, j.scale);
      // the previous item's bulk store has read the staging rows
      if (lane == 0) bulk_wait_read<0>();
      __syncwarp();
      box_put_row64(bq, lane, g);
      fence_smem_async();
      __syncwarp();
      if (lane == 0 && !dead) {
        tma_store_2d(j.map_dqkv, bq, h * HD, b * j.S + qb * 128 + q * 32);
        bulk_commit();
      }
      __syncwarp();
    }
    // every dQ row has landed before the phase ends
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  __syncthreads();
  s.next(items);
}

}  // namespace attn_tm
