// attn_tc.cuh - causal attention on tensor cores (bf16 operands, fp32
// accumulation and softmax) for head_dim 64: the pages' bf16_sdpa.sdpa
// ("How a training megakernel works", section "1 - Describe the model and
// update"; long-sequence attention is "Open problems", Performance item 4).
//
// Forward: one item = 128 query rows of one (batch, head); 8 warps own 16
// rows each; 64-key blocks of K and V are staged in XOR-swizzled shared
// memory (cp.async), S = Q K^T and O += P V run as mma.sync m16n8k16 with
// ldmatrix operands; the softmax is online in registers (exp2 domain) and
// the row log-sum-exp is saved.
// Backward (P recomputed from the log-sum-exp, D = rowsum(dO * O) from the
// dO product's epilogue), two item families so that every output is
// written once without atomics:
//   dK/dV: 128 keys per item (16 per warp), loop over 64-query blocks;
//   dQ   : 128 queries per item (16 per warp), loop over 64-key blocks.
// The rotary embedding is undone on dq and dk before they are stored.
#pragma once
#include "common.cuh"
#include "attn_simt.cuh"

namespace attn_tc {

typedef __nv_bfloat16 bf;
constexpr int HD = 64;
constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ uint32_t s_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// c[4] += a[4] (16x16, row) * b (16x8, col)
__device__ __forceinline__ void mma(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Tile of `rows` x 64 bf16 (128-byte rows); the 16-byte chunk c of row r is
// stored at chunk c ^ (r & 7) so that ldmatrix row groups hit distinct banks.
__device__ __forceinline__ uint32_t sw(uint32_t base, int r, int col) {
  return base + r * 128 + ((((col >> 3) ^ r) & 7) << 4) + ((col & 7) << 1);
}
__device__ __forceinline__ void load_tile(uint32_t base, const bf* g, long long ld, int rows) {
  for (int c = threadIdx.x; c < rows * 8; c += MT_THREADS) {
    const int r = c >> 3, ch = c & 7;
    cp_async16(base + r * 128 + (((ch ^ r) & 7) << 4), g + (long long)r * ld + ch * 8);
  }
}
// A fragment (16 x 16) at rows r0.., cols k0.. of a swizzled tile
__device__ __forceinline__ void frag_a(uint32_t base, int r0, int k0, uint32_t* a) {
  const int l = threadIdx.x & 31;
  ldsm_x4(sw(base, r0 + (l & 7) + ((l >> 3) & 1) * 8, k0 + (l >> 4) * 8), a);
}
// B fragments of n-tiles n0 and n0+8 (k16 at k0) from a tile stored [n][k]
__device__ __forceinline__ void frag_b(uint32_t base, int n0, int k0, uint32_t* b) {
  const int l = threadIdx.x & 31;
  ldsm_x4(sw(base, n0 + (l & 7) + (l >> 4) * 8, k0 + ((l >> 3) & 1) * 8), b);
}
// B fragments of n-tiles n0 and n0+8 (k16 at k0) from a tile stored [k][n]
__device__ __forceinline__ void frag_bt(uint32_t base, int k0, int n0, uint32_t* b) {
  const int l = threadIdx.x & 31;
  ldsm_x4_t(sw(base, k0 + (l & 7) + ((l >> 3) & 1) * 8, n0 + (l >> 4) * 8), b);
}
// C (16 x 64, 8 n-tiles) += A (16 x 64 along k, 4 frags) * B; B from tile [n][k] (trans = false)
// or [k][n] (trans = true), n and k both 64 wide.
template <bool TRANS>
__device__ __forceinline__ void mm16x64x64(float (*c)[4], const uint32_t (*a)[4], uint32_t bbase) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      uint32_t b[4];
      if (TRANS) frag_bt(bbase, kk * 16, np * 16, b);
      else frag_b(bbase, np * 16, kk * 16, b);
      mma(c[2 * np], a[kk], b[0], b[1]);
      mma(c[2 * np + 1], a[kk], b[2], b[3]);
    }
  }
}
// C accumulator (16 x 64 fp32) -> four bf16 A fragments along k
__device__ __forceinline__ void c_to_a(const float (*c)[4], uint32_t (*a)[4]) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    a[kk][0] = pack_bf16(c[2 * kk][0], c[2 * kk][1]);
    a[kk][1] = pack_bf16(c[2 * kk][2], c[2 * kk][3]);
    a[kk][2] = pack_bf16(c[2 * kk + 1][0], c[2 * kk + 1][1]);
    a[kk][3] = pack_bf16(c[2 * kk + 1][2], c[2 * kk + 1][3]);
  }
}
__device__ __forceinline__ void zero(float (*c)[4]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.f;
}

// Undo the rotary embedding on a 16 x 64 accumulator (rows row0 + g and
// row0 + g + 8, positions pos0, pos1): dim i pairs with i + 32, i.e. n-tile
// j with n-tile j + 4 of the same thread.
__device__ __forceinline__ void rope_undo_frag(float (*c)[4], const float* tab, int pos0, int pos1) {
  const int t = threadIdx.x & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = j * 8 + 2 * t + (e & 1);
      const int pos = (e < 2) ? pos0 : pos1;
      const float cs = tab[((long long)pos * 32 + i) * 2 + 0];
      const float sn = tab[((long long)pos * 32 + i) * 2 + 1];
      const float d1 = c[j][e], d2 = c[j + 4][e];
      c[j][e] = d1 * cs + d2 * sn;
      c[j + 4][e] = d2 * cs - d1 * sn;
    }
}
// store a 16 x 64 fp32 accumulator as bf16 rows (row stride ld)
__device__ __forceinline__ void store_frag(bf* base, long long ld, const float (*c)[4]) {
  const int l = threadIdx.x & 31, g = l >> 2, t = l & 3;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    *reinterpret_cast<uint32_t*>(base + (long long)g * ld + j * 8 + 2 * t) = pack_bf16(c[j][0], c[j][1]);
    *reinterpret_cast<uint32_t*>(base + (long long)(g + 8) * ld + j * 8 + 2 * t) = pack_bf16(c[j][2], c[j][3]);
  }
}

struct Args {
  const bf* qkv;   // [T][3hq]
  bf* o;           // [T][hq]
  float* lse;      // [B*H][S]
  const bf* dout;  // [T][hq]
  const float* dsum;  // [B*H][S] rowsum(dO * O)
  bf* dqkv;        // [T][3hq]
  const float* rope;  // [S][32][2]
  int B, H, S, hq;
  float scale;
};

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ---------------------------------------------------------------------------
// Every loop below double-buffers its streamed tiles: block i+1 is fetched
// with cp.async while block i is multiplied.
static __device__ void fwd_item(const Args& a, int b, int h, int qb, char* smem) {
  const uint32_t sQ = s_u32(smem);
  const uint32_t sKV = sQ + 128 * 128;                 // [2][K 64 rows | V 64 rows]
  const int warp = threadIdx.x >> 5, l = threadIdx.x & 31, g = l >> 2, t = l & 3;
  const long long ld = 3LL * a.hq;
  const bf* base = a.qkv + (long long)b * a.S * ld;
  const int q0 = qb * 128, qw = q0 + warp * 16;
  const int nkb = (q0 + 128) / 64;
  auto fetch = [&](int kb) {
    const uint32_t buf = sKV + (kb & 1) * (2 * 64 * 128);
    load_tile(buf, base + (long long)kb * 64 * ld + a.hq + h * HD, ld, 64);
    load_tile(buf + 64 * 128, base + (long long)kb * 64 * ld + 2 * a.hq + h * HD, ld, 64);
    cp_async_commit();
  };
  load_tile(sQ, base + (long long)q0 * ld + h * HD, ld, 128);
  fetch(0);
  uint32_t qa[4][4];
  float o[8][4];
  zero(o);
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const float sc = a.scale * LOG2E;
  for (int kb = 0; kb < nkb; ++kb) {
    if (kb + 1 < nkb) { fetch(kb + 1); cp_async_wait<1>(); }
    else cp_async_wait<0>();
    __syncthreads();
    if (kb == 0) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) frag_a(sQ, warp * 16, kk * 16, qa[kk]);
    }
    const int k0 = kb * 64;
    const uint32_t sK = sKV + (kb & 1) * (2 * 64 * 128), sV = sK + 64 * 128;
    if (k0 <= qw + 15) {                 // some key of this block precedes this warp's rows
      float s[8][4];
      zero(s);
      mm16x64x64<false>(s, qa, sK);
      const bool diag = (k0 + 63 > qw);
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = s[j][e] * sc;
          if (diag) {
            const int key = k0 + j * 8 + 2 * t + (e & 1);
            const int row = qw + g + ((e >> 1) << 3);
            if (key > row) v = -INFINITY;
          }
          s[j][e] = v;
          if (e < 2) mx0 = fmaxf(mx0, v); else mx1 = fmaxf(mx1, v);
        }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float nm0 = fmaxf(m0, mx0), nm1 = fmaxf(m1, mx1);
      const float c0 = (m0 == -INFINITY) ? 0.f : exp2f(m0 - nm0);
      const float c1 = (m1 == -INFINITY) ? 0.f : exp2f(m1 - nm1);
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        s[j][0] = exp2f(s[j][0] - nm0);
        s[j][1] = exp2f(s[j][1] - nm0);
        s[j][2] = exp2f(s[j][2] - nm1);
        s[j][3] = exp2f(s[j][3] - nm1);
        ls0 += s[j][0] + s[j][1];
        ls1 += s[j][2] + s[j][3];
      }
      ls0 += __shfl_xor_sync(0xffffffffu, ls0, 1);
      ls0 += __shfl_xor_sync(0xffffffffu, ls0, 2);
      ls1 += __shfl_xor_sync(0xffffffffu, ls1, 1);
      ls1 += __shfl_xor_sync(0xffffffffu, ls1, 2);
      l0 = l0 * c0 + ls0;
      l1 = l1 * c1 + ls1;
      m0 = nm0;
      m1 = nm1;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        o[j][0] *= c0; o[j][1] *= c0; o[j][2] *= c1; o[j][3] *= c1;
      }
      uint32_t pa[4][4];
      c_to_a(s, pa);
      mm16x64x64<true>(o, pa, sV);
    }
    __syncthreads();                     // buffer kb & 1 is refilled by the next iteration's fetch
  }
  const float i0 = 1.f / l0, i1 = 1.f / l1;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    o[j][0] *= i0; o[j][1] *= i0; o[j][2] *= i1; o[j][3] *= i1;
  }
  store_frag(a.o + ((long long)b * a.S + qw) * a.hq + h * HD, a.hq, o);
  if (t == 0) {
    float* L = a.lse + ((long long)b * a.H + h) * a.S;
    L[qw + g] = (m0 + log2f(l0)) / LOG2E;
    L[qw + g + 8] = (m1 + log2f(l1)) / LOG2E;
  }
}

// dQ for 128 query rows
static __device__ void dq_item(const Args& a, int b, int h, int qb, char* smem) {
  const uint32_t sQ = s_u32(smem), sD = sQ + 128 * 128;
  const uint32_t sKV = sD + 128 * 128;                 // [2][K 64 rows | V 64 rows]
  const int warp = threadIdx.x >> 5, l = threadIdx.x & 31, g = l >> 2, t = l & 3;
  const long long ld = 3LL * a.hq;
  const bf* base = a.qkv + (long long)b * a.S * ld;
  const int q0 = qb * 128, qw = q0 + warp * 16;
  const int nkb = (q0 + 128) / 64;
  auto fetch = [&](int kb) {
    const uint32_t buf = sKV + (kb & 1) * (2 * 64 * 128);
    load_tile(buf, base + (long long)kb * 64 * ld + a.hq + h * HD, ld, 64);
    load_tile(buf + 64 * 128, base + (long long)kb * 64 * ld + 2 * a.hq + h * HD, ld, 64);
    cp_async_commit();
  };
  load_tile(sQ, base + (long long)q0 * ld + h * HD, ld, 128);
  load_tile(sD, a.dout + ((long long)b * a.S + q0) * a.hq + h * HD, a.hq, 128);
  fetch(0);
  const float* Lr = a.lse + ((long long)b * a.H + h) * a.S;
  const float lse0 = Lr[qw + g] * LOG2E, lse1 = Lr[qw + g + 8] * LOG2E;
  const float* Dr = a.dsum + ((long long)b * a.H + h) * a.S;
  const float D0 = Dr[qw + g], D1 = Dr[qw + g + 8];
  uint32_t qa[4][4], da[4][4];
  float dq[8][4];
  zero(dq);
  const float sc = a.scale * LOG2E;
  for (int kb = 0; kb < nkb; ++kb) {
    if (kb + 1 < nkb) { fetch(kb + 1); cp_async_wait<1>(); }
    else cp_async_wait<0>();
    __syncthreads();
    if (kb == 0) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        frag_a(sQ, warp * 16, kk * 16, qa[kk]);
        frag_a(sD, warp * 16, kk * 16, da[kk]);
      }
    }
    const int k0 = kb * 64;
    const uint32_t sK = sKV + (kb & 1) * (2 * 64 * 128), sV = sK + 64 * 128;
    if (k0 <= qw + 15) {
      float s[8][4], dp[8][4];
      zero(s);
      zero(dp);
      mm16x64x64<false>(s, qa, sK);
      mm16x64x64<false>(dp, da, sV);
      const bool diag = (k0 + 63 > qw);
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = k0 + j * 8 + 2 * t + (e & 1);
          const int row = qw + g + ((e >> 1) << 3);
          float p = exp2f(s[j][e] * sc - ((e >> 1) ? lse1 : lse0));
          if (diag && key > row) p = 0.f;
          s[j][e] = p * (dp[j][e] - ((e >> 1) ? D1 : D0));
        }
      uint32_t sa[4][4];
      c_to_a(s, sa);
      mm16x64x64<true>(dq, sa, sK);
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    dq[j][0] *= a.scale; dq[j][1] *= a.scale; dq[j][2] *= a.scale; dq[j][3] *= a.scale;
  }
  rope_undo_frag(dq, a.rope, qw + g, qw + g + 8);
  store_frag(a.dqkv + ((long long)b * a.S + qw) * (3LL * a.hq) + h * HD, 3LL * a.hq, dq);
}

// dK and dV for 128 keys
static __device__ void dkdv_item(const Args& a, int b, int h, int kb, char* smem) {
  const uint32_t sK = s_u32(smem), sV = sK + 128 * 128;
  const uint32_t sQD = sV + 128 * 128;                  // [2][Q 64 rows | dO 64 rows]
  float* sLD = reinterpret_cast<float*>(smem + 2 * 128 * 128 + 2 * 2 * 64 * 128);   // [2][lse 64 | D 64]
  const int warp = threadIdx.x >> 5, l = threadIdx.x & 31, g = l >> 2, t = l & 3;
  const long long ld = 3LL * a.hq;
  const bf* base = a.qkv + (long long)b * a.S * ld;
  const int k0 = kb * 128, kw = k0 + warp * 16;
  const float* Lr = a.lse + ((long long)b * a.H + h) * a.S;
  const float* Dr = a.dsum + ((long long)b * a.H + h) * a.S;
  const int nqb = (a.S - k0) / 64;
  auto fetch = [&](int i) {
    const int q0 = k0 + i * 64;
    const uint32_t buf = sQD + (i & 1) * (2 * 64 * 128);
    load_tile(buf, base + (long long)q0 * ld + h * HD, ld, 64);
    load_tile(buf + 64 * 128, a.dout + ((long long)b * a.S + q0) * a.hq + h * HD, a.hq, 64);
    cp_async_commit();
    float* ldbuf = sLD + (i & 1) * 128;
    if (threadIdx.x < 64) {
      ldbuf[threadIdx.x] = Lr[q0 + threadIdx.x] * LOG2E;
      ldbuf[64 + threadIdx.x] = Dr[q0 + threadIdx.x];
    }
  };
  load_tile(sK, base + (long long)k0 * ld + a.hq + h * HD, ld, 128);
  load_tile(sV, base + (long long)k0 * ld + 2 * a.hq + h * HD, ld, 128);
  fetch(0);
  uint32_t ka[4][4], va[4][4];
  float dk[8][4], dv[8][4];
  zero(dk);
  zero(dv);
  const float sc = a.scale * LOG2E;
  for (int i = 0; i < nqb; ++i) {
    if (i + 1 < nqb) { fetch(i + 1); cp_async_wait<1>(); }
    else cp_async_wait<0>();
    __syncthreads();
    if (i == 0) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        frag_a(sK, warp * 16, kk * 16, ka[kk]);
        frag_a(sV, warp * 16, kk * 16, va[kk]);
      }
    }
    const int q0 = k0 + i * 64;
    const uint32_t sQ = sQD + (i & 1) * (2 * 64 * 128), sD = sQ + 64 * 128;
    const float* sL = sLD + (i & 1) * 128;
    const float* sDs = sL + 64;
    if (q0 + 63 >= kw) {                 // some query of this block follows this warp's keys
      float s[8][4], dp[8][4];
      zero(s);
      zero(dp);
      mm16x64x64<false>(s, ka, sQ);      // S^T: keys x queries
      mm16x64x64<false>(dp, va, sD);     // dP^T
      const bool diag = (q0 < kw + 15);
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int qi = j * 8 + 2 * t + (e & 1);
          const int key = kw + g + ((e >> 1) << 3);
          float p = exp2f(s[j][e] * sc - sL[qi]);
          if (diag && q0 + qi < key) p = 0.f;
          s[j][e] = p;
          dp[j][e] = p * (dp[j][e] - sDs[qi]);
        }
      uint32_t pa[4][4], dsa[4][4];
      c_to_a(s, pa);
      c_to_a(dp, dsa);
      mm16x64x64<true>(dv, pa, sD);
      mm16x64x64<true>(dk, dsa, sQ);
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    dk[j][0] *= a.scale; dk[j][1] *= a.scale; dk[j][2] *= a.scale; dk[j][3] *= a.scale;
  }
  rope_undo_frag(dk, a.rope, kw + g, kw + g + 8);
  bf* row = a.dqkv + ((long long)b * a.S + kw) * (3LL * a.hq);
  store_frag(row + a.hq + h * HD, 3LL * a.hq, dk);
  store_frag(row + 2 * a.hq + h * HD, 3LL * a.hq, dv);
}

}  // namespace attn_tc

// Dynamic scheduling and dependency counters of the attention jobs (all
// null: static rotation, phases fenced by grid barriers).
struct AttnDeps {
  unsigned* ticket;        // item numbers are drawn from this counter
  const unsigned* wait;    // per 128-row block of q,k,v: stored column tiles
  unsigned wtarget;
  unsigned* sig;           // per 128-row block of the output: +1 per stored head
  ArenaHdr* hdr;
  long long timeout_ns;
};

// Item number k of this CTA: a drawn ticket, or the static rotation.
__device__ __forceinline__ int attn_next_item(const AttnDeps& dp, const Sched& s, int k) {
  return dp.ticket ? draw_ticket(dp.ticket) : s.first() + k * s.G;
}

template <class OP>
__device__ void attn_tc_fwd_job(const attn_tc::Args& a, Sched& s, char* smem, const AttnDeps& dp) {
  const int nqb = a.S / 128;
  const int items = a.B * a.H * nqb;
  for (int k = 0;; ++k) {
    const int it = attn_next_item(dp, s, k);
    if (it >= items) break;
    int b, h, qb;
    if (dp.ticket) {
      // sequence by sequence (following the q,k,v product's row order),
      // longest rows first within a sequence
      b = it / (a.H * nqb);
      const int r = it % (a.H * nqb);
      qb = nqb - 1 - r / a.H; h = r % a.H;
    } else {
      // static rotation: longest rows first over the whole batch
      qb = nqb - 1 - it / (a.B * a.H);
      const int bh = it % (a.B * a.H);
      b = bh / a.H; h = bh % a.H;
    }
    if (dp.wait) {
      if (threadIdx.x <= qb) dep_wait(dp.hdr, dp.wait + b * nqb + threadIdx.x, dp.wtarget, dp.timeout_ns);
      __syncthreads();
    }
    attn_tc::fwd_item(a, b, h, qb, smem);
    __syncthreads();
    if (dp.sig && threadIdx.x == 0) dep_signal(dp.sig + b * nqb + qb);
  }
  s.next(items);
}

template <class OP>
__device__ void attn_tc_bwd_job(const attn_tc::Args& a, Sched& s, char* smem, const AttnDeps& dp) {
  const int nb = a.S / 128;
  const int per = a.B * a.H * nb;
  const int items = 2 * per;
  for (int k = 0;; ++k) {
    const int it = attn_next_item(dp, s, k);
    if (it >= items) break;
    // dK,dV items and dQ items alternate, longest first
    const int fam = it & 1, j = it >> 1;
    const int step = j / (a.B * a.H), bh = j % (a.B * a.H);
    if (fam == 0) attn_tc::dkdv_item(a, bh / a.H, bh % a.H, step, smem);
    else attn_tc::dq_item(a, bh / a.H, bh % a.H, nb - 1 - step, smem);
    __syncthreads();
  }
  s.next(items);
}
