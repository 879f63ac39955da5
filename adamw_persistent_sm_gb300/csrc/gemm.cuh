// gemm.cuh - one description of every matrix product of the update, and the
// CUDA-core implementation (exact fp32 FMAs; used for the fp32 tiny model
// and as a cross-check of the tensor-core path).
//
// D[m, n] = sum_k A(m, k) * B(n, k), followed by a fused epilogue.
// Three shapes occur ("How a training megakernel works", section "1 -
// Describe the model and update": dense products and ragged_mm):
//   dense     - one M x N x K product;
//   ragged M  - rows of A / D are split into expert segments (padded to 128
//               rows by route_order); B is the segment's expert weight;
//   ragged K  - the reduction runs over one expert's rows (weight
//               gradients); D is the expert's gradient tensor.
#pragma once
#include "common.cuh"

enum EpiKind {
  EPI_STORE_OP = 0,   // out(op)[m][n] = acc
  EPI_STORE_F32,      // out(f32)[m][n] = acc
  EPI_RESID,          // out(f32)[m][n] = aux(f32)[m][n] + acc
  EPI_ROPE,           // out(op) = acc with rotary embedding on the q and k columns
  EPI_SWIGLU,         // tile = [64 gate | 64 up] columns -> g, u (out) and silu(g)*u (out2)
  EPI_SWIGLU_BWD,     // acc = d(silu(g)*u); aux = [g | u] -> out = [dg | du]
  EPI_GRAD,           // out(f32) = acc (+ out if accumulate); rows >= osplit go to out1
  EPI_STORE_OP_D,     // out(op) = acc, and out2(f32)[batch][head][position] of row m = sum over the
                      // head's 64 columns of op(acc) * aux(op)  (attention's D = rowsum(dO * O));
                      // ldo2 = number of heads, S = positions per sequence
  EPI_NONE,           // test harness: accumulators are read and dropped
  EPI_LOGITS          // out(op) = acc (LM-head logits); per row and column tile, (max, sum exp(acc -
                      // max)) into cepart[m][n0 / tile width]; the target token's fp32 logit into cetgt[m]
};

enum RagKind { RAG_NONE = 0, RAG_M = 1, RAG_K = 2 };

// One operand: element (r, k) where r indexes rows of A (m) or of B (n).
struct GOperand {
  const void* p0;
  const void* p1;       // second source (two-source weights)
  long long ld;         // row stride of the 2-D storage, elements
  long long seg;        // element offset per expert segment (ragged-M B operand)
  int mn;               // 0: (r,k) at p[r*ld + k] (K-major); 1: at p[k*ld + r] (MN-major)
  int two;              // 0 single source; 1 rows interleaved by 64 between p0/p1;
                        // 2 reduction split: k >= split reads p1 at k - split
  int split;
  // tensor-map coordinates (tcgen05 path): map index and outer-coordinate base
  int map0, map1;
  int y0;               // outer (row) coordinate of element (0,0) in map0/map1
  int yseg;             // outer-coordinate step per expert segment
  int rows_per_box = 64; // K-major single-source operands: rows per TMA box of map0 (64, 128 or 256)
};

struct GemmDesc {
  int M, N, K;
  int rag;              // RagKind
  const int* offs;      // [nseg + 1] padded segment starts (ragged kinds)
  int nseg;
  GOperand A, B;
  int epi;
  void* out; long long ldo; long long oseg;   // ragged K: output offset per segment
  void* out1; int osplit;                     // EPI_GRAD: rows >= osplit -> out1
  void* out2; long long ldo2;                 // EPI_SWIGLU: silu(g)*u
  const void* aux; long long ldaux;           // EPI_RESID (f32) / EPI_SWIGLU_BWD ([g|u], op)
  int accumulate;                             // EPI_GRAD: add into out
  int F;                                      // expert width (swiglu epilogues)
  int S, hd, hq;                              // EPI_ROPE
  const float* rope;                          // [S][hd/2][2] cos, sin
  const int* tok;                             // EPI_LOGITS: token ids (target of row m = tok[m + 1])
  float* cepart;                              // EPI_LOGITS: [M][ceparts][2]
  float* cetgt;                               // EPI_LOGITS: [M]
  int ceparts;
  int ksplit;                                 // tensor-core path, dense products: the K range is cut
                                              // into ksplit slices, slice s writes out + s * oseg
  // Dependency counters (tensor-core path; null where a grid barrier fences
  // the product), one per 128-row block:
  const unsigned* dwait; unsigned dtarget;    // A rows: wait before loading a tile's operands
  const unsigned* dwait_aux; unsigned dtarget_aux;  // aux rows: wait before the epilogue reads aux
  unsigned* dsig;                             // output rows: +1 per stored tile
  // Epilogue tensor maps (tensor-core path; -1: plain stores / loads):
  // out and out2 by bulk tensor stores, aux by bulk tensor loads.  Row m of
  // the product is row y0 + m of the map.
  int omap, omap2, amap;
  int oy0, oy02, ay0;
  // Tile order (tensor-core path): null - tile t on CTA (t + base) % G;
  // else tiles are drawn from this counter (zero at the start of the launch)
  // by the CTAs as they become free.
  unsigned* ticket;
};

// Target column of logits row m (next token), or -1 for the last position.
__device__ __forceinline__ int ce_target(const GemmDesc& g, int m) {
  if (m % g.S == g.S - 1) return -1;
  const int v = g.tok[m + 1];
  return (v >= 0 && v < g.N) ? v : 0;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }
__device__ __forceinline__ float silu_grad_f(float g) {
  float s = 1.0f / (1.0f + expf(-g));
  return s * (1.0f + g * (1.0f - s));
}

// Element (r, k) of an operand, segment `seg`, as float.  Out-of-range
// elements (r >= rmax or k >= kmax) read as zero.
template <class OP>
__device__ __forceinline__ float op_elem(const GOperand& o, int seg, int r, int k, int rmax, int kmax) {
  if (r >= rmax || k >= kmax) return 0.f;
  const OP* p = (const OP*)o.p0;
  long long rr = r, kk = k;
  if (o.two == 1) {
    if ((r >> 6) & 1) p = (const OP*)o.p1;
    rr = ((long long)(r >> 7) << 6) | (r & 63);
  } else if (o.two == 2 && k >= o.split) {
    p = (const OP*)o.p1;
    kk = k - o.split;
  }
  p += (long long)seg * o.seg;
  return to_f(o.mn ? p[kk * o.ld + rr] : p[rr * o.ld + kk]);
}

// Segment of a row of a ragged-M product / number of tiles.
__device__ __forceinline__ int seg_of_row(const int* offs, int nseg, int row) {
  int e = 0;
  while (e + 1 < nseg && offs[e + 1] <= row) ++e;
  return e;
}

// ---------------------------------------------------------------------------
// Epilogue on one output element group (shared by the SIMT and tcgen05 paths)
// ---------------------------------------------------------------------------
// Rotary embedding on a pair (x_i, x_{i+hd/2}) at position pos.
__device__ __forceinline__ void rope_pair(const float* tab, int hd, int pos, int i, float x1, float x2,
                                          float& y1, float& y2) {
  const float c = tab[((long long)pos * (hd / 2) + i) * 2 + 0];
  const float s = tab[((long long)pos * (hd / 2) + i) * 2 + 1];
  y1 = x1 * c - x2 * s;
  y2 = x2 * c + x1 * s;
}

template <class OP>
__device__ __forceinline__ void grad_store(const GemmDesc& g, int seg, int m, int n, float v) {
  float* out = (float*)g.out;
  int mm = m;
  if (g.osplit > 0 && m >= g.osplit) { out = (float*)g.out1; mm = m - g.osplit; }
  out += (long long)seg * g.oseg;
  float* p = out + (long long)mm * g.ldo + n;
  *p = g.accumulate ? (*p + v) : v;
}

// SIMT tile: 64 x 128 outputs, BK = 16, 256 threads each owning 4 rows x 8 cols.
#define SG_BM 64
#define SG_BN 128
#define SG_BK 16
#define SG_CPAD 132

template <class OP>
__device__ void gemm_simt_tile(const GemmDesc& g, int seg, int m0, int n0, int k0, int k1,
                               int mmax, float* sm) {
  float* As = sm;                        // [BK][BM]
  float* Bs = sm + SG_BK * SG_BM;        // [BK][BN]
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  const int bseg = (g.rag == RAG_M) ? seg : 0;
  for (int k = k0; k < k1; k += SG_BK) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int e = tid + i * 256;
      int r, kk;
      if (!g.A.mn) { r = e >> 4; kk = e & 15; } else { kk = e >> 6; r = e & 63; }
      As[kk * SG_BM + r] = op_elem<OP>(g.A, 0, m0 + r, k + kk, mmax, k1);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int e = tid + i * 256;
      int r, kk;
      if (!g.B.mn) { r = e >> 4; kk = e & 15; } else { kk = e >> 7; r = e & 127; }
      Bs[kk * SG_BN + r] = op_elem<OP>(g.B, bseg, n0 + r, k + kk, g.N, k1);
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SG_BK; ++kk) {
      float a[4], b[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk * SG_BM + ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b[j] = Bs[kk * SG_BN + tx * 4 + j];
        b[4 + j] = Bs[kk * SG_BN + 64 + tx * 4 + j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  // stage the tile so that every epilogue sees whole tile rows
  float* Cs = sm;   // [BM][CPAD], aliases the operand tiles
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      Cs[(ty * 4 + i) * SG_CPAD + tx * 4 + j] = acc[i][j];
      Cs[(ty * 4 + i) * SG_CPAD + 64 + tx * 4 + j] = acc[i][4 + j];
    }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  if (g.epi == EPI_LOGITS) {
    for (int r = warp; r < SG_BM; r += MT_WARPS) {
      const int m = m0 + r;
      if (m >= mmax) continue;
      const float* crow = Cs + r * SG_CPAD;
      const int tgt = ce_target(g, m);
      float mx = -INFINITY;
      for (int c = lane; c < SG_BN; c += 32) {
        const int n = n0 + c;
        if (n >= g.N) continue;
        ((OP*)g.out)[(long long)m * g.ldo + n] = from_f<OP>(crow[c]);
        mx = fmaxf(mx, crow[c]);
        if (n == tgt) g.cetgt[m] = crow[c];
      }
      mx = warp_max(mx);
      float sm = 0.f;
      for (int c = lane; c < SG_BN; c += 32)
        if (n0 + c < g.N) sm += expf(crow[c] - mx);
      sm = warp_sum(sm);
      if (lane == 0) {
        float* pp = g.cepart + ((long long)m * g.ceparts + n0 / SG_BN) * 2;
        pp[0] = mx;
        pp[1] = sm;
      }
    }
    __syncthreads();
    return;
  }
  if (g.epi == EPI_STORE_OP_D) {
    // 64-column heads: lane owns columns lane, lane+32 of each head
    for (int r = warp; r < SG_BM; r += MT_WARPS) {
      const int m = m0 + r;
      if (m >= mmax) continue;
      const float* crow = Cs + r * SG_CPAD;
      for (int hh = 0; hh < SG_BN / 64; ++hh) {
        float dot = 0.f;
        for (int c = hh * 64 + lane; c < hh * 64 + 64; c += 32) {
          const int n = n0 + c;
          if (n >= g.N) continue;
          const OP q = from_f<OP>(crow[c]);
          ((OP*)g.out)[(long long)m * g.ldo + n] = q;
          dot = fmaf(to_f(q), to_f(((const OP*)g.aux)[(long long)m * g.ldaux + n]), dot);
        }
        dot = warp_sum(dot);
        const int n = n0 + hh * 64;
        if (lane == 0 && n < g.N)
          ((float*)g.out2)[((long long)(m / g.S) * g.ldo2 + n / 64) * g.S + (m % g.S)] = dot;
      }
    }
    __syncthreads();
    return;
  }
  for (int r = warp; r < SG_BM; r += MT_WARPS) {
    const int m = m0 + r;
    if (m >= mmax) continue;
    const float* crow = Cs + r * SG_CPAD;
    for (int c = lane; c < SG_BN; c += 32) {
      const int n = n0 + c;
      const float v = crow[c];
      switch (g.epi) {
        case EPI_STORE_OP:
          if (n < g.N) ((OP*)g.out)[(long long)m * g.ldo + n] = from_f<OP>(v);
          break;
        case EPI_STORE_F32:
          if (n < g.N) ((float*)g.out)[(long long)m * g.ldo + n] = v;
          break;
        case EPI_RESID:
          if (n < g.N)
            ((float*)g.out)[(long long)m * g.ldo + n] =
                ((const float*)g.aux)[(long long)m * g.ldaux + n] + v;
          break;
        case EPI_ROPE: {
          if (n >= g.N) break;
          float y = v;
          if (n < 2 * g.hq) {
            const int i = n % g.hd, half = g.hd / 2;
            const int pos = m % g.S;
            if (i < half) {
              float y2;
              rope_pair(g.rope, g.hd, pos, i, v, crow[c + half], y, y2);
            } else {
              float y1;
              rope_pair(g.rope, g.hd, pos, i - half, crow[c - half], v, y1, y);
            }
          }
          ((OP*)g.out)[(long long)m * g.ldo + n] = from_f<OP>(y);
          break;
        }
        case EPI_SWIGLU: {
          if (c >= 64) break;
          const int f = (n0 >> 7) * 64 + c;
          if (f >= g.F) break;
          const float gg = v, uu = crow[c + 64];
          OP* gu = (OP*)g.out + (long long)m * g.ldo;
          gu[f] = from_f<OP>(gg);
          gu[g.F + f] = from_f<OP>(uu);
          ((OP*)g.out2)[(long long)m * g.ldo2 + f] = from_f<OP>(silu_f(gg) * uu);
          break;
        }
        case EPI_SWIGLU_BWD: {
          if (n >= g.N) break;
          const OP* gu = (const OP*)g.aux + (long long)m * g.ldaux;
          const float gg = to_f(gu[n]), uu = to_f(gu[g.F + n]);
          OP* d = (OP*)g.out + (long long)m * g.ldo;
          d[n] = from_f<OP>(v * uu * silu_grad_f(gg));
          d[g.F + n] = from_f<OP>(v * silu_f(gg));
          break;
        }
        case EPI_GRAD:
          if (n < g.N) grad_store<OP>(g, seg, m, n, v);
          break;
      }
    }
  }
  __syncthreads();
}

// Number of (M-tile, N-tile[, segment]) items for a tile shape.
__device__ __forceinline__ int gemm_items(const GemmDesc& g, int bm, int bn) {
  const int nt = (g.N + bn - 1) / bn;
  if (g.rag == RAG_M) return (g.offs[g.nseg] / bm) * nt;
  const int mt = (g.M + bm - 1) / bm;
  if (g.rag == RAG_K) return g.nseg * mt * nt;
  return mt * nt;
}

template <class OP>
__device__ __noinline__ void gemm_simt_job(const GemmDesc& g, Sched& s, float* sm) {
  const int nt = (g.N + SG_BN - 1) / SG_BN;
  const int items = gemm_items(g, SG_BM, SG_BN);
  for (int it = s.first(); it < items; it += s.G) {
    if (g.rag == RAG_K) {
      const int mt = (g.M + SG_BM - 1) / SG_BM;
      const int seg = it / (mt * nt);
      const int rem = it % (mt * nt);
      const int m0 = (rem / nt) * SG_BM, n0 = (rem % nt) * SG_BN;
      gemm_simt_tile<OP>(g, seg, m0, n0, g.offs[seg], g.offs[seg + 1], g.M, sm);
    } else {
      const int m0 = (it / nt) * SG_BM, n0 = (it % nt) * SG_BN;
      const int mmax = g.rag == RAG_M ? g.offs[g.nseg] : g.M;
      const int seg = g.rag == RAG_M ? seg_of_row(g.offs, g.nseg, m0) : 0;
      gemm_simt_tile<OP>(g, seg, m0, n0, 0, g.K, mmax, sm);
    }
  }
  s.next(items);
}
