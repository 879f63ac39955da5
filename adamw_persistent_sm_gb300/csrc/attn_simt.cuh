// attn_simt.cuh - causal attention forward and backward on CUDA cores (fp32
// arithmetic), one 64-row block of one (batch, head) per work item.
//
// The pages' bf16_sdpa.sdpa ("How a training megakernel works", section
// "1 - Describe the model and update"): o = softmax(q k^T / sqrt(hd) with
// keys j <= query i) v, saving the row log-sum-exp for the backward pass.
// The backward pass recomputes P from the saved log-sum-exp and runs as two
// independent item families - dK/dV per key block and dQ per query block -
// so every output element is written once, in a fixed order, without
// atomics.
#pragma once
#include "common.cuh"

#define AT_B 64

struct AttnArgs {
  const void* qkv;     // op [T][3hq]: q, k after RoPE, v
  void* o;             // op [T][hq]
  float* lse;          // [B*H][S]
  const void* dout;    // op [T][hq]
  void* dqkv;          // op [T][3hq] (dq, dk with RoPE undone)
  const float* rope;   // [S][hd/2][2]
  int B, H, S, hq;
  float scale;
};

template <class OP, int HD>
__device__ void load_tile(float* dst, int ld_dst, const OP* src, long long ld_src, int row0, int nrows_valid) {
  for (int e = threadIdx.x; e < AT_B * HD; e += MT_THREADS) {
    const int r = e / HD, c = e % HD;
    dst[r * ld_dst + c] = (r < nrows_valid) ? to_f(src[(long long)(row0 + r) * ld_src + c]) : 0.f;
  }
}

// ---------------------------------------------------------------------------
template <class OP, int HD>
__device__ void attn_fwd_item(const AttnArgs& a, int b, int h, int qb, float* sm) {
  constexpr int LD = HD + 1;
  constexpr int DPT = HD / 4;            // output dims per thread
  float* Qs = sm;
  float* Ks = Qs + AT_B * LD;
  float* Vs = Ks + AT_B * LD;
  float* Ps = Vs + AT_B * LD;            // [64][65]
  const int tid = threadIdx.x, r = tid >> 2, sub = tid & 3;
  const int S = a.S, hq = a.hq;
  const long long ld = 3LL * hq;
  const OP* base = (const OP*)a.qkv + (long long)b * S * ld;
  const int q0 = qb * AT_B;
  const int qi = q0 + r;
  load_tile<OP, HD>(Qs, LD, base + h * HD, ld, q0, S - q0);
  float m = -INFINITY, l = 0.f, o[DPT];
#pragma unroll
  for (int i = 0; i < DPT; ++i) o[i] = 0.f;
  for (int kt = 0; kt <= qb; ++kt) {
    const int k0 = kt * AT_B;
    __syncthreads();
    load_tile<OP, HD>(Ks, LD, base + hq + h * HD, ld, k0, S - k0);
    load_tile<OP, HD>(Vs, LD, base + 2 * hq + h * HD, ld, k0, S - k0);
    __syncthreads();
    float s[16];
    float mx = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      const int j = sub + 4 * jj, kj = k0 + j;
      float acc = 0.f;
#pragma unroll
      for (int d = 0; d < HD; ++d) acc = fmaf(Qs[r * LD + d], Ks[j * LD + d], acc);
      acc *= a.scale;
      s[jj] = (kj <= qi && kj < S) ? acc : -INFINITY;
      mx = fmaxf(mx, s[jj]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mnew = fmaxf(m, mx);
    const float corr = (m == -INFINITY) ? 0.f : expf(m - mnew);
    float ls = 0.f;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      const float p = (s[jj] == -INFINITY) ? 0.f : expf(s[jj] - mnew);
      Ps[r * 65 + sub + 4 * jj] = p;
      ls += p;
    }
    ls += __shfl_xor_sync(0xffffffffu, ls, 1);
    ls += __shfl_xor_sync(0xffffffffu, ls, 2);
    l = l * corr + ls;
    m = mnew;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < DPT; ++i) o[i] *= corr;
    for (int j = 0; j < AT_B; ++j) {
      const float p = Ps[r * 65 + j];
#pragma unroll
      for (int i = 0; i < DPT; ++i) o[i] = fmaf(p, Vs[j * LD + sub * DPT + i], o[i]);
    }
  }
  if (qi < S) {
    OP* orow = (OP*)a.o + ((long long)b * S + qi) * hq + h * HD + sub * DPT;
    const float inv = 1.f / l;
#pragma unroll
    for (int i = 0; i < DPT; ++i) orow[i] = from_f<OP>(o[i] * inv);
    if (sub == 0) a.lse[((long long)b * a.H + h) * S + qi] = m + logf(l);
  }
  __syncthreads();
}

// D_i = sum_d dO[i][d] * O[i][d] for the 64 rows of a query block, into Ds.
template <class OP, int HD>
__device__ void attn_rowdot(const AttnArgs& a, int b, int h, int q0, float* Ds) {
  const int tid = threadIdx.x, r = tid >> 2, sub = tid & 3;
  constexpr int DPT = HD / 4;
  float acc = 0.f;
  if (q0 + r < a.S) {
    const long long row = (long long)b * a.S + q0 + r;
    const OP* orow = (const OP*)a.o + row * a.hq + h * HD + sub * DPT;
    const OP* drow = (const OP*)a.dout + row * a.hq + h * HD + sub * DPT;
#pragma unroll
    for (int i = 0; i < DPT; ++i) acc = fmaf(to_f(orow[i]), to_f(drow[i]), acc);
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  if (sub == 0) Ds[r] = acc;
}

// Undo the rotary embedding on the DPT dims this thread owns; the partner
// dims (i +- hd/2) belong to lane ^ 2.
template <int HD>
__device__ __forceinline__ void rope_undo(float* v, const float* tab, int pos, int sub) {
  constexpr int DPT = HD / 4, HALF = HD / 2;
#pragma unroll
  for (int i = 0; i < DPT; ++i) {
    const float other = __shfl_xor_sync(0xffffffffu, v[i], 2);
    const int dim = sub * DPT + i;
    const int fi = dim % HALF;
    const float c = tab[((long long)pos * HALF + fi) * 2 + 0];
    const float s = tab[((long long)pos * HALF + fi) * 2 + 1];
    // forward: y1 = x1 c - x2 s, y2 = x2 c + x1 s; transpose:
    // dx1 = d1 c + d2 s, dx2 = d2 c - d1 s
    v[i] = (dim < HALF) ? (v[i] * c + other * s) : (v[i] * c - other * s);
  }
}

template <class OP, int HD>
__device__ void attn_bwd_dkdv_item(const AttnArgs& a, int b, int h, int kb, float* sm) {
  constexpr int LD = HD + 1;
  constexpr int DPT = HD / 4;
  float* Ks = sm;
  float* Vs = Ks + AT_B * LD;
  float* Qs = Vs + AT_B * LD;
  float* dOs = Qs + AT_B * LD;
  float* Ps = dOs + AT_B * LD;    // [64 keys][65]
  float* DSs = Ps + AT_B * 65;    // [64 keys][65]
  float* Ls = DSs + AT_B * 65;    // [64]
  float* Ds = Ls + AT_B;          // [64]
  const int tid = threadIdx.x, r = tid >> 2, sub = tid & 3;
  const int S = a.S, hq = a.hq;
  const long long ld = 3LL * hq;
  const OP* base = (const OP*)a.qkv + (long long)b * S * ld;
  const OP* dbase = (const OP*)a.dout + (long long)b * S * hq;
  const int k0 = kb * AT_B, kj = k0 + r;
  load_tile<OP, HD>(Ks, LD, base + hq + h * HD, ld, k0, S - k0);
  load_tile<OP, HD>(Vs, LD, base + 2 * hq + h * HD, ld, k0, S - k0);
  float dk[DPT], dv[DPT];
#pragma unroll
  for (int i = 0; i < DPT; ++i) dk[i] = dv[i] = 0.f;
  const int nqb = (S + AT_B - 1) / AT_B;
  for (int qb = kb; qb < nqb; ++qb) {
    const int q0 = qb * AT_B;
    __syncthreads();
    load_tile<OP, HD>(Qs, LD, base + h * HD, ld, q0, S - q0);
    load_tile<OP, HD>(dOs, LD, dbase + h * HD, hq, q0, S - q0);
    attn_rowdot<OP, HD>(a, b, h, q0, Ds);
    if (tid < AT_B) Ls[tid] = (q0 + tid < S) ? a.lse[((long long)b * a.H + h) * S + q0 + tid] : 0.f;
    __syncthreads();
#pragma unroll 4
    for (int ii = 0; ii < 16; ++ii) {
      const int i = sub + 4 * ii, qi = q0 + i;
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int d = 0; d < HD; ++d) {
        s = fmaf(Qs[i * LD + d], Ks[r * LD + d], s);
        dp = fmaf(dOs[i * LD + d], Vs[r * LD + d], dp);
      }
      const bool valid = (kj <= qi) && (qi < S) && (kj < S);
      const float p = valid ? expf(s * a.scale - Ls[i]) : 0.f;
      Ps[r * 65 + i] = p;
      DSs[r * 65 + i] = p * (dp - Ds[i]);
    }
    __syncwarp();
    for (int i = 0; i < AT_B; ++i) {
      const float p = Ps[r * 65 + i], ds = DSs[r * 65 + i];
#pragma unroll
      for (int t = 0; t < DPT; ++t) {
        dv[t] = fmaf(p, dOs[i * LD + sub * DPT + t], dv[t]);
        dk[t] = fmaf(ds, Qs[i * LD + sub * DPT + t], dk[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < DPT; ++t) dk[t] *= a.scale;
  rope_undo<HD>(dk, a.rope, kj < S ? kj : 0, sub);
  if (kj < S) {
    OP* row = (OP*)a.dqkv + ((long long)b * S + kj) * ld;
#pragma unroll
    for (int t = 0; t < DPT; ++t) {
      row[hq + h * HD + sub * DPT + t] = from_f<OP>(dk[t]);
      row[2 * hq + h * HD + sub * DPT + t] = from_f<OP>(dv[t]);
    }
  }
  __syncthreads();
}

template <class OP, int HD>
__device__ void attn_bwd_dq_item(const AttnArgs& a, int b, int h, int qb, float* sm) {
  constexpr int LD = HD + 1;
  constexpr int DPT = HD / 4;
  float* Qs = sm;
  float* dOs = Qs + AT_B * LD;
  float* Ks = dOs + AT_B * LD;
  float* Vs = Ks + AT_B * LD;
  float* DSs = Vs + AT_B * LD;    // [64 q][65]
  float* Ls = DSs + AT_B * 65;
  float* Ds = Ls + AT_B;
  const int tid = threadIdx.x, r = tid >> 2, sub = tid & 3;
  const int S = a.S, hq = a.hq;
  const long long ld = 3LL * hq;
  const OP* base = (const OP*)a.qkv + (long long)b * S * ld;
  const OP* dbase = (const OP*)a.dout + (long long)b * S * hq;
  const int q0 = qb * AT_B, qi = q0 + r;
  load_tile<OP, HD>(Qs, LD, base + h * HD, ld, q0, S - q0);
  load_tile<OP, HD>(dOs, LD, dbase + h * HD, hq, q0, S - q0);
  attn_rowdot<OP, HD>(a, b, h, q0, Ds);
  if (tid < AT_B) Ls[tid] = (q0 + tid < S) ? a.lse[((long long)b * a.H + h) * S + q0 + tid] : 0.f;
  float dq[DPT];
#pragma unroll
  for (int i = 0; i < DPT; ++i) dq[i] = 0.f;
  for (int kb = 0; kb <= qb; ++kb) {
    const int k0 = kb * AT_B;
    __syncthreads();
    load_tile<OP, HD>(Ks, LD, base + hq + h * HD, ld, k0, S - k0);
    load_tile<OP, HD>(Vs, LD, base + 2 * hq + h * HD, ld, k0, S - k0);
    __syncthreads();
    const float lse = Ls[r], Dr = Ds[r];
#pragma unroll 4
    for (int jj = 0; jj < 16; ++jj) {
      const int j = sub + 4 * jj, kj = k0 + j;
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int d = 0; d < HD; ++d) {
        s = fmaf(Qs[r * LD + d], Ks[j * LD + d], s);
        dp = fmaf(dOs[r * LD + d], Vs[j * LD + d], dp);
      }
      const bool valid = (kj <= qi) && (qi < S) && (kj < S);
      const float p = valid ? expf(s * a.scale - lse) : 0.f;
      DSs[r * 65 + j] = p * (dp - Dr);
    }
    __syncwarp();
    for (int j = 0; j < AT_B; ++j) {
      const float ds = DSs[r * 65 + j];
#pragma unroll
      for (int t = 0; t < DPT; ++t) dq[t] = fmaf(ds, Ks[j * LD + sub * DPT + t], dq[t]);
    }
  }
#pragma unroll
  for (int t = 0; t < DPT; ++t) dq[t] *= a.scale;
  rope_undo<HD>(dq, a.rope, qi < S ? qi : 0, sub);
  if (qi < S) {
    OP* row = (OP*)a.dqkv + ((long long)b * S + qi) * ld;
#pragma unroll
    for (int t = 0; t < DPT; ++t) row[h * HD + sub * DPT + t] = from_f<OP>(dq[t]);
  }
  __syncthreads();
}

template <class OP, int HD>
__device__ __noinline__ void attn_fwd_job(const AttnArgs& a, Sched& s, float* sm) {
  const int nqb = (a.S + AT_B - 1) / AT_B;
  const int items = a.B * a.H * nqb;
  for (int it = s.first(); it < items; it += s.G) {
    const int qb = nqb - 1 - it / (a.B * a.H);       // longest rows first
    const int bh = it % (a.B * a.H);
    attn_fwd_item<OP, HD>(a, bh / a.H, bh % a.H, qb, sm);
  }
  s.next(items);
}

template <class OP, int HD>
__device__ __noinline__ void attn_bwd_job(const AttnArgs& a, Sched& s, float* sm) {
  const int nqb = (a.S + AT_B - 1) / AT_B;
  const int per = a.B * a.H * nqb;
  const int items = 2 * per;
  for (int it = s.first(); it < items; it += s.G) {
    // interleave the two families, heaviest blocks first
    const int fam = it & 1, j = it >> 1;
    const int step = j / (a.B * a.H), bh = j % (a.B * a.H);
    if (fam == 0) attn_bwd_dkdv_item<OP, HD>(a, bh / a.H, bh % a.H, step, sm);
    else attn_bwd_dq_item<OP, HD>(a, bh / a.H, bh % a.H, nqb - 1 - step, sm);
  }
  s.next(items);
}
