// mega.cuh - the persistent training-update megakernel.
//
// One cooperative launch per microbatch, one CTA per SM, resident for the
// whole update ("How a training megakernel works", section "What Latch does":
// forward pass, loss, backward pass and weight update in one persistent GPU
// program).  The program at the bottom is a fixed sequence of phases; inside
// a phase every CTA takes work items of one or more jobs, and a grid-wide
// barrier separates phases whose results cross SMs (section "4 - Scheduling
// and storage").  Values that cross phases live in the caller's arena.
//
// OP is the operand type of the matrix products and attention: float for the
// exact-fp32 model, __nv_bfloat16 for the policy of the same section (FP32
// master weights and Adam moments, BF16 matrix products and attention).
#pragma once
#include "common.cuh"
#include "gemm.cuh"
#include "attn_simt.cuh"
#include "gemm_tc.cuh"

template <class T>
__device__ __forceinline__ T* abuf(const KArgs& a, int id) {
  return reinterpret_cast<T*>(a.arena + a.aoff[id]);
}
__device__ __forceinline__ const float* pmaster(const KArgs& a, int pid) { return a.master + a.poff[pid]; }
template <class OP>
__device__ __forceinline__ const OP* pweight(const KArgs& a, int pid) {
  if constexpr (sizeof(OP) == 4) return (const OP*)(a.master + a.poff[pid]);
  else return (const OP*)a.shadow + a.poff[pid];
}
__device__ __forceinline__ float* pgrad(const KArgs& a, int pid) { return a.grads + a.poff[pid]; }

// token chunk owned by CTA c in chunked jobs (routing, column reductions)
__device__ __forceinline__ int chunk_len(const MtDims& D, int G) { return (D.T + G - 1) / G; }

__device__ __forceinline__ float warp_rms_inv(const float* x, int d, float eps) {
  const int lane = threadIdx.x & 31;
  float ss = 0.f;
  for (int i = lane; i < d; i += 32) ss = fmaf(x[i], x[i], ss);
  ss = warp_sum(ss);
  return 1.0f / sqrtf(ss / (float)d + eps);
}

// ===========================================================================
// forward row jobs
// ===========================================================================
// Rotary table (angles in double precision) and x0 = emb[tok], plus the
// first layer's attention RMSNorm.
template <class OP>
__device__ void job_embed(const KArgs& a, Sched& s) {
  const MtDims& D = a.D;
  const int half = D.hd / 2;
  float* rope = abuf<float>(a, A_ROPE);
  const int me = s.first();
  for (int e = me * MT_THREADS + threadIdx.x; e < D.S * half; e += s.G * MT_THREADS) {
    const int pos = e / half, i = e % half;
    const double freq = pow((double)a.rope_theta, -2.0 * (double)i / (double)D.hd);
    double sv, cv;
    sincos((double)pos * freq, &sv, &cv);
    rope[2 * e] = (float)cv;
    rope[2 * e + 1] = (float)sv;
  }
  const int lane = threadIdx.x & 31;
  ArenaHdr* hdr = abuf<ArenaHdr>(a, A_HDR);
  const float* emb = pmaster(a, P_EMB);
  const float* g = pmaster(a, P_ATTN_NORM);
  float* X = abuf<float>(a, A_X);
  OP* R = abuf<OP>(a, A_R);
  float* inv1 = abuf<float>(a, A_INV1);
  const int nw = s.G * MT_WARPS;
  for (int t = me * MT_WARPS + (threadIdx.x >> 5); t < D.T; t += nw) {
    int v = a.tokens[t];
    if (v < 0 || v >= D.V) {
      if (lane == 0) set_error(hdr, MT_ERR_DEVICE_BOUNDS, SITE_TOKEN_RANGE);
      v = 0;
    }
    float* x = X + (long long)t * D.d;
    const float* er = emb + (long long)v * D.d;
    for (int i = lane; i < D.d; i += 32) x[i] = er[i];
    const float inv = warp_rms_inv(x, D.d, a.norm_eps);
    for (int i = lane; i < D.d; i += 32) R[(long long)t * D.d + i] = from_f<OP>(x[i] * inv * g[i]);
    if (lane == 0) inv1[t] = inv;
  }
  s.next(s.G);
}

// Warp-wide arg-max with ties going to the lower index.
__device__ __forceinline__ void warp_argmax(float& v, int& idx) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
    if (ov > v || (ov == v && oi < idx)) { v = ov; idx = oi; }
  }
}

// Expert RMSNorm, router logits, softmax and token_topk for CTA c's token
// chunk, then that chunk's per-expert counts (the histogram of route_order).
// Router logits use fp32 activations and fp32 master router weights; the
// top-k compares these fp32 logits (softmax is monotone), ties going to the
// lower expert index.
template <class OP>
__device__ void job_router(const KArgs& a, int l, float* sm) {
  const MtDims& D = a.D;
  const int c = blockIdx.x, G = gridDim.x;
  const int ch = chunk_len(D, G);
  const int t0 = c * ch, t1 = min(D.T, t0 + ch);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* XM = abuf<float>(a, A_XM) + (long long)l * D.T * D.d;
  float* inv2 = abuf<float>(a, A_INV2) + (long long)l * D.T;
  OP* R2 = abuf<OP>(a, A_R2) + (long long)l * D.T * D.d;
  float* Z = abuf<float>(a, A_Z) + (long long)l * D.T * D.E;
  int* IDX = abuf<int>(a, A_IDX) + (long long)l * D.T * D.K;
  float* WGT = abuf<float>(a, A_WGT) + (long long)l * D.T * D.K;
  const float* g = pmaster(a, P_MOE_NORM) + (long long)l * D.d;
  const float* Wr = pmaster(a, P_ROUTER) + (long long)l * D.E * D.d;
  float* row = sm + warp * D.d;
  for (int t = t0 + warp; t < t1; t += MT_WARPS) {
    const float* x = XM + (long long)t * D.d;
    const float inv = warp_rms_inv(x, D.d, a.norm_eps);
    for (int i = lane; i < D.d; i += 32) {
      const float r = x[i] * inv * g[i];
      row[i] = r;
      R2[(long long)t * D.d + i] = from_f<OP>(r);
    }
    __syncwarp();
    if (lane == 0) inv2[t] = inv;
    float z0 = -INFINITY, z1 = -INFINITY;   // experts lane and lane + 32
    for (int e = 0; e < D.E; ++e) {
      const float* w = Wr + (long long)e * D.d;
      float acc = 0.f;
      for (int i = lane; i < D.d; i += 32) acc = fmaf(row[i], w[i], acc);
      acc = warp_sum(acc);
      if (e == lane) z0 = acc;
      if (e == lane + 32) z1 = acc;
    }
    __syncwarp();
    if (lane < D.E) Z[(long long)t * D.E + lane] = z0;
    if (lane + 32 < D.E) Z[(long long)t * D.E + lane + 32] = z1;
    const float zmax = warp_max(fmaxf(z0, z1));
    const float p0 = (lane < D.E) ? expf(z0 - zmax) : 0.f;
    const float p1 = (lane + 32 < D.E) ? expf(z1 - zmax) : 0.f;
    // the softmax normaliser cancels in the renormalised weights
    float c0 = z0, c1 = z1;
    float chosen_p[8];
    int chosen_i[8];
    float psum = 0.f;
    for (int k = 0; k < D.K; ++k) {
      float v = c0;
      int idx = lane;
      if (c1 > v) { v = c1; idx = lane + 32; }
      warp_argmax(v, idx);
      chosen_i[k] = idx;
      const float pk = __shfl_sync(0xffffffffu, idx < 32 ? p0 : p1, idx & 31);
      chosen_p[k] = pk;
      psum += pk;
      if (idx == lane) c0 = -INFINITY;
      if (idx == lane + 32) c1 = -INFINITY;
    }
    if (lane == 0) {
      for (int k = 0; k < D.K; ++k) {
        IDX[(long long)t * D.K + k] = chosen_i[k];
        WGT[(long long)t * D.K + k] = chosen_p[k] / psum;
      }
    }
  }
  __syncthreads();
  if (t0 < D.T) {
    int* CNT = abuf<int>(a, A_CNT) + ((long long)l * D.nch + c) * D.E;
    for (int e = threadIdx.x; e < D.E; e += MT_THREADS) {
      int n = 0;
      for (int j = t0 * D.K; j < t1 * D.K; ++j) n += (IDX[j] == e);
      CNT[e] = n;
    }
  }
}

// route_order: stable counting sort of the T*K assignments by expert (the
// histogram comes from job_router), expert segments padded to MT_TILE_M rows,
// fused with the dispatch gather of the expert inputs.  Within an expert,
// assignments keep ascending a = t*K + k.
template <class OP>
__device__ void job_route(const KArgs& a, int l, int* ism) {
  const MtDims& D = a.D;
  const int c = blockIdx.x, G = gridDim.x;
  const int ch = chunk_len(D, G);
  const int nused = (D.T + ch - 1) / ch;
  const int t0 = c * ch, t1 = min(D.T, t0 + ch);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int* CNT = abuf<int>(a, A_CNT) + (long long)l * D.nch * D.E;
  int* OFFS = abuf<int>(a, A_OFFS) + (long long)l * (D.E + 1);
  int* PERM = abuf<int>(a, A_PERM) + (long long)l * D.Pmax;
  int* INVM = abuf<int>(a, A_INVM) + (long long)l * D.T * D.K;
  const int* IDX = abuf<int>(a, A_IDX) + (long long)l * D.T * D.K;
  const OP* R2 = abuf<OP>(a, A_R2) + (long long)l * D.T * D.d;
  OP* XS = abuf<OP>(a, A_XS) + (long long)l * D.Pmax * D.d;
  int* s_tot = ism;                 // [E]
  int* s_base = ism + 64;           // [E]
  int* s_offs = ism + 128;          // [E+1]
  for (int e = threadIdx.x; e < D.E; e += MT_THREADS) {
    int tot = 0, before = 0;
    for (int cc = 0; cc < nused; ++cc) {
      const int n = CNT[(long long)cc * D.E + e];
      tot += n;
      if (cc < c) before += n;
    }
    s_tot[e] = tot;
    s_base[e] = before;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int o = 0;
    for (int e = 0; e < D.E; ++e) {
      s_offs[e] = o;
      o += (s_tot[e] + MT_TILE_M - 1) / MT_TILE_M * MT_TILE_M;
    }
    s_offs[D.E] = o;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < D.E; e += MT_THREADS) s_base[e] += s_offs[e];
  if (c == 0) {
    for (int e = threadIdx.x; e <= D.E; e += MT_THREADS) OFFS[e] = s_offs[e];
    ArenaHdr* hdr = abuf<ArenaHdr>(a, A_HDR);
    if (l < MT_MAX_LAYERS)
      for (int e = threadIdx.x; e < D.E && e < MT_MAX_EXPERTS; e += MT_THREADS)
        hdr->expert_counts[l * MT_MAX_EXPERTS + e] = s_tot[e];
  }
  __syncthreads();
  // stable scatter of this chunk's assignments
  const int a0 = t0 * D.K, a1 = (t0 < D.T) ? t1 * D.K : a0;
  for (int e = warp; e < D.E; e += MT_WARPS) {
    int running = 0;
    const int base = s_base[e];
    for (int j0 = a0; j0 < a1; j0 += 32) {
      const int j = j0 + lane;
      const bool hit = (j < a1) && (IDX[j] == e);
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      if (hit) {
        const int pos = base + running + __popc(m & ((1u << lane) - 1u));
        PERM[pos] = j;
        INVM[j] = pos;
      }
      running += __popc(m);
    }
  }
  __syncthreads();
  // dispatch gather: XS[row] = R2[token]
  for (int j = a0 + warp; j < a1; j += MT_WARPS) {
    const int pos = INVM[j];
    const OP* src = R2 + (long long)(j / D.K) * D.d;
    OP* dst = XS + (long long)pos * D.d;
    for (int i = lane; i < D.d; i += 32) dst[i] = src[i];
  }
  // zero the pad rows of every segment (spread over all CTAs)
  const int gw = c * MT_WARPS + warp, nw = G * MT_WARPS;
  for (int e = 0; e < D.E; ++e) {
    const int p0 = s_offs[e] + s_tot[e], p1 = s_offs[e + 1];
    for (int p = p0 + gw; p < p1; p += nw) {
      OP* dst = XS + (long long)p * D.d;
      for (int i = lane; i < D.d; i += 32) dst[i] = from_f<OP>(0.f);
      if (lane == 0) PERM[p] = -1;
    }
  }
}

// x_{l+1} = x_mid + sum_k w_k y_k (fixed slot order), then the next
// RMSNorm (attention norm of layer l+1, or the final norm).
template <class OP>
__device__ void job_combine(const KArgs& a, int l, Sched& s) {
  const MtDims& D = a.D;
  const int lane = threadIdx.x & 31;
  const float* XM = abuf<float>(a, A_XM) + (long long)l * D.T * D.d;
  const float* Y = abuf<float>(a, A_Y) + (long long)l * D.Pmax * D.d;
  const float* WGT = abuf<float>(a, A_WGT) + (long long)l * D.T * D.K;
  const int* INVM = abuf<int>(a, A_INVM) + (long long)l * D.T * D.K;
  float* Xn = abuf<float>(a, A_X) + (long long)(l + 1) * D.T * D.d;
  const bool last = (l + 1 == D.L);
  const float* g = last ? pmaster(a, P_FINAL_NORM) : pmaster(a, P_ATTN_NORM) + (long long)(l + 1) * D.d;
  OP* Rn = last ? abuf<OP>(a, A_RF) : abuf<OP>(a, A_R) + (long long)(l + 1) * D.T * D.d;
  float* invn = last ? abuf<float>(a, A_INVF) : abuf<float>(a, A_INV1) + (long long)(l + 1) * D.T;
  const int nw = s.G * MT_WARPS;
  for (int t = s.first() * MT_WARPS + (threadIdx.x >> 5); t < D.T; t += nw) {
    float* x = Xn + (long long)t * D.d;
    const float* xm = XM + (long long)t * D.d;
    for (int i = lane; i < D.d; i += 32) {
      float acc = 0.f;
      for (int k = 0; k < D.K; ++k) {
        const int p = INVM[(long long)t * D.K + k];
        acc = fmaf(WGT[(long long)t * D.K + k], Y[(long long)p * D.d + i], acc);
      }
      x[i] = xm[i] + acc;
    }
    const float inv = warp_rms_inv(x, D.d, a.norm_eps);
    for (int i = lane; i < D.d; i += 32) Rn[(long long)t * D.d + i] = from_f<OP>(x[i] * inv * g[i]);
    if (lane == 0) invn[t] = inv;
  }
  s.next(s.G);
}

// Fused softmax cross-entropy with its gradient: per position, lse over the
// vocabulary, loss = coef * (lse - logit[target]) and
// dlogits = coef * (softmax - onehot).  Position s predicts token s+1; the
// last position of a sequence has no target (zero loss and gradient).
template <class OP>
__device__ void job_ce(const KArgs& a, Sched& s) {
  const MtDims& D = a.D;
  const int lane = threadIdx.x & 31;
  const float* LOG = abuf<float>(a, A_LOGITS);
  OP* DL = abuf<OP>(a, A_DLOGITS);
  float* TL = abuf<float>(a, A_TOKLOSS);
  const int nw = s.G * MT_WARPS;
  for (int t = s.first() * MT_WARPS + (threadIdx.x >> 5); t < D.T; t += nw) {
    const float* lg = LOG + (long long)t * D.V;
    OP* dl = DL + (long long)t * D.V;
    const bool has = (t % D.S) != D.S - 1;
    if (!has) {
      for (int j = lane; j < D.V; j += 32) dl[j] = from_f<OP>(0.f);
      if (lane == 0) TL[t] = 0.f;
      continue;
    }
    int target = a.tokens[t + 1];
    if (target < 0 || target >= D.V) target = 0;   // reported by job_embed; never read outside the row
    float m = -INFINITY, sum = 0.f;
    for (int j = lane; j < D.V; j += 32) {
      const float v = lg[j];
      if (v > m) { sum = sum * expf(m - v) + 1.f; m = v; }
      else sum += expf(v - m);
    }
    const float M = warp_max(m);
    sum = (m == -INFINITY) ? 0.f : sum * expf(m - M);
    sum = warp_sum(sum);
    const float lse = M + logf(sum);
    for (int j = lane; j < D.V; j += 32) {
      const float p = expf(lg[j] - lse);
      dl[j] = from_f<OP>(a.coef * (p - (j == target ? 1.f : 0.f)));
    }
    if (lane == 0) TL[t] = a.coef * (lse - lg[target]);
  }
  s.next(s.G);
}

// ===========================================================================
// backward row jobs
// ===========================================================================
// RMSNorm backward of one row: dx = inv * (a - xh * mean(a * xh)), a = dy*g.
// Adds into out (or overwrites when add == false).
__device__ __forceinline__ void warp_rmsnorm_bwd(const float* dy, const float* x, float inv,
                                                 const float* g, int d, float* out, bool add) {
  const int lane = threadIdx.x & 31;
  float dot = 0.f;
  for (int i = lane; i < d; i += 32) dot = fmaf(dy[i] * g[i], x[i] * inv, dot);
  dot = warp_sum(dot) / (float)d;
  for (int i = lane; i < d; i += 32) {
    const float v = inv * (dy[i] * g[i] - x[i] * inv * dot);
    out[i] = add ? out[i] + v : v;
  }
}

// dx = d(final RMSNorm) from d rf.
template <class OP>
__device__ void job_final_norm_bwd(const KArgs& a, Sched& s) {
  const MtDims& D = a.D;
  const float* DRF = abuf<float>(a, A_DRF);
  const float* X = abuf<float>(a, A_X) + (long long)D.L * D.T * D.d;
  const float* inv = abuf<float>(a, A_INVF);
  const float* g = pmaster(a, P_FINAL_NORM);
  float* DX = abuf<float>(a, A_DX);
  const int nw = s.G * MT_WARPS;
  for (int t = s.first() * MT_WARPS + (threadIdx.x >> 5); t < D.T; t += nw)
    warp_rmsnorm_bwd(DRF + (long long)t * D.d, X + (long long)t * D.d, inv[t], g, D.d,
                     DX + (long long)t * D.d, false);
  s.next(s.G);
}

// Expert-combine backward, part 1: dY[row] = w_k dx, dw_k = <dx, y_k>,
// router-logit gradient dz_i = w_i (dw_i - sum_j w_j dw_j) on the chosen
// experts (the renormalised weights are the softmax of the chosen logits),
// and zero pad rows of dY.
template <class OP>
__device__ void job_moe_bwd1(const KArgs& a, int l, Sched& s) {
  const MtDims& D = a.D;
  const int lane = threadIdx.x & 31;
  const float* DX = abuf<float>(a, A_DX);
  const float* Y = abuf<float>(a, A_Y) + (long long)l * D.Pmax * D.d;
  const float* WGT = abuf<float>(a, A_WGT) + (long long)l * D.T * D.K;
  const int* IDX = abuf<int>(a, A_IDX) + (long long)l * D.T * D.K;
  const int* INVM = abuf<int>(a, A_INVM) + (long long)l * D.T * D.K;
  const int* OFFS = abuf<int>(a, A_OFFS) + (long long)l * (D.E + 1);
  const int* PERM = abuf<int>(a, A_PERM) + (long long)l * D.Pmax;
  OP* DY = abuf<OP>(a, A_DY);
  float* DZ = abuf<float>(a, A_DZ);
  const int nw = s.G * MT_WARPS;
  const int me = s.first() * MT_WARPS + (threadIdx.x >> 5);
  for (int t = me; t < D.T; t += nw) {
    const float* dx = DX + (long long)t * D.d;
    float dw[8], w[8];
    for (int k = 0; k < D.K; ++k) {
      const int p = INVM[(long long)t * D.K + k];
      w[k] = WGT[(long long)t * D.K + k];
      const float* y = Y + (long long)p * D.d;
      OP* dy = DY + (long long)p * D.d;
      float acc = 0.f;
      for (int i = lane; i < D.d; i += 32) {
        acc = fmaf(dx[i], y[i], acc);
        dy[i] = from_f<OP>(w[k] * dx[i]);
      }
      dw[k] = warp_sum(acc);
    }
    float mean = 0.f;
    for (int k = 0; k < D.K; ++k) mean = fmaf(w[k], dw[k], mean);
    for (int e = lane; e < D.E; e += 32) {
      float v = 0.f;
      for (int k = 0; k < D.K; ++k)
        if (IDX[(long long)t * D.K + k] == e) v = w[k] * (dw[k] - mean);
      DZ[(long long)t * D.E + e] = v;
    }
  }
  // pad rows of dY: PERM == -1 inside [0, OFFS[E])
  const int nrows = OFFS[D.E];
  for (int p = me; p < nrows; p += nw) {
    if (PERM[p] >= 0) continue;
    OP* dy = DY + (long long)p * D.d;
    for (int i = lane; i < D.d; i += 32) dy[i] = from_f<OP>(0.f);
  }
  s.next(s.G);
}

// Expert-combine backward, part 2: the gather backward as a direct per-row
// sum (each token has exactly K contributions, summed in slot order, no
// atomics - "Open problems", Performance item 5), plus the router term
// dz Wr, then the expert RMSNorm backward into dx, and the operand copy of dx.
template <class OP>
__device__ void job_moe_bwd2(const KArgs& a, int l, Sched& s) {
  const MtDims& D = a.D;
  const int lane = threadIdx.x & 31;
  const float* DXS = abuf<float>(a, A_DXS);
  const float* DZ = abuf<float>(a, A_DZ);
  const int* INVM = abuf<int>(a, A_INVM) + (long long)l * D.T * D.K;
  const float* Wr = pmaster(a, P_ROUTER) + (long long)l * D.E * D.d;
  const float* XM = abuf<float>(a, A_XM) + (long long)l * D.T * D.d;
  const float* inv2 = abuf<float>(a, A_INV2) + (long long)l * D.T;
  const float* g = pmaster(a, P_MOE_NORM) + (long long)l * D.d;
  float* DR2 = abuf<float>(a, A_DR2);
  float* DX = abuf<float>(a, A_DX);
  OP* DXO = abuf<OP>(a, A_DXO);
  const int nw = s.G * MT_WARPS;
  for (int t = s.first() * MT_WARPS + (threadIdx.x >> 5); t < D.T; t += nw) {
    float* dr2 = DR2 + (long long)t * D.d;
    const float* dz = DZ + (long long)t * D.E;
    for (int i = lane; i < D.d; i += 32) {
      float acc = 0.f;
      for (int k = 0; k < D.K; ++k) acc += DXS[(long long)INVM[(long long)t * D.K + k] * D.d + i];
      float rz = 0.f;
      for (int e = 0; e < D.E; ++e) rz = fmaf(dz[e], Wr[(long long)e * D.d + i], rz);
      dr2[i] = acc + rz;
    }
    __syncwarp();
    float* dx = DX + (long long)t * D.d;
    warp_rmsnorm_bwd(dr2, XM + (long long)t * D.d, inv2[t], g, D.d, dx, true);
    __syncwarp();
    for (int i = lane; i < D.d; i += 32) DXO[(long long)t * D.d + i] = from_f<OP>(dx[i]);
  }
  s.next(s.G);
}

// Attention RMSNorm backward into dx.
template <class OP>
__device__ void job_attn_norm_bwd(const KArgs& a, int l, Sched& s) {
  const MtDims& D = a.D;
  const float* DR = abuf<float>(a, A_DR);
  const float* X = abuf<float>(a, A_X) + (long long)l * D.T * D.d;
  const float* inv = abuf<float>(a, A_INV1) + (long long)l * D.T;
  const float* g = pmaster(a, P_ATTN_NORM) + (long long)l * D.d;
  float* DX = abuf<float>(a, A_DX);
  const int nw = s.G * MT_WARPS;
  for (int t = s.first() * MT_WARPS + (threadIdx.x >> 5); t < D.T; t += nw)
    warp_rmsnorm_bwd(DR + (long long)t * D.d, X + (long long)t * D.d, inv[t], g, D.d,
                     DX + (long long)t * D.d, true);
  s.next(s.G);
}

// ===========================================================================
// deterministic column reductions over tokens (norm gains, router weights)
// ===========================================================================
// Partial sums over CTA chunk c of the tokens, in token order, written to
// PART[c][row][col]; a later phase adds the chunks in chunk order.
enum ColKind { COL_GAIN = 0, COL_MOE = 1 };
struct ColArgs {
  int kind;
  const float* dy;    // [T][d] gradient wrt the norm output
  const float* x;     // [T][d] norm input
  const float* inv;   // [T]
  const float* g;     // [d] gain (COL_MOE: r2 = x*inv*g for the router gradient)
  const float* dz;    // [T][E] (COL_MOE)
  int row0;           // first PART row written
};

static __device__ void job_colpart(const KArgs& a, const ColArgs& c, Sched& s) {
  const MtDims& D = a.D;
  const int G = s.G;
  const int ch = chunk_len(D, G);
  const int ncb = (D.d + 127) / 128;
  const int items = G * ncb;
  const int nrows = (c.kind == COL_MOE) ? D.E + 1 : 1;
  float* PART = abuf<float>(a, A_PART);
  const int col_l = threadIdx.x & 127, rg = threadIdx.x >> 7;   // 2 row groups
  for (int it = s.first(); it < items; it += G) {
    const int chunk = it / ncb, cb = it % ncb;
    const int col = cb * 128 + col_l;
    const int t0 = chunk * ch, t1 = min(D.T, t0 + ch);
    float acc[33];
#pragma unroll
    for (int r = 0; r < 33; ++r) acc[r] = 0.f;
    if (col < D.d) {
      for (int t = t0; t < t1; ++t) {
        const float xh = c.x[(long long)t * D.d + col] * c.inv[t];
        if (c.kind == COL_GAIN) {
          if (rg == 0) acc[0] = fmaf(c.dy[(long long)t * D.d + col], xh, acc[0]);
        } else {
          const float r2 = xh * c.g[col];
#pragma unroll
          for (int j = 0; j < 33; ++j) {
            const int e = rg + 2 * j;
            if (e < D.E) acc[j] = fmaf(c.dz[(long long)t * D.E + e], r2, acc[j]);
            else if (e == D.E) acc[j] = fmaf(c.dy[(long long)t * D.d + col], xh, acc[j]);
          }
        }
      }
      float* out = PART + ((long long)chunk * (D.E + 2) + c.row0) * D.d + col;
#pragma unroll
      for (int j = 0; j < 33; ++j) {
        const int r = rg + 2 * j;
        if (r < nrows) out[(long long)r * D.d] = acc[j];
      }
    }
  }
  s.next(items);
}

// out[r][col] (+)= sum over chunks of PART[chunk][row0 + r][col].
static __device__ void job_colfinal(const KArgs& a, int row0, int nrows, float* out_rows, float* out_last,
                             int last_is_separate, Sched& s) {
  const MtDims& D = a.D;
  const int G = s.G;
  const int ch = chunk_len(D, G);
  const int nused = (D.T + ch - 1) / ch;
  const float* PART = abuf<float>(a, A_PART);
  const int n = nrows * D.d;
  const bool acc = a.micro_index > 0;
  for (int e = s.first() * MT_THREADS + threadIdx.x; e < n; e += G * MT_THREADS) {
    const int r = e / D.d, col = e % D.d;
    float v = 0.f;
    for (int cc = 0; cc < nused; ++cc) v += PART[((long long)cc * (D.E + 2) + row0 + r) * D.d + col];
    float* dst = (last_is_separate && r == nrows - 1) ? out_last + col : out_rows + e;
    *dst = acc ? *dst + v : v;
  }
  s.next(G);
}

// ===========================================================================
// embedding backward: dE[v] (+)= sum over positions t with tok[t] = v of dx_t,
// in ascending t.  CTA c owns vocabulary rows [c*V/G, (c+1)*V/G).
// ===========================================================================
static __device__ void job_embed_bwd(const KArgs& a, int* ism) {
  const MtDims& D = a.D;
  const int c = blockIdx.x, G = gridDim.x;
  const int v0 = (int)((long long)D.V * c / G), v1 = (int)((long long)D.V * (c + 1) / G);
  float* dE = pgrad(a, P_EMB);
  const float* DX = abuf<float>(a, A_DX);
  if (a.micro_index == 0) {
    for (long long e = (long long)v0 * D.d + threadIdx.x; e < (long long)v1 * D.d; e += MT_THREADS) dE[e] = 0.f;
  }
  __syncthreads();
  int* flag = ism;   // [256]
  for (int tb = 0; tb < D.T; tb += MT_THREADS) {
    const int t = tb + threadIdx.x;
    int v = (t < D.T) ? a.tokens[t] : -1;
    flag[threadIdx.x] = (v >= v0 && v < v1) ? v : -1;
    __syncthreads();
    for (int j = 0; j < MT_THREADS; ++j) {
      const int vv = flag[j];
      if (vv < 0) continue;
      const float* dx = DX + (long long)(tb + j) * D.d;
      float* row = dE + (long long)vv * D.d;
      for (int i = threadIdx.x; i < D.d; i += MT_THREADS) row[i] += dx[i];
    }
    __syncthreads();
  }
}

// ===========================================================================
// loss reduction and optimizer
// ===========================================================================
static __device__ void job_loss(const KArgs& a) {
  if (blockIdx.x != 0 || threadIdx.x >= 32) return;
  const MtDims& D = a.D;
  const float* TL = abuf<float>(a, A_TOKLOSS);
  double acc = 0.0;
  for (int t = threadIdx.x; t < D.T; t += 32) acc += TL[t];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (threadIdx.x == 0) {
    ArenaHdr* h = abuf<ArenaHdr>(a, A_HDR);
    h->loss = (float)acc;
    h->loss_update = (a.micro_index == 0 ? 0.f : h->loss_update) + (float)acc;
  }
}

// Global gradient norm, first level: CTA c sums squares over its slice.
static __device__ void job_norm_partial(const KArgs& a, double* dsm) {
  const int c = blockIdx.x, G = gridDim.x;
  const long long n = a.n_params;
  const long long n4 = n / 4;
  const long long b0 = n4 * c / G, b1 = n4 * (c + 1) / G;
  const float4* g4 = reinterpret_cast<const float4*>(a.grads);
  double acc = 0.0;
  float facc = 0.f;
  int cnt = 0;
  for (long long i = b0 + threadIdx.x; i < b1; i += MT_THREADS) {
    const float4 v = g4[i];
    facc = fmaf(v.x, v.x, facc);
    facc = fmaf(v.y, v.y, facc);
    facc = fmaf(v.z, v.z, facc);
    facc = fmaf(v.w, v.w, facc);
    if (++cnt == 64) { acc += facc; facc = 0.f; cnt = 0; }
  }
  if (c == G - 1)
    for (long long i = n4 * 4 + threadIdx.x; i < n; i += MT_THREADS) facc = fmaf(a.grads[i], a.grads[i], facc);
  acc += facc;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) dsm[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < MT_WARPS; ++w) t += dsm[w];
    reinterpret_cast<double*>(abuf<float>(a, A_NORMPART))[c] = t;
  }
}

template <class OP>
__device__ __forceinline__ void adamw_elem(const KArgs& a, float c, float& p, float g, float& m, float& v) {
  g *= c;
  p *= 1.0f - a.lr * a.wd;
  m = a.beta1 * m + (1.0f - a.beta1) * g;
  v = a.beta2 * v + (1.0f - a.beta2) * g * g;
  const float mh = m / a.bc1;
  const float vh = v / a.bc2;
  p -= a.lr * mh / (sqrtf(vh) + a.eps);
}

// Clip coefficient from the ordered sum of the partials, then the AdamW sweep
// over CTA c's slice (float4 loads; writes p, m, v and the bf16 shadow).
template <class OP>
__device__ void job_adamw(const KArgs& a) {
  const int c = blockIdx.x, G = gridDim.x;
  const double* parts = reinterpret_cast<const double*>(abuf<float>(a, A_NORMPART));
  double tot = 0.0;
  for (int i = 0; i < G; ++i) tot += parts[i];
  const float norm = (float)sqrt(tot);
  const float coef = fminf(1.0f, a.clip / (norm + a.clip_eps));
  if (c == 0 && threadIdx.x == 0) {
    ArenaHdr* h = abuf<ArenaHdr>(a, A_HDR);
    h->grad_norm = norm;
    h->clip_coef = coef;
    h->optimizer_ran = 1;
  }
  const long long n = a.n_params;
  const long long n4 = n / 4;
  const long long b0 = n4 * c / G, b1 = n4 * (c + 1) / G;
  float4* p4 = reinterpret_cast<float4*>(a.master);
  const float4* g4 = reinterpret_cast<const float4*>(a.grads);
  float4* m4 = reinterpret_cast<float4*>(a.adam_m);
  float4* v4 = reinterpret_cast<float4*>(a.adam_v);
  __nv_bfloat16* sh = (sizeof(OP) == 2) ? (__nv_bfloat16*)a.shadow : nullptr;
  for (long long i = b0 + threadIdx.x; i < b1; i += MT_THREADS) {
    float4 p = p4[i], m = m4[i], v = v4[i];
    const float4 g = g4[i];
    adamw_elem<OP>(a, coef, p.x, g.x, m.x, v.x);
    adamw_elem<OP>(a, coef, p.y, g.y, m.y, v.y);
    adamw_elem<OP>(a, coef, p.z, g.z, m.z, v.z);
    adamw_elem<OP>(a, coef, p.w, g.w, m.w, v.w);
    p4[i] = p;
    m4[i] = m;
    v4[i] = v;
    if (sh) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(p.x, p.y), hi = __floats2bfloat162_rn(p.z, p.w);
      reinterpret_cast<__nv_bfloat162*>(sh)[2 * i] = lo;
      reinterpret_cast<__nv_bfloat162*>(sh)[2 * i + 1] = hi;
    }
  }
  if (c == G - 1) {
    for (long long i = n4 * 4 + threadIdx.x; i < n; i += MT_THREADS) {
      float p = a.master[i], m = a.adam_m[i], v = a.adam_v[i];
      adamw_elem<OP>(a, coef, p, a.grads[i], m, v);
      a.master[i] = p;
      a.adam_m[i] = m;
      a.adam_v[i] = v;
      if (sh) sh[i] = __float2bfloat16_rn(p);
    }
  }
}

// ===========================================================================
// matrix products of the update
// ===========================================================================
template <class OP>
struct Gemms {
  const KArgs& a;
  const MtDims& D;
  __device__ Gemms(const KArgs& a_) : a(a_), D(a_.D) {}

  __device__ GOperand opnd(const void* p, long long ld, int mn) const {
    GOperand o;
    o.p0 = p; o.p1 = nullptr; o.ld = ld; o.seg = 0; o.mn = mn; o.two = 0; o.split = 0;
    o.map0 = o.map1 = -1; o.y0 = 0; o.yseg = 0;
    return o;
  }
  __device__ GemmDesc base(int M, int N, int K, int epi) const {
    GemmDesc g;
    g.M = M; g.N = N; g.K = K; g.rag = RAG_NONE; g.offs = nullptr; g.nseg = 0; g.epi = epi;
    g.out = g.out1 = g.out2 = nullptr; g.ldo = g.ldo2 = 0; g.oseg = 0; g.osplit = 0;
    g.aux = nullptr; g.ldaux = 0; g.accumulate = 0; g.F = D.F; g.S = D.S; g.hd = D.hd; g.hq = D.hq;
    g.rope = nullptr;
    return g;
  }
  __device__ const int* offs(int l) const { return abuf<int>(a, A_OFFS) + (long long)l * (D.E + 1); }

  // forward
  __device__ GemmDesc qkv(int l) const {
    GemmDesc g = base(D.T, 3 * D.hq, D.d, EPI_ROPE);
    g.A = opnd(abuf<OP>(a, A_R) + (long long)l * D.T * D.d, D.d, 0);
    g.A.map0 = MAP_R; g.A.y0 = l * D.T;
    g.B = opnd(pweight<OP>(a, P_WQKV) + (long long)l * 3 * D.hq * D.d, D.d, 0);
    g.B.map0 = MAP_WQKV; g.B.y0 = l * 3 * D.hq;
    g.out = abuf<OP>(a, A_QKV) + (long long)l * D.T * 3 * D.hq; g.ldo = 3 * D.hq;
    g.rope = abuf<float>(a, A_ROPE);
    return g;
  }
  __device__ GemmDesc wo(int l) const {
    GemmDesc g = base(D.T, D.d, D.hq, EPI_RESID);
    g.A = opnd(abuf<OP>(a, A_O) + (long long)l * D.T * D.hq, D.hq, 0);
    g.A.map0 = MAP_O; g.A.y0 = l * D.T;
    g.B = opnd(pweight<OP>(a, P_WO) + (long long)l * D.d * D.hq, D.hq, 0);
    g.B.map0 = MAP_WO; g.B.y0 = l * D.d;
    g.out = abuf<float>(a, A_XM) + (long long)l * D.T * D.d; g.ldo = D.d;
    g.aux = abuf<float>(a, A_X) + (long long)l * D.T * D.d; g.ldaux = D.d;
    return g;
  }
  __device__ GemmDesc gateup(int l) const {
    GemmDesc g = base(D.Pmax, 2 * D.F, D.d, EPI_SWIGLU);
    g.rag = RAG_M; g.offs = offs(l); g.nseg = D.E;
    g.A = opnd(abuf<OP>(a, A_XS) + (long long)l * D.Pmax * D.d, D.d, 0);
    g.A.map0 = MAP_XS; g.A.y0 = l * D.Pmax;
    g.B = opnd(pweight<OP>(a, P_WGATE) + (long long)l * D.E * D.F * D.d, D.d, 0);
    g.B.p1 = pweight<OP>(a, P_WUP) + (long long)l * D.E * D.F * D.d;
    g.B.two = 1; g.B.seg = (long long)D.F * D.d;
    g.B.map0 = MAP_WGATE; g.B.map1 = MAP_WUP; g.B.y0 = l * D.E * D.F; g.B.yseg = D.F;
    g.out = abuf<OP>(a, A_GU) + (long long)l * D.Pmax * 2 * D.F; g.ldo = 2 * D.F;
    g.out2 = abuf<OP>(a, A_ACT) + (long long)l * D.Pmax * D.F; g.ldo2 = D.F;
    return g;
  }
  __device__ GemmDesc down(int l) const {
    GemmDesc g = base(D.Pmax, D.d, D.F, EPI_STORE_F32);
    g.rag = RAG_M; g.offs = offs(l); g.nseg = D.E;
    g.A = opnd(abuf<OP>(a, A_ACT) + (long long)l * D.Pmax * D.F, D.F, 0);
    g.A.map0 = MAP_ACT; g.A.y0 = l * D.Pmax;
    g.B = opnd(pweight<OP>(a, P_WDOWN) + (long long)l * D.E * D.d * D.F, D.F, 0);
    g.B.seg = (long long)D.d * D.F;
    g.B.map0 = MAP_WDOWN; g.B.y0 = l * D.E * D.d; g.B.yseg = D.d;
    g.out = abuf<float>(a, A_Y) + (long long)l * D.Pmax * D.d; g.ldo = D.d;
    return g;
  }
  __device__ GemmDesc lm() const {
    GemmDesc g = base(D.T, D.V, D.d, EPI_STORE_F32);
    g.A = opnd(abuf<OP>(a, A_RF), D.d, 0); g.A.map0 = MAP_RF;
    g.B = opnd(pweight<OP>(a, P_LM_HEAD), D.d, 0); g.B.map0 = MAP_WLM;
    g.out = abuf<float>(a, A_LOGITS); g.ldo = D.V;
    return g;
  }
  // backward
  __device__ GemmDesc lm_dgrad() const {
    GemmDesc g = base(D.T, D.d, D.V, EPI_STORE_F32);
    g.A = opnd(abuf<OP>(a, A_DLOGITS), D.V, 0); g.A.map0 = MAP_DLOGITS;
    g.B = opnd(pweight<OP>(a, P_LM_HEAD), D.d, 1); g.B.map0 = MAP_WLM;
    g.out = abuf<float>(a, A_DRF); g.ldo = D.d;
    return g;
  }
  __device__ GemmDesc lm_wgrad() const {
    GemmDesc g = base(D.V, D.d, D.T, EPI_GRAD);
    g.A = opnd(abuf<OP>(a, A_DLOGITS), D.V, 1); g.A.map0 = MAP_DLOGITS;
    g.B = opnd(abuf<OP>(a, A_RF), D.d, 1); g.B.map0 = MAP_RF;
    g.out = pgrad(a, P_LM_HEAD); g.ldo = D.d; g.accumulate = a.micro_index > 0;
    return g;
  }
  __device__ GemmDesc down_dgrad(int l) const {
    GemmDesc g = base(D.Pmax, D.F, D.d, EPI_SWIGLU_BWD);
    g.rag = RAG_M; g.offs = offs(l); g.nseg = D.E;
    g.A = opnd(abuf<OP>(a, A_DY), D.d, 0); g.A.map0 = MAP_DY;
    g.B = opnd(pweight<OP>(a, P_WDOWN) + (long long)l * D.E * D.d * D.F, D.F, 1);
    g.B.seg = (long long)D.d * D.F;
    g.B.map0 = MAP_WDOWN; g.B.y0 = l * D.E * D.d; g.B.yseg = D.d;
    g.out = abuf<OP>(a, A_DGU); g.ldo = 2 * D.F;
    g.aux = abuf<OP>(a, A_GU) + (long long)l * D.Pmax * 2 * D.F; g.ldaux = 2 * D.F;
    return g;
  }
  __device__ GemmDesc down_wgrad(int l) const {
    GemmDesc g = base(D.d, D.F, 0, EPI_GRAD);
    g.rag = RAG_K; g.offs = offs(l); g.nseg = D.E;
    g.A = opnd(abuf<OP>(a, A_DY), D.d, 1); g.A.map0 = MAP_DY;
    g.B = opnd(abuf<OP>(a, A_ACT) + (long long)l * D.Pmax * D.F, D.F, 1);
    g.B.map0 = MAP_ACT; g.B.y0 = l * D.Pmax;
    g.out = pgrad(a, P_WDOWN) + (long long)l * D.E * D.d * D.F; g.ldo = D.F;
    g.oseg = (long long)D.d * D.F; g.accumulate = a.micro_index > 0;
    return g;
  }
  __device__ GemmDesc gateup_dgrad(int l) const {
    GemmDesc g = base(D.Pmax, D.d, 2 * D.F, EPI_STORE_F32);
    g.rag = RAG_M; g.offs = offs(l); g.nseg = D.E;
    g.A = opnd(abuf<OP>(a, A_DGU), 2 * D.F, 0); g.A.map0 = MAP_DGU;
    g.B = opnd(pweight<OP>(a, P_WGATE) + (long long)l * D.E * D.F * D.d, D.d, 1);
    g.B.p1 = pweight<OP>(a, P_WUP) + (long long)l * D.E * D.F * D.d;
    g.B.two = 2; g.B.split = D.F; g.B.seg = (long long)D.F * D.d;
    g.B.map0 = MAP_WGATE; g.B.map1 = MAP_WUP; g.B.y0 = l * D.E * D.F; g.B.yseg = D.F;
    g.out = abuf<float>(a, A_DXS); g.ldo = D.d;
    return g;
  }
  __device__ GemmDesc gateup_wgrad(int l) const {
    GemmDesc g = base(2 * D.F, D.d, 0, EPI_GRAD);
    g.rag = RAG_K; g.offs = offs(l); g.nseg = D.E;
    g.A = opnd(abuf<OP>(a, A_DGU), 2 * D.F, 1); g.A.map0 = MAP_DGU;
    g.B = opnd(abuf<OP>(a, A_XS) + (long long)l * D.Pmax * D.d, D.d, 1);
    g.B.map0 = MAP_XS; g.B.y0 = l * D.Pmax;
    g.out = pgrad(a, P_WGATE) + (long long)l * D.E * D.F * D.d;
    g.out1 = pgrad(a, P_WUP) + (long long)l * D.E * D.F * D.d;
    g.osplit = D.F; g.ldo = D.d; g.oseg = (long long)D.F * D.d; g.accumulate = a.micro_index > 0;
    return g;
  }
  __device__ GemmDesc wo_dgrad(int l) const {
    GemmDesc g = base(D.T, D.hq, D.d, EPI_STORE_OP);
    g.A = opnd(abuf<OP>(a, A_DXO), D.d, 0); g.A.map0 = MAP_DXO;
    g.B = opnd(pweight<OP>(a, P_WO) + (long long)l * D.d * D.hq, D.hq, 1);
    g.B.map0 = MAP_WO; g.B.y0 = l * D.d;
    g.out = abuf<OP>(a, A_DO); g.ldo = D.hq;
    return g;
  }
  __device__ GemmDesc wo_wgrad(int l) const {
    GemmDesc g = base(D.d, D.hq, D.T, EPI_GRAD);
    g.A = opnd(abuf<OP>(a, A_DXO), D.d, 1); g.A.map0 = MAP_DXO;
    g.B = opnd(abuf<OP>(a, A_O) + (long long)l * D.T * D.hq, D.hq, 1);
    g.B.map0 = MAP_O; g.B.y0 = l * D.T;
    g.out = pgrad(a, P_WO) + (long long)l * D.d * D.hq; g.ldo = D.hq; g.accumulate = a.micro_index > 0;
    return g;
  }
  __device__ GemmDesc qkv_dgrad(int l) const {
    GemmDesc g = base(D.T, D.d, 3 * D.hq, EPI_STORE_F32);
    g.A = opnd(abuf<OP>(a, A_DQKV), 3 * D.hq, 0); g.A.map0 = MAP_DQKV;
    g.B = opnd(pweight<OP>(a, P_WQKV) + (long long)l * 3 * D.hq * D.d, D.d, 1);
    g.B.map0 = MAP_WQKV; g.B.y0 = l * 3 * D.hq;
    g.out = abuf<float>(a, A_DR); g.ldo = D.d;
    return g;
  }
  __device__ GemmDesc qkv_wgrad(int l) const {
    GemmDesc g = base(3 * D.hq, D.d, D.T, EPI_GRAD);
    g.A = opnd(abuf<OP>(a, A_DQKV), 3 * D.hq, 1); g.A.map0 = MAP_DQKV;
    g.B = opnd(abuf<OP>(a, A_R) + (long long)l * D.T * D.d, D.d, 1);
    g.B.map0 = MAP_R; g.B.y0 = l * D.T;
    g.out = pgrad(a, P_WQKV) + (long long)l * 3 * D.hq * D.d; g.ldo = D.d; g.accumulate = a.micro_index > 0;
    return g;
  }
};

template <class OP>
__device__ __forceinline__ void run_gemm(const KArgs& a, const GemmDesc& g, Sched& s, char* smem, TcState& tc) {
  if constexpr (sizeof(OP) == 2) {
    if (a.use_tc) { gemm_tc_job(a, g, s, smem, tc); return; }
  }
  gemm_simt_job<OP>(g, s, reinterpret_cast<float*>(smem));
}

template <class OP>
__device__ __forceinline__ AttnArgs attn_args(const KArgs& a, int l) {
  const MtDims& D = a.D;
  AttnArgs t;
  t.qkv = abuf<OP>(a, A_QKV) + (long long)l * D.T * 3 * D.hq;
  t.o = abuf<OP>(a, A_O) + (long long)l * D.T * D.hq;
  t.lse = abuf<float>(a, A_LSE) + (long long)l * D.B * D.H * D.S;
  t.dout = abuf<OP>(a, A_DO);
  t.dqkv = abuf<OP>(a, A_DQKV);
  t.rope = abuf<float>(a, A_ROPE);
  t.B = D.B; t.H = D.H; t.S = D.S; t.hq = D.hq;
  t.scale = 1.0f / sqrtf((float)D.hd);
  return t;
}

template <class OP>
__device__ __forceinline__ void run_attn_fwd(const KArgs& a, int l, Sched& s, char* smem) {
  const AttnArgs t = attn_args<OP>(a, l);
  if (a.D.hd == 64) attn_fwd_job<OP, 64>(t, s, (float*)smem);
  else attn_fwd_job<OP, 16>(t, s, (float*)smem);
}
template <class OP>
__device__ __forceinline__ void run_attn_bwd(const KArgs& a, int l, Sched& s, char* smem) {
  const AttnArgs t = attn_args<OP>(a, l);
  if (a.D.hd == 64) attn_bwd_job<OP, 64>(t, s, (float*)smem);
  else attn_bwd_job<OP, 16>(t, s, (float*)smem);
}

// ===========================================================================
// the program
// ===========================================================================
// One microbatch: forward, loss, backward, and on the last microbatch the
// optimizer.  Returns early (every CTA) when a grid barrier reports an error.
template <class OP>
__device__ void run_update(const KArgs& a, char* smem, TcState& tc, Sched& s) {
  const MtDims& D = a.D;
  ArenaHdr* hdr = abuf<ArenaHdr>(a, A_HDR);
  const unsigned G = gridDim.x;
  const bool trace = (a.flags & MT_FLAG_TRACE) != 0;
  long long* tr = trace ? abuf<long long>(a, A_TRACE) + (long long)blockIdx.x * MT_MAX_PHASES * 2 : nullptr;
  int phase = 0;
  Gemms<OP> gm(a);
  const bool stall = (a.flags & MT_FLAG_TEST_STALL) && blockIdx.x == 0;

#define MT_SYNC()                                                                                      \
  do {                                                                                                 \
    if (!grid_barrier(hdr, G, a.timeout_ns, (tr && phase < MT_MAX_PHASES) ? tr + 2 * phase : nullptr, \
                      stall))                                                                          \
      return;                                                                                          \
    ++phase;                                                                                           \
  } while (0)

  // ---------------- forward ----------------
  job_embed<OP>(a, s);
  MT_SYNC();
  for (int l = 0; l < D.L; ++l) {
    run_gemm<OP>(a, gm.qkv(l), s, smem, tc);
    MT_SYNC();
    run_attn_fwd<OP>(a, l, s, smem);
    MT_SYNC();
    run_gemm<OP>(a, gm.wo(l), s, smem, tc);
    MT_SYNC();
    job_router<OP>(a, l, (float*)smem);
    MT_SYNC();
    job_route<OP>(a, l, (int*)smem);
    MT_SYNC();
    run_gemm<OP>(a, gm.gateup(l), s, smem, tc);
    MT_SYNC();
    run_gemm<OP>(a, gm.down(l), s, smem, tc);
    MT_SYNC();
    job_combine<OP>(a, l, s);
    MT_SYNC();
  }
  run_gemm<OP>(a, gm.lm(), s, smem, tc);
  MT_SYNC();
  job_ce<OP>(a, s);
  MT_SYNC();

  // ---------------- backward ----------------
  job_loss(a);
  run_gemm<OP>(a, gm.lm_dgrad(), s, smem, tc);
  run_gemm<OP>(a, gm.lm_wgrad(), s, smem, tc);
  MT_SYNC();
  job_final_norm_bwd<OP>(a, s);
  MT_SYNC();
  {
    // final-norm gain partials (DRF stays valid until the next LM-head use)
    ColArgs c{COL_GAIN, abuf<float>(a, A_DRF), abuf<float>(a, A_X) + (long long)D.L * D.T * D.d,
              abuf<float>(a, A_INVF), nullptr, nullptr, D.E + 1};
    job_colpart(a, c, s);
  }
  for (int l = D.L - 1; l >= 0; --l) {
    job_moe_bwd1<OP>(a, l, s);
    if (l < D.L - 1) {
      // attention-norm gain partials of layer l+1 (DR of layer l+1 is still live)
      ColArgs c{COL_GAIN, abuf<float>(a, A_DR), abuf<float>(a, A_X) + (long long)(l + 1) * D.T * D.d,
                abuf<float>(a, A_INV1) + (long long)(l + 1) * D.T, nullptr, nullptr, D.E + 1};
      job_colpart(a, c, s);
    }
    MT_SYNC();
    if (l == D.L - 1) job_colfinal(a, D.E + 1, 1, pgrad(a, P_FINAL_NORM), nullptr, 0, s);
    else job_colfinal(a, D.E + 1, 1, pgrad(a, P_ATTN_NORM) + (long long)(l + 1) * D.d, nullptr, 0, s);
    run_gemm<OP>(a, gm.down_dgrad(l), s, smem, tc);
    run_gemm<OP>(a, gm.down_wgrad(l), s, smem, tc);
    MT_SYNC();
    run_gemm<OP>(a, gm.gateup_dgrad(l), s, smem, tc);
    run_gemm<OP>(a, gm.gateup_wgrad(l), s, smem, tc);
    MT_SYNC();
    job_moe_bwd2<OP>(a, l, s);
    MT_SYNC();
    {
      ColArgs c{COL_MOE, abuf<float>(a, A_DR2), abuf<float>(a, A_XM) + (long long)l * D.T * D.d,
                abuf<float>(a, A_INV2) + (long long)l * D.T, pmaster(a, P_MOE_NORM) + (long long)l * D.d,
                abuf<float>(a, A_DZ), 0};
      job_colpart(a, c, s);
    }
    run_gemm<OP>(a, gm.wo_dgrad(l), s, smem, tc);
    run_gemm<OP>(a, gm.wo_wgrad(l), s, smem, tc);
    MT_SYNC();
    job_colfinal(a, 0, D.E + 1, pgrad(a, P_ROUTER) + (long long)l * D.E * D.d,
                 pgrad(a, P_MOE_NORM) + (long long)l * D.d, 1, s);
    run_attn_bwd<OP>(a, l, s, smem);
    MT_SYNC();
    run_gemm<OP>(a, gm.qkv_dgrad(l), s, smem, tc);
    run_gemm<OP>(a, gm.qkv_wgrad(l), s, smem, tc);
    MT_SYNC();
    job_attn_norm_bwd<OP>(a, l, s);
    MT_SYNC();
  }
  {
    ColArgs c{COL_GAIN, abuf<float>(a, A_DR), abuf<float>(a, A_X), abuf<float>(a, A_INV1), nullptr,
              nullptr, D.E + 1};
    job_colpart(a, c, s);
  }
  job_embed_bwd(a, (int*)smem);
  MT_SYNC();
  job_colfinal(a, D.E + 1, 1, pgrad(a, P_ATTN_NORM), nullptr, 0, s);

  // ---------------- optimizer (last microbatch) ----------------
  if (a.run_opt) {
    MT_SYNC();
    job_norm_partial(a, (double*)smem);
    MT_SYNC();
    job_adamw<OP>(a);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    hdr->micro_index = a.micro_index;
    if (!a.run_opt) hdr->optimizer_ran = 0;
    hdr->n_ctas = (int)G;
    hdr->n_phases = phase;
  }
#undef MT_SYNC
}

// Test harness: one product C = A B^T (fp32 out) described by the debug
// fields of the arguments; A in map MAP_R, B in map MAP_WQKV.
template <class OP>
__device__ void run_debug_gemm(const KArgs& a, char* smem, TcState& tc, Sched& s) {
  GemmDesc g;
  g.M = a.dbg_m; g.N = a.dbg_n; g.K = a.dbg_k; g.rag = a.dbg_rag; g.offs = a.dbg_offs; g.nseg = a.dbg_nseg;
  g.epi = (g.rag == RAG_K) ? EPI_GRAD : EPI_STORE_F32;
  g.out = a.dbg_c; g.out1 = nullptr; g.out2 = nullptr; g.ldo = g.N; g.ldo2 = 0; g.osplit = 0;
  g.oseg = (long long)g.M * g.N; g.aux = nullptr; g.ldaux = 0; g.accumulate = 0;
  g.F = 0; g.S = 1; g.hd = 64; g.hq = 0; g.rope = nullptr;
  GOperand A, B;
  A.p0 = a.dbg_a; A.p1 = nullptr; A.mn = a.dbg_a_mn; A.ld = A.mn ? g.M : g.K; A.seg = 0; A.two = 0;
  A.split = 0; A.map0 = MAP_R; A.map1 = -1; A.y0 = 0; A.yseg = 0;
  B.p0 = a.dbg_b; B.p1 = nullptr; B.mn = a.dbg_b_mn; B.ld = B.mn ? g.N : g.K;
  B.seg = (long long)g.N * g.K; B.two = 0; B.split = 0; B.map0 = MAP_WQKV; B.map1 = -1; B.y0 = 0;
  B.yseg = B.mn ? g.K : g.N;
  g.A = A;
  g.B = B;
  run_gemm<OP>(a, g, s, smem, tc);
  ArenaHdr* hdr = abuf<ArenaHdr>(a, A_HDR);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    hdr->n_ctas = (int)gridDim.x;
    hdr->n_phases = 0;
  }
}

template <class OP>
__global__ void __launch_bounds__(MT_THREADS, 1) mt_megakernel(const __grid_constant__ KArgs a) {
  extern __shared__ __align__(1024) char smem[];
  Sched s{(int)blockIdx.x, (int)gridDim.x, 0};
  TcState tc;
  tc_setup<OP>(a, smem, tc);
  if (a.debug_gemm) run_debug_gemm<OP>(a, smem, tc, s);
  else run_update<OP>(a, smem, tc, s);
  tc_teardown<OP>(a, smem, tc);
}
