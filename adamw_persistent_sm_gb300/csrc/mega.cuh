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
#include "attn_tm.cuh"
#include "rows.cuh"
#include "rowpipe.cuh"
#include <type_traits>

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
// Whether this launch adds tensor pid's gradient into the buffer (else it
// overwrites it): every tensor after the first microbatch of an update, and
// under selective updates only the expert tensors.
__device__ __forceinline__ bool acc_of(const KArgs& a, int pid) { return (a.acc_mask >> pid) & 1u; }
// Weight slot of layer visit l: the looped model applies its U distinct
// layers in turn (visit l uses slot l mod U; U = L without looping).
__device__ __forceinline__ int wslot(const KArgs& a, int l) { return l % a.D.U; }
// Gradient write of layer visit l into its slot: the backward meets the
// visits in decreasing order, so every visit but the last U (the first ones
// processed) adds into what a later visit already wrote.
__device__ __forceinline__ bool acc_visit(const KArgs& a, int pid, int l) {
  return acc_of(a, pid) || l < a.D.L - a.D.U;
}

// Column tiles of the LM-head product (one cross-entropy partial each).
template <class OP>
__device__ __forceinline__ int ce_parts(const KArgs& a) {
  const int w = (sizeof(OP) == 2 && a.use_tc) ? 256 : 128;
  return (a.D.V + w - 1) / w;
}

// Slices of a weight-gradient reduction over K tokens on the tensor-core
// path: enough tiles for every SM, K/64 divisible by the count, and the
// slices must fit in A_KPART (8 x 3hq x d floats).
__device__ __forceinline__ int ksplit_of(const KArgs& a, int M, int N, int K) {
  if (!a.use_tc || M % 128 || N % 256 || K % 64) return 1;
  const int tiles = (M / 128) * (N / 256);
  int ks = (int)gridDim.x / tiles;
  const long long cap = 8LL * 3 * a.D.hq * a.D.d / ((long long)M * N);
  if (ks > cap) ks = (int)cap;
  if (ks > 16) ks = 16;
  while (ks > 1 && (K / 64) % ks) --ks;
  return ks < 1 ? 1 : ks;
}

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
// CTA me's share of the rotary table (cos, sin of pos * theta^(-2i/hd), in
// double precision) and of the zeroing of the dependency counters and
// tickets, which start at zero in every launch (first used after the first
// grid barrier).
__device__ __forceinline__ void launch_prologue(const KArgs& a, int me, int G) {
  const MtDims& D = a.D;
  const int half = D.hd / 2;
  float* rope = abuf<float>(a, A_ROPE);
  for (int e = me * MT_THREADS + threadIdx.x; e < D.S * half; e += G * MT_THREADS) {
    const int pos = e / half, i = e % half;
    const double freq = pow((double)a.rope_theta, -2.0 * (double)i / (double)D.hd);
    double sv, cv;
    sincos((double)pos * freq, &sv, &cv);
    rope[2 * e] = (float)cv;
    rope[2 * e + 1] = (float)sv;
  }
  unsigned* dep = abuf<unsigned>(a, A_DEP);
  const long long ndep = dep_words(D);
  for (long long i = (long long)me * MT_THREADS + threadIdx.x; i < ndep; i += (long long)G * MT_THREADS) dep[i] = 0u;
}

template <class OP>
__device__ __noinline__ void job_embed(const KArgs& a, Sched& s) {
  const MtDims& D = a.D;
  const int me = s.first();
  launch_prologue(a, me, s.G);
  ArenaHdr* hdr = abuf<ArenaHdr>(a, A_HDR);
  const float* emb = pmaster(a, P_EMB);
  float* X = abuf<float>(a, A_X);
  OP* R = abuf<OP>(a, A_R);
  float* inv1 = abuf<float>(a, A_INV1);
  const int n4 = D.d / 4, nw = s.G * MT_WARPS, lane = threadIdx.x & 31;
  with_nc(D.d, [&](auto NCc) {
    constexpr int NC = decltype(NCc)::value;
    Row<NC> g, x, r;
    row_ld(g, pmaster(a, P_ATTN_NORM), n4);
    for (int t = me * MT_WARPS + (threadIdx.x >> 5); t < D.T; t += nw) {
      int v = a.tokens[t];
      if (v < 0 || v >= D.V) {
        if (lane == 0) set_error(hdr, MT_ERR_DEVICE_BOUNDS, SITE_TOKEN_RANGE);
        v = 0;
      }
      row_ld(x, emb + (long long)v * D.d, n4);
      row_st(X + (long long)t * D.d, x, n4);
      const float inv = row_rms_inv(x, D.d, a.norm_eps);
      row_norm_apply(r, x, inv, g);
      row_st_op(R + (long long)t * D.d, r, n4);
      if (lane == 0) inv1[t] = inv;
    }
  });
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
__device__ __noinline__ void job_router(const KArgs& a, int l, char* smem, const unsigned* dw, unsigned dtarget,
                                        long long* wait_stamp) {
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
  const float* g = pmaster(a, P_MOE_NORM) + (long long)wslot(a, l) * D.d;
  const float* Wr = pmaster(a, P_ROUTER) + (long long)wslot(a, l) * D.E * D.d;
  const uint32_t rowb = (uint32_t)D.d * 4u;
  // shared memory: [mbarriers of the row rings | router weights (fp32, E x d)
  // | per-expert counts | row rings]
  float* sm = reinterpret_cast<float*>(smem + RP_WIN_OFF);
  const uint32_t swr = smem_u32(sm);
  int* s_cnt = reinterpret_cast<int*>(sm + (long long)D.E * D.d);
  const uint32_t win = (RP_WIN_OFF + (uint32_t)D.E * rowb + 4u * 64u + 127u) & ~127u;
  // two tokens per stage: each router-weight value read from shared memory
  // serves both (the logits are bound by shared-memory reads otherwise)
  const RowPipe p = rp_make(smem, win, (uint32_t)a.smem_bytes, 2u * rowb);
  if (p.ns > 0) rp_begin(p);
  else __syncthreads();
  for (int i = threadIdx.x; i < D.E * D.d / 4; i += MT_THREADS)
    reinterpret_cast<float4*>(sm)[i] = reinterpret_cast<const float4*>(Wr)[i];
  for (int e = threadIdx.x; e < D.E; e += MT_THREADS) s_cnt[e] = 0;
  if (dw && t0 < t1) {
    // the chunk's x_mid rows are stored by out-projection tiles of other CTAs
    const int b0 = t0 / MT_TILE_M, nb = (t1 - 1) / MT_TILE_M - b0 + 1;
    if (threadIdx.x < nb) dep_wait(abuf<ArenaHdr>(a, A_HDR), dw + b0 + threadIdx.x, dtarget, a.timeout_ns);
  }
  __syncthreads();
  if (wait_stamp && threadIdx.x == 0) {
    // trace: the end of the wait for the out-projection tiles
    wait_stamp[0] = (long long)globaltimer();
    wait_stamp[1] = 36;
  }
  if (p.ns > 0 && lane == 0) asm volatile("fence.proxy.async;" ::: "memory");   // after the acquire
  const int n4 = D.d / 4;
  bool ok = true;
  with_nc(D.d, [&](auto NCc) {
  constexpr int NC = decltype(NCc)::value;
  Row<NC> gr, xa, xb;
  row_ld(gr, g, n4);
  // softmax, token_topk and renormalised weights of one token from its logits
  // (lane e holds expert e in z0, expert e + 32 in z1)
  auto pick = [&](int t, float z0, float z1) {
    if (lane < D.E) Z[(long long)t * D.E + lane] = z0;
    if (lane + 32 < D.E) Z[(long long)t * D.E + lane + 32] = z1;
    const float zmax = warp_max(fmaxf(z0, z1));
    const float p0 = (lane < D.E) ? __expf(z0 - zmax) : 0.f;
    const float p1 = (lane + 32 < D.E) ? __expf(z1 - zmax) : 0.f;
    // the softmax normaliser cancels in the renormalised weights; slot k is
    // kept by lane k
    float c0 = z0, c1 = z1;
    float my_p = 0.f;
    int my_i = 0;
    float psum = 0.f;
    for (int k = 0; k < D.K; ++k) {
      float v = c0;
      int idx = lane;
      if (c1 > v) { v = c1; idx = lane + 32; }
      warp_argmax(v, idx);
      const float pk = __shfl_sync(0xffffffffu, idx < 32 ? p0 : p1, idx & 31);
      if (lane == k) { my_i = idx; my_p = pk; }
      psum += pk;
      if (idx == lane) c0 = -INFINITY;
      if (idx == lane + 32) c1 = -INFINITY;
    }
    if (lane < D.K) {
      IDX[(long long)t * D.K + lane] = my_i;
      WGT[(long long)t * D.K + lane] = my_p / psum;
      atomicAdd(&s_cnt[my_i], 1);
    }
  };
  // expert RMSNorm of tokens ta and tb (tb < 0: none), their operand rows,
  // then the logits four experts per step: lane-partial dot products over the
  // lane's columns and one warp sum each.  The expert loop is not unrolled,
  // so that the code stays small in the instruction cache.
  auto tokens2 = [&](int ta, int tb) {
    const float inva = row_rms_inv(xa, D.d, a.norm_eps);
    const float invb = row_rms_inv(xb, D.d, a.norm_eps);
    row_norm_apply(xa, xa, inva, gr);
    row_norm_apply(xb, xb, invb, gr);
    row_st_op(R2 + (long long)ta * D.d, xa, n4);
    if (lane == 0) inv2[ta] = inva;
    if (tb >= 0) {
      row_st_op(R2 + (long long)tb * D.d, xb, n4);
      if (lane == 0) inv2[tb] = invb;
    }
    float za0 = -INFINITY, za1 = -INFINITY, zb0 = -INFINITY, zb1 = -INFINITY;
    // Lane l's logit sums of group e0 end up in red: the eight partials
    // (token a: experts e0..e0+3, token b: the same) are reduce-scattered over
    // lane bits 4, 3, 2 (one value left per lane) and summed over bits 1, 0:
    // lane l holds partial index ((l >> 4) & 1) * 4 + ((l >> 3) & 1) * 2 + ((l >> 2) & 1).
#pragma unroll 2
    for (int e0 = 0; e0 < D.E; e0 += 4) {
      float aa[4], ab[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        aa[q] = 0.f;
        ab[q] = 0.f;
        if (e0 + q < D.E) {
          const uint32_t wa = swr + (uint32_t)(e0 + q) * (uint32_t)D.d * 4u + 16u * (uint32_t)lane;
#pragma unroll
          for (int i = 0; i < NC; ++i) {
            if (lane + 32 * i < n4) {
              const float4 w4 = lds4(wa + 512u * (uint32_t)i);
              aa[q] = fmaf(xa.v[i].x, w4.x, aa[q]);
              aa[q] = fmaf(xa.v[i].y, w4.y, aa[q]);
              aa[q] = fmaf(xa.v[i].z, w4.z, aa[q]);
              aa[q] = fmaf(xa.v[i].w, w4.w, aa[q]);
              ab[q] = fmaf(xb.v[i].x, w4.x, ab[q]);
              ab[q] = fmaf(xb.v[i].y, w4.y, ab[q]);
              ab[q] = fmaf(xb.v[i].z, w4.z, ab[q]);
              ab[q] = fmaf(xb.v[i].w, w4.w, ab[q]);
            }
          }
        }
      }
      float v8[8] = {aa[0], aa[1], aa[2], aa[3], ab[0], ab[1], ab[2], ab[3]};
      const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
#pragma unroll
      for (int i = 0; i < 4; ++i) {        // bit 4: keep the half of index bit 2
        const float send = b4 ? v8[i] : v8[i + 4], keep = b4 ? v8[i + 4] : v8[i];
        v8[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {        // bit 3
        const float send = b3 ? v8[i] : v8[i + 2], keep = b3 ? v8[i + 2] : v8[i];
        v8[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
      }
      {                                    // bit 2
        const float send = b2 ? v8[0] : v8[1], keep = b2 ? v8[1] : v8[0];
        v8[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
      }
      v8[0] += __shfl_xor_sync(0xffffffffu, v8[0], 2);
      v8[0] += __shfl_xor_sync(0xffffffffu, v8[0], 1);
      // lane e (and e + 32) collects expert e of both tokens: index (e & 3)
      // of token a lives in lane 8 ((e >> 1) & 1) + 4 (e & 1), of token b 16 lanes up
      const int src = 8 * ((lane >> 1) & 1) + 4 * (lane & 1);
      const float ga = __shfl_sync(0xffffffffu, v8[0], src);
      const float gb = __shfl_sync(0xffffffffu, v8[0], src + 16);
      if ((lane & ~3) == e0 && lane < D.E) { za0 = ga; zb0 = gb; }
      if (((lane + 32) & ~3) == e0 && lane + 32 < D.E) { za1 = ga; zb1 = gb; }
    }
    pick(ta, za0, za1);
    if (tb >= 0) pick(tb, zb0, zb1);
  };
  // this warp's tokens t0 + warp + 8 i, in pairs (i = 2j, 2j + 1)
  const int nt = t0 + warp < t1 ? (t1 - 1 - t0 - warp) / MT_WARPS + 1 : 0;
  if (p.ns > 0) {
    // staged: the x_mid rows of a token pair; header: both tokens (-1: none)
    ok = rp_run(
        p, (nt + 1) / 2, abuf<ArenaHdr>(a, A_HDR), a.timeout_ns / 2, SITE_ROWPIPE + 0,
        [&](int j, uint32_t st, uint32_t bar) {
          const int ta = t0 + warp + 2 * j * MT_WARPS;
          const int tb = (2 * j + 1 < nt) ? ta + MT_WARPS : -1;
          sts_i32(st, ta);
          sts_i32(st + 4u, tb);
          mbar_expect_tx(bar, (tb >= 0 ? 2u : 1u) * rowb);
          bulk_g2s(st + RP_HDR, XM + (long long)ta * D.d, rowb, bar);
          if (tb >= 0) bulk_g2s(st + RP_HDR + rowb, XM + (long long)tb * D.d, rowb, bar);
        },
        [&](int j, uint32_t st) {
          const int ta = lds_i32(st), tb = lds_i32(st + 4u);
          row_lds(xa, st + RP_HDR, n4);
          if (tb >= 0) row_lds(xb, st + RP_HDR + rowb, n4);
          else row_scale(xb, xa, 0.f);
          tokens2(ta, tb);
        },
        [&](int) {});
  } else {
    for (int i = 0; i < nt; i += 2) {
      const int ta = t0 + warp + i * MT_WARPS;
      const int tb = (i + 1 < nt) ? ta + MT_WARPS : -1;
      row_ld(xa, XM + (long long)ta * D.d, n4);
      if (tb >= 0) row_ld(xb, XM + (long long)tb * D.d, n4);
      else row_scale(xb, xa, 0.f);
      tokens2(ta, tb);
    }
  }
  });
  if (p.ns > 0) rp_end(p, ok);
  else __syncthreads();
  if (t0 < D.T) {
    int* CNT = abuf<int>(a, A_CNT) + ((long long)l * D.nch + c) * D.E;
    for (int e = threadIdx.x; e < D.E; e += MT_THREADS) CNT[e] = s_cnt[e];
  }
  __syncthreads();
}

// route_order: stable counting sort of the T*K assignments by expert (the
// histogram comes from job_router), expert segments padded to MT_TILE_M rows,
// fused with the dispatch gather of the expert inputs.  Within an expert,
// assignments keep ascending a = t*K + k.
template <class OP>
__device__ __noinline__ void job_route(const KArgs& a, int l, char* smem) {
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
  // shared memory: [mbarriers of the row rings | counting-sort scratch | rings]
  int* ism = reinterpret_cast<int*>(smem + RP_WIN_OFF);
  int* s_tot = ism;                 // [E]
  int* s_base = ism + 64;           // [E]
  int* s_offs = ism + 128;          // [E+1]
  int* s_cnt = ism + 256;           // [nused][E] chunk counts
  const uint32_t rowb = (uint32_t)D.d * (uint32_t)sizeof(OP);
  const uint32_t win = (RP_WIN_OFF + 4u * (256u + (uint32_t)(nused * D.E)) + 127u) & ~127u;
  const RowPipe rp = rp_make(smem, win, (uint32_t)a.smem_bytes, rowb);
  if (rp.ns > 0) rp_begin(rp);
  for (int i = threadIdx.x; i < nused * D.E; i += MT_THREADS) s_cnt[i] = CNT[i];
  __syncthreads();
  for (int e = threadIdx.x; e < D.E; e += MT_THREADS) {
    int tot = 0, before = 0;
    for (int cc = 0; cc < nused; ++cc) {
      const int n = s_cnt[cc * D.E + e];
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
  const int n16 = D.d * (int)sizeof(OP) / 16;
  // dispatch gather: XS[row] = R2[token].  With a ring, lane 0 of each warp
  // copies the warp's token rows into shared memory (cp.async.bulk) and
  // stores each to its K sorted rows with bulk stores; the stage of token j
  // is refilled once the stores of token j have been read out.
  if (rp.ns > 0) {
    if (lane == 0) {
      const int n = t0 + warp < t1 ? (t1 - 1 - t0 - warp) / MT_WARPS + 1 : 0;
      auto load = [&](int j) {
        mbar_expect_tx(rp.sbar(j), rowb);
        bulk_g2s(rp.stage(j) + RP_HDR, R2 + (long long)(t0 + warp + j * MT_WARPS) * D.d, rowb, rp.sbar(j));
      };
      for (int j = 0; j < n && j < rp.ns; ++j) load(j);
      bool ok = true;
      for (int j = 0; j < n && ok; ++j) {
        if (!mbar_wait(rp.sbar(j), rp.parity(j), a.timeout_ns / 2)) {
          set_error(abuf<ArenaHdr>(a, A_HDR), MT_ERR_DEVICE_TIMEOUT, SITE_ROWPIPE + 1);
          ok = false;
          break;
        }
        const int t = t0 + warp + j * MT_WARPS;
        for (int k = 0; k < D.K; ++k)
          bulk_s2g(XS + (long long)INVM[(long long)t * D.K + k] * D.d, rp.stage(j) + RP_HDR, rowb);
        bulk_commit();
        if (j + rp.ns < n) {
          bulk_wait_read0();
          load(j + rp.ns);
        }
      }
      bulk_wait_all0();
      // the bulk stores (async proxy) come before the release at the next barrier
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    __syncwarp();
  } else {
    for (int j = a0 + warp; j < a1; j += MT_WARPS) {
      const int pos = INVM[j];
      const uint4* src = reinterpret_cast<const uint4*>(R2 + (long long)(j / D.K) * D.d);
      uint4* dst = reinterpret_cast<uint4*>(XS + (long long)pos * D.d);
      for (int i = lane; i < n16; i += 32) dst[i] = src[i];
    }
  }
  // zero the pad rows of every segment (spread over all CTAs)
  const int gw = c * MT_WARPS + warp, nw = G * MT_WARPS;
  for (int e = 0; e < D.E; ++e) {
    const int p0 = s_offs[e] + s_tot[e], p1 = s_offs[e + 1];
    for (int p = p0 + gw; p < p1; p += nw) {
      uint4* dst = reinterpret_cast<uint4*>(XS + (long long)p * D.d);
      for (int i = lane; i < n16; i += 32) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      if (lane == 0) PERM[p] = -1;
    }
  }
  if (rp.ns > 0) rp_end(rp, true);
}

// x_{l+1} = x_mid + sum_k w_k y_k (fixed slot order), then the next
// RMSNorm (attention norm of layer l+1, or the final norm).
template <class OP>
__device__ __noinline__ void job_combine(const KArgs& a, int l, Sched& s, unsigned* dsig, char* smem) {
  const MtDims& D = a.D;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n4 = D.d / 4;
  const float* XM = abuf<float>(a, A_XM) + (long long)l * D.T * D.d;
  const float* Y = abuf<float>(a, A_Y) + (long long)l * D.Pmax * D.d;
  const float* WGT = abuf<float>(a, A_WGT) + (long long)l * D.T * D.K;
  const int* INVM = abuf<int>(a, A_INVM) + (long long)l * D.T * D.K;
  float* Xn = abuf<float>(a, A_X) + (long long)(l + 1) * D.T * D.d;
  const bool last = (l + 1 == D.L);
  const float* gp = last ? pmaster(a, P_FINAL_NORM) : pmaster(a, P_ATTN_NORM) + (long long)wslot(a, l + 1) * D.d;
  OP* Rn = last ? abuf<OP>(a, A_RF) : abuf<OP>(a, A_R) + (long long)(l + 1) * D.T * D.d;
  float* invn = last ? abuf<float>(a, A_INVF) : abuf<float>(a, A_INV1) + (long long)(l + 1) * D.T;
  // items: groups of MT_DEP_GROUP tokens (each warp takes every 8th token of
  // its CTA's group); with counters on, each finished group is published
  const int ng = (D.T + MT_DEP_GROUP - 1) / MT_DEP_GROUP;
  const uint32_t rowb = (uint32_t)D.d * 4u;
  // index table: per token of the warp (first RP_TBL), its K sorted rows and K weights
  const RowPipe p = rp_make(smem, RP_WIN_OFF, (uint32_t)a.smem_bytes, (uint32_t)(1 + D.K) * rowb,
                            (uint32_t)(RP_TBL * 2 * D.K * 4));
  if (p.ns > 0 && D.K <= 8) {
    // staged: x_mid row and the K expert-output rows of each token
    constexpr int PER = MT_DEP_GROUP / MT_WARPS;
    const int first = s.first();
    const int mine = first < ng ? (ng - 1 - first) / s.G + 1 : 0;
    auto tok = [&](int j) {
      const int t = (first + (j / PER) * s.G) * MT_DEP_GROUP + warp + MT_WARPS * (j % PER);
      return t < D.T ? t : -1;
    };
    rp_begin(p);
    const int n = mine * PER;
    {
      // index table: lane j reads token j's rows and weights (one round trip)
      const int t = lane < n ? tok(lane) : -1;
      if (lane < RP_TBL && t >= 0)
        for (int k = 0; k < D.K; ++k) {
          sts_i32(p.tbl + 4u * (uint32_t)(lane * 2 * D.K + k), INVM[(long long)t * D.K + k]);
          sts_f32(p.tbl + 4u * (uint32_t)(lane * 2 * D.K + D.K + k), WGT[(long long)t * D.K + k]);
        }
      __syncwarp();
    }
    bool ok = true;
    with_nc(D.d, [&](auto NCc) {
      constexpr int NC = decltype(NCc)::value;
      Row<NC> g, x, acc, y, r;
      row_ld(g, gp, n4);
      ok = rp_run(
          p, n, abuf<ArenaHdr>(a, A_HDR), a.timeout_ns / 2, SITE_ROWPIPE + 2,
          [&](int j, uint32_t st, uint32_t bar) {
            // header: t, then K weights
            const int t = tok(j);
            sts_i32(st, t);
            if (t < 0) { mbar_arrive(bar); return; }
            mbar_expect_tx(bar, (uint32_t)(1 + D.K) * rowb);
            bulk_g2s(st + RP_HDR, XM + (long long)t * D.d, rowb, bar);
            for (int k = 0; k < D.K; ++k) {
              int pr;
              float w;
              if (j < RP_TBL) {
                pr = lds_i32(p.tbl + 4u * (uint32_t)(j * 2 * D.K + k));
                w = lds_f32(p.tbl + 4u * (uint32_t)(j * 2 * D.K + D.K + k));
              } else {
                pr = INVM[(long long)t * D.K + k];
                w = WGT[(long long)t * D.K + k];
              }
              sts_f32(st + 4u * (1 + k), w);
              bulk_g2s(st + RP_HDR + (1 + k) * rowb, Y + (long long)pr * D.d, rowb, bar);
            }
          },
          [&](int j, uint32_t st) {
            const int t = lds_i32(st);
            if (t < 0) return;
            row_lds(x, st + RP_HDR, n4);
            row_scale(acc, x, 0.f);
            for (int k = 0; k < D.K; ++k) {
              row_lds(y, st + RP_HDR + (1 + k) * rowb, n4);
              row_axpy(acc, y, lds_f32(st + 4u * (1 + k)));
            }
            row_add(x, acc);
            row_st(Xn + (long long)t * D.d, x, n4);
            const float inv = row_rms_inv(x, D.d, a.norm_eps);
            row_norm_apply(r, x, inv, g);
            row_st_op(Rn + (long long)t * D.d, r, n4);
            if (lane == 0) invn[t] = inv;
          },
          [&](int j) {
            if (dsig && j % PER == PER - 1) {
              __syncthreads();
              if (threadIdx.x == 0) dep_signal(dsig + (first + (j / PER) * s.G) * MT_DEP_GROUP / MT_TILE_M);
            }
          });
    });
    rp_end(p, ok);
    s.next(ng);
    return;
  }
  with_nc(D.d, [&](auto NCc) {
    constexpr int NC = decltype(NCc)::value;
    Row<NC> g, x, acc, y, r;
    row_ld(g, gp, n4);
    for (int gi = s.first(); gi < ng; gi += s.G) {
    const int tend = min(D.T, (gi + 1) * MT_DEP_GROUP);
    for (int t = gi * MT_DEP_GROUP + (threadIdx.x >> 5); t < tend; t += MT_WARPS) {
      row_ld(x, XM + (long long)t * D.d, n4);
      row_scale(acc, x, 0.f);
      for (int k = 0; k < D.K; ++k) {
        const int p = INVM[(long long)t * D.K + k];
        row_ld(y, Y + (long long)p * D.d, n4);
        row_axpy(acc, y, WGT[(long long)t * D.K + k]);
      }
      row_add(x, acc);
      row_st(Xn + (long long)t * D.d, x, n4);
      const float inv = row_rms_inv(x, D.d, a.norm_eps);
      row_norm_apply(r, x, inv, g);
      row_st_op(Rn + (long long)t * D.d, r, n4);
      if (lane == 0) invn[t] = inv;
    }
    if (dsig) {
      __syncthreads();
      if (threadIdx.x == 0) dep_signal(dsig + gi * MT_DEP_GROUP / MT_TILE_M);
    }
    }
  });
  s.next(ng);
}

// Cross-entropy with its gradient, fused with the LM-head product: the
// product's epilogue left the logits (operand type) and, per column tile,
// the max and sum of exp(logit - max) of the fp32 accumulators, plus the
// target's fp32 logit.  Per position: lse from the tile partials,
// loss = coef * (lse - logit[target]), and the logits row is overwritten in
// place by dlogits = coef * (softmax - onehot).  Position s predicts token
// s+1; the last position of a sequence has no target (zero loss and gradient).
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4(__nv_bfloat16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}
template <class OP>
__device__ __noinline__ void job_ce(const KArgs& a, Sched& s, char* smem) {
  const MtDims& D = a.D;
  const int lane = threadIdx.x & 31;
  OP* DL = abuf<OP>(a, A_DLOGITS);
  const float* PART = abuf<float>(a, A_CEPART);
  const float* TGT = abuf<float>(a, A_CETGT);
  float* TL = abuf<float>(a, A_TOKLOSS);
  const int np = ce_parts<OP>(a);
  const int nw = s.G * MT_WARPS;
  const int v4 = D.V / 4;                 // V % 8 == 0 (checked on the host)
  if constexpr (sizeof(OP) == 2) {
    // bf16 logits: each warp streams its rows in chunks of CK logits through
    // a ring of shared-memory stages - bulk load, dlogits computed in place,
    // bulk store back over the logits; the next row's column-tile partials
    // are fetched into registers while the current row streams
    constexpr int CK = 4096;
    constexpr int PQ = 8;                 // partials per lane (np <= 256)
    const RowPipe p = rp_make(smem, RP_WIN_OFF, (uint32_t)a.smem_bytes, CK * 2u);
    if (p.ns > 0 && np <= 32 * PQ) {
      const int nck = (D.V + CK - 1) / CK;
      const int r0 = s.first() * MT_WARPS + (threadIdx.x >> 5);
      const int nrow = r0 < D.T ? (D.T - 1 - r0) / nw + 1 : 0;
      const int n = nrow * nck;
      auto row_of = [&](int j) { return r0 + (j / nck) * nw; };
      auto gptr = [&](int j) { return DL + (long long)row_of(j) * D.V + (long long)(j % nck) * CK; };
      auto nbytes = [&](int j) { return (uint32_t)min(CK, D.V - (j % nck) * CK) * 2u; };
      auto load = [&](int j) {              // lane 0
        mbar_expect_tx(p.sbar(j), nbytes(j));
        bulk_g2s(p.stage(j), gptr(j), nbytes(j), p.sbar(j));
      };
      float pm[PQ], ps[PQ];
      auto fetch_parts = [&](int t) {
#pragma unroll
        for (int q = 0; q < PQ; ++q) {
          const int i = lane + 32 * q;
          pm[q] = (i < np) ? PART[((long long)t * np + i) * 2] : -INFINITY;
          ps[q] = (i < np) ? PART[((long long)t * np + i) * 2 + 1] : 0.f;
        }
      };
      rp_begin(p);
      if (lane == 0)
        for (int j = 0; j < n && j < p.ns; ++j) load(j);
      __syncwarp();
      if (nrow > 0) fetch_parts(r0);
      bool ok = true;
      float lse = 0.f;
      int target = -1;
      bool has = false;
      for (int j = 0; j < n; ++j) {
        const int k = j % nck, t = row_of(j);
        if (k == 0) {
          // log-sum-exp of row t from its partials (the same order as the
          // register path), then the next row's partials
          has = (t % D.S) != D.S - 1;
          target = has ? a.tokens[t + 1] : -1;
          if (has && (target < 0 || target >= D.V)) target = 0;
          float m = -INFINITY, sum = 0.f;
#pragma unroll
          for (int q = 0; q < PQ; ++q) {
            const float nm = fmaxf(m, pm[q]);
            sum = (m == -INFINITY ? 0.f : sum * expf(m - nm)) + (pm[q] == -INFINITY ? 0.f : ps[q] * expf(pm[q] - nm));
            m = nm;
          }
          const float M = warp_max(m);
          sum = (m == -INFINITY) ? 0.f : sum * expf(m - M);
          sum = warp_sum(sum);
          lse = M + logf(sum);
          if (j + nck < n) fetch_parts(row_of(j + nck));
          if (lane == 0) TL[t] = has ? a.coef * (lse - TGT[t]) : 0.f;
        }
        if (ok && !mbar_wait(p.sbar(j), p.parity(j), a.timeout_ns)) {
          set_error(abuf<ArenaHdr>(a, A_HDR), MT_ERR_DEVICE_TIMEOUT, SITE_ROWPIPE + 10);
          ok = false;
        }
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          const uint32_t st = p.stage(j);
          const int nu = (int)(nbytes(j) / 16u), c0 = k * CK;
          // coef exp(x - lse) = 2^(x log2 e + (log2 coef - lse log2 e)): one
          // two-wide FMA per pair of logits and the special-function unit's
          // 2^x; a row without a target gets zeros
          const float sh = has ? log2f(a.coef) - lse * EPI_LOG2E : -INFINITY;
          const uint64_t l2e2 = f2(EPI_LOG2E, EPI_LOG2E), sh2 = f2(sh, sh);
          const int tu = (target - c0) >> 3;     // the 16-byte group holding the target (if any)
          for (int u = lane; u < nu; u += 32) {
            uint4 q;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(q.x), "=r"(q.y), "=r"(q.z), "=r"(q.w) : "r"(st + 16u * u));
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
            float pv[8];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              float t0, t1;
              unf2(fma2(f2(__uint_as_float(w[h] << 16), __uint_as_float(w[h] & 0xFFFF0000u)),
                                          l2e2, sh2), t0, t1);
              pv[2 * h] = epi_ex2(t0);
              pv[2 * h + 1] = epi_ex2(t1);
            }
            if (u == tu && target >= 0) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (c0 + 8 * u + i == target) pv[i] -= a.coef;
            }
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(st + 16u * u), "r"(bf2(pv[0], pv[1])),
                         "r"(bf2(pv[2], pv[3])), "r"(bf2(pv[4], pv[5])), "r"(bf2(pv[6], pv[7])) : "memory");
          }
          // the dlogits of the stage are read by the bulk store (async proxy)
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if (lane == 0 && ok) {
          bulk_s2g(gptr(j), p.stage(j), nbytes(j));
          bulk_commit();
          if (j + p.ns < n) {
            bulk_wait_read0();
            load(j + p.ns);
          }
        }
        __syncwarp();
      }
      if (lane == 0) {
        bulk_wait_all0();
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      rp_end(p, ok);
      s.next(s.G);
      return;
    }
  }
  constexpr int U = sizeof(OP) == 2 ? 16 : 8;   // 16-byte loads in flight per lane
  for (int t = s.first() * MT_WARPS + (threadIdx.x >> 5); t < D.T; t += nw) {
    OP* row = DL + (long long)t * D.V;
    const bool has = (t % D.S) != D.S - 1;
    if (!has) {
      for (int j = lane; j < v4; j += 32) st4(row + 4 * j, make_float4(0.f, 0.f, 0.f, 0.f));
      if (lane == 0) TL[t] = 0.f;
      continue;
    }
    int target = a.tokens[t + 1];
    if (target < 0 || target >= D.V) target = 0;   // reported by job_embed; never read outside the row
    float m = -INFINITY, sum = 0.f;
    for (int i = lane; i < np; i += 32) {
      const float pm = PART[((long long)t * np + i) * 2], ps = PART[((long long)t * np + i) * 2 + 1];
      const float nm = fmaxf(m, pm);
      sum = (m == -INFINITY ? 0.f : sum * expf(m - nm)) + (pm == -INFINITY ? 0.f : ps * expf(pm - nm));
      m = nm;
    }
    const float M = warp_max(m);
    sum = (m == -INFINITY) ? 0.f : sum * expf(m - M);
    sum = warp_sum(sum);
    const float lse = M + logf(sum);
    if constexpr (sizeof(OP) == 2) {
      // bf16 logits: 16-byte groups of 8, U groups in flight per lane
      const int v8 = D.V / 8;
      for (int j0 = 0; j0 < v8; j0 += 32 * U) {
        uint4 q[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = j0 + lane + 32 * u;
          if (j < v8) q[u] = reinterpret_cast<const uint4*>(row)[j];
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = j0 + lane + 32 * u;
          if (j < v8) {
            const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
            uint32_t o[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[h]));
              float p0 = a.coef * __expf(x.x - lse), p1 = a.coef * __expf(x.y - lse);
              if (target == 8 * j + 2 * h) p0 -= a.coef;
              if (target == 8 * j + 2 * h + 1) p1 -= a.coef;
              __nv_bfloat162 r = __floats2bfloat162_rn(p0, p1);
              o[h] = *reinterpret_cast<uint32_t*>(&r);
            }
            reinterpret_cast<uint4*>(row)[j] = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      }
    } else {
      for (int j0 = 0; j0 < v4; j0 += 32 * U) {
        float4 q[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = j0 + lane + 32 * u;
          if (j < v4) q[u] = ld4(row + 4 * j);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = j0 + lane + 32 * u;
          if (j < v4) {
            float4 p = make_float4(a.coef * __expf(q[u].x - lse), a.coef * __expf(q[u].y - lse),
                                   a.coef * __expf(q[u].z - lse), a.coef * __expf(q[u].w - lse));
            if ((target >> 2) == j) {
              const int c = target & 3;
              if (c == 0) p.x -= a.coef;
              else if (c == 1) p.y -= a.coef;
              else if (c == 2) p.z -= a.coef;
              else p.w -= a.coef;
            }
            st4(row + 4 * j, p);
          }
        }
      }
    }
    if (lane == 0) TL[t] = a.coef * (lse - TGT[t]);
  }
  s.next(s.G);
}

// ===========================================================================
// backward row jobs
// ===========================================================================
// Norm-gain gradient sum_t dy_t * xhat_t, fused with the norm backward:
// each warp keeps a register partial over its tokens (token order); at the
// end of the job the CTA adds its warps' partials in warp order and stores
// them as PART[cta][E+1][:]; a later phase sums the CTAs in CTA order.
template <int NC>
__device__ __forceinline__ void row_gain_acc(Row<NC>& acc, const Row<NC>& dy, const Row<NC>& x, float inv) {
  const uint64_t i2 = f2(inv, inv);
#pragma unroll
  for (int i = 0; i < NC; ++i)
    acc.v[i] = join2(fma2(lo2(dy.v[i]), mul2(lo2(x.v[i]), i2), lo2(acc.v[i])),
                     fma2(hi2(dy.v[i]), mul2(hi2(x.v[i]), i2), hi2(acc.v[i])));
}
template <int NC>
__device__ __forceinline__ void gain_partial_store(const KArgs& a, const Row<NC>& acc, char* smem) {
  const MtDims& D = a.D;
  const int warp = threadIdx.x >> 5, n4 = D.d / 4;
  float* sw = reinterpret_cast<float*>(smem + RP_WIN_OFF);   // [MT_WARPS][d]
  __syncthreads();
  row_st(sw + warp * D.d, acc, n4);
  __syncthreads();
  float* out = abuf<float>(a, A_PART) + ((long long)blockIdx.x * (D.E + 2) + D.E + 1) * D.d;
  for (int c = threadIdx.x; c < D.d; c += MT_THREADS) {
    float v = 0.f;
    for (int w = 0; w < MT_WARPS; ++w) v += sw[w * D.d + c];
    out[c] = v;
  }
  __syncthreads();
}

// dx = d(final RMSNorm) from d rf.
template <class OP>
__device__ __noinline__ void job_final_norm_bwd(const KArgs& a, Sched& s, char* smem) {
  const MtDims& D = a.D;
  const float* DRF = abuf<float>(a, A_DRF);
  const float* X = abuf<float>(a, A_X) + (long long)D.L * D.T * D.d;
  const float* inv = abuf<float>(a, A_INVF);
  float* DX = abuf<float>(a, A_DX);
  const int n4 = D.d / 4, nw = s.G * MT_WARPS;
  const int me = s.first() * MT_WARPS + (threadIdx.x >> 5);
  const uint32_t rowb = (uint32_t)D.d * 4u;
  const RowPipe p = rp_make(smem, RP_WIN_OFF, (uint32_t)a.smem_bytes, 2u * rowb);
  if (p.ns > 0) rp_begin(p);
  bool ok = true;
  with_nc(D.d, [&](auto NCc) {
    constexpr int NC = decltype(NCc)::value;
    Row<NC> g, dy, x, dx, acc;
    row_ld(g, pmaster(a, P_FINAL_NORM), n4);
    row_scale(acc, g, 0.f);
    if (p.ns > 0) {
      // staged: d rf and x rows of each token; header: t, 1/rms
      const int n = me < D.T ? (D.T - 1 - me) / nw + 1 : 0;
      ok = rp_run(
          p, n, abuf<ArenaHdr>(a, A_HDR), a.timeout_ns / 2, SITE_ROWPIPE + 7,
          [&](int j, uint32_t st, uint32_t bar) {
            const int t = me + j * nw;
            sts_i32(st, t);
            sts_f32(st + 4u, inv[t]);
            mbar_expect_tx(bar, 2u * rowb);
            bulk_g2s(st + RP_HDR, DRF + (long long)t * D.d, rowb, bar);
            bulk_g2s(st + RP_HDR + rowb, X + (long long)t * D.d, rowb, bar);
          },
          [&](int j, uint32_t st) {
            const int t = lds_i32(st);
            const float iv = lds_f32(st + 4u);
            row_lds(dy, st + RP_HDR, n4);
            row_lds(x, st + RP_HDR + rowb, n4);
            row_norm_bwd(dx, dy, x, iv, g, D.d);
            row_st(DX + (long long)t * D.d, dx, n4);
            row_gain_acc(acc, dy, x, iv);
          },
          [&](int) {});
    } else {
      for (int t = me; t < D.T; t += nw) {
        row_ld(dy, DRF + (long long)t * D.d, n4);
        row_ld(x, X + (long long)t * D.d, n4);
        const float iv = inv[t];
        row_norm_bwd(dx, dy, x, iv, g, D.d);
        row_st(DX + (long long)t * D.d, dx, n4);
        row_gain_acc(acc, dy, x, iv);
      }
    }
    if (p.ns > 0) rp_end(p, ok);
    gain_partial_store(a, acc, smem);
  });
  s.next(s.G);
}

// Expert-combine backward, part 1: dY[row] = w_k dx, dw_k = <dx, y_k>,
// router-logit gradient dz_i = w_i (dw_i - sum_j w_j dw_j) on the chosen
// experts (the renormalised weights are the softmax of the chosen logits),
// and zero pad rows of dY.  CTA c takes the token chunk the attention-norm
// backward gives it, so that every dx row it reads was written by the same
// CTA: the hand-off from the layer above needs no grid barrier.
template <class OP>
__device__ __noinline__ void job_moe_bwd1(const KArgs& a, int l, Sched& s, char* smem) {
  const MtDims& D = a.D;
  const int lane = threadIdx.x & 31, n4 = D.d / 4;
  const float* DX = abuf<float>(a, A_DX);
  const float* Y = abuf<float>(a, A_Y) + (long long)l * D.Pmax * D.d;
  const float* WGT = abuf<float>(a, A_WGT) + (long long)l * D.T * D.K;
  const int* IDX = abuf<int>(a, A_IDX) + (long long)l * D.T * D.K;
  const int* INVM = abuf<int>(a, A_INVM) + (long long)l * D.T * D.K;
  const int* OFFS = abuf<int>(a, A_OFFS) + (long long)l * (D.E + 1);
  OP* DY = abuf<OP>(a, A_DY);
  float* DZ = abuf<float>(a, A_DZ);
  __nv_bfloat16* DZB = abuf<__nv_bfloat16>(a, A_DZB);
  // tokens: the chunk [c ch, (c+1) ch) of CTA c, warp w its tokens t0 + w + 8 j
  const int ch = chunk_len(D, gridDim.x);
  const int t0 = (int)blockIdx.x * ch, t1 = min(D.T, t0 + ch);
  const int me = t0 + (threadIdx.x >> 5), nw = MT_WARPS;
  // pad rows of dY: spread over every warp of the grid
  const int gnw = s.G * MT_WARPS, gme = s.first() * MT_WARPS + (threadIdx.x >> 5);
  const uint32_t rowb = (uint32_t)D.d * 4u;
  // index table: per token of the warp (first RP_TBL), its K sorted rows,
  // K weights and K experts (the layout of the stage header after t)
  const RowPipe p = rp_make(smem, RP_WIN_OFF, (uint32_t)a.smem_bytes, (uint32_t)(1 + D.K) * rowb,
                            (uint32_t)(RP_TBL * 3 * D.K * 4));
  const bool piped = p.ns > 0 && D.K <= 8;
  // the chunk's dx rows were stored by this CTA's warps in the previous job
  // (rp_begin also orders them before the bulk loads)
  if (piped) rp_begin(p);
  else __syncthreads();
  bool ok = true;
  with_nc(D.d, [&](auto NCc) {
    constexpr int NC = decltype(NCc)::value;
    Row<NC> dx, y, dy;
    if (piped) {
      // staged: the dx row and the K expert-output rows of each token;
      // header: t, then K sorted rows, K weights, K experts
      const int n = me < t1 ? (t1 - 1 - me) / nw + 1 : 0;
      if (lane < RP_TBL && lane < n) {
        const int t = me + lane * nw;
        for (int k = 0; k < D.K; ++k) {
          sts_i32(p.tbl + 4u * (uint32_t)(lane * 3 * D.K + k), INVM[(long long)t * D.K + k]);
          sts_f32(p.tbl + 4u * (uint32_t)(lane * 3 * D.K + D.K + k), WGT[(long long)t * D.K + k]);
          sts_i32(p.tbl + 4u * (uint32_t)(lane * 3 * D.K + 2 * D.K + k), IDX[(long long)t * D.K + k]);
        }
      }
      __syncwarp();
      ok = rp_run(
          p, n, abuf<ArenaHdr>(a, A_HDR), a.timeout_ns / 2, SITE_ROWPIPE + 3,
          [&](int j, uint32_t st, uint32_t bar) {
            const int t = me + j * nw;
            sts_i32(st, t);
            mbar_expect_tx(bar, (uint32_t)(1 + D.K) * rowb);
            bulk_g2s(st + RP_HDR, DX + (long long)t * D.d, rowb, bar);
            for (int k = 0; k < D.K; ++k) {
              int pr, e;
              float w;
              if (j < RP_TBL) {
                const uint32_t tr = p.tbl + 4u * (uint32_t)(j * 3 * D.K);
                pr = lds_i32(tr + 4u * k);
                w = lds_f32(tr + 4u * (D.K + k));
                e = lds_i32(tr + 4u * (2 * D.K + k));
              } else {
                pr = INVM[(long long)t * D.K + k];
                w = WGT[(long long)t * D.K + k];
                e = IDX[(long long)t * D.K + k];
              }
              sts_i32(st + 4u * (1 + k), pr);
              sts_f32(st + 4u * (1 + D.K + k), w);
              sts_i32(st + 4u * (1 + 2 * D.K + k), e);
              bulk_g2s(st + RP_HDR + (1 + k) * rowb, Y + (long long)pr * D.d, rowb, bar);
            }
          },
          [&](int j, uint32_t st) {
            const int t = lds_i32(st);
            row_lds(dx, st + RP_HDR, n4);
            // sum_k w_k dw_k, then dz_e = w_k (dw_k - mean) for the chosen e
            float mean = 0.f;
            float dzl = 0.f, dzh = 0.f;   // experts lane and lane + 32
            float dwk[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              if (k < D.K) {
                row_lds(y, st + RP_HDR + (1 + k) * rowb, n4);
                const float w = lds_f32(st + 4u * (1 + D.K + k));
                dwk[k] = row_dot(dx, y);
                mean = fmaf(w, dwk[k], mean);
                row_scale(dy, dx, w);
                row_st_op(DY + (long long)lds_i32(st + 4u * (1 + k)) * D.d, dy, n4);
              }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              if (k < D.K) {
                const int e = lds_i32(st + 4u * (1 + 2 * D.K + k));
                const float v = lds_f32(st + 4u * (1 + D.K + k)) * (dwk[k] - mean);
                if (e == lane) dzl = v;
                if (e == lane + 32) dzh = v;
              }
            }
            if (lane < D.E) DZ[(long long)t * D.E + lane] = dzl;
            if (lane + 32 < D.E) DZ[(long long)t * D.E + lane + 32] = dzh;
            if constexpr (sizeof(OP) == 2) {
              // bf16 operand copy for the router-weight gradient product
              // (the lanes of absent experts hold 0)
              DZB[(long long)t * 64 + lane] = __float2bfloat16_rn(dzl);
              DZB[(long long)t * 64 + lane + 32] = __float2bfloat16_rn(dzh);
            }
          },
          [&](int) {});
    } else {
      for (int t = me; t < t1; t += nw) {
        row_ld(dx, DX + (long long)t * D.d, n4);
        float dw[8], w[8];
        for (int k = 0; k < D.K; ++k) {
          const int p = INVM[(long long)t * D.K + k];
          w[k] = WGT[(long long)t * D.K + k];
          row_ld(y, Y + (long long)p * D.d, n4);
          dw[k] = row_dot(dx, y);
          row_scale(dy, dx, w[k]);
          row_st_op(DY + (long long)p * D.d, dy, n4);
        }
        float mean = 0.f;
        for (int k = 0; k < D.K; ++k) mean = fmaf(w[k], dw[k], mean);
        for (int e = lane; e < 64; e += 32) {
          float v = 0.f;
          for (int k = 0; k < D.K; ++k)
            if (IDX[(long long)t * D.K + k] == e) v = w[k] * (dw[k] - mean);
          if (e < D.E) DZ[(long long)t * D.E + e] = v;
          if constexpr (sizeof(OP) == 2) DZB[(long long)t * 64 + e] = __float2bfloat16_rn(v);
        }
      }
    }
    // pad rows of dY: [OFFS[e] + n_e, OFFS[e+1]) of every expert segment,
    // n_e = rows routed to e (the route job's totals); the segment bounds
    // are read once per warp, two experts per lane
#pragma unroll
    for (int i = 0; i < NC; ++i) dy.v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int* ncnt = abuf<ArenaHdr>(a, A_HDR)->expert_counts + l * MT_MAX_EXPERTS;
    int lo0 = 0, hi0 = 0, lo1 = 0, hi1 = 0;
    if (lane < D.E) { lo0 = OFFS[lane] + ncnt[lane]; hi0 = OFFS[lane + 1]; }
    if (lane + 32 < D.E) { lo1 = OFFS[lane + 32] + ncnt[lane + 32]; hi1 = OFFS[lane + 33]; }
    for (int e = 0; e < D.E; ++e) {
      const int p0 = __shfl_sync(0xffffffffu, e < 32 ? lo0 : lo1, e & 31);
      const int p1 = __shfl_sync(0xffffffffu, e < 32 ? hi0 : hi1, e & 31);
      for (int p = p0 + gme; p < p1; p += gnw) row_st_op(DY + (long long)p * D.d, dy, n4);
    }
  });
  if (piped) rp_end(p, ok);
  s.next(s.G);
}

// Expert-combine backward, part 2: the gather backward as a direct per-row
// sum (each token has exactly K contributions, summed in slot order, no
// atomics - "Open problems", Performance item 5), plus the router term
// dz Wr, then the expert RMSNorm backward into dx, and the operand copy of dx.
template <class OP>
__device__ __noinline__ void job_moe_bwd2(const KArgs& a, int l, Sched& s, char* smem) {
  const MtDims& D = a.D;
  const int n4 = D.d / 4;
  const int lane = threadIdx.x & 31;
  const float* DXS = abuf<float>(a, A_DXS);
  const float* DZ = abuf<float>(a, A_DZ);
  const int* INVM = abuf<int>(a, A_INVM) + (long long)l * D.T * D.K;
  const int* IDX = abuf<int>(a, A_IDX) + (long long)l * D.T * D.K;
  const float* Wr = pmaster(a, P_ROUTER) + (long long)wslot(a, l) * D.E * D.d;
  const float* XM = abuf<float>(a, A_XM) + (long long)l * D.T * D.d;
  const float* inv2 = abuf<float>(a, A_INV2) + (long long)l * D.T;
  float* DX = abuf<float>(a, A_DX);
  OP* DXO = abuf<OP>(a, A_DXO);
  const int nw = s.G * MT_WARPS;
  const int me = s.first() * MT_WARPS + (threadIdx.x >> 5);
  const uint32_t rowb = (uint32_t)D.d * 4u;
  // index table: per token of the warp (first RP_TBL), 1/rms, then its K
  // sorted rows, experts (ascending) and router-logit gradients
  const RowPipe p = rp_make(smem, RP_WIN_OFF, (uint32_t)a.smem_bytes, (uint32_t)(D.K + 2) * rowb,
                            (uint32_t)(RP_TBL * (1 + 3 * D.K) * 4));
  const bool piped = p.ns > 0 && D.K <= 8;
  if (piped) rp_begin(p);
  bool ok = true;
  with_nc(D.d, [&](auto NCc) {
    constexpr int NC = decltype(NCc)::value;
    Row<NC> g, dr2, tmp, x, dx, gacc;
    row_ld(g, pmaster(a, P_MOE_NORM) + (long long)wslot(a, l) * D.d, n4);
    row_scale(gacc, g, 0.f);
    if (piped) {
      // staged: the K expert-input gradient rows, x_mid and dx of each token;
      // header: t, 1/rms, then the chosen experts in ascending order with
      // their router-logit gradients
      const int n = me < D.T ? (D.T - 1 - me) / nw + 1 : 0;
      // index table row of token j: [1/rms, K sorted rows, K experts ascending,
      // K router-logit gradients] - lane j fills row j (two round trips)
      auto fill = [&](int j, uint32_t row) {
        const int t = me + j * nw;
        sts_f32(row, inv2[t]);
        int ex[8];
        for (int k = 0; k < D.K; ++k) {
          sts_i32(row + 4u * (1 + k), INVM[(long long)t * D.K + k]);
          int e = IDX[(long long)t * D.K + k], q = k;
          while (q > 0 && ex[q - 1] > e) { ex[q] = ex[q - 1]; --q; }
          ex[q] = e;
        }
        for (int k = 0; k < D.K; ++k) {
          sts_i32(row + 4u * (1 + D.K + k), ex[k]);
          sts_f32(row + 4u * (1 + 2 * D.K + k), DZ[(long long)t * D.E + ex[k]]);
        }
      };
      const uint32_t tw = 4u * (uint32_t)(1 + 3 * D.K);   // table row bytes
      if (lane < RP_TBL && lane < n) fill(lane, p.tbl + (uint32_t)lane * tw);
      __syncwarp();
      ok = rp_run(
          p, n, abuf<ArenaHdr>(a, A_HDR), a.timeout_ns / 2, SITE_ROWPIPE + 4,
          [&](int j, uint32_t st, uint32_t bar) {
            const int t = me + j * nw;
            // the header takes the table row; tokens past the table reuse row
            // j % RP_TBL (its token was issued long before) and fill it here
            const uint32_t row = p.tbl + (uint32_t)(j % RP_TBL) * tw;
            if (j >= RP_TBL) fill(j, row);
            sts_i32(st, t);
            sts_f32(st + 4u, lds_f32(row));
            mbar_expect_tx(bar, (uint32_t)(D.K + 2) * rowb);
            for (int k = 0; k < D.K; ++k)
              bulk_g2s(st + RP_HDR + k * rowb, DXS + (long long)lds_i32(row + 4u * (1 + k)) * D.d, rowb, bar);
            bulk_g2s(st + RP_HDR + D.K * rowb, XM + (long long)t * D.d, rowb, bar);
            bulk_g2s(st + RP_HDR + (D.K + 1) * rowb, DX + (long long)t * D.d, rowb, bar);
            for (int k = 0; k < D.K; ++k) {
              sts_i32(st + 4u * (2 + k), lds_i32(row + 4u * (1 + D.K + k)));
              sts_f32(st + 4u * (2 + D.K + k), lds_f32(row + 4u * (1 + 2 * D.K + k)));
            }
          },
          [&](int j, uint32_t st) {
            const int t = lds_i32(st);
            row_lds(dr2, st + RP_HDR, n4);
            for (int k = 1; k < D.K; ++k) row_add_lds(dr2, st + RP_HDR + k * rowb, n4);
            for (int k = 0; k < D.K; ++k) {
              const float ze = lds_f32(st + 4u * (2 + D.K + k));
              if (ze != 0.f) {
                row_ld(tmp, Wr + (long long)lds_i32(st + 4u * (2 + k)) * D.d, n4);
                row_axpy(dr2, tmp, ze);
              }
            }
            row_lds(x, st + RP_HDR + D.K * rowb, n4);
            const float iv = lds_f32(st + 4u);
            row_gain_acc(gacc, dr2, x, iv);
            row_lds(dx, st + RP_HDR + (D.K + 1) * rowb, n4);
            row_norm_bwd_add(dx, dr2, x, iv, g, D.d);
            row_st(DX + (long long)t * D.d, dx, n4);
            row_st_op(DXO + (long long)t * D.d, dx, n4);
          },
          [&](int) {});
    } else {
      for (int t = me; t < D.T; t += nw) {
        row_scale(dr2, g, 0.f);
        for (int k = 0; k < D.K; ++k) {
          row_ld(tmp, DXS + (long long)INVM[(long long)t * D.K + k] * D.d, n4);
          row_add(dr2, tmp);
        }
        const float* dz = DZ + (long long)t * D.E;
        for (int e = 0; e < D.E; ++e) {
          const float ze = dz[e];
          if (ze != 0.f) {
            row_ld(tmp, Wr + (long long)e * D.d, n4);
            row_axpy(dr2, tmp, ze);
          }
        }
        row_ld(x, XM + (long long)t * D.d, n4);
        row_ld(dx, DX + (long long)t * D.d, n4);
        const float iv = inv2[t];
        row_gain_acc(gacc, dr2, x, iv);
        row_norm_bwd_add(dx, dr2, x, iv, g, D.d);
        row_st(DX + (long long)t * D.d, dx, n4);
        row_st_op(DXO + (long long)t * D.d, dx, n4);
      }
    }
    if (piped) rp_end(p, ok);
    gain_partial_store(a, gacc, smem);
  });
  s.next(s.G);
}

// Attention RMSNorm backward into dx.
template <class OP>
__device__ __noinline__ void job_attn_norm_bwd(const KArgs& a, int l, Sched& s, char* smem, const unsigned* dw,
                                              unsigned dtarget) {
  const MtDims& D = a.D;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* DR = abuf<float>(a, A_DR);
  const float* X = abuf<float>(a, A_X) + (long long)l * D.T * D.d;
  const float* inv = abuf<float>(a, A_INV1) + (long long)l * D.T;
  float* DX = abuf<float>(a, A_DX);
  const int n4 = D.d / 4;
  // CTA c takes the token chunk [c ch, (c+1) ch); warp w its tokens t0 + w + 8 j
  const int c = blockIdx.x, ch = chunk_len(D, gridDim.x);
  const int t0 = c * ch, t1 = min(D.T, t0 + ch);
  const int me = t0 + warp, nw = MT_WARPS;
  const uint32_t rowb = (uint32_t)D.d * 4u;
  const RowPipe p = rp_make(smem, RP_WIN_OFF, (uint32_t)a.smem_bytes, 3u * rowb, RP_TBL * 4u);
  if (p.ns > 0) rp_begin(p);
  else __syncthreads();
  if (dw && t0 < t1) {
    // the chunk's dR rows are stored by qkv dgrad tiles of other CTAs
    const int b0 = t0 / MT_TILE_M, nb = (t1 - 1) / MT_TILE_M - b0 + 1;
    if (threadIdx.x < nb) dep_wait(abuf<ArenaHdr>(a, A_HDR), dw + b0 + threadIdx.x, dtarget, a.timeout_ns);
  }
  __syncthreads();
  if (dw && p.ns > 0 && lane == 0) asm volatile("fence.proxy.async;" ::: "memory");   // bulk loads after the acquire
  bool ok = true;
  with_nc(D.d, [&](auto NCc) {
    constexpr int NC = decltype(NCc)::value;
    Row<NC> g, dy, x, dx, acc, gacc;
    row_ld(g, pmaster(a, P_ATTN_NORM) + (long long)wslot(a, l) * D.d, n4);
    row_scale(gacc, g, 0.f);
    if (p.ns > 0) {
      // staged: dr, x and dx rows of each token; header: t, 1/rms (1/rms of
      // the warp's first RP_TBL tokens read up front into the table)
      const int n = me < t1 ? (t1 - 1 - me) / nw + 1 : 0;
      if (lane < RP_TBL && lane < n) sts_f32(p.tbl + 4u * lane, inv[me + lane * nw]);
      __syncwarp();
      ok = rp_run(
          p, n, abuf<ArenaHdr>(a, A_HDR), a.timeout_ns / 2, SITE_ROWPIPE + 5,
          [&](int j, uint32_t st, uint32_t bar) {
            const int t = me + j * nw;
            sts_i32(st, t);
            sts_f32(st + 4u, j < RP_TBL ? lds_f32(p.tbl + 4u * j) : inv[t]);
            mbar_expect_tx(bar, 3u * rowb);
            bulk_g2s(st + RP_HDR, DR + (long long)t * D.d, rowb, bar);
            bulk_g2s(st + RP_HDR + rowb, X + (long long)t * D.d, rowb, bar);
            bulk_g2s(st + RP_HDR + 2u * rowb, DX + (long long)t * D.d, rowb, bar);
          },
          [&](int j, uint32_t st) {
            const int t = lds_i32(st);
            row_lds(dy, st + RP_HDR, n4);
            row_lds(x, st + RP_HDR + rowb, n4);
            row_lds(acc, st + RP_HDR + 2u * rowb, n4);
            const float iv = lds_f32(st + 4u);
            row_norm_bwd(dx, dy, x, iv, g, D.d);
            row_add(acc, dx);
            row_st(DX + (long long)t * D.d, acc, n4);
            row_gain_acc(gacc, dy, x, iv);
          },
          [&](int) {});
    } else {
      for (int t = me; t < t1; t += nw) {
        row_ld(dy, DR + (long long)t * D.d, n4);
        row_ld(x, X + (long long)t * D.d, n4);
        row_ld(acc, DX + (long long)t * D.d, n4);
        const float iv = inv[t];
        row_norm_bwd(dx, dy, x, iv, g, D.d);
        row_add(acc, dx);
        row_st(DX + (long long)t * D.d, acc, n4);
        row_gain_acc(gacc, dy, x, iv);
      }
    }
    if (p.ns > 0) rp_end(p, ok);
    gain_partial_store(a, gacc, smem);
  });
  s.next(s.G);
}

// ===========================================================================
// deterministic column reductions over tokens (norm gains, router weights)
// ===========================================================================
// Partial sums over token chunks written to PART[chunk][row][col]; a later
// phase adds the chunks in chunk order.  Inside a chunk, four token lanes
// each sum every fourth token in token order and are then added in lane
// order, so for a given grid the result is the same in every launch.  A
// thread owns CW adjacent columns and every output row of them (ER router
// rows plus the gain row); CW shrinks as the router rows grow so that the
// accumulators stay in registers.
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

#define COL_LANES 4
// columns per thread for a reduction with E router rows (0: gain only)
__device__ __forceinline__ int col_width(int E) { return E <= 16 ? 4 : (E <= 32 ? 2 : 1); }
// token chunks: about two items per CTA
__device__ __forceinline__ int col_nchunks(const MtDims& D, int G, int E) {
  const int cb = (MT_THREADS / COL_LANES) * col_width(E);
  const int ncb = (D.d + cb - 1) / cb;
  int n = (2 * G + ncb - 1) / ncb;
  if (n > D.nch) n = D.nch;
  if (n > D.T) n = D.T;
  return n < 1 ? 1 : n;
}

template <int CW>
__device__ __forceinline__ void ld_cols(float (&v)[CW], const float* p) {
  if constexpr (CW == 4) {
    const float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  } else if constexpr (CW == 2) {
    const float2 q = *reinterpret_cast<const float2*>(p);
    v[0] = q.x; v[1] = q.y;
  } else {
    v[0] = *p;
  }
}

template <int ER, int CW>
__device__ void colpart_items(const KArgs& a, const ColArgs& c, Sched& s, char* smem) {
  constexpr int TPL = MT_THREADS / COL_LANES;   // threads per token lane
  constexpr int CB = TPL * CW;                  // columns per item
  constexpr int U = 1;                          // tokens in flight per thread
  constexpr int SUB = 256;                      // tokens staged at a time
  const MtDims& D = a.D;
  const int G = s.G;
  const bool moe = (c.kind == COL_MOE);
  const bool gain = c.dy != nullptr;            // the gain row (else router rows only)
  const int E = moe ? D.E : 0;
  const int ncb = (D.d + CB - 1) / CB;
  const int nchunk = col_nchunks(D, G, E);
  const int ch = (D.T + nchunk - 1) / nchunk;
  const int items = ncb * nchunk;
  float* PART = abuf<float>(a, A_PART);
  float* s_inv = reinterpret_cast<float*>(smem + RP_WIN_OFF);   // [SUB]
  float* s_dz = s_inv + SUB;                    // [SUB][E]
  float* s_red = s_dz + SUB * E;                // [COL_LANES - 1][ER + 1][CB]
  const int tl = threadIdx.x / TPL, tc = threadIdx.x % TPL;
  for (int it = s.first(); it < items; it += G) {
    const int chunk = it / ncb, cb = it % ncb;
    const int col = cb * CB + tc * CW;
    const bool active = col < D.d;
    const int t0 = chunk * ch, t1 = min(D.T, t0 + ch);
    float acc[ER + 1][CW];
#pragma unroll
    for (int r = 0; r <= ER; ++r)
#pragma unroll
      for (int j = 0; j < CW; ++j) acc[r][j] = 0.f;
    float gcol[CW];
#pragma unroll
    for (int j = 0; j < CW; ++j) gcol[j] = 0.f;
    if (moe && active) ld_cols<CW>(gcol, c.g + col);
    for (int s0 = t0; s0 < t1; s0 += SUB) {
      const int n = min(SUB, t1 - s0);
      __syncthreads();
      for (int i = threadIdx.x; i < n; i += MT_THREADS) s_inv[i] = c.inv[s0 + i];
      if (moe)
        for (int i = threadIdx.x; i < n * E; i += MT_THREADS) s_dz[i] = c.dz[(long long)s0 * E + i];
      __syncthreads();
      if (!active) continue;
      for (int tb = tl; tb < n; tb += COL_LANES * U) {
        float xv[U][CW], dyv[U][CW];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int tk = tb + u * COL_LANES;
          if (tk < n) {
            const long long off = (long long)(s0 + tk) * D.d + col;
            ld_cols<CW>(xv[u], c.x + off);
            if (gain) ld_cols<CW>(dyv[u], c.dy + off);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int tk = tb + u * COL_LANES;
          if (tk < n) {
            const float iv = s_inv[tk];
#pragma unroll
            for (int j = 0; j < CW; ++j) {
              const float xh = xv[u][j] * iv;
              if (gain) acc[ER][j] = fmaf(dyv[u][j], xh, acc[ER][j]);      // gain gradient row
              if (ER > 0) {
                const float r2 = xh * gcol[j];
                const float* dz = s_dz + tk * E;
#pragma unroll
                for (int e = 0; e < ER; ++e)
                  if (e < E) acc[e][j] = fmaf(dz[e], r2, acc[e][j]);
              }
            }
          }
        }
      }
    }
    // add the token lanes in lane order
    if (tl > 0 && active) {
#pragma unroll
      for (int r = 0; r <= ER; ++r)
#pragma unroll
        for (int j = 0; j < CW; ++j) s_red[((tl - 1) * (ER + 1) + r) * CB + tc * CW + j] = acc[r][j];
    }
    __syncthreads();
    if (tl == 0 && active) {
      float* out = PART + ((long long)chunk * (D.E + 2) + c.row0) * D.d + col;
#pragma unroll
      for (int r = 0; r <= ER; ++r) {
        if (r < ER && r >= E) continue;
        if (r == ER && !gain) continue;
        const int orow = (r == ER) ? E : r;
#pragma unroll
        for (int j = 0; j < CW; ++j) {
          float v = acc[r][j];
#pragma unroll
          for (int q = 0; q < COL_LANES - 1; ++q) v += s_red[(q * (ER + 1) + r) * CB + tc * CW + j];
          out[(long long)orow * D.d + j] = v;
        }
      }
    }
    // the next item may be an empty chunk (no staging barrier) that writes s_red at once
    __syncthreads();
  }
  s.next(items);
}

static __device__ __noinline__ void job_colpart(const KArgs& a, const ColArgs& c, Sched& s, char* sm) {
  const int E = (c.kind == COL_MOE) ? a.D.E : 0;
  if (E <= 4) colpart_items<4, 4>(a, c, s, sm);
  else if (E <= 16) colpart_items<16, 4>(a, c, s, sm);
  else if (E <= 32) colpart_items<32, 2>(a, c, s, sm);
  else colpart_items<64, 1>(a, c, s, sm);
}

// Router-weight gradient partials dWr[e][c] = sum_t dz[t][e] r2[t][c] with
// r2 = x_mid * (1/rms) * g in fp32.  CTA c takes the token chunk of the
// routing jobs; its x_mid rows (and dz rows) are staged RG_TB tokens at a
// time by cp.async.bulk into a ring of CTA-wide stages; warp w owns the
// columns [w d/8, (w+1) d/8) and each lane keeps EM x 3 accumulators over
// the chunk in token order, then stores PART[cta][e][col] (no cross-warp
// reduction: the warps own disjoint columns).  Returns false when the ring
// does not fit (the caller then takes the column pass).
#define RG_TB 16
template <int EM>
__device__ __forceinline__ bool router_grad_cta(const KArgs& a, int l, char* smem) {
  const MtDims& D = a.D;
  const int c = blockIdx.x, G = gridDim.x;
  const int ch = chunk_len(D, G);
  const int t0 = c * ch, t1 = min(D.T, t0 + ch);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rowb = (uint32_t)D.d * 4u, dzb = (uint32_t)D.E * 4u;
  const uint32_t stage_bytes = ((uint32_t)RG_TB * (rowb + dzb) + 127u) & ~127u;
  int ns = (int)(((uint32_t)a.smem_bytes - RP_WIN_OFF) / stage_bytes);
  if (ns > 4) ns = 4;
  if (ns < 2 || (dzb & 15u)) return false;
  const float* XM = abuf<float>(a, A_XM) + (long long)l * D.T * D.d;
  const float* inv2 = abuf<float>(a, A_INV2) + (long long)l * D.T;
  const float* DZ = abuf<float>(a, A_DZ);
  const float* g = pmaster(a, P_MOE_NORM) + (long long)wslot(a, l) * D.d;
  constexpr int NCOL = 3;                       // columns per lane (d <= 768)
  const int cpw = D.d / MT_WARPS;
  int col[NCOL];
  float gc[NCOL];
#pragma unroll
  for (int i = 0; i < NCOL; ++i) {
    col[i] = warp * cpw + lane + 32 * i;
    gc[i] = (lane + 32 * i < cpw) ? g[col[i]] : 0.f;
  }
  float acc[EM][NCOL];
#pragma unroll
  for (int e = 0; e < EM; ++e)
#pragma unroll
    for (int i = 0; i < NCOL; ++i) acc[e][i] = 0.f;
  const uint32_t ring = smem_u32(smem) + RP_WIN_OFF, bar0 = smem_u32(&rp_bars[0]);
  ArenaHdr* hdr = abuf<ArenaHdr>(a, A_HDR);
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 0; i < ns; ++i) mbar_init(bar0 + 8u * i, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async;" ::: "memory");
  }
  __syncthreads();
  const int nb = t1 > t0 ? (t1 - t0 + RG_TB - 1) / RG_TB : 0;
  auto issue = [&](int b) {      // thread 0
    const int tb = t0 + b * RG_TB, nt = min(RG_TB, t1 - tb);
    const uint32_t st = ring + (uint32_t)(b % ns) * stage_bytes, bar = bar0 + 8u * (uint32_t)(b % ns);
    mbar_expect_tx(bar, (uint32_t)nt * (rowb + dzb));
    bulk_g2s(st + (uint32_t)RG_TB * rowb, DZ + (long long)tb * D.E, (uint32_t)nt * dzb, bar);
    bulk_g2s(st, XM + (long long)tb * D.d, (uint32_t)nt * rowb, bar);    // the batch's rows are contiguous
  };
  if (threadIdx.x == 0)
    for (int b = 0; b < nb && b < ns; ++b) issue(b);
  bool ok = true;
  for (int b = 0; b < nb; ++b) {
    const int tb = t0 + b * RG_TB, nt = min(RG_TB, t1 - tb);
    const float ivl = lane < nt ? inv2[tb + lane] : 0.f;     // 1/rms of the batch, lane r holds token r
    if (ok && !mbar_wait(bar0 + 8u * (uint32_t)(b % ns), (uint32_t)(b / ns) & 1u, a.timeout_ns)) {
      set_error(hdr, MT_ERR_DEVICE_TIMEOUT, SITE_ROWPIPE + 8);
      ok = false;
    }
    if (ok) {
      const uint32_t st = ring + (uint32_t)(b % ns) * stage_bytes;
      const uint32_t dzs = st + (uint32_t)RG_TB * rowb;
      for (int r = 0; r < nt; ++r) {
        const float iv = __shfl_sync(0xffffffffu, ivl, r);
        float rr[NCOL];
#pragma unroll
        for (int i = 0; i < NCOL; ++i)
          rr[i] = (lane + 32 * i < cpw) ? lds_f32(st + (uint32_t)r * rowb + 4u * (uint32_t)col[i]) * iv * gc[i] : 0.f;
#pragma unroll
        for (int e4 = 0; e4 < EM; e4 += 4) {
          if (e4 < D.E) {
            const float4 z = lds4(dzs + (uint32_t)(r * D.E + e4) * 4u);
            const float zz[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
              for (int i = 0; i < NCOL; ++i) acc[e4 + q][i] = fmaf(zz[q], rr[i], acc[e4 + q][i]);
          }
        }
      }
    }
    __syncthreads();
    if (ok && threadIdx.x == 0 && b + ns < nb) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the reads of this stage come first
      issue(b + ns);
    }
  }
  if (threadIdx.x == 0 && ok)
    for (int i = 0; i < ns; ++i) asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar0 + 8u * i) : "memory");
  float* out = abuf<float>(a, A_PART) + (long long)c * (D.E + 2) * D.d;
#pragma unroll
  for (int e = 0; e < EM; ++e)
    if (e < D.E)
#pragma unroll
      for (int i = 0; i < NCOL; ++i)
        if (lane + 32 * i < cpw) out[(long long)e * D.d + col[i]] = acc[e][i];
  __syncthreads();
  return true;
}
// Router-weight gradient partials of layer l: per-CTA rows (PART[cta][0..E))
// when the staged form fits, else the column pass (PART[chunk][0..E)).
// Returns the number of partial chunks for job_colfinal.
static __device__ __noinline__ int job_router_grad(const KArgs& a, int l, Sched& s, char* smem) {
  const MtDims& D = a.D;
  bool done = false;
  if (D.E % 4 == 0 && D.d % (8 * MT_WARPS) == 0 && D.d <= 768) {
    if (D.E <= 16) done = router_grad_cta<16>(a, l, smem);
    else if (D.E <= 32) done = router_grad_cta<32>(a, l, smem);
  }
  if (done) return (int)gridDim.x;
  ColArgs c{COL_MOE, nullptr, abuf<float>(a, A_XM) + (long long)l * D.T * D.d,
            abuf<float>(a, A_INV2) + (long long)l * D.T, pmaster(a, P_MOE_NORM) + (long long)wslot(a, l) * D.d,
            abuf<float>(a, A_DZ), 0};
  job_colpart(a, c, s, smem);
  return 0;
}


// out[r][col] (+)= sum over chunks of PART[chunk][row0 + r][col]; E_kind is
// the router-row count of the reduction that wrote those rows (0: gain only).
static __device__ __noinline__ void job_colfinal(const KArgs& a, int row0, int nrows, int E_kind, float* out_rows,
                                                 float* out_last, int last_is_separate, Sched& s, int nchunks,
                                                 bool acc) {
  const MtDims& D = a.D;
  const int G = s.G;
  const int nused = nchunks > 0 ? nchunks : col_nchunks(D, G, E_kind);
  const float* PART = abuf<float>(a, A_PART);
  const int n = nrows * D.d;
  // eight lanes per output: lane j of the group adds chunks j, j+8, ... in
  // order, then the group sums its eight partials by a fixed butterfly (so
  // every CTA takes part; a whole warp steps together for the shuffles)
  const long long total = (long long)n * 8;
  const long long nthr = (long long)G * MT_THREADS;
  const int lane = threadIdx.x & 31;
  for (long long base = (long long)s.first() * MT_THREADS + (threadIdx.x & ~31); base < total; base += nthr) {
    const long long w = base + lane;
    const int e = (int)(w >> 3), sub = (int)(w & 7);
    float v = 0.f;
    if (e < n) {
      const int r = e / D.d, col = e % D.d;
      for (int cc = sub; cc < nused; cc += 8) v += PART[((long long)cc * (D.E + 2) + row0 + r) * D.d + col];
    }
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    if (sub == 0 && e < n) {
      const int r = e / D.d, col = e % D.d;
      float* dst = (last_is_separate && r == nrows - 1) ? out_last + col : out_rows + e;
      *dst = acc ? *dst + v : v;
    }
  }
  s.next(G);
}

// ===========================================================================
// embedding backward: dE[v] (+)= sum over positions t with tok[t] = v of dx_t,
// in ascending t.  CTA c owns vocabulary rows [c*V/G, (c+1)*V/G).
// ===========================================================================
static __device__ __noinline__ void job_embed_bwd(const KArgs& a, int* ism) {
  const MtDims& D = a.D;
  const int c = blockIdx.x, G = gridDim.x;
  const int v0 = (int)((long long)D.V * c / G), v1 = (int)((long long)D.V * (c + 1) / G);
  float* dE = pgrad(a, P_EMB);
  const float* DX = abuf<float>(a, A_DX);
  const int n4 = D.d / 4;
  if (!acc_of(a, P_EMB)) {
    float4* z = reinterpret_cast<float4*>(dE + (long long)v0 * D.d);
    const long long nz = (long long)(v1 - v0) * n4;
    for (long long e = threadIdx.x; e < nz; e += MT_THREADS) z[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncthreads();
  // The matches (tokens in this CTA's vocabulary rows) are compacted in
  // ascending position order into a list of up to RB_CAP entries, eight
  // consecutive token ids per thread and round (few rounds, each waiting on
  // one load of ids); then the CTA adds them in list order, thread i taking
  // float4 i of every row (a row's matches are summed in position order by
  // the same threads, whatever the token distribution).
  constexpr int RB_CAP = 4096, TPT = 8;
  int* list = ism;                 // [RB_CAP] positions
  int* vid = ism + RB_CAP;         // [RB_CAP] vocabulary rows
  int* cnt = ism + 2 * RB_CAP;     // [8] per-warp match counts of a round
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int n = 0;                       // entries in the list (the same in every thread)
  auto flush = [&]() {
    __syncthreads();
    for (int j = 0; j < n; ++j) {
      const float4* src = reinterpret_cast<const float4*>(DX + (long long)list[j] * D.d);
      float4* row = reinterpret_cast<float4*>(dE + (long long)vid[j] * D.d);
      for (int i = threadIdx.x; i < n4; i += MT_THREADS) {
        const float4 x = src[i];
        float4 y = row[i];
        y.x += x.x; y.y += x.y; y.z += x.z; y.w += x.w;
        row[i] = y;
      }
    }
    __syncthreads();
    n = 0;
  };
  for (int tb = 0; tb < D.T; tb += MT_THREADS * TPT) {
    const int tt = tb + (int)threadIdx.x * TPT;
    int vv[TPT];
    int nh = 0;
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
      vv[i] = (tt + i < D.T) ? a.tokens[tt + i] : -1;
      nh += (vv[i] >= v0 && vv[i] < v1) ? 1 : 0;
    }
    // exclusive prefix of the match counts in thread order (= position order)
    int incl = nh;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) cnt[warp] = incl;
    __syncthreads();
    int base = 0, total = 0;
    for (int w = 0; w < MT_WARPS; ++w) {
      const int cw = cnt[w];
      if (w < warp) base += cw;
      total += cw;
    }
    if (n + total > RB_CAP) flush();
    int pos = n + base + incl - nh;
#pragma unroll
    for (int i = 0; i < TPT; ++i)
      if (vv[i] >= v0 && vv[i] < v1) {
        list[pos] = tt + i;
        vid[pos] = vv[i];
        ++pos;
      }
    n += total;
    __syncthreads();
  }
  flush();
}

// ===========================================================================
// loss reduction and optimizer
// ===========================================================================
static __device__ __noinline__ void job_loss(const KArgs& a) {
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

// Global gradient norm, first level: CTA c sums squares over its slice of
// optimizer range ri (the range's partials go to slot ri).
static __device__ __noinline__ void job_norm_partial(const KArgs& a, double* dsm, int ri) {
  const int c = blockIdx.x, G = gridDim.x;
  const OptRange& R = a.orng[ri];
  const float* gr = a.grads + R.off;
  const long long n = R.n;
  const long long n4 = n / 4;
  const long long b0 = n4 * c / G, b1 = n4 * (c + 1) / G;
  const float4* g4 = reinterpret_cast<const float4*>(gr);
  double acc = 0.0;
  float facc = 0.f;
  // four float4 loads in flight per thread; fp32 partial sums of 16 squares
  // are added into the fp64 accumulator in a fixed order
  long long i = b0 + threadIdx.x;
  for (; i + 3 * MT_THREADS < b1; i += 4 * MT_THREADS) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = g4[i + u * MT_THREADS];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      facc = fmaf(v[u].x, v[u].x, facc);
      facc = fmaf(v[u].y, v[u].y, facc);
      facc = fmaf(v[u].z, v[u].z, facc);
      facc = fmaf(v[u].w, v[u].w, facc);
    }
    acc += facc;
    facc = 0.f;
  }
  for (; i < b1; i += MT_THREADS) {
    const float4 v = g4[i];
    facc = fmaf(v.x, v.x, facc);
    facc = fmaf(v.y, v.y, facc);
    facc = fmaf(v.z, v.z, facc);
    facc = fmaf(v.w, v.w, facc);
  }
  if (c == G - 1)
    for (long long i = n4 * 4 + threadIdx.x; i < n; i += MT_THREADS) facc = fmaf(gr[i], gr[i], facc);
  acc += facc;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) dsm[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < MT_WARPS; ++w) t += dsm[w];
    reinterpret_cast<double*>(abuf<float>(a, A_NORMPART))[(long long)ri * MT_MAX_CTAS + c] = t;
  }
}

// AdamW constants of one sweep, held in registers.
struct AwConst {
  float c;                  // clip coefficient
  float decay;              // 1 - lr * wd (decoupled decay, applied first)
  float b1, omb1, b2, omb2; // beta1, 1 - beta1, beta2, 1 - beta2
  float ibc1, ibc2;         // 1 / (1 - beta^t)
  float lr, eps;
};
__device__ __forceinline__ AwConst aw_const(const KArgs& a, const OptGroup& og, float c) {
  AwConst k;
  k.c = c; k.decay = a.decay; k.b1 = a.beta1; k.omb1 = 1.0f - a.beta1; k.b2 = a.beta2; k.omb2 = 1.0f - a.beta2;
  k.ibc1 = og.ibc1; k.ibc2 = og.ibc2; k.lr = a.lr; k.eps = a.eps;
  return k;
}
// One parameter: g <- c g; p <- (1 - lr wd) p; m, v moving averages;
// p <- p - lr m^ / (sqrt(v^) + eps) with the bias-corrected moments.  The
// bias corrections multiply by host reciprocals and the step divides with
// the fast division (relative error ~1e-7 on a step of ~lr).
__device__ __forceinline__ void adamw_elem(const AwConst& k, float& p, float g, float& m, float& v) {
  g *= k.c;
  p *= k.decay;
  m = k.b1 * m + k.omb1 * g;
  v = k.b2 * v + k.omb2 * g * g;
  const float mh = m * k.ibc1;
  const float vh = v * k.ibc2;
  p -= __fdividef(k.lr * mh, sqrtf(vh) + k.eps);
}

// Clip coefficient of range ri's group from the ordered sum of the group's
// partials, then the AdamW sweep over the range (float4 loads; writes p, m, v
// and the bf16 shadow).  The group's step uses gscale * g, clipped.
template <class OP>
__device__ __noinline__ void job_adamw(const KArgs& a, char* smem, int ri) {
  const int c = blockIdx.x, G = gridDim.x;
  const OptRange& R = a.orng[ri];
  const OptGroup& og = a.ogrp[R.group];
  const double* parts = reinterpret_cast<const double*>(abuf<float>(a, A_NORMPART));
  double tot = 0.0;
  for (int r = og.r0; r < og.r0 + og.nr; ++r)
    for (int i = 0; i < G; ++i) tot += parts[(long long)r * MT_MAX_CTAS + i];
  const float norm = (float)sqrt(tot) * og.gscale;
  const float coef = fminf(1.0f, a.clip / (norm + a.clip_eps));
  const AwConst ak = aw_const(a, og, coef * og.gscale);
  if (c == 0 && threadIdx.x == 0 && R.first) {
    ArenaHdr* h = abuf<ArenaHdr>(a, A_HDR);
    if (R.group == 0) {
      h->grad_norm = norm;
      h->clip_coef = coef;
      h->optimizer_ran = 1;
    } else {
      h->expert_grad_norm = norm;
      h->expert_clip_coef = coef;
      h->experts_updated = 1;
    }
  }
  const long long n = R.n;
  const long long n4 = n / 4;
  float* const pm = a.master + R.off;
  const float* const gr = a.grads + R.off;
  float* const mm_ = a.adam_m + R.off;
  float* const vv_ = a.adam_v + R.off;
  float4* p4 = reinterpret_cast<float4*>(pm);
  const float4* g4 = reinterpret_cast<const float4*>(gr);
  float4* m4 = reinterpret_cast<float4*>(mm_);
  float4* v4 = reinterpret_cast<float4*>(vv_);
  __nv_bfloat16* sh = (sizeof(OP) == 2) ? (__nv_bfloat16*)a.shadow + R.off : nullptr;
  auto step4 = [&](long long j, float4 p, const float4 g, float4 m, float4 v) {
    adamw_elem(ak, p.x, g.x, m.x, v.x);
    adamw_elem(ak, p.y, g.y, m.y, v.y);
    adamw_elem(ak, p.z, g.z, m.z, v.z);
    adamw_elem(ak, p.w, g.w, m.w, v.w);
    p4[j] = p;
    m4[j] = m;
    v4[j] = v;
    if (sh) {
      uint2 u;
      __nv_bfloat162 lo = __floats2bfloat162_rn(p.x, p.y), hi = __floats2bfloat162_rn(p.z, p.w);
      u.x = *reinterpret_cast<uint32_t*>(&lo);
      u.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(sh)[j] = u;
    }
  };
  // The sweep is elementwise, so any split gives the same result.  Chunks
  // of AW_T float4 groups are drawn from a ticket counter (zeroed at the
  // start of the launch; the next ticket is drawn one chunk ahead), so that
  // SMs that stream faster take more chunks.  Each chunk streams through
  // AW_NS shared-memory stages of AW_G groups: thread 0 copies a stage's p,
  // m, v and g in with cp.async.bulk, every thread updates the stage in place
  // (and writes the bf16 shadow next to it), and thread 0 stores p, m, v and
  // the shadow back with bulk stores.  After the stores of iteration i are
  // issued, the stage of iteration i-1 (whose stores have had a whole
  // iteration to read it out) is refilled.  Groups past the last whole chunk
  // take the register path on the last CTA.
  constexpr int AW_G = 512, AW_NS = 6, AW_T = 4096;
  const uint32_t SEG = (uint32_t)AW_G * 16u;
  const uint32_t STB = 4u * SEG + (uint32_t)AW_G * 8u;   // p | m | v | g | shadow
  const bool bulk = RP_WIN_OFF + (uint32_t)AW_NS * STB <= (uint32_t)a.smem_bytes;
  const long long nfull = bulk ? n4 / AW_T : 0;          // whole chunks
  unsigned* ticket = abuf<unsigned>(a, A_DEP) + ticket_offset(a.D, a.D.L, ri == 0 ? TK_ADAMW : ri == 1 ? TK_ADAMW_R1 : TK_ADAMW_R2);
  if (bulk) {
    const uint32_t ring = smem_u32(smem) + RP_WIN_OFF;
    const uint32_t bar0 = smem_u32(&rp_bars[0]);
    long long* s_g0 = reinterpret_cast<long long*>(smem + 64);   // first group of each stage (-1: none)
    ArenaHdr* hdr = abuf<ArenaHdr>(a, A_HDR);
    // thread 0's stream position: current chunk, next sub-chunk, prefetched ticket
    long long cur = 0, nxt = 0;
    int sub = AW_T / AW_G;
    __syncthreads();
    auto refill = [&](int st) {        // thread 0: the next sub-chunk into stage st
      if (sub == AW_T / AW_G) {
        cur = nxt;
        if (cur < nfull) nxt = (long long)atomicAdd(ticket, 1u);
        sub = 0;
      }
      if (cur >= nfull) { s_g0[st] = -1; return; }
      const long long g0 = cur * AW_T + (long long)(sub++) * AW_G;
      s_g0[st] = g0;
      const uint32_t dst = ring + (uint32_t)st * STB, bar = bar0 + 8u * (uint32_t)st;
      mbar_expect_tx(bar, 4u * SEG);
      bulk_g2s(dst, p4 + g0, SEG, bar);
      bulk_g2s(dst + SEG, m4 + g0, SEG, bar);
      bulk_g2s(dst + 2u * SEG, v4 + g0, SEG, bar);
      bulk_g2s(dst + 3u * SEG, g4 + g0, SEG, bar);
    };
    if (threadIdx.x == 0) {
      for (int st = 0; st < AW_NS; ++st) mbar_init(bar0 + 8u * st, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      asm volatile("fence.proxy.async;" ::: "memory");
      nxt = (long long)atomicAdd(ticket, 1u);
      for (int st = 0; st < AW_NS; ++st) refill(st);
    }
    __syncthreads();
    bool ok = true;
    for (int it = 0;; ++it) {
      const int st = it % AW_NS;
      const long long g0 = s_g0[st];
      if (g0 < 0) break;
      if (ok && !mbar_wait(bar0 + 8u * (uint32_t)st, (uint32_t)(it / AW_NS) & 1u, a.timeout_ns)) {
        set_error(hdr, MT_ERR_DEVICE_TIMEOUT, SITE_ROWPIPE + 9);
        ok = false;
      }
      const uint32_t base = ring + (uint32_t)st * STB;
      if (ok) {
        for (int k = threadIdx.x; k < AW_G; k += MT_THREADS) {
          const uint32_t o = 16u * (uint32_t)k;
          float4 pp = lds4(base + o), mm = lds4(base + SEG + o), vv = lds4(base + 2u * SEG + o);
          const float4 gg = lds4(base + 3u * SEG + o);
          adamw_elem(ak, pp.x, gg.x, mm.x, vv.x);
          adamw_elem(ak, pp.y, gg.y, mm.y, vv.y);
          adamw_elem(ak, pp.z, gg.z, mm.z, vv.z);
          adamw_elem(ak, pp.w, gg.w, mm.w, vv.w);
          sts4(base + o, pp);
          sts4(base + SEG + o, mm);
          sts4(base + 2u * SEG + o, vv);
          if (sh) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(pp.x, pp.y), hi = __floats2bfloat162_rn(pp.z, pp.w);
            sts_u2(base + 4u * SEG + 8u * (uint32_t)k, *reinterpret_cast<uint32_t*>(&lo),
                   *reinterpret_cast<uint32_t*>(&hi));
          }
        }
      }
      // the stage's new values are read by the bulk stores (async proxy)
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncthreads();
      if (threadIdx.x == 0) {
        if (ok) {
          bulk_s2g(p4 + g0, base, SEG);
          bulk_s2g(m4 + g0, base + SEG, SEG);
          bulk_s2g(v4 + g0, base + 2u * SEG, SEG);
          if (sh) bulk_s2g(reinterpret_cast<uint2*>(sh) + g0, base + 4u * SEG, (uint32_t)AW_G * 8u);
          bulk_commit();
        }
        if (it > 0) {
          // the previous iteration's stores have read their stage: refill it
          bulk_wait_read1();
          const int pst = (it - 1) % AW_NS;
          if (ok) refill(pst);
          else s_g0[pst] = -1;
        }
        if (!ok) s_g0[st] = -1;
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      bulk_wait_all0();
      asm volatile("fence.proxy.async.global;" ::: "memory");
      if (ok)
        for (int st = 0; st < AW_NS; ++st)
          asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar0 + 8u * st) : "memory");
    }
    __syncthreads();
  }
  // groups past the last whole chunk (all groups when the stages do not fit)
  constexpr int UA = 4;                 // float4 groups per thread in flight (16 loads)
  const long long rest0 = nfull * AW_T;
  if (!bulk || c == G - 1) {
    const long long r0 = bulk ? rest0 : (n4 * c / G), r1 = bulk ? n4 : (n4 * (c + 1) / G);
    long long i = r0 + threadIdx.x;
    for (; i + (UA - 1) * MT_THREADS < r1; i += UA * MT_THREADS) {
      float4 pp[UA], mm[UA], vv[UA], gg[UA];
#pragma unroll
      for (int u = 0; u < UA; ++u) {
        const long long j = i + u * MT_THREADS;
        pp[u] = p4[j]; mm[u] = m4[j]; vv[u] = v4[j]; gg[u] = g4[j];
      }
#pragma unroll
      for (int u = 0; u < UA; ++u) step4(i + u * MT_THREADS, pp[u], gg[u], mm[u], vv[u]);
    }
    for (; i < r1; i += MT_THREADS) step4(i, p4[i], g4[i], m4[i], v4[i]);
  }
  if (c == G - 1) {
    for (long long i = n4 * 4 + threadIdx.x; i < n; i += MT_THREADS) {
      float p = pm[i], m = mm_[i], v = vv_[i];
      adamw_elem(ak, p, gr[i], m, v);
      pm[i] = p;
      mm_[i] = m;
      vv_[i] = v;
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
  // slot of layer l in the expert-activation buffers [g | u] and silu(g) u
  __device__ int al(int l) const { return a.act_layers == D.L ? l : 0; }

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
    g.tok = nullptr; g.cepart = nullptr; g.cetgt = nullptr; g.ceparts = 0; g.ksplit = 1;
    g.dwait = nullptr; g.dtarget = 0; g.dwait_aux = nullptr; g.dtarget_aux = 0; g.dsig = nullptr;
    g.omap = g.omap2 = g.amap = -1; g.oy0 = g.oy02 = g.ay0 = 0;
    g.ticket = nullptr;
    return g;
  }
  __device__ const int* offs(int l) const { return abuf<int>(a, A_OFFS) + (long long)l * (D.E + 1); }

  // forward
  __device__ GemmDesc qkv(int l) const {
    GemmDesc g = base(D.T, 3 * D.hq, D.d, EPI_ROPE);
    g.A = opnd(abuf<OP>(a, A_R) + (long long)l * D.T * D.d, D.d, 0);
    g.A.map0 = MAP_R; g.A.y0 = l * D.T;
    g.B = opnd(pweight<OP>(a, P_WQKV) + (long long)wslot(a, l) * 3 * D.hq * D.d, D.d, 0);
    g.B.map0 = MAP_WQKV; g.B.y0 = wslot(a, l) * 3 * D.hq;
    g.out = abuf<OP>(a, A_QKV) + (long long)l * D.T * 3 * D.hq; g.ldo = 3 * D.hq;
    g.omap = MAP_E_QKV64; g.oy0 = l * D.T;
    g.rope = abuf<float>(a, A_ROPE);
    return g;
  }
  __device__ GemmDesc wo(int l) const {
    GemmDesc g = base(D.T, D.d, D.hq, EPI_RESID);
    g.A = opnd(abuf<OP>(a, A_O) + (long long)l * D.T * D.hq, D.hq, 0);
    g.A.map0 = MAP_O; g.A.y0 = l * D.T;
    g.B = opnd(pweight<OP>(a, P_WO) + (long long)wslot(a, l) * D.d * D.hq, D.hq, 0);
    g.B.map0 = MAP_WO; g.B.y0 = wslot(a, l) * D.d;
    g.out = abuf<float>(a, A_XM) + (long long)l * D.T * D.d; g.ldo = D.d;
    g.aux = abuf<float>(a, A_X) + (long long)l * D.T * D.d; g.ldaux = D.d;
    g.omap = MAP_E_XM; g.oy0 = l * D.T; g.amap = MAP_E_X; g.ay0 = l * D.T;
    return g;
  }
  __device__ GemmDesc gateup(int l) const {
    GemmDesc g = base(D.Pmax, 2 * D.F, D.d, EPI_SWIGLU);
    g.rag = RAG_M; g.offs = offs(l); g.nseg = D.E;
    g.A = opnd(abuf<OP>(a, A_XS) + (long long)l * D.Pmax * D.d, D.d, 0);
    g.A.map0 = MAP_XS; g.A.y0 = l * D.Pmax;
    g.B = opnd(pweight<OP>(a, P_WGATE) + (long long)wslot(a, l) * D.E * D.F * D.d, D.d, 0);
    g.B.p1 = pweight<OP>(a, P_WUP) + (long long)wslot(a, l) * D.E * D.F * D.d;
    g.B.two = 1; g.B.seg = (long long)D.F * D.d;
    g.B.map0 = MAP_WGATE; g.B.map1 = MAP_WUP; g.B.y0 = wslot(a, l) * D.E * D.F; g.B.yseg = D.F;
    g.out = abuf<OP>(a, A_GU) + (long long)al(l) * D.Pmax * 2 * D.F; g.ldo = 2 * D.F;
    g.out2 = abuf<OP>(a, A_ACT) + (long long)al(l) * D.Pmax * D.F; g.ldo2 = D.F;
    g.omap = MAP_E_GU; g.oy0 = al(l) * D.Pmax; g.omap2 = MAP_E_ACT; g.oy02 = al(l) * D.Pmax;
    return g;
  }
  __device__ GemmDesc down(int l) const {
    GemmDesc g = base(D.Pmax, D.d, D.F, EPI_STORE_F32);
    g.rag = RAG_M; g.offs = offs(l); g.nseg = D.E;
    g.A = opnd(abuf<OP>(a, A_ACT) + (long long)al(l) * D.Pmax * D.F, D.F, 0);
    g.A.map0 = MAP_ACT; g.A.y0 = al(l) * D.Pmax;
    g.B = opnd(pweight<OP>(a, P_WDOWN) + (long long)wslot(a, l) * D.E * D.d * D.F, D.F, 0);
    g.B.seg = (long long)D.d * D.F;
    g.B.map0 = MAP_WDOWN; g.B.y0 = wslot(a, l) * D.E * D.d; g.B.yseg = D.d;
    g.out = abuf<float>(a, A_Y) + (long long)l * D.Pmax * D.d; g.ldo = D.d;
    g.omap = MAP_E_Y; g.oy0 = l * D.Pmax;
    return g;
  }
  __device__ GemmDesc lm() const {
    GemmDesc g = base(D.T, D.V, D.d, EPI_LOGITS);
    g.A = opnd(abuf<OP>(a, A_RF), D.d, 0); g.A.map0 = MAP_RF;
    g.B = opnd(pweight<OP>(a, P_LM_HEAD), D.d, 0); g.B.map0 = MAP_WLM;
    g.out = abuf<OP>(a, A_DLOGITS); g.ldo = D.V;
    g.tok = a.tokens; g.cepart = abuf<float>(a, A_CEPART); g.cetgt = abuf<float>(a, A_CETGT);
    g.ceparts = ce_parts<OP>(a);
    g.omap = MAP_E_DLOGITS;
    return g;
  }
  // backward
  __device__ GemmDesc lm_dgrad() const {
    GemmDesc g = base(D.T, D.d, D.V, EPI_STORE_F32);
    g.A = opnd(abuf<OP>(a, A_DLOGITS), D.V, 0); g.A.map0 = MAP_DLOGITS;
    g.B = opnd(pweight<OP>(a, P_LM_HEAD), D.d, 1); g.B.map0 = MAP_WLM;
    g.out = abuf<float>(a, A_DRF); g.ldo = D.d;
    g.omap = MAP_E_DRF;
    return g;
  }
  __device__ GemmDesc lm_wgrad() const {
    GemmDesc g = base(D.V, D.d, D.T, EPI_GRAD);
    g.A = opnd(abuf<OP>(a, A_DLOGITS), D.V, 1); g.A.map0 = MAP_DLOGITS;
    g.B = opnd(abuf<OP>(a, A_RF), D.d, 1); g.B.map0 = MAP_RF;
    g.out = pgrad(a, P_LM_HEAD); g.ldo = D.d; g.accumulate = acc_of(a, P_LM_HEAD);
    return g;
  }
  __device__ GemmDesc down_dgrad(int l) const {
    GemmDesc g = base(D.Pmax, D.F, D.d, EPI_SWIGLU_BWD);
    g.rag = RAG_M; g.offs = offs(l); g.nseg = D.E;
    g.A = opnd(abuf<OP>(a, A_DY), D.d, 0); g.A.map0 = MAP_DY;
    g.B = opnd(pweight<OP>(a, P_WDOWN) + (long long)wslot(a, l) * D.E * D.d * D.F, D.F, 1);
    g.B.seg = (long long)D.d * D.F;
    g.B.map0 = MAP_WDOWN; g.B.y0 = wslot(a, l) * D.E * D.d; g.B.yseg = D.d;
    g.out = abuf<OP>(a, A_DGU); g.ldo = 2 * D.F;
    g.aux = abuf<OP>(a, A_GU) + (long long)al(l) * D.Pmax * 2 * D.F; g.ldaux = 2 * D.F;
    g.omap = MAP_E_DGU; g.amap = MAP_E_GU; g.ay0 = al(l) * D.Pmax;
    return g;
  }
  __device__ GemmDesc down_wgrad(int l) const {
    GemmDesc g = base(D.d, D.F, 0, EPI_GRAD);
    g.rag = RAG_K; g.offs = offs(l); g.nseg = D.E;
    g.A = opnd(abuf<OP>(a, A_DY), D.d, 1); g.A.map0 = MAP_DY;
    g.B = opnd(abuf<OP>(a, A_ACT) + (long long)al(l) * D.Pmax * D.F, D.F, 1);
    g.B.map0 = MAP_ACT; g.B.y0 = al(l) * D.Pmax;
    g.out = pgrad(a, P_WDOWN) + (long long)wslot(a, l) * D.E * D.d * D.F; g.ldo = D.F;
    g.oseg = (long long)D.d * D.F; g.accumulate = acc_visit(a, P_WDOWN, l);
    return g;
  }
  __device__ GemmDesc gateup_dgrad(int l) const {
    GemmDesc g = base(D.Pmax, D.d, 2 * D.F, EPI_STORE_F32);
    g.rag = RAG_M; g.offs = offs(l); g.nseg = D.E;
    g.A = opnd(abuf<OP>(a, A_DGU), 2 * D.F, 0); g.A.map0 = MAP_DGU;
    g.B = opnd(pweight<OP>(a, P_WGATE) + (long long)wslot(a, l) * D.E * D.F * D.d, D.d, 1);
    g.B.p1 = pweight<OP>(a, P_WUP) + (long long)wslot(a, l) * D.E * D.F * D.d;
    g.B.two = 2; g.B.split = D.F; g.B.seg = (long long)D.F * D.d;
    g.B.map0 = MAP_WGATE; g.B.map1 = MAP_WUP; g.B.y0 = wslot(a, l) * D.E * D.F; g.B.yseg = D.F;
    g.out = abuf<float>(a, A_DXS); g.ldo = D.d;
    g.omap = MAP_E_DXS;
    return g;
  }
  __device__ GemmDesc gateup_wgrad(int l) const {
    GemmDesc g = base(2 * D.F, D.d, 0, EPI_GRAD);
    g.rag = RAG_K; g.offs = offs(l); g.nseg = D.E;
    g.A = opnd(abuf<OP>(a, A_DGU), 2 * D.F, 1); g.A.map0 = MAP_DGU;
    g.B = opnd(abuf<OP>(a, A_XS) + (long long)l * D.Pmax * D.d, D.d, 1);
    g.B.map0 = MAP_XS; g.B.y0 = l * D.Pmax;
    g.out = pgrad(a, P_WGATE) + (long long)wslot(a, l) * D.E * D.F * D.d;
    g.out1 = pgrad(a, P_WUP) + (long long)wslot(a, l) * D.E * D.F * D.d;
    g.osplit = D.F; g.ldo = D.d; g.oseg = (long long)D.F * D.d; g.accumulate = acc_visit(a, P_WGATE, l);
    return g;
  }
  __device__ GemmDesc wo_dgrad(int l) const {
    GemmDesc g = base(D.T, D.hq, D.d, EPI_STORE_OP_D);
    g.A = opnd(abuf<OP>(a, A_DXO), D.d, 0); g.A.map0 = MAP_DXO;
    g.B = opnd(pweight<OP>(a, P_WO) + (long long)wslot(a, l) * D.d * D.hq, D.hq, 1);
    g.B.map0 = MAP_WO; g.B.y0 = wslot(a, l) * D.d;
    g.out = abuf<OP>(a, A_DO); g.ldo = D.hq;
    g.aux = abuf<OP>(a, A_O) + (long long)l * D.T * D.hq; g.ldaux = D.hq;
    g.out2 = abuf<float>(a, A_DSUM); g.ldo2 = D.H;
    g.omap = MAP_E_DO; g.amap = MAP_E_O; g.ay0 = l * D.T;
    return g;
  }
  // Weight gradients with few output tiles cut their token reduction into
  // slices (tensor-core path); the slices land in A_KPART and job_ksplit_sum
  // adds them in slice order.
  __device__ void split(GemmDesc& g) const {
    const int ks = ksplit_of(a, g.M, g.N, g.K);
    if (ks <= 1) return;
    g.ksplit = ks;
    g.out = abuf<float>(a, A_KPART); g.out1 = nullptr; g.osplit = 0;
    g.ldo = g.N; g.oseg = (long long)g.M * g.N; g.accumulate = 0;
  }
  __device__ GemmDesc wo_wgrad(int l) const {
    GemmDesc g = base(D.d, D.hq, D.T, EPI_GRAD);
    g.A = opnd(abuf<OP>(a, A_DXO), D.d, 1); g.A.map0 = MAP_DXO;
    g.B = opnd(abuf<OP>(a, A_O) + (long long)l * D.T * D.hq, D.hq, 1);
    g.B.map0 = MAP_O; g.B.y0 = l * D.T;
    g.out = pgrad(a, P_WO) + (long long)wslot(a, l) * D.d * D.hq; g.ldo = D.hq; g.accumulate = acc_visit(a, P_WO, l);
    split(g);
    return g;
  }
  __device__ GemmDesc qkv_dgrad(int l) const {
    GemmDesc g = base(D.T, D.d, 3 * D.hq, EPI_STORE_F32);
    g.A = opnd(abuf<OP>(a, A_DQKV), 3 * D.hq, 0); g.A.map0 = MAP_DQKV;
    g.B = opnd(pweight<OP>(a, P_WQKV) + (long long)wslot(a, l) * 3 * D.hq * D.d, D.d, 1);
    g.B.map0 = MAP_WQKV; g.B.y0 = wslot(a, l) * 3 * D.hq;
    g.out = abuf<float>(a, A_DR); g.ldo = D.d;
    g.omap = MAP_E_DR;
    return g;
  }
  // Router-weight gradient dWr[e][c] = sum_t dz[t][e] r2[t][c] as a product
  // over the tokens: the E rows padded to one 128-row tile (the operand
  // columns beyond the bf16 dz copy's 64 read as zeros), the token reduction
  // split into slices of 128 x d at `off` floats into A_KPART.
  __device__ GemmDesc router_wgrad(int l, long long off) const {
    GemmDesc g = base(TC_BM, D.d, D.T, EPI_GRAD);
    g.A = opnd(abuf<__nv_bfloat16>(a, A_DZB), 64, 1); g.A.map0 = MAP_DZB;
    g.B = opnd(abuf<OP>(a, A_R2) + (long long)l * D.T * D.d, D.d, 1);
    g.B.map0 = MAP_R2; g.B.y0 = l * D.T;
    g.ksplit = ksplit_of(a, TC_BM, D.d, D.T);
    g.out = abuf<float>(a, A_KPART) + off; g.ldo = D.d; g.oseg = (long long)TC_BM * D.d; g.accumulate = 0;
    return g;
  }
  __device__ GemmDesc qkv_wgrad(int l) const {
    GemmDesc g = base(3 * D.hq, D.d, D.T, EPI_GRAD);
    g.A = opnd(abuf<OP>(a, A_DQKV), 3 * D.hq, 1); g.A.map0 = MAP_DQKV;
    g.B = opnd(abuf<OP>(a, A_R) + (long long)l * D.T * D.d, D.d, 1);
    g.B.map0 = MAP_R; g.B.y0 = l * D.T;
    g.out = pgrad(a, P_WQKV) + (long long)wslot(a, l) * 3 * D.hq * D.d; g.ldo = D.d; g.accumulate = acc_visit(a, P_WQKV, l);
    split(g);
    return g;
  }
};

// out[i] (+)= sum over slices k < ks (in order) of src[k * stride + i], i < n
// (n and stride multiples of 4).
static __device__ __noinline__ void job_slices_sum(float* out, const float* src, long long n, long long stride, int ks,
                                                   Sched& s, bool acc) {
  const float4* P = reinterpret_cast<const float4*>(src);
  float4* o = reinterpret_cast<float4*>(out);
  const long long n4 = n / 4, s4 = stride / 4;
  for (long long i = (long long)s.first() * MT_THREADS + threadIdx.x; i < n4; i += (long long)s.G * MT_THREADS) {
    float4 v = acc ? o[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < ks; ++k) {
      const float4 p = P[(long long)k * s4 + i];
      v.x += p.x; v.y += p.y; v.z += p.z; v.w += p.w;
    }
    o[i] = v;
  }
  s.next(s.G);
}
// out[i] (+)= sum over slices s (in order) of KPART[s][i], i < M*N.
static __device__ __forceinline__ void job_ksplit_sum(const KArgs& a, float* out, int M, int N, Sched& s, bool acc) {
  const int ks = ksplit_of(a, M, N, a.D.T);
  if (ks <= 1) return;
  job_slices_sum(out, abuf<float>(a, A_KPART), (long long)M * N, (long long)M * N, ks, s, acc);
}
// Offset (floats) in A_KPART of the router-weight gradient's slices, after
// the out-projection weight gradient's (both run in one phase), or -1 when
// the product form does not apply (CUDA-core model, or the slices do not fit).
__device__ __forceinline__ long long router_kpart_off(const KArgs& a) {
  const MtDims& D = a.D;
  const int ks = ksplit_of(a, TC_BM, D.d, D.T);
  if (ks <= 1) return -1;
  const int kw = ksplit_of(a, D.d, D.hq, D.T);
  const long long off = kw > 1 ? (long long)kw * D.d * D.hq : 0;
  if (off + (long long)ks * TC_BM * D.d > 8LL * 3 * D.hq * D.d) return -1;
  return off;
}

// Products: tcgen05 for bf16 operands, exact fp32 FMAs on the CUDA cores for
// the fp32 model.  There is no other path: bf16 shapes the tensor-core tiles
// do not cover are refused on the host.
template <class OP>
__device__ __forceinline__ void run_gemm(const KArgs& a, const GemmDesc& g, Sched& s, char* smem, TcState& tc) {
  if constexpr (sizeof(OP) == 2) gemm_tc_job(a, g, s, smem, tc);
  else gemm_simt_job<OP>(g, s, reinterpret_cast<float*>(smem));
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
__device__ __forceinline__ void run_attn_fwd(const KArgs& a, int l, Sched& s, char* smem, const TcState& tc,
                                             const AttnDeps& dp) {
  if constexpr (sizeof(OP) == 2) {
    const MtDims& D = a.D;
    attn_tm::Job j{&a.maps[MAP_QKV], &a.maps[MAP_E_OROW], l * D.T, abuf<__nv_bfloat16>(a, A_O) + (long long)l * D.T * D.hq,
                   abuf<float>(a, A_LSE) + (long long)l * D.B * D.H * D.S, D.B, D.H, D.S, D.hq,
                   1.0f / sqrtf((float)D.hd), dp.wait, dp.wtarget, dp.sig, dp.hdr, dp.timeout_ns};
    attn_tm::fwd_job(j, s, smem, tc);
  } else {
    const AttnArgs t = attn_args<OP>(a, l);
    if (a.D.hd == 64) attn_fwd_job<OP, 64>(t, s, (float*)smem);
    else attn_fwd_job<OP, 16>(t, s, (float*)smem);
  }
}
// The tcgen05 attention backward's job description for layer l.
__device__ __forceinline__ attn_tm::BwdJob tm_bwd_job(const KArgs& a, int l, const AttnDeps& dp) {
  const MtDims& D = a.D;
  return attn_tm::BwdJob{&a.maps[MAP_QKV], &a.maps[MAP_DOUT], &a.maps[MAP_E_DQKV], &a.maps[MAP_E_DS],
                         &a.maps[MAP_E_DSL], a.use_dsg, l * D.T,
                         abuf<float>(a, A_LSE) + (long long)l * D.B * D.H * D.S, abuf<float>(a, A_DSUM),
                         abuf<__nv_bfloat16>(a, A_DQKV), abuf<float>(a, A_ROPE), D.B, D.H, D.S, D.hq,
                         1.0f / sqrtf((float)D.hd), dp.hdr, dp.timeout_ns};
}

template <class OP, class Stamp>
__device__ __forceinline__ void run_attn_bwd(const KArgs& a, int l, Sched& s, char* smem, const TcState& tc,
                                             const AttnDeps& dp, Stamp&& stamp) {
  if constexpr (sizeof(OP) == 2) {
    const attn_tm::BwdJob j = tm_bwd_job(a, l, dp);
    attn_tm::dkdv_job(j, s, smem, tc);
    stamp();
    attn_tm::dq_job(j, s, smem, tc);
  } else {
    const AttnArgs t = attn_args<OP>(a, l);
    if (a.D.hd == 64) attn_bwd_job<OP, 64>(t, s, (float*)smem);
    else attn_bwd_job<OP, 16>(t, s, (float*)smem);
  }
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
  long long* tr = trace ? abuf<long long>(a, A_TRACE) + (long long)blockIdx.x * MT_TRACE_WORDS : nullptr;
  int phase = 0;
  Gemms<OP> gm(a);
  const bool stall = (a.flags & MT_FLAG_TEST_STALL) && blockIdx.x == 0;
  // per-job trace: (end time, job id) pairs in the second half of the CTA's trace
  int nj = 0;
  auto TJ = [&](int id) {
    if (tr) {
      __syncthreads();
      if (threadIdx.x == 0 && nj < MT_TRACE_JOBS) {
        tr[2 * MT_TRACE_PHASES + 2 * nj] = (long long)globaltimer();
        tr[2 * MT_TRACE_PHASES + 2 * nj + 1] = id;
      }
      ++nj;
    }
  };

#define MT_SYNC()                                                                                      \
  do {                                                                                                 \
    if (!grid_barrier(hdr, G, a.timeout_ns, (tr && phase < MT_TRACE_PHASES) ? tr + 2 * phase : nullptr, \
                      stall))                                                                          \
      return;                                                                                          \
    ++phase;                                                                                           \
    TJ(0);                                                                                             \
  } while (0)

  // Hand-offs between consecutive phases either wait at a grid barrier or,
  // with dependency counters, per 128-row block: the consumer waits only for
  // the producer parts of the blocks it reads (a.deps is grid-uniform).
  const bool dep = a.deps != 0;
  unsigned* depc = abuf<unsigned>(a, A_DEP);
  auto DEPC = [&](int l, int kind) { return depc + dep_offset(D, l, kind); };
  auto attn_deps = [&](int l, bool fwd) {
    AttnDeps dp{nullptr, 0u, nullptr, hdr, a.timeout_ns};
    if (dep) {
      if (fwd) {
        dp.wait = DEPC(l, DEP_QKV); dp.wtarget = (unsigned)(3 * D.hq / TC_BN);
        dp.sig = DEPC(l, DEP_O);
      }
    }
    return dp;
  };
  const unsigned rn_target = MT_TILE_M / MT_DEP_GROUP;
  // tensor-core products draw their tiles (longest products first in a phase)
  auto TK = [&](GemmDesc g, int l, int id) {
    g.ticket = depc + ticket_offset(D, l, id);
    return g;
  };

  // ---------------- forward ----------------
  job_embed<OP>(a, s); TJ(1);
  MT_SYNC();
  for (int l = 0; l < D.L; ++l) {
    {
      GemmDesc g = TK(gm.qkv(l), l, TK_QKV);
      if (dep) {
        if (l > 0) { g.dwait = DEPC(l - 1, DEP_RN); g.dtarget = rn_target; }
        g.dsig = DEPC(l, DEP_QKV);
      }
      run_gemm<OP>(a, g, s, smem, tc); TJ(2);
    }
    if (!dep) MT_SYNC();
    run_attn_fwd<OP>(a, l, s, smem, tc, attn_deps(l, true)); TJ(3);
    if (!dep) MT_SYNC();
    {
      GemmDesc g = TK(gm.wo(l), l, TK_WO);
      if (dep) {
        g.dwait = DEPC(l, DEP_O); g.dtarget = (unsigned)D.H;
        if (l > 0) { g.dwait_aux = DEPC(l - 1, DEP_RN); g.dtarget_aux = rn_target; }
        g.dsig = DEPC(l, DEP_XMID);
      }
      run_gemm<OP>(a, g, s, smem, tc); TJ(4);
    }
    if (!dep) MT_SYNC();
    {
      long long* ws = (tr && nj < MT_TRACE_JOBS) ? tr + 2 * MT_TRACE_PHASES + 2 * nj : nullptr;
      if (tr) ++nj;
      job_router<OP>(a, l, smem, dep ? DEPC(l, DEP_XMID) : nullptr, (unsigned)(D.d / TC_BN), ws); TJ(5);
    }
    MT_SYNC();
    job_route<OP>(a, l, smem); TJ(6);
    MT_SYNC();
    {
      GemmDesc g = TK(gm.gateup(l), l, TK_GATEUP);
      if (dep) g.dsig = DEPC(l, DEP_ACT);
      run_gemm<OP>(a, g, s, smem, tc); TJ(7);
    }
    if (!dep) MT_SYNC();
    {
      GemmDesc g = TK(gm.down(l), l, TK_DOWN);
      if (dep) { g.dwait = DEPC(l, DEP_ACT); g.dtarget = (unsigned)(2 * D.F / TC_BN); }
      run_gemm<OP>(a, g, s, smem, tc); TJ(8);
    }
    MT_SYNC();
    job_combine<OP>(a, l, s, dep ? DEPC(l, DEP_RN) : nullptr, smem); TJ(9);
    if (!dep) MT_SYNC();
  }
  {
    GemmDesc g = TK(gm.lm(), D.L, TK_LM);
    if (dep) { g.dwait = DEPC(D.L - 1, DEP_RN); g.dtarget = rn_target; }
    run_gemm<OP>(a, g, s, smem, tc); TJ(10);
  }
  MT_SYNC();
  job_ce<OP>(a, s, smem); TJ(11);
  MT_SYNC();

  // ---------------- backward ----------------
  job_loss(a); TJ(12);
  run_gemm<OP>(a, TK(gm.lm_wgrad(), D.L, TK_LM_WGRAD), s, smem, tc); TJ(14);
  run_gemm<OP>(a, TK(gm.lm_dgrad(), D.L, TK_LM_DGRAD), s, smem, tc); TJ(13);
  MT_SYNC();
  // the norm-gain gradients: per-CTA partials (PART row E+1) left by the
  // norm backward jobs, summed in CTA order by job_colfinal
  job_final_norm_bwd<OP>(a, s, smem); TJ(15);
  MT_SYNC();
  for (int l = D.L - 1; l >= 0; --l) {
    job_moe_bwd1<OP>(a, l, s, smem); TJ(17);
    // memory rule: the arena keeps one layer's expert activations; re-run
    // this layer's gate/up product (same inputs, same tiles: the same values).
    // Its tiles come from a ticket; the rotating item map of the later jobs
    // (whose per-CTA partial sums follow it) is left as without the rule.
    if (a.act_layers != D.L) {
      const int rot = s.base;
      run_gemm<OP>(a, TK(gm.gateup(l), l, TK_GATEUP_AGAIN), s, smem, tc); TJ(37);
      s.base = rot;
    }
    MT_SYNC();
    // the split-K slices of layer l+1's qkv weight gradient (complete since
    // the grid barrier above; the buffer is next written by layer l's
    // out-projection weight gradient)
    if (l + 1 < D.L) {
      job_ksplit_sum(a, pgrad(a, P_WQKV) + (long long)wslot(a, l + 1) * 3 * D.hq * D.d, 3 * D.hq, D.d, s,
                     acc_visit(a, P_WQKV, l + 1));
      TJ(33);
    }
    if (l == D.L - 1) job_colfinal(a, D.E + 1, 1, 0, pgrad(a, P_FINAL_NORM), nullptr, 0, s, (int)G, acc_of(a, P_FINAL_NORM));
    else job_colfinal(a, D.E + 1, 1, 0, pgrad(a, P_ATTN_NORM) + (long long)wslot(a, l + 1) * D.d, nullptr, 0, s, (int)G,
                      acc_visit(a, P_ATTN_NORM, l + 1));
    TJ(18);
    run_gemm<OP>(a, TK(gm.down_wgrad(l), l, TK_DOWN_WGRAD), s, smem, tc); TJ(20);
    run_gemm<OP>(a, TK(gm.down_dgrad(l), l, TK_DOWN_DGRAD), s, smem, tc); TJ(19);
    MT_SYNC();
    run_gemm<OP>(a, TK(gm.gateup_wgrad(l), l, TK_GU_WGRAD), s, smem, tc); TJ(22);
    run_gemm<OP>(a, TK(gm.gateup_dgrad(l), l, TK_GU_DGRAD), s, smem, tc); TJ(21);
    MT_SYNC();
    job_moe_bwd2<OP>(a, l, s, smem); TJ(23);
    MT_SYNC();
    // router-weight gradient: a tensor-core product over the tokens whose
    // slices are summed after the barrier, else (fp32 model) per-CTA partials
    // on the CUDA cores (rows 0..E-1); the expert-norm gain partial was left
    // by job_moe_bwd2
    const long long rg_off = router_kpart_off(a);
    int rg_chunks = 0;
    if (rg_off >= 0) run_gemm<OP>(a, TK(gm.router_wgrad(l, rg_off), l, TK_ROUTER_WGRAD), s, smem, tc);
    else rg_chunks = job_router_grad(a, l, s, smem);
    TJ(16);
    run_gemm<OP>(a, TK(gm.wo_wgrad(l), l, TK_WO_WGRAD), s, smem, tc); TJ(25);
    run_gemm<OP>(a, TK(gm.wo_dgrad(l), l, TK_WO_DGRAD), s, smem, tc); TJ(24);
    MT_SYNC();
    if (rg_off >= 0)
      job_slices_sum(pgrad(a, P_ROUTER) + (long long)wslot(a, l) * D.E * D.d, abuf<float>(a, A_KPART) + rg_off,
                     (long long)D.E * D.d, (long long)TC_BM * D.d, ksplit_of(a, TC_BM, D.d, D.T), s,
                     acc_visit(a, P_ROUTER, l));
    else
      job_colfinal(a, 0, D.E, D.E, pgrad(a, P_ROUTER) + (long long)wslot(a, l) * D.E * D.d, nullptr, 0, s, rg_chunks,
                   acc_visit(a, P_ROUTER, l));
    job_colfinal(a, D.E + 1, 1, 0, pgrad(a, P_MOE_NORM) + (long long)wslot(a, l) * D.d, nullptr, 0, s, (int)G,
                 acc_visit(a, P_MOE_NORM, l)); TJ(18);
    job_ksplit_sum(a, pgrad(a, P_WO) + (long long)wslot(a, l) * D.d * D.hq, D.d, D.hq, s, acc_visit(a, P_WO, l)); TJ(32);
    if constexpr (sizeof(OP) == 2) {
      if (a.use_dsg) {
        // dK/dV stores dS^T; after a grid barrier dQ is a product over it
        const attn_tm::BwdJob j = tm_bwd_job(a, l, attn_deps(l, false));
        attn_tm::dkdv_job(j, s, smem, tc); TJ(35);
        MT_SYNC();
        attn_tm::dqs_job(j, s, smem, tc); TJ(26);
      }
    }
    if (!a.use_dsg) { run_attn_bwd<OP>(a, l, s, smem, tc, attn_deps(l, false), [&] { TJ(35); }); TJ(26); }
    MT_SYNC();
    run_gemm<OP>(a, TK(gm.qkv_wgrad(l), l, TK_QKV_WGRAD), s, smem, tc); TJ(28);
    {
      GemmDesc g = TK(gm.qkv_dgrad(l), l, TK_QKV_DGRAD);
      if (dep) g.dsig = DEPC(l, DEP_DR);
      run_gemm<OP>(a, g, s, smem, tc); TJ(27);
    }
    // the norm backward of a token chunk starts once the chunk's dR rows are
    // stored (counters), else after a grid barrier
    if (!dep) MT_SYNC();
    job_attn_norm_bwd<OP>(a, l, s, smem, dep ? DEPC(l, DEP_DR) : nullptr, (unsigned)(D.d / TC_BN)); TJ(29);
    // the next layer's expert-combine backward reads only dx rows that this
    // job stored on the same CTA (same token chunks); its other inputs are
    // forward activations, and what it writes is read after a grid barrier
    if (!dep || l == 0) MT_SYNC();
  }
  // the split-K slices of layer 0's qkv weight gradient (the other layers'
  // are summed in the next layer's first backward phase)
  job_ksplit_sum(a, pgrad(a, P_WQKV), 3 * D.hq, D.d, s, acc_visit(a, P_WQKV, 0)); TJ(33);
  job_embed_bwd(a, (int*)smem); TJ(30);
  MT_SYNC();
  job_colfinal(a, D.E + 1, 1, 0, pgrad(a, P_ATTN_NORM), nullptr, 0, s, (int)G, acc_visit(a, P_ATTN_NORM, 0)); TJ(18);

  // ---------------- optimizer (last microbatch) ----------------
  if (a.n_ranges > 0) {
    MT_SYNC();
    for (int r = 0; r < a.n_ranges; ++r) job_norm_partial(a, (double*)smem, r);
    TJ(31);
    MT_SYNC();
    for (int r = 0; r < a.n_ranges; ++r) job_adamw<OP>(a, smem, r);
    TJ(34);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    hdr->micro_index = a.micro_index;
    bool g0 = false, g1 = false;
    for (int r = 0; r < a.n_ranges; ++r) (a.orng[r].group ? g1 : g0) = true;
    if (!g0) hdr->optimizer_ran = 0;
    if (!g1) hdr->experts_updated = 0;
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
  g.epi = (g.rag == RAG_K) ? EPI_GRAD : (a.dbg_out_mode == 1 ? EPI_STORE_OP : EPI_STORE_F32);
  if (a.dbg_out_mode == 2) g.epi = EPI_NONE;
  g.out = a.dbg_c; g.out1 = nullptr; g.out2 = nullptr; g.ldo = g.N; g.ldo2 = 0; g.osplit = 0;
  g.oseg = (long long)g.M * g.N; g.aux = nullptr; g.ldaux = 0; g.accumulate = 0;
  g.F = 0; g.S = 1; g.hd = 64; g.hq = 0; g.rope = nullptr;
  g.tok = nullptr; g.cepart = nullptr; g.cetgt = nullptr; g.ceparts = 0; g.ksplit = 1;
  g.dwait = nullptr; g.dtarget = 0; g.dwait_aux = nullptr; g.dtarget_aux = 0; g.dsig = nullptr;
  g.omap = g.omap2 = g.amap = -1; g.oy0 = g.oy02 = g.ay0 = 0;
  g.ticket = nullptr;
  if (a.dbg_tma && g.rag != RAG_K && a.dbg_out_mode < 2) g.omap = a.dbg_out_mode == 1 ? MAP_E_QKV : MAP_E_Y;
  GOperand A, B;
  A.p0 = a.dbg_a; A.p1 = nullptr; A.mn = a.dbg_a_mn; A.ld = A.mn ? g.M : g.K; A.seg = 0; A.two = 0;
  A.split = 0; A.map0 = MAP_R; A.map1 = -1; A.y0 = 0; A.yseg = 0;
  B.p0 = a.dbg_b; B.p1 = nullptr; B.mn = a.dbg_b_mn; B.ld = B.mn ? g.N : g.K;
  B.seg = (long long)g.N * g.K; B.two = 0; B.split = 0; B.map0 = MAP_WQKV; B.map1 = -1; B.y0 = 0;
  B.yseg = B.mn ? g.K : g.N;
  A.rows_per_box = a.dbg_a_rpb > 0 ? a.dbg_a_rpb : 64;
  B.rows_per_box = a.dbg_b_rpb > 0 ? a.dbg_b_rpb : 64;
  g.A = A;
  g.B = B;
  run_gemm<OP>(a, g, s, smem, tc);
  ArenaHdr* hdr = abuf<ArenaHdr>(a, A_HDR);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    hdr->n_ctas = (int)gridDim.x;
    hdr->n_phases = 0;
  }
}

// ===========================================================================
// single-op harness (mt_debug_run): one step of the update on inputs the
// caller placed in the arena, run by the same jobs as the update
// ===========================================================================
// D = rowsum(dO * O) per (batch, head, position) from the stored dO and O
// (the update forms it in the epilogue of the product that makes dO).
template <class OP>
__device__ __noinline__ void job_dsum(const KArgs& a, int l, Sched& s) {
  const MtDims& D = a.D;
  const OP* O = abuf<OP>(a, A_O) + (long long)l * D.T * D.hq;
  const OP* dO = abuf<OP>(a, A_DO);
  float* Ds = abuf<float>(a, A_DSUM);
  const int lane = threadIdx.x & 31;
  const long long n = (long long)D.T * D.H;
  for (long long i = (long long)s.first() * MT_WARPS + (threadIdx.x >> 5); i < n; i += (long long)s.G * MT_WARPS) {
    const int t = (int)(i / D.H), h = (int)(i % D.H);
    float dot = 0.f;
    for (int j = lane; j < D.hd; j += 32) {
      const long long o = (long long)t * D.hq + (long long)h * D.hd + j;
      dot = fmaf(to_f(dO[o]), to_f(O[o]), dot);
    }
    dot = warp_sum(dot);
    if (lane == 0) Ds[((long long)(t / D.S) * D.H + h) * D.S + (t % D.S)] = dot;
  }
  s.next(s.G);
}

template <class OP>
__device__ __noinline__ void run_op(const KArgs& a, char* smem, TcState& tc, Sched& s) {
  const MtDims& D = a.D;
  ArenaHdr* hdr = abuf<ArenaHdr>(a, A_HDR);
  const unsigned G = gridDim.x;
  const int l = a.dbg_layer;
  int phase = 0;
#define OP_SYNC()                                                          \
  do {                                                                     \
    if (!grid_barrier(hdr, G, a.timeout_ns, nullptr, false)) return;       \
    ++phase;                                                               \
  } while (0)
  launch_prologue(a, s.first(), s.G);
  OP_SYNC();
  Gemms<OP> gm(a);
  const AttnDeps nodeps{nullptr, 0u, nullptr, hdr, a.timeout_ns};
  switch (a.debug_op) {
    case MT_OP_ATTN_FWD:
      run_attn_fwd<OP>(a, l, s, smem, tc, nodeps);
      break;
    case MT_OP_ATTN_BWD:
      job_dsum<OP>(a, l, s);
      OP_SYNC();
      if constexpr (sizeof(OP) == 2) {
        if (a.use_dsg) {
          const attn_tm::BwdJob j = tm_bwd_job(a, l, nodeps);
          attn_tm::dkdv_job(j, s, smem, tc);
          OP_SYNC();
          attn_tm::dqs_job(j, s, smem, tc);
          break;
        }
      }
      run_attn_bwd<OP>(a, l, s, smem, tc, nodeps, [] {});
      break;
    case MT_OP_ROUTER:
      job_router<OP>(a, l, smem, nullptr, 0u, nullptr);
      OP_SYNC();
      job_route<OP>(a, l, smem);
      break;
    case MT_OP_LM_CE: {
      GemmDesc g = gm.lm();
      g.ticket = abuf<unsigned>(a, A_DEP) + ticket_offset(D, D.L, TK_LM);
      run_gemm<OP>(a, g, s, smem, tc);
      OP_SYNC();
      job_ce<OP>(a, s, smem);
      OP_SYNC();
      job_loss(a);
      break;
    }
    case MT_OP_CLIP_ADAMW:
      for (int r = 0; r < a.n_ranges; ++r) job_norm_partial(a, (double*)smem, r);
      OP_SYNC();
      for (int r = 0; r < a.n_ranges; ++r) job_adamw<OP>(a, smem, r);
      break;
    default:
      break;
  }
#undef OP_SYNC
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    hdr->micro_index = a.micro_index;
    hdr->n_ctas = (int)G;
    hdr->n_phases = phase;
  }
}

// The single-op harness is its own kernel, so the update kernel's code is
// the same with or without it.
template <class OP>
__global__ void __launch_bounds__(MT_THREADS, 1) mt_opkernel(const __grid_constant__ KArgs a) {
  extern __shared__ __align__(1024) char smem[];
  Sched s{(int)blockIdx.x, (int)gridDim.x, 0};
  TcState tc;
  tc_setup<OP>(a, smem, tc);
  run_op<OP>(a, smem, tc, s);
  tc_teardown<OP>(a, smem, tc);
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
