// rows.cuh - per-token row jobs of the megakernel, one warp per token with
// the token's d-wide rows held in registers as float4 chunks (lane l owns
// chunks l, l+32, ...).  All loads of a row are issued before its values are
// used, so each warp keeps several 16-byte loads in flight per lane.
//
// NC is the number of chunks per lane (d/4/32 rounded up); the jobs are
// instantiated for NC in {1, 6} (d <= 128 and d <= 768) and dispatched on d.
#pragma once
#include "common.cuh"

template <int NC>
struct Row {
  float4 v[NC];
};

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

template <int NC>
__device__ __forceinline__ void row_ld(Row<NC>& r, const float* p, int n4) {
  const int l = lane_id();
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const int c = l + 32 * i;
    r.v[i] = (c < n4) ? reinterpret_cast<const float4*>(p)[c] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}
template <int NC>
__device__ __forceinline__ void row_st(float* p, const Row<NC>& r, int n4) {
  const int l = lane_id();
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const int c = l + 32 * i;
    if (c < n4) reinterpret_cast<float4*>(p)[c] = r.v[i];
  }
}
// operand-type rows (fp32 or bf16)
template <int NC>
__device__ __forceinline__ void row_ld_op(Row<NC>& r, const float* p, int n4) { row_ld(r, p, n4); }
template <int NC>
__device__ __forceinline__ void row_ld_op(Row<NC>& r, const __nv_bfloat16* p, int n4) {
  const int l = lane_id();
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const int c = l + 32 * i;
    if (c < n4) {
      const uint2 u = reinterpret_cast<const uint2*>(p)[c];
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
      r.v[i] = make_float4(a.x, a.y, b.x, b.y);
    } else {
      r.v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}
template <int NC>
__device__ __forceinline__ void row_st_op(float* p, const Row<NC>& r, int n4) { row_st(p, r, n4); }
template <int NC>
__device__ __forceinline__ void row_st_op(__nv_bfloat16* p, const Row<NC>& r, int n4) {
  const int l = lane_id();
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const int c = l + 32 * i;
    if (c < n4) {
      __nv_bfloat162 a = __floats2bfloat162_rn(r.v[i].x, r.v[i].y);
      __nv_bfloat162 b = __floats2bfloat162_rn(r.v[i].z, r.v[i].w);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&a);
      u.y = *reinterpret_cast<uint32_t*>(&b);
      reinterpret_cast<uint2*>(p)[c] = u;
    }
  }
}
// The arithmetic below runs on two-wide fp32 instructions: each float4 chunk
// is two (x, y), (z, w) pairs.  Elementwise results equal the scalar ones;
// dot products keep two partial sums (even and odd columns) per lane.
__device__ __forceinline__ uint64_t lo2(const float4& v) { return f2(v.x, v.y); }
__device__ __forceinline__ uint64_t hi2(const float4& v) { return f2(v.z, v.w); }
__device__ __forceinline__ float4 join2(uint64_t lo, uint64_t hi) {
  float4 r;
  unf2(lo, r.x, r.y);
  unf2(hi, r.z, r.w);
  return r;
}
__device__ __forceinline__ float sum2(uint64_t v) {
  float a, b;
  unf2(v, a, b);
  return a + b;
}
template <int NC>
__device__ __forceinline__ float row_dot(const Row<NC>& a, const Row<NC>& b) {
  uint64_t s = f2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    s = fma2(lo2(a.v[i]), lo2(b.v[i]), s);
    s = fma2(hi2(a.v[i]), hi2(b.v[i]), s);
  }
  return warp_sum(sum2(s));
}
// r = a * s (elementwise scalar)
template <int NC>
__device__ __forceinline__ void row_scale(Row<NC>& r, const Row<NC>& a, float s) {
  const uint64_t s2 = f2(s, s);
#pragma unroll
  for (int i = 0; i < NC; ++i) r.v[i] = join2(mul2(lo2(a.v[i]), s2), mul2(hi2(a.v[i]), s2));
}
// r += a * s
template <int NC>
__device__ __forceinline__ void row_axpy(Row<NC>& r, const Row<NC>& a, float s) {
  const uint64_t s2 = f2(s, s);
#pragma unroll
  for (int i = 0; i < NC; ++i)
    r.v[i] = join2(fma2(lo2(a.v[i]), s2, lo2(r.v[i])), fma2(hi2(a.v[i]), s2, hi2(r.v[i])));
}
// y = x * inv * g
template <int NC>
__device__ __forceinline__ void row_norm_apply(Row<NC>& y, const Row<NC>& x, float inv, const Row<NC>& g) {
  const uint64_t i2 = f2(inv, inv);
#pragma unroll
  for (int i = 0; i < NC; ++i)
    y.v[i] = join2(mul2(mul2(lo2(x.v[i]), i2), lo2(g.v[i])), mul2(mul2(hi2(x.v[i]), i2), hi2(g.v[i])));
}
// sum over the row of (dy * g) * (x * inv), over the warp
template <int NC>
__device__ __forceinline__ float row_norm_dot(const Row<NC>& dy, const Row<NC>& x, float inv, const Row<NC>& g) {
  const uint64_t i2 = f2(inv, inv);
  uint64_t s = f2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    s = fma2(mul2(lo2(dy.v[i]), lo2(g.v[i])), mul2(lo2(x.v[i]), i2), s);
    s = fma2(mul2(hi2(dy.v[i]), hi2(g.v[i])), mul2(hi2(x.v[i]), i2), s);
  }
  return warp_sum(sum2(s));
}
// inv * (dy * g - (x * inv) * mean) for one pair
__device__ __forceinline__ uint64_t norm_bwd2(uint64_t dy, uint64_t g, uint64_t x, uint64_t i2, uint64_t m2) {
  return mul2(i2, sub2(mul2(dy, g), mul2(mul2(x, i2), m2)));
}
// RMSNorm backward: returns dx = inv * (dy*g - xh * mean(dy*g*xh)), xh = x*inv
template <int NC>
__device__ __forceinline__ void row_norm_bwd(Row<NC>& dx, const Row<NC>& dy, const Row<NC>& x, float inv,
                                             const Row<NC>& g, int d) {
  const float mean = row_norm_dot(dy, x, inv, g) / (float)d;
  const uint64_t i2 = f2(inv, inv), m2 = f2(mean, mean);
#pragma unroll
  for (int i = 0; i < NC; ++i)
    dx.v[i] = join2(norm_bwd2(lo2(dy.v[i]), lo2(g.v[i]), lo2(x.v[i]), i2, m2),
                    norm_bwd2(hi2(dy.v[i]), hi2(g.v[i]), hi2(x.v[i]), i2, m2));
}
// dx += RMSNorm backward of dy (as row_norm_bwd, added in place)
template <int NC>
__device__ __forceinline__ void row_norm_bwd_add(Row<NC>& dx, const Row<NC>& dy, const Row<NC>& x, float inv,
                                                 const Row<NC>& g, int d) {
  const float mean = row_norm_dot(dy, x, inv, g) / (float)d;
  const uint64_t i2 = f2(inv, inv), m2 = f2(mean, mean);
#pragma unroll
  for (int i = 0; i < NC; ++i)
    dx.v[i] = join2(add2(lo2(dx.v[i]), norm_bwd2(lo2(dy.v[i]), lo2(g.v[i]), lo2(x.v[i]), i2, m2)),
                    add2(hi2(dx.v[i]), norm_bwd2(hi2(dy.v[i]), hi2(g.v[i]), hi2(x.v[i]), i2, m2)));
}
template <int NC>
__device__ __forceinline__ void row_add(Row<NC>& r, const Row<NC>& a) {
#pragma unroll
  for (int i = 0; i < NC; ++i) r.v[i] = join2(add2(lo2(r.v[i]), lo2(a.v[i])), add2(hi2(r.v[i]), hi2(a.v[i])));
}
template <int NC>
__device__ __forceinline__ float row_rms_inv(const Row<NC>& x, int d, float eps) {
  return 1.0f / sqrtf(row_dot(x, x) / (float)d + eps);
}

// Run f(integral_constant<int, NC>) with the NC that covers d (d <= 768,
// checked on the host: six rows of NC = 6 chunks still fit in registers).
template <class F>
__device__ __forceinline__ void with_nc(int d, F&& f) {
  const int n4 = d / 4;
  if (n4 <= 32) f(std::integral_constant<int, 1>());
  else f(std::integral_constant<int, 6>());
}
