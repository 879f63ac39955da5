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
template <int NC>
__device__ __forceinline__ float row_dot(const Row<NC>& a, const Row<NC>& b) {
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    s = fmaf(a.v[i].x, b.v[i].x, s);
    s = fmaf(a.v[i].y, b.v[i].y, s);
    s = fmaf(a.v[i].z, b.v[i].z, s);
    s = fmaf(a.v[i].w, b.v[i].w, s);
  }
  return warp_sum(s);
}
// r = a * s (elementwise scalar)
template <int NC>
__device__ __forceinline__ void row_scale(Row<NC>& r, const Row<NC>& a, float s) {
#pragma unroll
  for (int i = 0; i < NC; ++i) r.v[i] = make_float4(a.v[i].x * s, a.v[i].y * s, a.v[i].z * s, a.v[i].w * s);
}
// r += a * s
template <int NC>
__device__ __forceinline__ void row_axpy(Row<NC>& r, const Row<NC>& a, float s) {
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    r.v[i].x = fmaf(a.v[i].x, s, r.v[i].x);
    r.v[i].y = fmaf(a.v[i].y, s, r.v[i].y);
    r.v[i].z = fmaf(a.v[i].z, s, r.v[i].z);
    r.v[i].w = fmaf(a.v[i].w, s, r.v[i].w);
  }
}
// y = x * inv * g
template <int NC>
__device__ __forceinline__ void row_norm_apply(Row<NC>& y, const Row<NC>& x, float inv, const Row<NC>& g) {
#pragma unroll
  for (int i = 0; i < NC; ++i)
    y.v[i] = make_float4(x.v[i].x * inv * g.v[i].x, x.v[i].y * inv * g.v[i].y, x.v[i].z * inv * g.v[i].z,
                         x.v[i].w * inv * g.v[i].w);
}
// RMSNorm backward: returns dx = inv * (dy*g - xh * mean(dy*g*xh)), xh = x*inv
template <int NC>
__device__ __forceinline__ void row_norm_bwd(Row<NC>& dx, const Row<NC>& dy, const Row<NC>& x, float inv,
                                             const Row<NC>& g, int d) {
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    s = fmaf(dy.v[i].x * g.v[i].x, x.v[i].x * inv, s);
    s = fmaf(dy.v[i].y * g.v[i].y, x.v[i].y * inv, s);
    s = fmaf(dy.v[i].z * g.v[i].z, x.v[i].z * inv, s);
    s = fmaf(dy.v[i].w * g.v[i].w, x.v[i].w * inv, s);
  }
  const float mean = warp_sum(s) / (float)d;
#pragma unroll
  for (int i = 0; i < NC; ++i)
    dx.v[i] = make_float4(inv * (dy.v[i].x * g.v[i].x - x.v[i].x * inv * mean),
                          inv * (dy.v[i].y * g.v[i].y - x.v[i].y * inv * mean),
                          inv * (dy.v[i].z * g.v[i].z - x.v[i].z * inv * mean),
                          inv * (dy.v[i].w * g.v[i].w - x.v[i].w * inv * mean));
}
// dx += RMSNorm backward of dy (as row_norm_bwd, added in place)
template <int NC>
__device__ __forceinline__ void row_norm_bwd_add(Row<NC>& dx, const Row<NC>& dy, const Row<NC>& x, float inv,
                                                 const Row<NC>& g, int d) {
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    s = fmaf(dy.v[i].x * g.v[i].x, x.v[i].x * inv, s);
    s = fmaf(dy.v[i].y * g.v[i].y, x.v[i].y * inv, s);
    s = fmaf(dy.v[i].z * g.v[i].z, x.v[i].z * inv, s);
    s = fmaf(dy.v[i].w * g.v[i].w, x.v[i].w * inv, s);
  }
  const float mean = warp_sum(s) / (float)d;
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    dx.v[i].x += inv * (dy.v[i].x * g.v[i].x - x.v[i].x * inv * mean);
    dx.v[i].y += inv * (dy.v[i].y * g.v[i].y - x.v[i].y * inv * mean);
    dx.v[i].z += inv * (dy.v[i].z * g.v[i].z - x.v[i].z * inv * mean);
    dx.v[i].w += inv * (dy.v[i].w * g.v[i].w - x.v[i].w * inv * mean);
  }
}
template <int NC>
__device__ __forceinline__ void row_add(Row<NC>& r, const Row<NC>& a) {
#pragma unroll
  for (int i = 0; i < NC; ++i)
    r.v[i] = make_float4(r.v[i].x + a.v[i].x, r.v[i].y + a.v[i].y, r.v[i].z + a.v[i].z, r.v[i].w + a.v[i].w);
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
