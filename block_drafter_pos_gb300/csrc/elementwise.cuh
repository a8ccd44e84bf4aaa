// Element-wise helpers of the channel kernels: 16-bit activation stores (with the
// optional low-order plane), 4-channel loads, split-plane sums, per-chunk sums of
// squares, and the per-channel arithmetic of the convolution after a sublayer and
// of SwiGLU.
#pragma once

#include "common.cuh"

namespace df2 {
namespace ew {

DF2_DEV void put_act(void* act, size_t lo, int fmt, size_t idx, float v) {
  if (fmt == 0) {
    __nv_bfloat16* p = reinterpret_cast<__nv_bfloat16*>(act);
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    p[idx] = h;
    if (lo) p[lo + idx] = __float2bfloat16_rn(v - __bfloat162float(h));
  } else {
    __half* p = reinterpret_cast<__half*>(act);
    const __half h = __float2half_rn(v);
    p[idx] = h;
    if (lo) p[lo + idx] = __float2half_rn(v - __half2float(h));
  }
}

DF2_DEV float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
DF2_DEV float4 ld_bf16x4(const uint16_t* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                     __uint_as_float(u.y & 0xFFFF0000u));
}
DF2_DEV float4 add4(float4 a, float4 b) { return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }
DF2_DEV float4 mul4(float4 a, float4 b) { return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w); }
DF2_DEV float4 scale4(float4 a, float s) { return make_float4(a.x * s, a.y * s, a.z * s, a.w * s); }

// Sum of the split planes p[s * plane] of 4 channels, s = 0..S-1, added in split order
// (the same order, per channel, as plane_sum); up to 8 planes' loads in flight.
DF2_DEV float4 plane_sum4(const float* p, size_t plane, int S) {
  float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < S; s0 += 8) {
    float4 t[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) t[j] = (s0 + j < S) ? ld4(p + static_cast<size_t>(s0 + j) * plane) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 8; ++j) y = add4(y, t[j]);
  }
  return y;
}

// Four consecutive activations (col a multiple of 4: contiguous in both layouts of
// act_offset) as 16-bit values, one 8-byte store per plane.
DF2_DEV void put_act4(void* act, size_t lo, int fmt, size_t idx, float4 v) {
  uint2 hi, low;
  if (fmt == 0) {
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x, v.y), h1 = __floats2bfloat162_rn(v.z, v.w);
    hi = make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
    if (lo) {
      const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
      const __nv_bfloat162 l0 = __floats2bfloat162_rn(v.x - f0.x, v.y - f0.y),
                           l1 = __floats2bfloat162_rn(v.z - f1.x, v.w - f1.y);
      low = make_uint2(*reinterpret_cast<const uint32_t*>(&l0), *reinterpret_cast<const uint32_t*>(&l1));
    }
  } else {
    const __half2 h0 = __floats2half2_rn(v.x, v.y), h1 = __floats2half2_rn(v.z, v.w);
    hi = make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
    if (lo) {
      const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
      const __half2 l0 = __floats2half2_rn(v.x - f0.x, v.y - f0.y), l1 = __floats2half2_rn(v.z - f1.x, v.w - f1.y);
      low = make_uint2(*reinterpret_cast<const uint32_t*>(&l0), *reinterpret_cast<const uint32_t*>(&l1));
    }
  }
  uint16_t* p = reinterpret_cast<uint16_t*>(act);
  *reinterpret_cast<uint2*>(p + idx) = hi;
  if (lo) *reinterpret_cast<uint2*>(p + lo + idx) = low;
}

// Per-row sums of squares of 32-channel chunks (8 lanes x 4 channels each) ->
// ss[row][c / 32]: each lane's 4 squares in order, then a fixed shuffle tree.
DF2_DEV void emit_ss4(float4 v, int row, float* ss, int nch, int c) {
  float s = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  s += __shfl_xor_sync(0xffffffffu, s, 4);
  if ((threadIdx.x & 7) == 0) ss[static_cast<size_t>(row) * nch + (c >> 5)] = s;
}

// Conv after a sublayer + residual, per channel: x + (b2 + d2) y + (b3 + d3) y_prev.
DF2_DEV float4 conv_out4(float4 x0, float4 y, float4 yp, float4 b2, float4 b3, float d2, float d3) {
  float4 xv;
  xv.x = x0.x + (b2.x + d2) * y.x + (b3.x + d3) * yp.x;
  xv.y = x0.y + (b2.y + d2) * y.y + (b3.y + d3) * yp.y;
  xv.z = x0.z + (b2.z + d2) * y.z + (b3.z + d3) * yp.z;
  xv.w = x0.w + (b2.w + d2) * y.w + (b3.w + d3) * yp.w;
  return xv;
}

// SwiGLU per channel: silu(g) * u.
DF2_DEV float4 swiglu4(float4 g, float4 u) {
  float4 h;
  h.x = g.x / (1.f + __expf(-g.x)) * u.x;
  h.y = g.y / (1.f + __expf(-g.y)) * u.y;
  h.z = g.z / (1.f + __expf(-g.z)) * u.z;
  h.w = g.w / (1.f + __expf(-g.w)) * u.w;
  return h;
}

}  // namespace ew
}  // namespace df2
