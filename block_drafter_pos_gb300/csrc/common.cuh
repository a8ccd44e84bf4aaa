// Device helpers shared by the DFlash2 kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define DF2_DEV __device__ __forceinline__

namespace df2 {

constexpr int kWarp = 32;

// Streaming 16-byte load for data read once per step (weights): skip L1.
DF2_DEV uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Cached 16-byte load for data many warps reuse (activations).
DF2_DEV uint4 ld_cached(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulators.
DF2_DEV void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                      uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A * B, m16n8k16, fp16 inputs, fp32 accumulators.
DF2_DEV void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                     uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two signed int8 codes (bytes sel of a word) -> half2 holding their exact values.
// The byte is biased to u = q + 128, placed under the fp16 exponent of 1024
// (0x64uu = 1024 + u exactly), and 1152 is subtracted.
DF2_DEV uint32_t codes_to_half2(uint32_t w_biased, uint32_t sel) {
  uint32_t h = __byte_perm(w_biased, 0x64646464u, sel);
  __half2 v = *reinterpret_cast<__half2*>(&h);
  const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  v = __hsub2(v, off);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Element offset of activation (row, col) in a buffer of row width K: row-major when
// T == 0; when T > 0 the tensor-core GEMM's operand layout, slices of 64 columns of
// T rows each ([K/64][T][64]), the 16-byte pieces of a row placed under the
// 128-byte swizzle (piece p of row r at p ^ (r mod 8)), so that one 64-column
// slice of the first rows is one contiguous block, ready for a single bulk copy.
DF2_DEV size_t act_offset(int row, int col, int K, int T) {
  if (T == 0) return static_cast<size_t>(row) * K + col;
  const int w = col & 63;
  return (static_cast<size_t>(col >> 6) * T + row) * 64 + ((((w >> 3) ^ (row & 7)) << 3) | (w & 7));
}

// Programmatic dependent launch: wait until the previous kernel in the stream has
// completed (its writes visible), and let the next kernel start being scheduled.
// Both are no-ops for a kernel launched without the attribute.
DF2_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
DF2_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
DF2_DEV void pdl_begin() {
  pdl_wait();
  pdl_trigger();
}
// For a kernel whose successor does nothing before its own wait but read weights and
// set up its shared memory: the successor launches at once, so its CTAs take the
// SMs the current weight stream frees and start their weight copies there.
DF2_DEV void pdl_begin_early() {
  pdl_trigger();
  pdl_wait();
}

// 1/rms of one row from nch per-chunk sums of squares, computed by a whole warp
// (fixed lane order and shuffle tree: bit-reproducible).  All lanes get the value.
DF2_DEV float warp_inv_rms(const float* ss, int row, int nch, int H, float eps);

DF2_DEV float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

DF2_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

DF2_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

DF2_DEV float warp_inv_rms(const float* ss, int row, int nch, int H, float eps) {
  const float* p = ss + static_cast<size_t>(row) * nch + (threadIdx.x & 31);
  float s = 0.f;
  for (int j0 = 0; j0 < nch; j0 += 256) {  // up to 8 loads per lane in flight, added in order
    float t[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) t[u] = (j0 + 32 * u + static_cast<int>(threadIdx.x & 31) < nch) ? p[j0 + 32 * u] : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) s += t[u];
  }
  s = warp_sum(s);
  return rsqrtf(s / static_cast<float>(H) + eps);
}

// Block-wide sum; `red` holds >= 32 floats of shared memory.  All threads get the sum.
DF2_DEV float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = (threadIdx.x < nw) ? red[threadIdx.x] : 0.f;
  if (wid == 0) t = warp_sum(t);
  if (threadIdx.x == 0) red[0] = t;
  __syncthreads();
  return red[0];
}

// Total order on float logits used by the top-k ("LSE docs/DFLASH2.md", top-k
// paragraph): NaN above everything, then the usual order with +/-inf, and for
// equal values the smaller index first.  Key = (ordered value << 32) | ~index.
DF2_DEV uint32_t float_order(float x) {
  uint32_t b = __float_as_uint(x);
  if (isnan(x)) return 0xFFFFFFFFu;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
DF2_DEV float order_to_float(uint32_t o) {
  if (o == 0xFFFFFFFFu) return __uint_as_float(0x7FC00000u);
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
DF2_DEV unsigned long long topk_key(float x, uint32_t idx) {
  return (static_cast<unsigned long long>(float_order(x)) << 32) | (0xFFFFFFFFu - idx);
}
DF2_DEV uint32_t key_index(unsigned long long k) { return 0xFFFFFFFFu - static_cast<uint32_t>(k); }
DF2_DEV float key_value(unsigned long long k) { return order_to_float(static_cast<uint32_t>(k >> 32)); }

DF2_DEV unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

}  // namespace df2
