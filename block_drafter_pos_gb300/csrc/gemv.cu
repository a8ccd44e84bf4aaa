// Weight-streaming GEMV / skinny GEMM for the drafter projections (a1, a3, a4, a6,
// a7, a9 of the step): out[n][m] = sum_k W[m][k] x[n][k] for a handful of
// activation rows (8 per request).
//
// Design (sm_103a): the weights are read exactly once per step, so the kernel is
// bound by HBM bandwidth.  Each warp owns a 16-row weight tile and one K split;
// every lane streams 16 contiguous bytes of a weight row per load
// (ld.global.nc.L1::no_allocate.v4) and feeds them straight into mma.sync
// m16n8k16 as the A operand.  The order of the K sum inside one MMA is free, so
// the physical K positions a lane holds are assigned to the MMA's logical K
// slots, and the activation (B) fragment is loaded with the same permutation.
// Split-K partial sums go to scratch; the consumer adds them in a fixed order,
// which keeps every result bit-reproducible.
//
// Q8/group64: codes are exact in fp16, so each 64-wide group is one fp16 MMA
// chain from zero; its result is folded as scale * (sum q x) + bias * (sum x)
// ("LSE docs/DFLASH2.md", Q8 paragraph: w = scale * q + bias per group of 64).
#include "common.cuh"
#include "internal.h"

namespace df2 {

namespace {

constexpr int kWarpsPerCta = 16;
constexpr int kKStep = 128;  // K elements per inner iteration (4 x 32)

__device__ __forceinline__ int find_seg(const GemvArgs& a, int u) {
  int s = 0;
#pragma unroll
  for (int i = 1; i < kMaxSeg; ++i)
    if (i < a.nseg && u >= a.seg[i].unit_begin) s = i;
  return s;
}

template <int NT>
__device__ __forceinline__ void store_tile(const GemvSeg& sg, int split, int row0, int nt, const float (&acc)[NT][4],
                                           int lane) {
  const int g = lane >> 2, q = lane & 3;
  float* out = sg.out + static_cast<size_t>(split) * (sg.n_tiles * 8) * sg.M;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    if (t < nt) {
      const int n0 = t * 8 + 2 * q;
      out[static_cast<size_t>(n0) * sg.M + row0 + g] = acc[t][0];
      out[static_cast<size_t>(n0 + 1) * sg.M + row0 + g] = acc[t][1];
      out[static_cast<size_t>(n0) * sg.M + row0 + g + 8] = acc[t][2];
      out[static_cast<size_t>(n0 + 1) * sg.M + row0 + g + 8] = acc[t][3];
    }
  }
}

// ------------------------------------------------------------------ BF16 weights
template <int NT>
__global__ void __launch_bounds__(kWarpsPerCta * 32) gemv_bf16_kernel(const __grid_constant__ GemvArgs a) {
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kWarpsPerCta;
  const int g = lane >> 2, q = lane & 3;
  for (int u = warp; u < a.total_units; u += nwarps) {
    const GemvSeg& sg = a.seg[find_seg(a, u)];
    const int local = u - sg.unit_begin;
    const int tiles = sg.M >> 4;
    const int tile = local % tiles, split = local / tiles;
    const int kchunk = sg.K / sg.splits;
    const int k0 = split * kchunk;
    const int row0 = tile * 16;
    const int nt = sg.n_tiles;
    const __nv_bfloat16* w0 = reinterpret_cast<const __nv_bfloat16*>(sg.w) + static_cast<size_t>(row0 + g) * sg.K + k0 + 8 * q;
    const __nv_bfloat16* w1 = w0 + static_cast<size_t>(8) * sg.K;
    const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(sg.x) + static_cast<size_t>(g) * sg.ldx + k0 + 8 * q;
    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    uint4 ra[4], rb[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      ra[j] = ld_stream(w0 + 32 * j);
      rb[j] = ld_stream(w1 + 32 * j);
    }
    for (int k = 0; k < kchunk; k += kKStep) {
      uint4 ca[4], cb[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        ca[j] = ra[j];
        cb[j] = rb[j];
      }
      if (k + kKStep < kchunk) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          ra[j] = ld_stream(w0 + k + kKStep + 32 * j);
          rb[j] = ld_stream(w1 + k + kKStep + 32 * j);
        }
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t < nt) {
          const __nv_bfloat16* xt = xb + static_cast<size_t>(t * 8) * sg.ldx + k;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 x = ld_cached(xt + 32 * j);
            mma_bf16(acc[t], ca[j].x, cb[j].x, ca[j].y, cb[j].y, x.x, x.y);
            mma_bf16(acc[t], ca[j].z, cb[j].z, ca[j].w, cb[j].w, x.z, x.w);
          }
        }
      }
    }
    store_tile<NT>(sg, split, row0, nt, acc, lane);
  }
}

// ------------------------------------------------------------------ Q8/group64 weights
template <int NT>
__global__ void __launch_bounds__(kWarpsPerCta * 32) gemv_q8_kernel(const __grid_constant__ GemvArgs a) {
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kWarpsPerCta;
  const int g = lane >> 2, q = lane & 3;
  for (int u = warp; u < a.total_units; u += nwarps) {
    const GemvSeg& sg = a.seg[find_seg(a, u)];
    const int local = u - sg.unit_begin;
    const int tiles = sg.M >> 4;
    const int tile = local % tiles, split = local / tiles;
    const int kchunk = sg.K / sg.splits;
    const int k0 = split * kchunk;
    const int row0 = tile * 16;
    const int nt = sg.n_tiles;
    const int KG = sg.K >> 6;
    const int8_t* c0p = reinterpret_cast<const int8_t*>(sg.w) + static_cast<size_t>(row0 + g) * sg.K + k0 + 16 * q;
    const int8_t* c1p = c0p + static_cast<size_t>(8) * sg.K;
    const uint16_t* s0p = sg.scale + static_cast<size_t>(row0 + g) * KG + (k0 >> 6);
    const uint16_t* b0p = sg.bias + static_cast<size_t>(row0 + g) * KG + (k0 >> 6);
    const size_t rs8 = static_cast<size_t>(8) * KG;
    const __half* xb = reinterpret_cast<const __half*>(sg.x) + static_cast<size_t>(g) * sg.ldx + k0 + 16 * q;
    const float* xs = sg.xsum + (k0 >> 6);
    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    const int ngroups = kchunk >> 6;
    uint4 rc0[2], rc1[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      rc0[j] = ld_stream(c0p + 64 * j);
      rc1[j] = ld_stream(c1p + 64 * j);
    }
    for (int gi = 0; gi < ngroups; gi += 2) {
      uint4 cc0[2], cc1[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        cc0[j] = rc0[j];
        cc1[j] = rc1[j];
      }
      if (gi + 2 < ngroups) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          rc0[j] = ld_stream(c0p + 64 * (gi + 2 + j));
          rc1[j] = ld_stream(c1p + 64 * (gi + 2 + j));
        }
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int grp = gi + j;
        const float s0 = bf16_to_f32(__ldg(s0p + grp)), s1 = bf16_to_f32(__ldg(s0p + rs8 + grp));
        const float b0 = bf16_to_f32(__ldg(b0p + grp)), b1 = bf16_to_f32(__ldg(b0p + rs8 + grp));
        const uint32_t u0[4] = {cc0[j].x ^ 0x80808080u, cc0[j].y ^ 0x80808080u, cc0[j].z ^ 0x80808080u,
                                cc0[j].w ^ 0x80808080u};
        const uint32_t u1[4] = {cc1[j].x ^ 0x80808080u, cc1[j].y ^ 0x80808080u, cc1[j].z ^ 0x80808080u,
                                cc1[j].w ^ 0x80808080u};
        uint32_t A[4][4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          A[m][0] = codes_to_half2(u0[m], 0x4140);
          A[m][1] = codes_to_half2(u1[m], 0x4140);
          A[m][2] = codes_to_half2(u0[m], 0x4342);
          A[m][3] = codes_to_half2(u1[m], 0x4342);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t < nt) {
            const __half* xt = xb + static_cast<size_t>(t * 8) * sg.ldx + 64 * grp;
            const uint4 xa = ld_cached(xt);
            const uint4 xc = ld_cached(xt + 8);
            float cg[4] = {0.f, 0.f, 0.f, 0.f};
            mma_f16(cg, A[0][0], A[0][1], A[0][2], A[0][3], xa.x, xa.y);
            mma_f16(cg, A[1][0], A[1][1], A[1][2], A[1][3], xa.z, xa.w);
            mma_f16(cg, A[2][0], A[2][1], A[2][2], A[2][3], xc.x, xc.y);
            mma_f16(cg, A[3][0], A[3][1], A[3][2], A[3][3], xc.z, xc.w);
            const int n0 = t * 8 + 2 * q;
            const float xs0 = __ldg(xs + static_cast<size_t>(n0) * KG + grp);
            const float xs1 = __ldg(xs + static_cast<size_t>(n0 + 1) * KG + grp);
            acc[t][0] += s0 * cg[0] + b0 * xs0;
            acc[t][1] += s0 * cg[1] + b0 * xs1;
            acc[t][2] += s1 * cg[2] + b1 * xs0;
            acc[t][3] += s1 * cg[3] + b1 * xs1;
          }
        }
      }
    }
    store_tile<NT>(sg, split, row0, nt, acc, lane);
  }
}

template <int NT>
cudaError_t launch_nt(const GemvArgs& a, int fmt, int num_sms, cudaStream_t st) {
  // persistent grid: exactly the CTAs that are resident at once (a grid-stride loop
  // over work units must not leave CTAs waiting for a second wave)
  static int occ[2] = {0, 0};
  if (occ[fmt] == 0) {
    cudaError_t e = fmt == 0 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[0], gemv_bf16_kernel<NT>, kWarpsPerCta * 32, 0)
                             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[1], gemv_q8_kernel<NT>, kWarpsPerCta * 32, 0);
    if (e != cudaSuccess) return e;
    if (occ[fmt] < 1) occ[fmt] = 1;
  }
  int ctas = num_sms * occ[fmt];
  const int need = (a.total_units + kWarpsPerCta - 1) / kWarpsPerCta;
  if (ctas > need) ctas = need;
  if (ctas < 1) ctas = 1;
  if (fmt == 0)
    gemv_bf16_kernel<NT><<<ctas, kWarpsPerCta * 32, 0, st>>>(a);
  else
    gemv_q8_kernel<NT><<<ctas, kWarpsPerCta * 32, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const GemvArgs& a, int fmt, int max_tiles, int num_sms, cudaStream_t st) {
  if (max_tiles <= 1) return launch_nt<1>(a, fmt, num_sms, st);
  if (max_tiles <= 2) return launch_nt<2>(a, fmt, num_sms, st);
  if (max_tiles <= 4) return launch_nt<4>(a, fmt, num_sms, st);
  if (max_tiles <= 8) return launch_nt<8>(a, fmt, num_sms, st);
  return cudaErrorInvalidValue;
}

}  // namespace df2
