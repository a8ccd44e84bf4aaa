// Weight-streaming GEMV / skinny GEMM for the drafter projections (steps a1, a3,
// a4, a6, a7, a9): y[n][m] = sum_k W[m][k] x[n][k] for 8 activation rows per request.
//
// Design (sm_103a):
//  * The weights are read exactly once per step, so the kernel is bound by HBM
//    bandwidth.  A work unit is a 16-row weight tile times one K split; every warp
//    of a persistent grid (one 16-warp CTA per SM) walks its units grid-stride, the
//    warps of one CTA on consecutive tiles of the same split.  One lane streams 16
//    contiguous bytes of a weight row per load (ld.global.nc.L1::no_allocate.v4)
//    straight into mma.sync m16n8k16 as the A operand.  The order of the K sum
//    inside one MMA is free, so the physical K positions a lane holds fill the
//    MMA's logical K slots and the activation (B) fragment is loaded with the same
//    permutation.
//  * Weight loads run one batch (4 x 32 K) ahead of the MMAs; independent
//    accumulator chains keep the MMA dependency latency off the critical path.
//  * Each split's partial goes to its own output plane with plain stores (no
//    fences or atomics on the streaming path); the consumer kernel adds the planes
//    in split order, so every result is bit-reproducible.  The split count comes
//    from a cost model over the grid (gemv_choose_splits).
//  * Activations may carry a low-order plane (x = hi + lo) for ~16-bit accuracy.
//  * Programmatic dependent launch: the first weight loads are issued before
//    griddepcontrol.wait, so the weight stream starts while the previous kernel
//    drains.
//  * Q8/group64 ("LSE docs/DFLASH2.md", Q8 paragraph: w = scale * q + bias per
//    group of 64): codes are exact in fp16; each group is one fp16 MMA chain from
//    zero, folded as scale * (sum q x) + bias * (sum x), with sum x taken by one
//    more MMA chain against a row of ones.
#include "common.cuh"
#include "internal.h"

namespace df2 {

namespace {

constexpr int kWarpsPerCta = 16;
constexpr int kKStep = 128;  // K elements per batch (4 x 32)

DF2_DEV int find_seg(const GemvArgs& a, int u) {
  int s = 0;
#pragma unroll
  for (int i = 1; i < kMaxSeg; ++i)
    if (i < a.nseg && u >= a.seg[i].unit_begin) s = i;
  return s;
}

template <int NT>
DF2_DEV void store_tile(const GemvSeg& sg, int split, int row0, int nt, const float (&acc)[NT][4], int lane) {
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
#ifndef DF2_GEMV_NO_PDL
  pdl_trigger();
  bool waited = false;
#endif
  for (int u = warp; u < a.total_units; u += nwarps) {
    const GemvSeg& sg = a.seg[find_seg(a, u)];
    const int local = u - sg.unit_begin;
    const int tiles = sg.M >> 4;
    const int tile = local % tiles, split = local / tiles;
    const int kchunk = sg.K / sg.splits;
    const int k0 = split * kchunk;
    const int row0 = tile * 16;
    const int nt = sg.n_tiles;
    const __nv_bfloat16* w0 =
        reinterpret_cast<const __nv_bfloat16*>(sg.w) + static_cast<size_t>(row0 + g) * sg.K + k0 + 8 * q;
    const __nv_bfloat16* w1 = w0 + static_cast<size_t>(8) * sg.K;
    const __nv_bfloat16* xb =
        reinterpret_cast<const __nv_bfloat16*>(sg.x) + static_cast<size_t>(g) * sg.ldx + k0 + 8 * q;
    const size_t xlo = sg.xlo_off;
    // independent chains: (hi, lo plane) x (first, second 16 K of a 32 step)
    float acc[NT][4], acc2[NT][4], acc3[NT][4], acc4[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[t][e] = acc2[t][e] = acc3[t][e] = acc4[t][e] = 0.f;
    uint4 ra[4], rb[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      ra[j] = ld_stream(w0 + 32 * j);
      rb[j] = ld_stream(w1 + 32 * j);
    }
#ifndef DF2_GEMV_NO_PDL
    if (!waited) {  // weights are independent of earlier kernels; activations are not
      pdl_wait();
      waited = true;
    }
#endif
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
            mma_bf16(acc2[t], ca[j].z, cb[j].z, ca[j].w, cb[j].w, x.z, x.w);
            if (xlo) {
              const uint4 y = ld_cached(xt + xlo + 32 * j);
              mma_bf16(acc3[t], ca[j].x, cb[j].x, ca[j].y, cb[j].y, y.x, y.y);
              mma_bf16(acc4[t], ca[j].z, cb[j].z, ca[j].w, cb[j].w, y.z, y.w);
            }
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[t][e] = (acc[t][e] + acc2[t][e]) + (acc3[t][e] + acc4[t][e]);
    store_tile<NT>(sg, split, row0, nt, acc, lane);
  }
#ifndef DF2_GEMV_NO_PDL
  if (!waited) pdl_wait();  // every CTA orders itself after the previous kernel
#endif
}

// ------------------------------------------------------------------ Q8/group64 weights
template <int NT>
__global__ void __launch_bounds__(kWarpsPerCta * 32) gemv_q8_kernel(const __grid_constant__ GemvArgs a) {
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kWarpsPerCta;
  const int g = lane >> 2, q = lane & 3;
  const uint32_t one2 = 0x3C003C00u;  // half2(1, 1)
#ifndef DF2_GEMV_NO_PDL
  pdl_trigger();
  bool waited = false;
#endif
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
    const size_t xlo = sg.xlo_off;
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
#ifndef DF2_GEMV_NO_PDL
    if (!waited) {
      pdl_wait();
      waited = true;
    }
#endif
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
            // independent chains: codes x hi, ones x hi (column sums), codes x lo, ones x lo
            float cg[4] = {0.f, 0.f, 0.f, 0.f}, cs[4] = {0.f, 0.f, 0.f, 0.f};
            float cgl[4] = {0.f, 0.f, 0.f, 0.f}, csl[4] = {0.f, 0.f, 0.f, 0.f};
            mma_f16(cg, A[0][0], A[0][1], A[0][2], A[0][3], xa.x, xa.y);
            mma_f16(cs, one2, one2, one2, one2, xa.x, xa.y);
            mma_f16(cg, A[1][0], A[1][1], A[1][2], A[1][3], xa.z, xa.w);
            mma_f16(cs, one2, one2, one2, one2, xa.z, xa.w);
            mma_f16(cg, A[2][0], A[2][1], A[2][2], A[2][3], xc.x, xc.y);
            mma_f16(cs, one2, one2, one2, one2, xc.x, xc.y);
            mma_f16(cg, A[3][0], A[3][1], A[3][2], A[3][3], xc.z, xc.w);
            mma_f16(cs, one2, one2, one2, one2, xc.z, xc.w);
            if (xlo) {
              const uint4 ya = ld_cached(xt + xlo);
              const uint4 yc = ld_cached(xt + xlo + 8);
              mma_f16(cgl, A[0][0], A[0][1], A[0][2], A[0][3], ya.x, ya.y);
              mma_f16(csl, one2, one2, one2, one2, ya.x, ya.y);
              mma_f16(cgl, A[1][0], A[1][1], A[1][2], A[1][3], ya.z, ya.w);
              mma_f16(csl, one2, one2, one2, one2, ya.z, ya.w);
              mma_f16(cgl, A[2][0], A[2][1], A[2][2], A[2][3], yc.x, yc.y);
              mma_f16(csl, one2, one2, one2, one2, yc.x, yc.y);
              mma_f16(cgl, A[3][0], A[3][1], A[3][2], A[3][3], yc.z, yc.w);
              mma_f16(csl, one2, one2, one2, one2, yc.z, yc.w);
            }
            acc[t][0] += s0 * (cg[0] + cgl[0]) + b0 * (cs[0] + csl[0]);
            acc[t][1] += s0 * (cg[1] + cgl[1]) + b0 * (cs[1] + csl[1]);
            acc[t][2] += s1 * (cg[2] + cgl[2]) + b1 * (cs[2] + csl[2]);
            acc[t][3] += s1 * (cg[3] + cgl[3]) + b1 * (cs[3] + csl[3]);
          }
        }
      }
    }
    store_tile<NT>(sg, split, row0, nt, acc, lane);
  }
#ifndef DF2_GEMV_NO_PDL
  if (!waited) pdl_wait();
#endif
}

template <int NT>
cudaError_t launch_nt(const GemvArgs& a, int fmt, int num_sms, bool pdl, cudaStream_t st) {
  int ctas = num_sms;  // one 16-warp CTA per SM (the kernels use up to 128 registers a thread)
  const int need = (a.total_units + kWarpsPerCta - 1) / kWarpsPerCta;
  if (ctas > need) ctas = need;
  if (ctas < 1) ctas = 1;
  if (fmt == 0) return launch_ex(gemv_bf16_kernel<NT>, dim3(ctas), dim3(kWarpsPerCta * 32), 0, st, pdl, a);
  return launch_ex(gemv_q8_kernel<NT>, dim3(ctas), dim3(kWarpsPerCta * 32), 0, st, pdl, a);
}

}  // namespace

int gemv_choose_splits(int tiles, int K, int num_sms) {
  const long long W = static_cast<long long>(num_sms) * kWarpsPerCta;
  const int chunks = K / kKStep;
  int best_s = 1;
  double best = -1.0;
  for (int s = 1; s <= chunks; ++s) {
    if (chunks % s) continue;
    const long long rounds = (static_cast<long long>(tiles) * s + W - 1) / W;
    // a warp's batches (+1 pipeline start per unit) and the consumer's per-plane reads
    const double cost = static_cast<double>(rounds) * (chunks / s + 1) + 0.25 * s;
    if (best < 0.0 || cost < best) {
      best = cost;
      best_s = s;
    }
  }
  return best_s;
}

cudaError_t launch_gemv(GemvArgs& a, int fmt, int max_tiles, int num_sms, bool pdl, cudaStream_t st) {
  int units = 0;
  for (int i = 0; i < a.nseg; ++i) {
    GemvSeg& sg = a.seg[i];
    if (sg.splits < 1 || sg.M % 16 || sg.K % sg.splits || (sg.K / sg.splits) % kKStep) return cudaErrorInvalidValue;
    sg.unit_begin = units;
    units += (sg.M / 16) * sg.splits;
  }
  a.total_units = units;
  if (max_tiles <= 1) return launch_nt<1>(a, fmt, num_sms, pdl, st);
  if (max_tiles <= 2) return launch_nt<2>(a, fmt, num_sms, pdl, st);
  if (max_tiles <= 4) return launch_nt<4>(a, fmt, num_sms, pdl, st);
  if (max_tiles <= 8) return launch_nt<8>(a, fmt, num_sms, pdl, st);
  return cudaErrorInvalidValue;
}

}  // namespace df2
