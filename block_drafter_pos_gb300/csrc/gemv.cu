// Weight-streaming GEMV / skinny GEMM for the drafter projections (steps a1, a3,
// a4, a6, a7, a9): y[n][m] = sum_k W[m][k] x[n][k] for 8 activation rows per request.
//
// Design (sm_103a):
//  * The weights are read exactly once per step, so the kernel is bound by HBM
//    bandwidth.  A work unit is a 16-row weight tile times one K split; every warp
//    of a persistent grid walks its units (grid stride), warps of one CTA on
//    consecutive tiles of the same split.  One lane streams 16 contiguous bytes of
//    a weight row per load (ld.global.nc.L1::no_allocate.v4) straight into
//    mma.sync m16n8k16 as the A operand.  The order of the K sum inside one MMA is
//    free, so the physical K positions a lane holds fill the MMA's logical K slots
//    and the activation (B) fragment is loaded with the same permutation.
//  * Loads run one batch (4 x 32 K) ahead of the MMAs, across unit boundaries, so
//    a warp never waits for a cold start between units; independent accumulator
//    chains keep the MMA dependency latency off the critical path.
//  * The split count of each launch comes from a cost model (rounds of units over
//    the grid plus per-unit and per-partial overheads).  The partials of a tile go
//    to fixed slots (one per split); the warp that completes the tile (atomic
//    counter) adds them in split order - bit-reproducible - and runs the
//    epilogue: plain store, SwiGLU (a tile holds 8 gate rows and the same 8 up
//    rows), or the dynamic convolution after a sublayer + residual add + the next
//    norm's input and sums of squares.
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

DF2_DEV int find_seg(const GemvArgs& a, int u) {
  int r = 0;
#pragma unroll
  for (int i = 1; i < kMaxSeg; ++i)
    if (i < a.nseg && u >= a.seg[i].unit_begin) r = i;
  return r;
}

DF2_DEV float silu(float v) { return v / (1.f + __expf(-v)); }

// Writes one activation value (hi, and lo when lo != 0) in bf16 (fmt 0) or fp16.
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

// ------------------------------------------------------------------ epilogues
// acc[t] is the warp's C fragment of n-tile t: lane (g, q) holds rows g, g+8 and
// columns 8t + 2q, 8t + 2q + 1 of the 16-row tile.
template <int NT>
DF2_DEV void epilogue(const GemvSeg& sg, int tile, const float (&acc)[NT][4], int lane) {
  const int g = lane >> 2, q = lane & 3;
  const int nt = sg.n_tiles;
  if (sg.epi == kEpiStore) {
    const int r0 = tile * 16 + g;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < nt) {
        const size_t n0 = static_cast<size_t>(t * 8 + 2 * q);
        sg.out[n0 * sg.ldo + r0] = acc[t][0];
        sg.out[(n0 + 1) * sg.ldo + r0] = acc[t][1];
        sg.out[n0 * sg.ldo + r0 + 8] = acc[t][2];
        sg.out[(n0 + 1) * sg.ldo + r0 + 8] = acc[t][3];
      }
    }
  } else if (sg.epi == kEpiSwiglu) {
    const int f = tile * 8 + g;  // rows g: gate f, rows g+8: up f
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < nt) {
        const size_t n0 = static_cast<size_t>(t * 8 + 2 * q);
        put_act(sg.act, sg.act_lo, sg.act_fmt, n0 * sg.ld_act + f, silu(acc[t][0]) * acc[t][2]);
        put_act(sg.act, sg.act_lo, sg.act_fmt, (n0 + 1) * sg.ld_act + f, silu(acc[t][1]) * acc[t][3]);
      }
    }
  } else {  // kEpiConvOut: the tile's 16 output channels are one conv group (group = tile)
    const int H = sg.ld_act, G = sg.G;
    const int ca = tile * 16 + g, cb = ca + 8;
    const float b2a = bf16_to_f32(sg.base[2 * H + ca]), b3a = bf16_to_f32(sg.base[3 * H + ca]);
    const float b2b = bf16_to_f32(sg.base[2 * H + cb]), b3b = bf16_to_f32(sg.base[3 * H + cb]);
    const float wa = bf16_to_f32(sg.norm_w[ca]), wb = bf16_to_f32(sg.norm_w[cb]);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < nt) {
        // block positions i = 2q and 2q+1 of request t; y_{i-1} of position 2q sits in lane q-1
        float pa = __shfl_up_sync(0xffffffffu, acc[t][1], 1);
        float pb = __shfl_up_sync(0xffffffffu, acc[t][3], 1);
        if (q == 0) pa = pb = 0.f;
        const size_t n0 = static_cast<size_t>(t * 8 + 2 * q), n1 = n0 + 1;
        const float* d0 = sg.delta + n0 * (4 * G);
        const float* d1 = sg.delta + n1 * (4 * G);
        const float ya0 = acc[t][0], ya1 = acc[t][1], yb0 = acc[t][2], yb1 = acc[t][3];
        const float c20 = d0[2 * G + tile], c30 = d0[3 * G + tile], c21 = d1[2 * G + tile], c31 = d1[3 * G + tile];
        float* xr0 = sg.xres + n0 * H;
        float* xr1 = sg.xres + n1 * H;
        const float xa0 = xr0[ca] + (b2a + c20) * ya0 + (b3a + c30) * pa;
        const float xa1 = xr1[ca] + (b2a + c21) * ya1 + (b3a + c31) * ya0;
        const float xb0 = xr0[cb] + (b2b + c20) * yb0 + (b3b + c30) * pb;
        const float xb1 = xr1[cb] + (b2b + c21) * yb1 + (b3b + c31) * yb0;
        xr0[ca] = xa0;
        xr1[ca] = xa1;
        xr0[cb] = xb0;
        xr1[cb] = xb1;
        put_act(sg.act, sg.act_lo, sg.act_fmt, n0 * H + ca, xa0 * wa);
        put_act(sg.act, sg.act_lo, sg.act_fmt, n1 * H + ca, xa1 * wa);
        put_act(sg.act, sg.act_lo, sg.act_fmt, n0 * H + cb, xb0 * wb);
        put_act(sg.act, sg.act_lo, sg.act_fmt, n1 * H + cb, xb1 * wb);
        if (sg.act2 != nullptr) {
          put_act(sg.act2, sg.act2_lo, 0, n0 * H + ca, xa0 * wa);
          put_act(sg.act2, sg.act2_lo, 0, n1 * H + ca, xa1 * wa);
          put_act(sg.act2, sg.act2_lo, 0, n0 * H + cb, xb0 * wb);
          put_act(sg.act2, sg.act2_lo, 0, n1 * H + cb, xb1 * wb);
        }
        // sums of squares over the tile's 16 channels (lanes with equal q)
        float s0 = xa0 * xa0 + xb0 * xb0, s1 = xa1 * xa1 + xb1 * xb1;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          s0 += __shfl_xor_sync(0xffffffffu, s0, o);
          s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        }
        if (g == 0) {
          const int ntl = H / 16;
          sg.ss[n0 * ntl + tile] = s0;
          sg.ss[n1 * ntl + tile] = s1;
        }
      }
    }
  }
}

// Stores a warp's partial of one tile (split `split`); the warp that completes the
// tile adds all splits in order and runs the epilogue.
// Not inlined: the epilogues' temporaries stay out of the streaming loop's registers.
template <int NT>
__device__ __noinline__ void finish_unit(const GemvArgs& a, const GemvSeg& sg, int tile, int split,
                                         const float (&acc)[NT][4], int lane) {
  if (sg.splits == 1) {
    epilogue<NT>(sg, tile, acc, lane);
    return;
  }
  const int gt = sg.tile_begin + tile;
  const size_t slot0 = static_cast<size_t>(gt) * a.max_splits * (NT * 128);
  float* mine = a.part + slot0 + static_cast<size_t>(split) * (NT * 128) + lane * 4;
#pragma unroll
  for (int t = 0; t < NT; ++t)
    if (t < sg.n_tiles)
      *reinterpret_cast<float4*>(mine + t * 128) = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
  __threadfence();
  __syncwarp();
  int old = 0;
  if (lane == 0) old = atomicAdd(a.counters + gt, 1);
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old != sg.splits - 1) return;
  __threadfence();
  float sum[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) sum[t][0] = sum[t][1] = sum[t][2] = sum[t][3] = 0.f;
  // splits are added in order; their loads are issued 8 at a time
  for (int j0 = 0; j0 < sg.splits; j0 += 8) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < sg.n_tiles) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j0 + j < sg.splits)
            v[j] = __ldcg(reinterpret_cast<const float4*>(a.part + slot0 + static_cast<size_t>(j0 + j) * (NT * 128) +
                                                          t * 128 + lane * 4));
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j0 + j < sg.splits) {
            sum[t][0] += v[j].x;
            sum[t][1] += v[j].y;
            sum[t][2] += v[j].z;
            sum[t][3] += v[j].w;
          }
        }
      }
    }
  }
  if (lane == 0) a.counters[gt] = 0;  // ready for the next launch (stream ordered)
  epilogue<NT>(sg, tile, sum, lane);
}

// A warp's view of one unit: where its lane's weight rows, activations start.
struct UnitBf16 {
  int seg, tile, split, nb;
  const __nv_bfloat16* w0;
  const __nv_bfloat16* w1;
  const __nv_bfloat16* xb;
};

DF2_DEV UnitBf16 unit_bf16(const GemvArgs& a, int u, int g, int q) {
  UnitBf16 r;
  r.seg = find_seg(a, u);
  const GemvSeg& sg = a.seg[r.seg];
  const int local = u - sg.unit_begin;
  r.tile = local % sg.tiles;
  r.split = local / sg.tiles;
  const int kchunk = sg.K / sg.splits;
  const int k0 = r.split * kchunk;
  r.nb = kchunk / 128;
  if (sg.epi == kEpiSwiglu) {
    r.w0 = reinterpret_cast<const __nv_bfloat16*>(sg.w) + static_cast<size_t>(r.tile * 8 + g) * sg.K;
    r.w1 = reinterpret_cast<const __nv_bfloat16*>(sg.w2) + static_cast<size_t>(r.tile * 8 + g) * sg.K;
  } else {
    r.w0 = reinterpret_cast<const __nv_bfloat16*>(sg.w) + static_cast<size_t>(r.tile * 16 + g) * sg.K;
    r.w1 = r.w0 + static_cast<size_t>(8) * sg.K;
  }
  r.w0 += k0 + 8 * q;
  r.w1 += k0 + 8 * q;
  r.xb = reinterpret_cast<const __nv_bfloat16*>(sg.x) + static_cast<size_t>(g) * sg.ldx + k0 + 8 * q;
  return r;
}

// ------------------------------------------------------------------ BF16 weights
template <int NT>
__global__ void __launch_bounds__(kWarpsPerCta * 32, 1) gemv_bf16_kernel(const __grid_constant__ GemvArgs a) {
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kWarpsPerCta;
  const int g = lane >> 2, q = lane & 3;
  pdl_trigger();
  int u = warp;
  if (u >= a.total_units) {
    pdl_wait();
    return;
  }
  UnitBf16 cur = unit_bf16(a, u, g, q);
  uint4 ra[4], rb[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    ra[j] = ld_stream(cur.w0 + 32 * j);
    rb[j] = ld_stream(cur.w1 + 32 * j);
  }
  pdl_wait();  // weights are independent of earlier kernels; activations are not
  // four independent accumulator chains: (hi, lo) x (first, second K half of a 32 step)
  float acc[4][NT][4];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[c][t][0] = acc[c][t][1] = acc[c][t][2] = acc[c][t][3] = 0.f;
  int b = 0;
  while (true) {
    uint4 ca[4], cb[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      ca[j] = ra[j];
      cb[j] = rb[j];
    }
    const bool last = b + 1 == cur.nb;
    const int un = u + nwarps;
    const bool more = un < a.total_units;
    if (!last) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        ra[j] = ld_stream(cur.w0 + (b + 1) * 128 + 32 * j);
        rb[j] = ld_stream(cur.w1 + (b + 1) * 128 + 32 * j);
      }
    } else if (more) {  // first batch of the next unit, in flight during this batch and the epilogue
      const UnitBf16 nxt = unit_bf16(a, un, g, q);  // recomputed at the switch: fewer live registers
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        ra[j] = ld_stream(nxt.w0 + 32 * j);
        rb[j] = ld_stream(nxt.w1 + 32 * j);
      }
    }
    const GemvSeg& sg = a.seg[cur.seg];
    const bool has_lo = sg.xlo_off != 0;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < sg.n_tiles) {
        const __nv_bfloat16* xt = cur.xb + static_cast<size_t>(t * 8) * sg.ldx + b * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 x = ld_cached(xt + 32 * j);
          mma_bf16(acc[0][t], ca[j].x, cb[j].x, ca[j].y, cb[j].y, x.x, x.y);
          mma_bf16(acc[1][t], ca[j].z, cb[j].z, ca[j].w, cb[j].w, x.z, x.w);
          if (has_lo) {
            const uint4 y = ld_cached(xt + sg.xlo_off + 32 * j);
            mma_bf16(acc[2][t], ca[j].x, cb[j].x, ca[j].y, cb[j].y, y.x, y.y);
            mma_bf16(acc[3][t], ca[j].z, cb[j].z, ca[j].w, cb[j].w, y.z, y.w);
          }
        }
      }
    }
    if (!last) {
      ++b;
      continue;
    }
    float sum[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sum[t][e] = (acc[0][t][e] + acc[1][t][e]) + (acc[2][t][e] + acc[3][t][e]);
        acc[0][t][e] = acc[1][t][e] = acc[2][t][e] = acc[3][t][e] = 0.f;
      }
    finish_unit<NT>(a, sg, cur.tile, cur.split, sum, lane);
    if (!more) break;
    u = un;
    cur = unit_bf16(a, u, g, q);
    b = 0;
  }
}

// ------------------------------------------------------------------ Q8/group64 weights
// A batch is 2 groups (128 K).
struct UnitQ8 {
  int seg, tile, split, nb;
  const int8_t* c0;
  const int8_t* c1;
  const uint16_t *s0, *s1, *b0, *b1;
  const __half* xb;
};

DF2_DEV UnitQ8 unit_q8(const GemvArgs& a, int u, int g, int q) {
  UnitQ8 r;
  r.seg = find_seg(a, u);
  const GemvSeg& sg = a.seg[r.seg];
  const int local = u - sg.unit_begin;
  r.tile = local % sg.tiles;
  r.split = local / sg.tiles;
  const int kchunk = sg.K / sg.splits;
  const int k0 = r.split * kchunk;
  const int KG = sg.K >> 6;
  r.nb = kchunk / 128;
  if (sg.epi == kEpiSwiglu) {
    const size_t row = static_cast<size_t>(r.tile * 8 + g);
    r.c0 = reinterpret_cast<const int8_t*>(sg.w) + row * sg.K;
    r.c1 = reinterpret_cast<const int8_t*>(sg.w2) + row * sg.K;
    r.s0 = sg.scale + row * KG;
    r.b0 = sg.bias + row * KG;
    r.s1 = sg.scale2 + row * KG;
    r.b1 = sg.bias2 + row * KG;
  } else {
    const size_t row = static_cast<size_t>(r.tile * 16 + g);
    r.c0 = reinterpret_cast<const int8_t*>(sg.w) + row * sg.K;
    r.c1 = r.c0 + static_cast<size_t>(8) * sg.K;
    r.s0 = sg.scale + row * KG;
    r.b0 = sg.bias + row * KG;
    r.s1 = r.s0 + static_cast<size_t>(8) * KG;
    r.b1 = r.b0 + static_cast<size_t>(8) * KG;
  }
  r.c0 += k0 + 16 * q;
  r.c1 += k0 + 16 * q;
  r.s0 += k0 >> 6;
  r.s1 += k0 >> 6;
  r.b0 += k0 >> 6;
  r.b1 += k0 >> 6;
  r.xb = reinterpret_cast<const __half*>(sg.x) + static_cast<size_t>(g) * sg.ldx + k0 + 16 * q;
  return r;
}

struct BatchQ8 {
  uint4 c0[2], c1[2];
  uint16_t s0[2], s1[2], b0[2], b1[2];
};

DF2_DEV void load_q8(BatchQ8& r, const UnitQ8& u, int b) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int gi = b * 2 + j;
    r.c0[j] = ld_stream(u.c0 + 64 * gi);
    r.c1[j] = ld_stream(u.c1 + 64 * gi);
    r.s0[j] = __ldg(u.s0 + gi);
    r.s1[j] = __ldg(u.s1 + gi);
    r.b0[j] = __ldg(u.b0 + gi);
    r.b1[j] = __ldg(u.b1 + gi);
  }
}

template <int NT>
__global__ void __launch_bounds__(kWarpsPerCta * 32, 1) gemv_q8_kernel(const __grid_constant__ GemvArgs a) {
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kWarpsPerCta;
  const int g = lane >> 2, q = lane & 3;
  const uint32_t one2 = 0x3C003C00u;  // half2(1, 1)
  pdl_trigger();
  int u = warp;
  if (u >= a.total_units) {
    pdl_wait();
    return;
  }
  UnitQ8 cur = unit_q8(a, u, g, q);
  BatchQ8 rb;
  load_q8(rb, cur, 0);
  pdl_wait();
  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  int b = 0;
  while (true) {
    const BatchQ8 cb = rb;
    const bool last = b + 1 == cur.nb;
    const int un = u + nwarps;
    const bool more = un < a.total_units;
    if (!last) {
      load_q8(rb, cur, b + 1);
    } else if (more) {
      const UnitQ8 nxt = unit_q8(a, un, g, q);  // recomputed at the switch: fewer live registers
      load_q8(rb, nxt, 0);
    }
    const GemvSeg& sg = a.seg[cur.seg];
    const bool has_lo = sg.xlo_off != 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int gi = b * 2 + j;
      const float s0 = bf16_to_f32(cb.s0[j]), s1 = bf16_to_f32(cb.s1[j]);
      const float b0 = bf16_to_f32(cb.b0[j]), b1 = bf16_to_f32(cb.b1[j]);
      const uint32_t u0[4] = {cb.c0[j].x ^ 0x80808080u, cb.c0[j].y ^ 0x80808080u, cb.c0[j].z ^ 0x80808080u,
                              cb.c0[j].w ^ 0x80808080u};
      const uint32_t u1[4] = {cb.c1[j].x ^ 0x80808080u, cb.c1[j].y ^ 0x80808080u, cb.c1[j].z ^ 0x80808080u,
                              cb.c1[j].w ^ 0x80808080u};
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
        if (t < sg.n_tiles) {
          const __half* xt = cur.xb + static_cast<size_t>(t * 8) * sg.ldx + 64 * gi;
          const uint4 xa = ld_cached(xt);
          const uint4 xc = ld_cached(xt + 8);
          // independent chains: codes x hi, ones x hi, codes x lo, ones x lo
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
          if (has_lo) {
            const uint4 ya = ld_cached(xt + sg.xlo_off);
            const uint4 yc = ld_cached(xt + sg.xlo_off + 8);
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
    if (!last) {
      ++b;
      continue;
    }
    float sum[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sum[t][e] = acc[t][e];
        acc[t][e] = 0.f;
      }
    finish_unit<NT>(a, sg, cur.tile, cur.split, sum, lane);
    if (!more) break;
    u = un;
    cur = unit_q8(a, u, g, q);
    b = 0;
  }
}

template <int NT>
cudaError_t launch_nt(const GemvArgs& a, int fmt, int num_sms, bool pdl, cudaStream_t st) {
  int ctas = num_sms;  // one 16-warp CTA per SM (128 registers a thread)
  const int need = (a.total_units + kWarpsPerCta - 1) / kWarpsPerCta;
  if (ctas > need) ctas = need;
  if (fmt == 0) return launch_ex(gemv_bf16_kernel<NT>, dim3(ctas), dim3(kWarpsPerCta * 32), 0, st, pdl, a);
  return launch_ex(gemv_q8_kernel<NT>, dim3(ctas), dim3(kWarpsPerCta * 32), 0, st, pdl, a);
}

}  // namespace

void gemv_plan(GemvArgs& a, int fmt, int num_sms, size_t* part_floats, int* n_counters) {
  (void)fmt;
  const long long W = static_cast<long long>(num_sms) * kWarpsPerCta;
  int units = 0, tiles = 0, max_s = 1;
  long long tiles_all = 0;
  for (int i = 0; i < a.nseg; ++i) tiles_all += a.seg[i].tiles;
  // one split count for the whole launch (all segments of a launch share K here)
  const int K = a.seg[0].K;
  const int chunks = K / 128;
  int best_s = 1;
  long long best_cost = -1;
  for (int s = 1; s <= chunks; ++s) {
    if (chunks % s) continue;
    const long long n_units = tiles_all * s;
    const long long rounds = (n_units + W - 1) / W;
    // K elements a warp streams, + per-unit restart and per-partial read overheads
    const long long cost = rounds * (K / s + 32) + (s > 1 ? 8LL * s : 0);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_s = s;
    }
  }
  for (int i = 0; i < a.nseg; ++i) {
    GemvSeg& s = a.seg[i];
    s.splits = best_s;
    s.unit_begin = units;
    s.tile_begin = tiles;
    units += s.tiles * s.splits;
    tiles += s.tiles;
    max_s = max_s > s.splits ? max_s : s.splits;
  }
  a.total_units = units;
  a.max_splits = max_s;
  if (part_floats) *part_floats = static_cast<size_t>(tiles) * max_s * 128 * 8;
  if (n_counters) *n_counters = tiles;
}

cudaError_t launch_gemv(GemvArgs& a, int fmt, int max_tiles, int num_sms, bool pdl, cudaStream_t st) {
  gemv_plan(a, fmt, num_sms, nullptr, nullptr);
  if (max_tiles <= 1) return launch_nt<1>(a, fmt, num_sms, pdl, st);
  if (max_tiles <= 2) return launch_nt<2>(a, fmt, num_sms, pdl, st);
  if (max_tiles <= 4) return launch_nt<4>(a, fmt, num_sms, pdl, st);
  if (max_tiles <= 8) return launch_nt<8>(a, fmt, num_sms, pdl, st);
  return cudaErrorInvalidValue;
}

}  // namespace df2
