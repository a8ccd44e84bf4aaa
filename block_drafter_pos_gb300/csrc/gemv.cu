// Weight-streaming GEMV / skinny GEMM for the drafter projections (steps a1, a3,
// a4, a6, a7, a9): y[n][m] = sum_k W[m][k] x[n][k] for 8 activation rows per request.
//
// Design (sm_103a):
//  * The weights are read exactly once per step, so the kernel is bound by HBM
//    bandwidth; what it needs is enough bytes in flight to cover HBM latency and
//    no other long-latency load on the consumers' path.
//  * A launch's work is the sequence of stages (64-row weight block x 128 K) of
//    its segments; CTA c of C (two per SM) takes the contiguous share
//    [c T / C, (c + 1) T / C) of the T stages (stream-K), so every CTA streams
//    the same bytes whatever the matrix shapes.  Each CTA has one producer warp
//    and four consumer warps.  The producer fills a ring of shared-memory stages with bulk tensor
//    copies (cp.async.bulk.tensor) completing on the stage's "full" mbarrier: 64
//    weight rows x 128 K, plus the matching activation slice, both planes, in
//    8-row boxes.  Copies move 64 K per row: 128-byte rows (128-byte swizzle) for
//    bf16 weights and for activations, 64-byte rows (64-byte swizzle) for int8
//    codes.  The copy engine's cost grows with the number of rows it fetches, so
//    rows are kept as long as the swizzle allows.  The consumers release a stage
//    through its "empty" mbarrier.  The weight copies of the first stages are
//    issued before griddepcontrol.wait (weights never depend on the previous
//    kernel); the activation copies after it.
//  * Each consumer warp owns 16 of the 64 rows: mma.sync m16n8k16 with the weights
//    as the A operand.  The order of the K sum inside one MMA is free: a lane
//    reads the same consecutive K of weight rows g and g + 8 and of activation row
//    g (16-byte shared-memory loads, bank-conflict-free under the swizzle), so A
//    and B agree on which K each MMA slot holds.
//  * A block whose stages are shared by several CTAs gets one partial plane per
//    CTA, written with plain stores at plane (CTA - first CTA of the block); the
//    consumer kernel adds the block's planes in order (gemv_plane_count gives
//    their number in closed form), so every result is bit-reproducible, with no
//    atomics and no inter-CTA signalling.
//  * bf16 activations carry a low-order plane (x = hi + lo) for ~16-bit accuracy,
//    with independent accumulator chains for the two planes; fp16 activations (int8
//    weights) round to 2^-12 relative and are one plane.
//  * Q8/group64 ("LSE docs/DFLASH2.md", Q8 paragraph: w = scale * q + bias per
//    group of 64 along K, bf16 scale and bias): the int8 codes become exact fp16
//    values by a byte permute against the 1024 exponent, and the affine map is
//    applied in fp16 (w = q * s + b, one fused multiply-add per pair).  A group's
//    scale and bias are loaded one stage ahead.  The fp16 activation slice uses
//    128-byte rows (64 K, 128-byte swizzle) so a lane's 16 consecutive K are two
//    conflict-free loads.
//  * Every mbarrier wait is bounded; a wait that gives up sets the error word, and
//    the producer lets its outstanding copies land (again bounded) before exiting.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "glue.h"
#include "internal.h"
#include "pipeline.cuh"

namespace df2 {

namespace {

using namespace pipe;

DF2_DEV int find_seg(const GemvArgs& a, long long t) {
  int s = 0;
#pragma unroll
  for (int i = 1; i < kMaxSeg; ++i)
    if (i < a.nseg && t >= a.seg[i].stage_begin) s = i;
  return s;
}

// Walks this CTA's stage range [t0, t1): for stage t the segment, 64-row block and
// K offset, and whether it opens or closes a piece (the CTA's share of a block).
struct Cursor {
  long long t, t1;
  int seg, row0, kabs, kst, kstage;
  bool valid;
  DF2_DEV void load(const GemvArgs& a) {
    valid = t < t1;
    if (!valid) return;
    seg = find_seg(a, t);
    const GemvSeg& sg = a.seg[seg];
    kst = sg.K / a.stage_k;
    const long long local = t - sg.stage_begin;
    row0 = static_cast<int>(local / kst) * kBlockRows;
    kstage = static_cast<int>(local % kst);
    kabs = kstage * a.stage_k;
  }
  DF2_DEV void start(const GemvArgs& a) {
    const long long T = a.total_stages, C = gridDim.x;
    t = (static_cast<long long>(blockIdx.x) * T) / C;
    t1 = (static_cast<long long>(blockIdx.x + 1) * T) / C;
    load(a);
  }
  DF2_DEV void next(const GemvArgs& a) {  // incremental: no division inside a segment
    if (++t >= t1) {
      valid = false;
      return;
    }
    if (++kstage < kst) {
      kabs += a.stage_k;
      return;
    }
    kstage = 0;
    kabs = 0;
    row0 += kBlockRows;
    if (row0 >= a.seg[seg].M) {
      ++seg;
      row0 = 0;
      kst = a.seg[seg].K / a.stage_k;
    }
  }
  DF2_DEV bool opens(long long t_first) const { return kstage == 0 || t == t_first; }
  DF2_DEV bool closes() const { return kstage == kst - 1 || t == t1 - 1; }
  // plane of this CTA's piece of the current block
  DF2_DEV int plane(const GemvArgs& a) const {
    const long long b0 = t - kstage;  // the block's first stage
    return static_cast<int>(blockIdx.x) - gemv_cta_of_stage(b0, gridDim.x, a.total_stages);
  }
};

template <int NT>
DF2_DEV void store_tile(const GemvSeg& sg, int plane, int row0, const float (&acc)[NT][4], int lane) {
  const int g = lane >> 2, q = lane & 3;
  float* out = sg.out + static_cast<size_t>(plane) * (sg.n_tiles * 8) * sg.M;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    if (t < sg.n_tiles) {
      const int n0 = t * 8 + 2 * q;
      out[static_cast<size_t>(n0) * sg.M + row0 + g] = acc[t][0];
      out[static_cast<size_t>(n0 + 1) * sg.M + row0 + g] = acc[t][1];
      out[static_cast<size_t>(n0) * sg.M + row0 + g + 8] = acc[t][2];
      out[static_cast<size_t>(n0 + 1) * sg.M + row0 + g + 8] = acc[t][3];
    }
  }
}

DF2_DEV __half2 bf16_bits_half2(uint16_t b) { return __float2half2_rn(bf16_to_f32(b)); }

DF2_DEV uint32_t dequant2(uint32_t codes_biased, uint32_t sel, __half2 s, __half2 b) {
  const uint32_t qh = codes_to_half2(codes_biased, sel);
  __half2 w = __hfma2(*reinterpret_cast<const __half2*>(&qh), s, b);
  return *reinterpret_cast<uint32_t*>(&w);
}

// Scale and bias (bf16 bits) of the two groups a lane meets in one Q8 stage (one per
// code box: group 2b + q/2 of the stage), for rows g and g + 8.
constexpr int kAffGroups = stage_k<1>() / wbox_k<1>();
struct Q8Affine {
  uint16_t s0[kAffGroups], s1[kAffGroups], b0[kAffGroups], b1[kAffGroups];
};

DF2_DEV Q8Affine load_affine(const GemvSeg& sg, int row, int kabs, int q) {
  const int KG = sg.K >> 6;
  const size_t i0 = static_cast<size_t>(row) * KG + (kabs >> 6) + (q >> 1);
  const size_t i1 = i0 + static_cast<size_t>(8) * KG;
  Q8Affine r;
#pragma unroll
  for (int j = 0; j < kAffGroups; ++j) {
    r.s0[j] = __ldg(reinterpret_cast<const unsigned short*>(sg.scale) + i0 + 2 * j);
    r.s1[j] = __ldg(reinterpret_cast<const unsigned short*>(sg.scale) + i1 + 2 * j);
    r.b0[j] = __ldg(reinterpret_cast<const unsigned short*>(sg.bias) + i0 + 2 * j);
    r.b1[j] = __ldg(reinterpret_cast<const unsigned short*>(sg.bias) + i1 + 2 * j);
  }
  return r;
}

// Q8 stage: codes in two boxes [128 K][kBlockRows rows] (128-byte rows, 128-byte
// swizzle); fp16 activations per tile and plane in four boxes [64 K][8 rows] (1 KB
// each, 128-byte swizzle).  In code box b, lane (g, q) takes K 32q .. 32q + 31 (one
// group of 64: 2b + q/2): pieces 2q and 2q + 1 of rows g and g + 8, and pieces
// 4(q & 1) .. 4(q & 1) + 3 of activation box 2b + q/2.  Lanes with q >= 2 take
// the two halves in the opposite order (weight pieces 2q + 1 then 2q, activation
// piece j ^ 2 in register j), which puts every quarter-warp's 16-byte loads on
// distinct banks; which K an MMA slot holds then depends on q alone, the same for
// A and B.  wa: row g of this warp in code box 0; xrow: row g of tile 0, box 0, hi.
template <int NT>
DF2_DEV void stage_q8(int n_tiles, uint32_t wa, uint32_t xrow, int g, int q, const Q8Affine& af,
                      float (&c0)[NT][4], float (&c1)[NT][4], float (&c2)[NT][4], float (&c3)[NT][4]) {
  constexpr int kXBoxes = stage_k<1>() / 64;
  constexpr int kWBoxes = stage_k<1>() / wbox_k<1>();
  const int sw = q & 2;
  const uint32_t pf = static_cast<uint32_t>(((2 * q + (sw >> 1)) ^ g) << 4);
  const uint32_t ps = static_cast<uint32_t>(((2 * q + 1 - (sw >> 1)) ^ g) << 4);
  uint32_t xo[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    xo[j] = static_cast<uint32_t>((((4 * (q & 1) + (j ^ sw)) ^ g) << 4) + (q >> 1) * 1024);
#pragma unroll
  for (int b = 0; b < kWBoxes; ++b) {
    const uint32_t wb = wa + b * wbox_bytes<1>();
    const uint4 w0[2] = {lds128(wb + pf), lds128(wb + ps)};                // row g, two halves
    const uint4 w1[2] = {lds128(wb + 1024 + pf), lds128(wb + 1024 + ps)};  // row g + 8
    const __half2 sg0 = bf16_bits_half2(af.s0[b]), sg1 = bf16_bits_half2(af.s1[b]);
    const __half2 bg0 = bf16_bits_half2(af.b0[b]), bg1 = bf16_bits_half2(af.b1[b]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t u0[4] = {w0[h].x ^ 0x80808080u, w0[h].y ^ 0x80808080u, w0[h].z ^ 0x80808080u,
                              w0[h].w ^ 0x80808080u};
      const uint32_t u1[4] = {w1[h].x ^ 0x80808080u, w1[h].y ^ 0x80808080u, w1[h].z ^ 0x80808080u,
                              w1[h].w ^ 0x80808080u};
      uint32_t A[4][4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        A[m][0] = dequant2(u0[m], 0x4140, sg0, bg0);
        A[m][1] = dequant2(u1[m], 0x4140, sg1, bg1);
        A[m][2] = dequant2(u0[m], 0x4342, sg0, bg0);
        A[m][3] = dequant2(u1[m], 0x4342, sg1, bg1);
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t < n_tiles) {
          const uint32_t xb = xrow + (t * kXBoxes + 2 * b) * 1024;
          const uint4 xa = lds128(xb + xo[2 * h]), xc = lds128(xb + xo[2 * h + 1]);  // 8 + 8 K of this half
          // one fp16 plane; four independent accumulator chains
          mma_f16(c0[t], A[0][0], A[0][1], A[0][2], A[0][3], xa.x, xa.y);
          mma_f16(c1[t], A[1][0], A[1][1], A[1][2], A[1][3], xa.z, xa.w);
          mma_f16(c2[t], A[2][0], A[2][1], A[2][2], A[2][3], xc.x, xc.y);
          mma_f16(c3[t], A[3][0], A[3][1], A[3][2], A[3][3], xc.z, xc.w);
        }
      }
    }
  }
}

template <int NT, int FMT>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) gemv_kernel(const __grid_constant__ GemvArgs a) {
  using Geo = StageGeo<FMT, NT>;
  constexpr int D = Geo::kDepth;
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[D], empty_bar[D];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t full0 = smem_u32(&full_bar[0]), empty0 = smem_u32(&empty_bar[0]);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < D; ++s) {
      mbar_init_count(full0 + 8 * s, 1);
      mbar_init_count(empty0 + 8 * s, kConsumers);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_trigger();

  if (wid == kConsumers) {
    // ---------------------------------------------------------------- producer warp
    const uint64_t policy = evict_first_policy();  // weights: streamed once
    const uint64_t xpolicy = evict_last_policy();  // activations: read by every CTA
    constexpr int kWBoxes = stage_k<FMT>() / wbox_k<FMT>();  // weight boxes per stage
    constexpr int kXBoxes = stage_k<FMT>() / 64;  // activation boxes per tile and plane (64 K x 8 rows)
    constexpr int kXBoxK = 64;
    constexpr int kXBoxBytes = 8 * kXBoxK * 2;
    auto issue_w = [&](const Cursor& c, int slot) {
      if (lane < kWBoxes)
        tma_load_2d(ring + slot * Geo::kBytes + lane * wbox_bytes<FMT>(), &a.seg[c.seg].wmap, c.kabs + lane * wbox_k<FMT>(),
                    c.row0, full0 + 8 * slot, policy);
    };
    // this lane's activation boxes (plane, tile, 64-K box): box indices lane and lane + 32,
    // recomputed when the segment changes
    constexpr int kXPerLane = (Geo::kXPlanes * NT * kXBoxes + 31) / 32;
    int xs_seg = -1, x_row[kXPerLane], x_b[kXPerLane];
    uint32_t x_dst[kXPerLane];
    bool x_on[kXPerLane];
    auto issue_x = [&](const Cursor& c, int slot) {
      const GemvSeg& sg = a.seg[c.seg];
      if (c.seg != xs_seg) {
        xs_seg = c.seg;
        const int per = sg.n_tiles * kXBoxes;  // boxes per plane
#pragma unroll
        for (int j = 0; j < kXPerLane; ++j) {
          const int box = lane + 32 * j;
          x_on[j] = box < Geo::kXPlanes * per;
          const int plane = box / per, rem = box % per, t = rem / kXBoxes;
          x_b[j] = rem % kXBoxes;
          x_dst[j] = Geo::kWBytes + plane * Geo::kXPlane + (t * kXBoxes + x_b[j]) * kXBoxBytes;
          x_row[j] = plane * sg.x_lo_row + t * 8;
        }
      }
#pragma unroll
      for (int j = 0; j < kXPerLane; ++j)
        if (x_on[j])
          tma_load_2d(ring + slot * Geo::kBytes + x_dst[j], &sg.xmap, c.kabs + x_b[j] * kXBoxK, x_row[j],
                      full0 + 8 * slot, xpolicy);
    };
    auto arm = [&](const Cursor& c, int slot) {
      const int xbytes = Geo::kXPlanes * a.seg[c.seg].n_tiles * kXBoxes * kXBoxBytes;
      if (lane == 0) mbar_expect_tx(full0 + 8 * slot, Geo::kWBytes + xbytes);
      __syncwarp();
    };
    Cursor cw;
    cw.start(a);
    int np = 0;
    while (np < D && cw.valid) {  // weights of the first stages: before the wait on the previous kernel
      arm(cw, np);
      issue_w(cw, np);
      cw.next(a);
      ++np;
    }
    pdl_wait();
    Cursor cx;
    cx.start(a);
    int it = 0;
    bool ok = true;
    while (cx.valid) {
      const int slot = it % D;
      if (it >= np) {
        const uint32_t parity = static_cast<uint32_t>(((it / D) + 1) & 1);
        if (!__all_sync(0xffffffffu, mbar_wait(empty0 + 8 * slot, parity))) {
          ok = false;
          break;
        }
        arm(cx, slot);
        issue_w(cx, slot);
      }
      issue_x(cx, slot);
      cx.next(a);
      ++it;
    }
    if (!ok && lane == 0 && a.err != nullptr) atomicExch(a.err, 1);
    // the copies of the last stages land before this CTA's shared memory is released (bounded);
    // a failed wait happens only after every earlier stage was fully issued
    const int issued = it;
    for (int j = issued > D ? issued - D : 0; j < issued; ++j)
      mbar_wait(full0 + 8 * (j % D), static_cast<uint32_t>((j / D) & 1));
    return;
  }

  // ------------------------------------------------------------------ consumer warps
  pdl_wait();
  const int g = lane >> 2, q = lane & 3;
  // row g of this warp in a weight box (128-byte rows; the stage functions choose the
  // pieces), and row g of an activation box
  const uint32_t wrow = static_cast<uint32_t>((wid * 16 + g) * 128);
  const uint32_t xrow = static_cast<uint32_t>(g * 128);
  float c0[NT][4], c1[NT][4], c2[NT][4], c3[NT][4];
  Cursor c;
  c.start(a);
  const long long t_first = c.t;
  Q8Affine af = {};
  if (FMT == 1 && c.valid) af = load_affine(a.seg[c.seg], c.row0 + wid * 16 + g, c.kabs, q);
  int it = 0;
  while (c.valid) {
    if (c.opens(t_first)) {
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) c0[t][e] = c1[t][e] = c2[t][e] = c3[t][e] = 0.f;
    }
    const int slot = it % D;
    const GemvSeg& sg = a.seg[c.seg];
    // scale and bias of the next stage, loaded while this one computes
    Cursor cn = c;
    cn.next(a);
    Q8Affine afn = af;
    if (FMT == 1 && cn.valid) afn = load_affine(a.seg[cn.seg], cn.row0 + wid * 16 + g, cn.kabs, q);
    if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * slot, static_cast<uint32_t>((it / D) & 1)))) {
      if (lane == 0 && a.err != nullptr) atomicExch(a.err, 1);
      break;
    }
    const uint32_t base = ring + slot * Geo::kBytes;
    if (FMT == 0)
      stage_bf16<NT>(sg.n_tiles, base + wrow, base + Geo::kWBytes + xrow, g, q, c0, c1, c2, c3);
    else
      stage_q8<NT>(sg.n_tiles, base + wrow, base + Geo::kWBytes + xrow, g, q, af, c0, c1, c2, c3);
    __syncwarp();  // every lane's reads of this stage are done before it is released
    if (lane == 0) mbar_arrive(empty0 + 8 * slot);
    if (c.closes()) {
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) c0[t][e] = (c0[t][e] + c1[t][e]) + (c2[t][e] + c3[t][e]);
      store_tile<NT>(sg, c.plane(a), c.row0 + wid * 16, c0, lane);
    }
    c = cn;
    af = afn;
    ++it;
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, int esz, const void* p, int inner, int rows, int box_inner,
               int box_rows, CUtensorMapSwizzle swz, CUtensorMapL2promotion promo) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr || p == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * esz};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(p), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, promo,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NT, int FMT>
cudaError_t launch_nt(const GemvArgs& a, int ctas, bool pdl, cudaStream_t st) {
  constexpr int smem = StageGeo<FMT, NT>::kSmem;
  static std::atomic<unsigned long long> attr_done{0};
  const cudaError_t e = set_smem_once(gemv_kernel<NT, FMT>, smem, attr_done);
  if (e != cudaSuccess) return e;
  return launch_ex(gemv_kernel<NT, FMT>, dim3(ctas), dim3(kThreads), smem, st, pdl, a);
}

}  // namespace

bool tma_encode_2d(CUtensorMap* map, CUtensorMapDataType dt, int esz, const void* p, int inner, int rows,
                   int box_inner, int box_rows, CUtensorMapSwizzle swz) {
  return encode_2d(map, dt, esz, p, inner, rows, box_inner, box_rows, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

bool gemv_encode_wmap(CUtensorMap* map, const void* w, int M, int K, int fmt) {
  if (M % kBlockRows || K % kStageK) return false;
  if (fmt == 0)
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, K, M, 64, kBlockRows, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w, K, M, wbox_k<1>(), kBlockRows, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

bool gemv_encode_xmap(CUtensorMap* map, const void* x, int rows, int K, int fmt) {
  if (rows % 8 || K % kStageK) return false;
  if (fmt == 0)
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, K, 2 * rows, 64, 8, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x, K, 2 * rows, 64, 8, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
}

bool lm_encode_map(CUtensorMap* map, const void* p, int inner, int rows, int box_rows) {
  if (inner % kStageK || rows < 1) return false;
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p, inner, rows, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

int gemv_plan(GemvArgs& a, int num_sms, int fmt) {
  a.stage_k = fmt == 0 ? stage_k<0>() : stage_k<1>();
  long long T = 0;
  for (int i = 0; i < a.nseg; ++i) {
    GemvSeg& sg = a.seg[i];
    sg.stage_begin = T;
    T += static_cast<long long>(sg.M / kBlockRows) * (sg.K / a.stage_k);
  }
  a.total_stages = T;
  const long long C = static_cast<long long>(num_sms) * kCtasPerSm;
  return static_cast<int>(C < T ? C : (T > 0 ? T : 1));
}

GemvPlanes gemv_planes(const GemvArgs& a, int i, int C) {
  GemvPlanes p;
  p.T = a.total_stages;
  p.base = a.seg[i].stage_begin;
  p.C = C;
  p.kst = a.seg[i].K / a.stage_k;
  p.bshift = 6;
  return p;
}

int gemv_max_planes(const GemvArgs& a, int i, int C) {
  const GemvPlanes p = gemv_planes(a, i, C);
  int mx = 0;
  for (int m = 0; m < a.seg[i].M; m += kBlockRows) mx = std::max(mx, gemv_plane_count(p, m));
  return mx;
}

cudaError_t launch_gemv(GemvArgs& a, int fmt, int max_tiles, int num_sms, bool pdl, cudaStream_t st) {
  const int ks = fmt == 0 ? stage_k<0>() : stage_k<1>();
  for (int i = 0; i < a.nseg; ++i) {
    const GemvSeg& sg = a.seg[i];
    if (sg.M % kBlockRows || sg.K % ks || sg.n_tiles < 1 || sg.n_tiles > max_tiles) return cudaErrorInvalidValue;
  }
  const int C = gemv_plan(a, num_sms, fmt);
  if (a.total_stages < 1) return cudaErrorInvalidValue;
  if (fmt == 0) {
    if (max_tiles <= 1) return launch_nt<1, 0>(a, C, pdl, st);
    if (max_tiles <= 2) return launch_nt<2, 0>(a, C, pdl, st);
    if (max_tiles <= 4) return launch_nt<4, 0>(a, C, pdl, st);
    if (max_tiles <= 8) return launch_nt<8, 0>(a, C, pdl, st);
  } else {
    if (max_tiles <= 1) return launch_nt<1, 1>(a, C, pdl, st);
    if (max_tiles <= 2) return launch_nt<2, 1>(a, C, pdl, st);
    if (max_tiles <= 4) return launch_nt<4, 1>(a, C, pdl, st);
    if (max_tiles <= 8) return launch_nt<8, 1>(a, C, pdl, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace df2
