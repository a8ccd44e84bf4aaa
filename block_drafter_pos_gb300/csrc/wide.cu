// Projections with many activation rows on the fifth-generation tensor cores
// (tcgen05): y[n][m] = sum_k W[m][k] x[n][k] for up to 256 activation rows, the
// shape of a step with more than four requests (8 block rows per request, plus the
// new context rows for the key and value projections).
//
// Design (sm_103a):
//  * Work is cut like the GEMV's: the stages (128-row weight block x 64 K) of the
//    launch's segments are split into contiguous runs, one per CTA (one CTA per SM,
//    stream-K), and a block shared by several CTAs gets one partial plane per CTA
//    (plane = CTA - first CTA of the block), which the next kernel adds in order.
//  * One CTA per SM with warp roles: warp 0 issues the bulk tensor copies of a stage
//    (the weight tile and the activation tile, 128-byte swizzle, completing on the
//    stage's "full" mbarrier); one thread of warp 1 issues tcgen05.mma (M = 128
//    weight rows, N = the activation rows rounded up to 16, K = 16 per instruction,
//    both operands from shared memory through matrix descriptors) into an fp32
//    accumulator in tensor memory, and tcgen05.commit releases the stage; warps 4..7
//    read a finished accumulator out of tensor memory (tcgen05.ld, one weight row
//    per thread) and store the partial plane.  The accumulator is double-buffered
//    (2 x 256 of the 512 tensor-memory columns), so the epilogue of one block
//    overlaps the products of the next.
//  * Q8/group64 weights ("LSE docs/DFLASH2.md", Q8 paragraph: w = scale * q + bias
//    per group of 64 along K): the copy brings the int8 codes (64-byte swizzle), and
//    warps 8..11 turn them into fp16 values in the operand layout (one weight row per
//    thread: byte permute against the 1024 exponent, w = q * s + b in fp16), then
//    hand the stage to the MMA thread through a second mbarrier after a proxy fence.
//    One stage is exactly one quantisation group along K.
//  * The activations are read as one 16-bit plane (bf16 for bf16 weights, fp16 for
//    Q8), the high plane of the buffers the element-wise kernels write.
//  * Every mbarrier wait is bounded; a wait that gives up sets the error word and
//    the CTA drains what it started (copies, products) before it frees the tensor
//    memory and exits.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "glue.h"
#include "internal.h"
#include "pipeline.cuh"

namespace df2 {

namespace {

using pipe::evict_first_policy;
using pipe::evict_last_policy;
using pipe::lds128;
using pipe::mbar_arrive;
using pipe::mbar_expect_tx;
using pipe::mbar_init_count;
using pipe::mbar_wait;
using pipe::smem_u32;
using pipe::tma_load_2d;

constexpr int kTM = 128;         // weight rows per block: the MMA's M
constexpr int kTK = 64;          // K per stage: one 128-byte swizzle atom of 16-bit values
constexpr int kMaxN = 256;       // activation rows per product: the MMA's largest N
constexpr int kTmemCols = 512;   // two accumulators of up to 256 fp32 columns
constexpr int kRingBytes = 200 * 1024;

// Shared-memory stage: A tile [128 rows][64 K] 16-bit (the weights, or their fp16
// values for Q8), B tile [up to 256 rows][64 K] 16-bit, and for Q8 the int8 codes
// [128 rows][64].  Every region starts on a 1 KB boundary (the swizzle atoms).
template <int FMT>
struct WideGeo {
  static constexpr int kA = kTM * kTK * 2;
  static constexpr int kB = kMaxN * kTK * 2;
  static constexpr int kCodes = FMT == 1 ? kTM * kTK : 0;
  static constexpr int kStage = kA + kB + kCodes;
  static constexpr int kDepth = kRingBytes / kStage;
  static constexpr int kSmem = kDepth * kStage + 1024;
  static constexpr int kWarps = FMT == 1 ? 12 : 8;
};

// Shared-memory matrix descriptor of a K-major tile of 128-byte rows under the
// 128-byte swizzle: start address, stride between 8-row groups 1024 bytes, the
// descriptor version of this architecture, swizzle mode 128B.  The leading offset is
// not used by this layout (one swizzle atom spans the tile's K) and is set to 1.
DF2_DEV uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B both bf16 (fmt 0)
// or both fp16 (fmt 1), both K-major, N and M.
DF2_DEV uint32_t instr_desc(int fmt, int n) {
  const uint32_t ab = fmt == 0 ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(kTM >> 4) << 24);
}

DF2_DEV void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier receives one arrival once every product issued before it has completed.
DF2_DEV void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

DF2_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DF2_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive fp32 columns of this thread's tensor-memory lane.
DF2_DEV void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

DF2_DEV void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Position in the launch's stage sequence: CTA c takes [c T / C, (c + 1) T / C).
struct WCursor {
  long long t, t1;
  int seg, row0, kstage, kst, kabs;
  bool valid;
  DF2_DEV void start(const GemvArgs& a) {
    const long long T = a.total_stages, C = gridDim.x;
    t = blockIdx.x * T / C;
    t1 = (blockIdx.x + 1) * T / C;
    valid = t < t1;
    if (!valid) return;
    seg = 0;
    while (seg + 1 < a.nseg && t >= a.seg[seg + 1].stage_begin) ++seg;
    const GemvSeg& sg = a.seg[seg];
    kst = sg.K / kTK;
    const long long local = t - sg.stage_begin;
    row0 = static_cast<int>(local / kst) * kTM;
    kstage = static_cast<int>(local % kst);
    kabs = kstage * kTK;
  }
  DF2_DEV void next(const GemvArgs& a) {
    if (++t >= t1) {
      valid = false;
      return;
    }
    if (++kstage < kst) {
      kabs += kTK;
      return;
    }
    kstage = 0;
    kabs = 0;
    row0 += kTM;
    if (row0 >= a.seg[seg].M) {
      ++seg;
      row0 = 0;
      kst = a.seg[seg].K / kTK;
    }
  }
  DF2_DEV bool opens(long long t_first) const { return kstage == 0 || t == t_first; }
  DF2_DEV bool closes() const { return kstage == kst - 1 || t == t1 - 1; }
  DF2_DEV int plane(const GemvArgs& a) const {
    return static_cast<int>(blockIdx.x) - gemv_cta_of_stage(t - kstage, gridDim.x, a.total_stages);
  }
};

DF2_DEV int n_mma_of(const GemvSeg& sg) { return (sg.n_tiles * 8 + 15) & ~15; }

DF2_DEV uint32_t dequant_pair(uint32_t codes_biased, uint32_t sel, __half2 s, __half2 b) {
  const uint32_t qh = codes_to_half2(codes_biased, sel);
  __half2 w = __hfma2(*reinterpret_cast<const __half2*>(&qh), s, b);
  return *reinterpret_cast<uint32_t*>(&w);
}

template <int FMT>
__global__ void __launch_bounds__(WideGeo<FMT>::kWarps * 32, 1) wide_kernel(const __grid_constant__ GemvArgs a) {
  using Geo = WideGeo<FMT>;
  constexpr int D = Geo::kDepth;
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[D], conv_bar[D], empty_bar[D], dfull_bar[2], dempty_bar[2], done_bar;
  __shared__ uint32_t tmem_base_sh;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t full0 = smem_u32(&full_bar[0]), conv0 = smem_u32(&conv_bar[0]);
  const uint32_t empty0 = smem_u32(&empty_bar[0]), dfull0 = smem_u32(&dfull_bar[0]);
  const uint32_t dempty0 = smem_u32(&dempty_bar[0]), done = smem_u32(&done_bar);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < D; ++s) {
      mbar_init_count(full0 + 8 * s, 1);
      mbar_init_count(conv0 + 8 * s, 4);
      mbar_init_count(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init_count(dfull0 + 8 * b, 1);
      mbar_init_count(dempty0 + 8 * b, 4);
    }
    mbar_init_count(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (wid == 1) {  // the whole warp allocates the accumulator columns (and frees them at the end)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_sh)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  pdl_trigger();
  bool ok = true;

  if (wid == 0) {
    // ------------------------------------------------------------ copy producer (one lane)
    if (lane == 0) {
      const uint64_t wpol = evict_first_policy();  // weights: streamed once
      const uint64_t xpol = evict_last_policy();   // activations: read by every CTA
      auto arm_w = [&](const WCursor& c, int slot) {
        const GemvSeg& sg = a.seg[c.seg];
        mbar_expect_tx(full0 + 8 * slot, (FMT == 0 ? Geo::kA : Geo::kCodes) + n_mma_of(sg) * kTK * 2);
        const uint32_t dst = ring + slot * Geo::kStage + (FMT == 0 ? 0 : Geo::kA + Geo::kB);
        tma_load_2d(dst, &sg.wmap, c.kabs, c.row0, full0 + 8 * slot, wpol);
      };
      WCursor cw;
      cw.start(a);
      int np = 0;
      while (np < D && cw.valid) {  // weights of the first stages: before the wait on the previous kernel
        arm_w(cw, np);
        cw.next(a);
        ++np;
      }
      pdl_wait();
      WCursor cx;
      cx.start(a);
      int it = 0;
      while (cx.valid) {
        const int slot = it % D;
        if (it >= np) {
          if (!mbar_wait(empty0 + 8 * slot, static_cast<uint32_t>(((it / D) + 1) & 1))) {
            ok = false;
            break;
          }
          arm_w(cx, slot);
        }
        tma_load_2d(ring + slot * Geo::kStage + Geo::kA, &a.seg[cx.seg].xmap, cx.kabs, 0, full0 + 8 * slot, xpol);
        cx.next(a);
        ++it;
      }
      // the copies of the last stages land before the shared memory is released (bounded)
      for (int j = it > D ? it - D : 0; j < it; ++j) mbar_wait(full0 + 8 * (j % D), static_cast<uint32_t>((j / D) & 1));
    }
  } else if (wid == 1) {
    // ------------------------------------------------------------ MMA issuer (one lane)
    if (lane == 0) {
      WCursor c;
      c.start(a);
      const long long t_first = c.t;
      int it = 0, tile = 0;
      uint32_t d_tmem = tmem, idesc = 0;
      while (c.valid) {
        const int slot = it % D;
        const uint32_t par = static_cast<uint32_t>((it / D) & 1);
        const bool first = c.opens(t_first);
        if (first) {
          const int buf = tile & 1;
          // the epilogue has drained this accumulator (block tile - 2)
          if (tile >= 2 && !mbar_wait(dempty0 + 8 * buf, static_cast<uint32_t>(((tile >> 1) + 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          d_tmem = tmem + static_cast<uint32_t>(buf * 256);
          idesc = instr_desc(FMT, n_mma_of(a.seg[c.seg]));
        }
        if (!mbar_wait(full0 + 8 * slot, par) || (FMT == 1 && !mbar_wait(conv0 + 8 * slot, par))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = ring + slot * Geo::kStage;
        const uint64_t ad = sw128_desc(sa), bd = sw128_desc(sa + Geo::kA);
#pragma unroll
        for (int k = 0; k < kTK / 16; ++k)  // 16 K = 32 bytes further along the swizzled rows
          umma_f16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (first && k == 0) ? 0u : 1u);
        umma_commit(empty0 + 8 * slot);  // the stage is free once these products are done
        if (c.closes()) {
          umma_commit(dfull0 + 8 * (tile & 1));
          ++tile;
        }
        c.next(a);
        ++it;
      }
      // every product issued has completed before the columns are freed (bounded)
      umma_commit(done);
      mbar_wait(done, 0);
    }
  } else if (wid >= 4 && wid < 8) {
    // ------------------------------------------------------------ epilogue: accumulator -> partial plane
    pdl_wait();  // the planes are written only after the previous kernel has completed
    const int quarter = wid & 3;  // tensor-memory lanes 32 quarter .. 32 quarter + 31
    WCursor c;
    c.start(a);
    int tile = 0;
    while (c.valid) {
      if (c.closes()) {
        const int buf = tile & 1;
        if (!mbar_wait(dfull0 + 8 * buf, static_cast<uint32_t>((tile >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const GemvSeg& sg = a.seg[c.seg];
        const int n_rows = sg.n_tiles * 8, nm = n_mma_of(sg);
        const int m = c.row0 + quarter * 32 + lane;
        float* out = sg.out + static_cast<size_t>(c.plane(a)) * n_rows * sg.M + m;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(buf * 256);
        for (int n0 = 0; n0 < nm; n0 += 16) {
          uint32_t r[16];
          tmem_ld16(taddr + n0, r);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (n0 + j < n_rows) out[static_cast<size_t>(n0 + j) * sg.M] = __uint_as_float(r[j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dempty0 + 8 * buf);
        ++tile;
      }
      c.next(a);
    }
  } else if (FMT == 1 && wid >= 8) {
    // ------------------------------------------------------------ int8 codes -> fp16 operand tile
    const int r = (wid - 8) * 32 + lane;  // weight row within the block
    WCursor c;
    c.start(a);
    auto affine = [&](const WCursor& cc, uint16_t& s, uint16_t& b) {
      const GemvSeg& sg = a.seg[cc.seg];
      const size_t i = static_cast<size_t>(cc.row0 + r) * (sg.K >> 6) + (cc.kabs >> 6);
      s = __ldg(reinterpret_cast<const unsigned short*>(sg.scale) + i);
      b = __ldg(reinterpret_cast<const unsigned short*>(sg.bias) + i);
    };
    uint16_t s_cur = 0, b_cur = 0;
    if (c.valid) affine(c, s_cur, b_cur);
    int it = 0;
    while (c.valid) {
      const int slot = it % D;
      WCursor cn = c;
      cn.next(a);
      uint16_t s_nx = s_cur, b_nx = b_cur;
      if (cn.valid) affine(cn, s_nx, b_nx);  // the next group's scale and bias, loaded during this stage
      if (!mbar_wait(full0 + 8 * slot, static_cast<uint32_t>((it / D) & 1))) {
        ok = false;
        break;
      }
      const uint32_t st = ring + slot * Geo::kStage;
      const uint32_t codes = st + Geo::kA + Geo::kB + r * 64;                    // 64-byte rows, 64-byte swizzle
      const uint32_t arow = st + (r >> 3) * 1024 + (r & 7) * 128;               // 128-byte rows, 128-byte swizzle
      const __half2 sh = __float2half2_rn(bf16_to_f32(s_cur)), bh = __float2half2_rn(bf16_to_f32(b_cur));
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {  // codes 16 ch .. 16 ch + 15
        const uint4 w = lds128(codes + ((ch ^ ((r >> 1) & 3)) << 4));
        const uint32_t u[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
        uint32_t h[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          h[2 * m] = dequant_pair(u[m], 0x4140, sh, bh);
          h[2 * m + 1] = dequant_pair(u[m], 0x4342, sh, bh);
        }
        sts128(arow + (((2 * ch) ^ (r & 7)) << 4), h[0], h[1], h[2], h[3]);
        sts128(arow + (((2 * ch + 1) ^ (r & 7)) << 4), h[4], h[5], h[6], h[7]);
      }
      // generic-proxy stores become visible to the tensor cores' reads before the hand-over
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(conv0 + 8 * slot);
      s_cur = s_nx;
      b_cur = b_nx;
      c = cn;
      ++it;
    }
  }
  if (!ok && a.err != nullptr) atomicExch(a.err, 1);
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (wid == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

template <int FMT>
cudaError_t launch_fmt(const GemvArgs& a, int ctas, bool pdl, cudaStream_t st) {
  constexpr int smem = WideGeo<FMT>::kSmem;
  static bool attr_set = false;  // set once, outside any later stream capture
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(wide_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(wide_kernel<FMT>, dim3(ctas), dim3(WideGeo<FMT>::kWarps * 32), smem, st, pdl, a);
}

}  // namespace

int wide_plan(GemvArgs& a, int num_sms) {
  a.stage_k = kTK;
  long long T = 0;
  for (int i = 0; i < a.nseg; ++i) {
    GemvSeg& sg = a.seg[i];
    sg.stage_begin = T;
    T += static_cast<long long>(sg.M / kTM) * (sg.K / kTK);
  }
  a.total_stages = T;
  const long long C = num_sms;
  return static_cast<int>(C < T ? C : (T > 0 ? T : 1));
}

GemvPlanes wide_planes(const GemvArgs& a, int i, int C) {
  GemvPlanes p;
  p.T = a.total_stages;
  p.base = a.seg[i].stage_begin;
  p.C = C;
  p.kst = a.seg[i].K / kTK;
  p.bshift = 7;
  return p;
}

int wide_max_planes(const GemvArgs& a, int i, int C) {
  const GemvPlanes p = wide_planes(a, i, C);
  int mx = 0;
  for (int m = 0; m < a.seg[i].M; m += kTM) {
    const int n = gemv_plane_count(p, m);
    mx = n > mx ? n : mx;
  }
  return mx;
}

bool wide_encode_wmap(CUtensorMap* map, const void* w, int M, int K, int fmt) {
  if (M % kTM || K % kTK) return false;
  if (fmt == 0)
    return tma_encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, K, M, kTK, kTM, CU_TENSOR_MAP_SWIZZLE_128B);
  return tma_encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w, K, M, kTK, kTM, CU_TENSOR_MAP_SWIZZLE_64B);
}

bool wide_encode_xmap(CUtensorMap* map, const void* x, int rows, int K, int fmt) {
  if (rows < 1 || rows > kMaxN || K % kTK) return false;
  const int nm = (rows + 15) & ~15;
  return tma_encode_2d(map, fmt == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x, K,
                       rows, kTK, nm, CU_TENSOR_MAP_SWIZZLE_128B);
}

cudaError_t launch_wide(GemvArgs& a, int fmt, int num_sms, bool pdl, cudaStream_t st) {
  for (int i = 0; i < a.nseg; ++i) {
    const GemvSeg& sg = a.seg[i];
    if (sg.M % kTM || sg.K % kTK || sg.n_tiles < 1 || sg.n_tiles * 8 > kMaxN) return cudaErrorInvalidValue;
    if (fmt == 1 && (sg.scale == nullptr || sg.bias == nullptr)) return cudaErrorInvalidValue;
  }
  const int C = wide_plan(a, num_sms);
  if (a.total_stages < 1) return cudaErrorInvalidValue;
  return fmt == 0 ? launch_fmt<0>(a, C, pdl, st) : launch_fmt<1>(a, C, pdl, st);
}

}  // namespace df2
