// Projections with many activation rows on the fifth-generation tensor cores
// (tcgen05): y[n][m] = sum_k W[m][k] x[n][k] for up to 256 activation rows, the
// shape of a step with many requests (8 block rows per request, plus the
// new context rows for the key and value projections).
//
// Design (sm_103a):
//  * Work is cut like the GEMV's: the stages (128-row weight block x 64 K) of the
//    launch's segments are split into contiguous runs, one per CTA (one CTA per SM,
//    stream-K), and a block shared by several CTAs gets one partial plane per CTA
//    (plane = CTA - first CTA of the block), which the next kernel adds in order.
//  * One CTA per SM with warp roles: warp 0 issues the bulk tensor copies of the
//    weight tiles into a deep ring (they come from HBM and never depend on the
//    previous kernel), warp 2 those of the activation tiles into a shallow one (they
//    stay in L2), each completing on its stage's "full" mbarrier (128-byte swizzle);
//    one thread of warp 1 issues tcgen05.mma (M = 128
//    weight rows, N = the activation rows rounded up to 16, K = 16 per instruction,
//    both operands from shared memory through matrix descriptors) into an fp32
//    accumulator in tensor memory, and tcgen05.commit releases the stage; warps 4..7
//    read a finished accumulator out of tensor memory (tcgen05.ld, one weight row
//    per thread) and store the partial plane.  The accumulator is double-buffered
//    (2 x 256 of the 512 tensor-memory columns), so the epilogue of one block
//    overlaps the products of the next.
//  * Q8/group64 weights ("LSE docs/DFLASH2.md", Q8 paragraph: w = scale * q + bias
//    per group of 64 along K): the copy brings the int8 codes (64-byte swizzle), and
//    warps 8..15 turn them into fp16 values in a ring of operand tiles (one weight
//    row and half the stage's K per thread: byte permute against the 1024 exponent,
//    w = q * s + b in fp16), release the code slot once the codes have been used,
//    and hand the operand tile to the MMA thread through its mbarrier after a
//    proxy fence.
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
constexpr int kAtomK = 64;       // K of one 128-byte swizzle atom of 16-bit values
constexpr int kMaxN = 256;       // activation rows per product: the MMA's largest N
constexpr int kMinStages = 4;    // shortest run of stages per CTA (small launches take fewer CTAs)

// K per stage: one bf16 weight copy of 128-byte rows (64 K), or one int8 copy of
// 128-byte rows (128 K: two atoms of fp16 operand).
template <int FMT>
constexpr int stage_k() { return FMT == 0 ? 64 : 128; }
// CTAs per SM: bf16 runs two independent pipelines per SM (each with half the
// tensor memory); int8 one, whose sixteen converter warps fill the register file.
constexpr int ctas_per_sm(int fmt) { return fmt == 0 ? 2 : 1; }

// Three rings of shared-memory stages, each region on a 1 KB boundary (the swizzle
// atoms): the weight copies W [128 rows][128 bytes] (bf16: the A operand itself;
// int8: codes), which come from HBM; for int8 the fp16 operand tiles A (two atoms
// [128 rows][64 K]) the converter warps write; and the activation tiles B
// (stage_k / 64 atoms [NMAX rows][64 K]), which come from L2.  The accumulators:
// kBufs of NMAX fp32 columns in tensor memory (two, so the epilogue of one block
// overlaps the products of the next, where the columns allow).
template <int FMT, int NMAX>
struct WideGeo {
  static constexpr int kKS = stage_k<FMT>();
  static constexpr int kAtoms = kKS / kAtomK;
  static constexpr int kW = kTM * 128;
  static constexpr int kA = FMT == 1 ? kTM * kKS * 2 : 0;
  static constexpr int kBAtom = NMAX * kAtomK * 2;
  static constexpr int kB = kAtoms * kBAtom;
  static constexpr int kCtas = ctas_per_sm(FMT);
  static constexpr int kTmemCols = 512 / kCtas;
  static constexpr int kBufs = kTmemCols / NMAX >= 2 ? 2 : 1;
  static constexpr int kDA = FMT == 1 ? 2 : 0;
  static constexpr int kDB = FMT == 1 ? 2 : (NMAX == 128 ? 2 : 1);
  static constexpr int kRing = (FMT == 0 ? 100 : NMAX == 256 ? 224 : 208) * 1024;
  static constexpr int kDW = (kRing - kDB * kB - kDA * kA) / kW;
  static constexpr int kOffA = kDW * kW;
  static constexpr int kOffB = kOffA + kDA * kA;
  static constexpr int kSmem = kOffB + kDB * kB + 1024;
  static constexpr int kConvGroups = 2;  // int8: converter warp groups, taking alternate stages
  static constexpr int kWarps = FMT == 1 ? 8 + 8 * kConvGroups : 8;
  static_assert(kDW >= 2, "weight ring");
  // int8: converter group g takes the stages i = g (mod kConvGroups) and waits on the
  // code slot i mod kDW with the parity of i's use of that slot.  That wait is only
  // sound if the slot's previous use (stage i - kDW) has landed, which holds when
  // each group owns its slots (kDW == kConvGroups), or when the operand-slot wait the
  // group passed at stage i - kConvGroups (the products of stage i - kConvGroups - kDA
  // are done) already covers stage i - kDW.
  static_assert(FMT == 0 || kDW == kConvGroups || kDW >= kDA + kConvGroups, "code ring depth vs converter groups");
  static_assert(kCtas * (kSmem + 1024) <= 228 * 1024, "shared memory per SM");
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
template <int KS>
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
    kst = sg.K / KS;
    const long long local = t - sg.stage_begin;
    row0 = static_cast<int>(local / kst) * kTM;
    kstage = static_cast<int>(local % kst);
    kabs = kstage * KS;
  }
  DF2_DEV void next(const GemvArgs& a) {
    if (++t >= t1) {
      valid = false;
      return;
    }
    if (++kstage < kst) {
      kabs += KS;
      return;
    }
    kstage = 0;
    kabs = 0;
    row0 += kTM;
    if (row0 >= a.seg[seg].M) {
      ++seg;
      row0 = 0;
      kst = a.seg[seg].K / KS;
    }
  }
  DF2_DEV bool opens(long long t_first) const { return kstage == 0 || t == t_first; }
  DF2_DEV bool closes() const { return kstage == kst - 1 || t == t1 - 1; }
  DF2_DEV int plane(const GemvArgs& a) const {
    return static_cast<int>(blockIdx.x) - gemv_cta_of_stage(t - kstage, gridDim.x, a.total_stages);
  }
};

DF2_DEV int n_mma_of(const GemvSeg& sg) { return (sg.n_tiles * 8 + 15) & ~15; }

// Bulk copy of `bytes` contiguous bytes into shared memory, completing on an mbarrier.
DF2_DEV void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

DF2_DEV uint32_t dequant_pair(uint32_t codes_biased, uint32_t sel, __half2 s, __half2 b) {
  const uint32_t qh = codes_to_half2(codes_biased, sel);
  __half2 w = __hfma2(*reinterpret_cast<const __half2*>(&qh), s, b);
  return *reinterpret_cast<uint32_t*>(&w);
}

template <int FMT, int NMAX>
__global__ void __launch_bounds__(WideGeo<FMT, NMAX>::kWarps * 32, WideGeo<FMT, NMAX>::kCtas) wide_kernel(const __grid_constant__ GemvArgs a) {
  using Geo = WideGeo<FMT, NMAX>;
  using Cur = WCursor<Geo::kKS>;
  constexpr int DW = Geo::kDW, DB = Geo::kDB, DA = Geo::kDA > 0 ? Geo::kDA : 1;
  constexpr int kConv = 8;  // converter warps per group (int8)
  constexpr int NB = Geo::kBufs;
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t wfull_b[DW], wempty_b[DW], bfull_b[DB], bempty_b[DB], afull_b[DA], aempty_b[DA];
  __shared__ __align__(8) uint64_t dfull_b[2], dempty_b[2], done_b;
  __shared__ uint32_t tmem_base_sh;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t wfull = smem_u32(&wfull_b[0]), wempty = smem_u32(&wempty_b[0]);
  const uint32_t bfull = smem_u32(&bfull_b[0]), bempty = smem_u32(&bempty_b[0]);
  const uint32_t afull = smem_u32(&afull_b[0]), aempty = smem_u32(&aempty_b[0]);
  const uint32_t dfull = smem_u32(&dfull_b[0]), dempty = smem_u32(&dempty_b[0]), done = smem_u32(&done_b);
  if (threadIdx.x == 0) {
    for (int s = 0; s < DW; ++s) {
      mbar_init_count(wfull + 8 * s, 1);
      mbar_init_count(wempty + 8 * s, FMT == 0 ? 1 : kConv);  // released by the products / the converters
    }
    for (int s = 0; s < DB; ++s) {
      mbar_init_count(bfull + 8 * s, 1);
      mbar_init_count(bempty + 8 * s, 1);
    }
    for (int s = 0; s < DA; ++s) {
      mbar_init_count(afull + 8 * s, kConv);
      mbar_init_count(aempty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init_count(dfull + 8 * b, 1);
      mbar_init_count(dempty + 8 * b, 4);
    }
    mbar_init_count(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (wid == 1) {  // the whole warp allocates the accumulator columns (and frees them at the end)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_sh)),
                 "r"(Geo::kTmemCols)
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
    // ------------------------------------------------------------ weight copies (one lane)
    // The weights never depend on the previous kernel: no wait on it here.
    if (lane == 0) {
      const uint64_t pol = evict_first_policy();  // streamed once
      Cur c;
      c.start(a);
      int i = 0;
      while (c.valid) {
        const int s = i % DW;
        if (i >= DW && !mbar_wait(wempty + 8 * s, static_cast<uint32_t>(((i / DW) + 1) & 1))) {
          ok = false;
          break;
        }
        mbar_expect_tx(wfull + 8 * s, Geo::kW);
        tma_load_2d(ring + s * Geo::kW, &a.seg[c.seg].wmap, c.kabs, c.row0, wfull + 8 * s, pol);
        c.next(a);
        ++i;
      }
      // the last copies land before the shared memory is released (bounded)
      for (int j = i > DW ? i - DW : 0; j < i; ++j) mbar_wait(wfull + 8 * (j % DW), static_cast<uint32_t>((j / DW) & 1));
    }
  } else if (wid == 2) {
    // ------------------------------------------------------------ activation copies (one lane)
    if (lane == 0) {
      pdl_wait();  // the activations are the previous kernel's output
      const uint64_t pol = evict_last_policy();  // read by every CTA
      Cur c;
      c.start(a);
      int i = 0;
      while (c.valid) {
        const int s = i % DB;
        if (i >= DB && !mbar_wait(bempty + 8 * s, static_cast<uint32_t>(((i / DB) + 1) & 1))) {
          ok = false;
          break;
        }
        const GemvSeg& sg = a.seg[c.seg];
        const int nm = n_mma_of(sg);
        mbar_expect_tx(bfull + 8 * s, Geo::kAtoms * nm * kAtomK * 2);
        const uint32_t dst = ring + Geo::kOffB + s * Geo::kB;
#pragma unroll
        for (int j = 0; j < Geo::kAtoms; ++j) {
          if (sg.xt != nullptr) {  // one contiguous block per 64-K slice: rows 0 .. nm - 1 of the slice
            const char* src = static_cast<const char*>(sg.xt) +
                              (static_cast<size_t>(c.kabs / kAtomK + j) * sg.xt_rows) * (kAtomK * 2);
            bulk_load(dst + j * Geo::kBAtom, src, static_cast<uint32_t>(nm * kAtomK * 2), bfull + 8 * s, pol);
          } else {
            tma_load_2d(dst + j * Geo::kBAtom, &sg.xmap, c.kabs + j * kAtomK, 0, bfull + 8 * s, pol);
          }
        }
        c.next(a);
        ++i;
      }
      for (int j = i > DB ? i - DB : 0; j < i; ++j) mbar_wait(bfull + 8 * (j % DB), static_cast<uint32_t>((j / DB) & 1));
    }
  } else if (wid == 1) {
    // ------------------------------------------------------------ MMA issuer (one lane)
    if (lane == 0) {
      Cur c;
      c.start(a);
      const long long t_first = c.t;
      int i = 0, tile = 0;
      uint32_t d_tmem = tmem, idesc = 0;
      while (c.valid) {
        const bool first = c.opens(t_first);
        if (first) {
          const int buf = tile % NB;
          // the epilogue has drained this accumulator (block tile - NB)
          if (tile >= NB && !mbar_wait(dempty + 8 * buf, static_cast<uint32_t>(((tile / NB) + 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          d_tmem = tmem + static_cast<uint32_t>(buf * NMAX);
          idesc = instr_desc(FMT, n_mma_of(a.seg[c.seg]));
        }
        const int sb = i % DB, sw = i % DW, sa = i % DA;
        const bool in = mbar_wait(bfull + 8 * sb, static_cast<uint32_t>((i / DB) & 1)) &&
                        (FMT == 0 ? mbar_wait(wfull + 8 * sw, static_cast<uint32_t>((i / DW) & 1))
                                  : mbar_wait(afull + 8 * sa, static_cast<uint32_t>((i / DA) & 1)));
        if (!in) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t aaddr = FMT == 0 ? ring + sw * Geo::kW : ring + Geo::kOffA + sa * Geo::kA;
        const uint32_t baddr = ring + Geo::kOffB + sb * Geo::kB;
#pragma unroll
        for (int j = 0; j < Geo::kAtoms; ++j) {
          const uint64_t ad = sw128_desc(aaddr + j * kTM * 128), bd = sw128_desc(baddr + j * Geo::kBAtom);
#pragma unroll
          for (int k = 0; k < kAtomK / 16; ++k)  // 16 K = 32 bytes further along the swizzled rows
            umma_f16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (first && j == 0 && k == 0) ? 0u : 1u);
        }
        // the stages are free once these products are done
        umma_commit(bempty + 8 * sb);
        umma_commit(FMT == 0 ? wempty + 8 * sw : aempty + 8 * sa);
        if (c.closes()) {
          umma_commit(dfull + 8 * (tile % NB));
          ++tile;
        }
        c.next(a);
        ++i;
      }
      // every product issued has completed before the columns are freed (bounded)
      umma_commit(done);
      mbar_wait(done, 0);
    }
  } else if (wid >= 4 && wid < 8) {
    // ------------------------------------------------------------ epilogue: accumulator -> partial plane
    pdl_wait();  // the planes are written only after the previous kernel has completed
    const int quarter = wid & 3;  // tensor-memory lanes 32 quarter .. 32 quarter + 31
    Cur c;
    c.start(a);
    int tile = 0;
    while (c.valid) {
      if (c.closes()) {
        const int buf = tile % NB;
        if (!mbar_wait(dfull + 8 * buf, static_cast<uint32_t>((tile / NB) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const GemvSeg& sg = a.seg[c.seg];
        const int n_rows = sg.n_tiles * 8, nm = n_mma_of(sg);
        const int m = c.row0 + quarter * 32 + lane;
        float* out = sg.out + static_cast<size_t>(c.plane(a)) * n_rows * sg.M + m;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(buf * NMAX);
        for (int n0 = 0; n0 < nm; n0 += 16) {
          uint32_t r[16];
          tmem_ld16(taddr + n0, r);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (n0 + j < n_rows) out[static_cast<size_t>(n0 + j) * sg.M] = __uint_as_float(r[j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dempty + 8 * buf);
        ++tile;
      }
      c.next(a);
    }
  } else if (FMT == 1 && wid >= 8) {
    // ------------------------------------------------------------ int8 codes -> fp16 operand tiles
    const int cw = wid - 8;
    const int grp = cw >> 3;                    // this group converts the stages i with i mod 2 == grp
    const int r = (cw & 3) * 32 + lane;         // weight row within the block
    const int hk = (cw >> 2) & 1;               // 64-K half of the stage: one quantisation group, one atom
    Cur c;
    c.start(a);
    if (grp == 1) c.next(a);
    auto affine = [&](const Cur& cc, uint16_t& s, uint16_t& b) {
      const GemvSeg& sg = a.seg[cc.seg];
      const size_t idx = static_cast<size_t>(cc.row0 + r) * (sg.K >> 6) + (cc.kabs >> 6) + hk;
      s = __ldg(reinterpret_cast<const unsigned short*>(sg.scale) + idx);
      b = __ldg(reinterpret_cast<const unsigned short*>(sg.bias) + idx);
    };
    uint16_t s_cur = 0, b_cur = 0;
    if (c.valid) affine(c, s_cur, b_cur);
    int i = grp;
    while (c.valid) {
      const int sw = i % DW, sa = i % DA;
      Cur cn = c;
      cn.next(a);
      if (cn.valid) cn.next(a);
      uint16_t s_nx = s_cur, b_nx = b_cur;
      if (cn.valid) affine(cn, s_nx, b_nx);  // the next group's scale and bias, loaded during this stage
      if (!mbar_wait(wfull + 8 * sw, static_cast<uint32_t>((i / DW) & 1))) {
        ok = false;
        break;
      }
      // 128-byte code rows under the 128-byte swizzle: piece p (16 codes) of row r at p ^ (r mod 8)
      const uint32_t crow = ring + sw * Geo::kW + r * 128;
      uint4 w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = lds128(crow + (((4 * hk + j) ^ (r & 7)) << 4));
      if (i >= DA && !mbar_wait(aempty + 8 * sa, static_cast<uint32_t>(((i / DA) + 1) & 1))) {
        ok = false;
        break;
      }
      // atom hk of the operand tile: 128-byte rows, 128-byte swizzle
      const uint32_t arow = ring + Geo::kOffA + sa * Geo::kA + hk * (kTM * 128) + (r >> 3) * 1024 + (r & 7) * 128;
      const __half2 sh = __float2half2_rn(bf16_to_f32(s_cur)), bh = __float2half2_rn(bf16_to_f32(b_cur));
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // codes 16 j .. 16 j + 15 of the group -> fp16 pieces 2 j, 2 j + 1
        const uint32_t u[4] = {w[j].x ^ 0x80808080u, w[j].y ^ 0x80808080u, w[j].z ^ 0x80808080u,
                               w[j].w ^ 0x80808080u};
        uint32_t hv[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          hv[2 * m] = dequant_pair(u[m], 0x4140, sh, bh);
          hv[2 * m + 1] = dequant_pair(u[m], 0x4342, sh, bh);
        }
        sts128(arow + (((2 * j) ^ (r & 7)) << 4), hv[0], hv[1], hv[2], hv[3]);
        sts128(arow + (((2 * j + 1) ^ (r & 7)) << 4), hv[4], hv[5], hv[6], hv[7]);
      }
      // Every lane has used its codes (the stores above depend on them), so none of
      // its loads of the code slot is still in flight: the slot is free for the next
      // copy.  Releasing it before the values are used would let the copy overwrite
      // a slot a load is still reading.
      __syncwarp();
      if (lane == 0) mbar_arrive(wempty + 8 * sw);
      // generic-proxy stores become visible to the tensor cores' reads before the hand-over
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(afull + 8 * sa);
      s_cur = s_nx;
      b_cur = b_nx;
      c = cn;
      i += 2;
    }
  }
  if (!ok && a.err != nullptr) atomicExch(a.err, 1);
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (wid == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(Geo::kTmemCols) : "memory");
  }
}

template <int FMT, int NMAX>
cudaError_t launch_fmt(const GemvArgs& a, int ctas, bool pdl, cudaStream_t st) {
  constexpr int smem = WideGeo<FMT, NMAX>::kSmem;
  static std::atomic<unsigned long long> attr_done{0};
  const cudaError_t e = set_smem_once(wide_kernel<FMT, NMAX>, smem, attr_done);
  if (e != cudaSuccess) return e;
  return launch_ex(wide_kernel<FMT, NMAX>, dim3(ctas), dim3(WideGeo<FMT, NMAX>::kWarps * 32), smem, st, pdl, a);
}

int ks_of(int fmt) { return fmt == 0 ? stage_k<0>() : stage_k<1>(); }

}  // namespace

int wide_plan(GemvArgs& a, int num_sms, int fmt) {
  a.stage_k = ks_of(fmt);
  long long T = 0;
  for (int i = 0; i < a.nseg; ++i) {
    GemvSeg& sg = a.seg[i];
    sg.stage_begin = T;
    T += static_cast<long long>(sg.M / kTM) * (sg.K / a.stage_k);
  }
  a.total_stages = T;
  // one run of stages per CTA, at least kMinStages long: a small launch on fewer
  // CTAs pays fewer prologues and leaves fewer partial planes to add
  long long C = static_cast<long long>(num_sms) * ctas_per_sm(fmt);
  const long long Cmin = (T + kMinStages - 1) / kMinStages;
  if (Cmin < C) C = Cmin;
  return static_cast<int>(C < T ? C : (T > 0 ? T : 1));
}

GemvPlanes wide_planes(const GemvArgs& a, int i, int C) {
  GemvPlanes p;
  p.T = a.total_stages;
  p.base = a.seg[i].stage_begin;
  p.C = C;
  p.kst = a.seg[i].K / a.stage_k;
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
  if (M % kTM || K % ks_of(fmt)) return false;
  if (fmt == 0)
    return tma_encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, K, M, 64, kTM, CU_TENSOR_MAP_SWIZZLE_128B);
  return tma_encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w, K, M, 128, kTM, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool wide_encode_xmap(CUtensorMap* map, const void* x, int rows, int K, int fmt) {
  if (rows < 1 || rows > kMaxN || K % kAtomK) return false;
  const int nm = (rows + 15) & ~15;
  return tma_encode_2d(map, fmt == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x, K,
                       rows, kAtomK, nm, CU_TENSOR_MAP_SWIZZLE_128B);
}

cudaError_t launch_wide(GemvArgs& a, int fmt, int num_sms, bool pdl, cudaStream_t st) {
  const int ks = ks_of(fmt);
  int nmax = 0;
  for (int i = 0; i < a.nseg; ++i) {
    const GemvSeg& sg = a.seg[i];
    if (sg.M % kTM || sg.K % ks || sg.n_tiles < 1 || sg.n_tiles * 8 > kMaxN) return cudaErrorInvalidValue;
    if (fmt == 1 && (sg.scale == nullptr || sg.bias == nullptr)) return cudaErrorInvalidValue;
    const int nm = (sg.n_tiles * 8 + 15) & ~15;
    if (sg.xt != nullptr && (sg.xt_rows < nm || (reinterpret_cast<uintptr_t>(sg.xt) & 15u))) return cudaErrorInvalidValue;
    nmax = nm > nmax ? nm : nmax;
  }
  const int C = wide_plan(a, num_sms, fmt);
  if (a.total_stages < 1) return cudaErrorInvalidValue;
  if (fmt == 0) return nmax <= 128 ? launch_fmt<0, 128>(a, C, pdl, st) : launch_fmt<0, 256>(a, C, pdl, st);
  return nmax <= 128 ? launch_fmt<1, 128>(a, C, pdl, st) : launch_fmt<1, 256>(a, C, pdl, st);
}

}  // namespace df2
