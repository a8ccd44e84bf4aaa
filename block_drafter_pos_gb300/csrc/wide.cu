// Projections with many activation rows on the fifth-generation tensor cores
// (tcgen05): y[n][m] = sum_k W[m][k] x[n][k] for up to 256 activation rows, the
// shape of a step with many requests (8 block rows per request, plus the
// new context rows for the key and value projections).
//
// Design (sm_103a):
//  * Work is cut like the GEMV's: the stages (weight block x stage K) of the
//    launch's segments are split into contiguous runs, one per CTA (stream-K), and a
//    block shared by several CTAs gets one partial plane per CTA (plane = CTA - first
//    CTA of the block), which the next kernel adds in order.
//  * Warp roles: warp 0 issues the bulk tensor copies of the weight tiles into a
//    deep ring (they come from HBM and never depend on the previous kernel), warp 2
//    those of the activation tiles into a shallow one (they stay in L2), each
//    completing on its stage's "full" mbarrier (128-byte swizzle); one thread of
//    warp 1 issues tcgen05.mma (M = 128 weight rows, N = the activation rows rounded
//    up to 16, K = 16 per instruction) into fp32 accumulators in tensor memory, and
//    tcgen05.commit releases the stage; warps 4..7 read a finished accumulator out
//    of tensor memory (tcgen05.ld, one weight row per thread) and store the partial
//    plane.  Accumulators are double-buffered where the columns allow, so the
//    epilogue of one block overlaps the products of the next.  The CTA's last piece
//    sits on the launch's tail: it is staged in the (by then idle) rings and leaves by
//    bulk copies (cp.async.bulk), which takes about half the time of plain stores.
//    With int8 weights the other pieces pass through 32 KB of staging the rings leave
//    free, 64 activation rows at a time, also by bulk copies.
//  * bf16 weights: two CTAs per SM, A and B both from shared memory through matrix
//    descriptors; stages of one 128-row block x 64 K.
//  * Q8/group64 weights ("LSE docs/DFLASH2.md", Q8 paragraph: w = scale * q + bias
//    per group of 64 along K): the copy brings the int8 codes, and sixteen converter
//    warps (two groups taking alternate stages) turn them into fp16 values
//    (byte permute against the 1024 exponent, w = q * s + b in fp16) written
//    straight into tensor memory (tcgen05.st), where the MMA reads its A operand.
//    No fp16 tile passes through shared memory: no store bank conflicts, and the
//    freed shared memory deepens the code ring.
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

constexpr int kTM = 128;         // weight rows per MMA: the MMA's M
constexpr int kAtomK = 64;       // K of one 128-byte swizzle atom of 16-bit values
constexpr int kMaxN = 256;       // activation rows per product: the MMA's largest N
constexpr int kMinStages = 4;    // shortest run of 128-K stages per CTA (small launches take fewer CTAs)

// K per stage: one bf16 weight copy of 128-byte rows (64 K); int8 codes in copies of
// 128-byte rows (128 K each): two per stage (256 K: four atoms of fp16 operand) for
// up to 128 activation rows, one (128 K) for more, whose activation tiles are twice
// the size.  Every stage costs the pipeline a fixed round of hand-offs (copies,
// converters, products, commits; about 0.45 us measured with the data movement
// taken out), so stages as long as the buffers allow keep it off the stream.
template <int FMT, int NMAX>
constexpr int stage_k() { return FMT == 0 ? 64 : (NMAX <= 128 ? 256 : 128); }
// CTAs per SM: bf16 runs two independent pipelines per SM (each with half the
// tensor memory); int8 one, whose sixteen converter warps fill the register file.
// (Measured with the operand in tensor memory: two int8 CTAs per SM with one
// converter group each, or pairs of weight blocks sharing an activation tile, are
// both slower.)
constexpr int ctas_per_sm(int fmt) { return fmt == 0 ? 2 : 1; }

// Shared memory: two rings, each region on a 1 KB boundary (the swizzle atoms):
// the weight copies W [128 rows][128 bytes] (bf16: the A operand itself; int8: the
// codes), which come from HBM, and the activation tiles B (stage_k / 64 atoms
// [NMAX rows][64 K]), which come from L2.  Tensor memory (columns of 128 lanes x
// 32 bits): for int8 kDA slots of the fp16 A operand (64 columns: 128 K per weight
// row, two values per column), then kBufs accumulators of NMAX fp32 columns.
template <int FMT, int NMAX>
struct WideGeo {
  static constexpr int kKS = stage_k<FMT, NMAX>();
  static constexpr int kAtoms = kKS / kAtomK;
  static constexpr int kW = kTM * (FMT == 0 ? 128 : kKS);  // bytes of one weight (code) stage
  static constexpr int kWBoxes = FMT == 0 ? 1 : kKS / 128;   // copies of 128-byte rows per stage
  static constexpr int kBAtom = NMAX * kAtomK * 2;
  static constexpr int kB = kAtoms * kBAtom;
  static constexpr int kCtas = ctas_per_sm(FMT);
  static constexpr int kTmemCols = 512 / kCtas;
  static constexpr int kDA = FMT == 1 ? 2 : 0;            // A-operand slots in tensor memory (int8)
  static constexpr int kACols = FMT == 1 ? kKS / 2 : 0;  // columns of one slot
  static constexpr int kDCol0 = kDA * kACols;             // first accumulator column
  static constexpr int kBufs = (kTmemCols - kDCol0) / NMAX >= 2 ? 2 : 1;
  static constexpr int kDB = FMT == 1 ? 2 : (NMAX == 128 ? 2 : 1);
  static constexpr int kRing = (FMT == 0 ? 100 : 224) * 1024;  // bf16: two CTAs per SM
  // int8: a code ring of 64 KB (2 stages of 256 K, or 4 of 128 K).  Measured at 16
  // requests with 128-K stages: gate/up 78 us at 2 or 4 stages, 80 at 6, 82 at 10.
  static constexpr int kDW = FMT == 1 ? 64 * 1024 / kW : (kRing - kDB * kB) / kW;
  static constexpr int kOffB = kDW * kW;
  // int8: the 32 KB the rings leave free stage the epilogue of the pieces before the last
  static constexpr int kEpiStage = FMT == 1 ? 32 * 1024 : 0;
  static constexpr int kSmem = kOffB + kDB * kB + kEpiStage + 1024;
  // Final epilogue: activation rows staged per pass, [n][128 weight rows] fp32 in the rings
  static constexpr int kFinCols = ((kOffB + kDB * kB) / (kTM * 4) < NMAX ? (kOffB + kDB * kB) / (kTM * 4) : NMAX) & ~15;
  // int8: sixteen converter warps, each converting 64 K of 32 weight rows per stage: one
  // group for 256-K stages, two taking alternate stages for 128-K stages
  static constexpr int kConvGroups = FMT == 1 ? (kKS == 256 ? 1 : 2) : 0;
  static constexpr int kConv = FMT == 1 ? 16 / kConvGroups : 4;  // converter warps per group
  static constexpr int kWarps = FMT == 1 ? 24 : 8;
  static_assert(kDCol0 + NMAX <= kTmemCols, "tensor memory columns");
  static_assert(kDW >= 2, "weight ring");
  // int8: converter group g takes the stages i = g (mod 2) and waits on the code slot
  // i mod kDW with the parity of i's use of that slot.  That wait is only sound if the
  // slot's previous use (stage i - kDW) has landed, which holds when the A-slot wait
  // the group passed at stage i - 2 (the products of stage i - 2 - kDA are done, so
  // their codes were converted) covers stage i - kDW.
  static_assert(FMT == 0 || kConvGroups == 1 || kDW == kConvGroups || kDW >= kDA + kConvGroups,
                "code ring depth vs converter groups");
  static_assert(FMT == 0 || kConv == 4 * (kKS / 64), "converter warps: four lane groups per 64 K");
  static_assert(kCtas * (kSmem + 1024) <= 228 * 1024, "shared memory per SM");
  static_assert(kSmem <= 227 * 1024, "dynamic shared memory per CTA");
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

// 32 consecutive 32-bit columns of this thread's tensor-memory lane (lane group of the
// warp: warp w reaches lanes 32 (w mod 4) .. 32 (w mod 4) + 31).
DF2_DEV void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
DF2_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D (tensor memory) += A (tensor memory, [128 rows][16 K], row i in lane i, two 16-bit
// values per column in K order) x B (shared memory descriptor).
DF2_DEV void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
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

// Bulk copy of `bytes` contiguous bytes from shared to global memory (16-byte aligned
// addresses, size a multiple of 16), tracked by this thread's bulk async-group.
DF2_DEV void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}
DF2_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Closes this thread's bulk async-group and waits until all its copies have completed.
DF2_DEV void bulk_commit_wait_all() {
  bulk_commit();
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Waits until all this thread's committed bulk copies have read their sources.
DF2_DEV void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
DF2_DEV void sts32(uint32_t addr, uint32_t v) { asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory"); }
// Orders this thread's shared-memory stores before later bulk copies that read them.
DF2_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

DF2_DEV uint32_t dequant_pair(uint32_t codes_biased, uint32_t sel, __half2 s, __half2 b) {
  const uint32_t qh = codes_to_half2(codes_biased, sel);
  __half2 w = __hfma2(*reinterpret_cast<const __half2*>(&qh), s, b);
  return *reinterpret_cast<uint32_t*>(&w);
}

template <int FMT, int NMAX>
__global__ void __launch_bounds__(WideGeo<FMT, NMAX>::kWarps * 32, WideGeo<FMT, NMAX>::kCtas)
    wide_kernel(const __grid_constant__ GemvArgs a) {
  using Geo = WideGeo<FMT, NMAX>;
  using Cur = WCursor<Geo::kKS>;
  constexpr int DW = Geo::kDW, DB = Geo::kDB, DA = Geo::kDA > 0 ? Geo::kDA : 1;
  constexpr int kConv = Geo::kConv;  // converter warps per group (int8)
  constexpr int NG = Geo::kConvGroups > 0 ? Geo::kConvGroups : 1;
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
  if (wid == 1) {  // the whole warp allocates the tensor-memory columns (and frees them at the end)
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
#pragma unroll
        for (int b = 0; b < Geo::kWBoxes; ++b)  // int8: 128 K per copy
          tma_load_2d(ring + s * Geo::kW + b * (kTM * 128), &a.seg[c.seg].wmap, c.kabs + 128 * b, c.row0,
                      wfull + 8 * s, pol);
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
          d_tmem = tmem + static_cast<uint32_t>(Geo::kDCol0 + buf * NMAX);
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
        const uint32_t baddr = ring + Geo::kOffB + sb * Geo::kB;
#pragma unroll
        for (int j = 0; j < Geo::kAtoms; ++j) {
          const uint64_t bd = sw128_desc(baddr + j * Geo::kBAtom);
          if (FMT == 0) {
            const uint64_t ad = sw128_desc(ring + sw * Geo::kW + j * kTM * 128);
#pragma unroll
            for (int k = 0; k < kAtomK / 16; ++k)  // 16 K = 32 bytes further along the swizzled rows
              umma_f16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (first && j == 0 && k == 0) ? 0u : 1u);
          } else {
            // A from tensor memory: slot sa, 8 columns per 16 K
            const uint32_t a_col = tmem + static_cast<uint32_t>(sa * Geo::kACols + j * (kAtomK / 2));
#pragma unroll
            for (int k = 0; k < kAtomK / 16; ++k)
              umma_f16_ts(d_tmem, a_col + static_cast<uint32_t>(8 * k), bd + 2 * k, idesc,
                          (first && j == 0 && k == 0) ? 0u : 1u);
          }
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
        float* out = sg.out + static_cast<size_t>(c.plane(a)) * n_rows * sg.M + c.row0 + quarter * 32;
        const uint32_t taddr =
            tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(Geo::kDCol0 + buf * NMAX);
        if (c.t == c.t1 - 1) {
          // The CTA's last piece, on the launch's tail: every stage has been consumed, so the
          // rings are free.  The warp's 32 weight rows go through shared memory ([n][32] fp32)
          // and leave by bulk copies of 128 bytes, one per activation row: about half the time
          // of plain stores from four warps.
          const uint32_t stg = ring + static_cast<uint32_t>(quarter * Geo::kFinCols * 128);
          for (int c0 = 0; c0 < n_rows; c0 += Geo::kFinCols) {
            const int cols = min(Geo::kFinCols, n_rows - c0);
            for (int n0 = 0; n0 < cols; n0 += 16) {
              uint32_t r[16];
              tmem_ld16(taddr + c0 + n0, r);
#pragma unroll
              for (int j = 0; j < 16; ++j) sts32(stg + static_cast<uint32_t>(((n0 + j) * 32 + lane) * 4), r[j]);
            }
            fence_proxy_async_smem();  // the bulk copies read what these stores wrote
            __syncwarp();
            for (int n = lane; n < cols; n += 32)
              bulk_store(out + static_cast<size_t>(c0 + n) * sg.M, stg + static_cast<uint32_t>(n * 128), 128);
            bulk_commit_wait_all();  // written before the staging is reused or the CTA exits
            __syncwarp();
          }
        } else if (Geo::kEpiStage > 0) {
          // Other pieces (the rings busy): through this warp's part of the epilogue staging,
          // kEpiRows activation rows a pass, by bulk copies as above.  The tensor memory is
          // read out before the accumulator is released; the copies may still be running.
          constexpr int kRows = Geo::kEpiStage / (4 * 128);
          const uint32_t stg = ring + static_cast<uint32_t>(Geo::kOffB + DB * Geo::kB + quarter * kRows * 128);
          for (int c0 = 0; c0 < n_rows; c0 += kRows) {
            const int cols = min(kRows, n_rows - c0);
            bulk_wait_read_all();  // the staging's previous copies have read it
            __syncwarp();
            for (int n0 = 0; n0 < cols; n0 += 16) {
              uint32_t r[16];
              tmem_ld16(taddr + c0 + n0, r);
#pragma unroll
              for (int j = 0; j < 16; ++j) sts32(stg + static_cast<uint32_t>(((n0 + j) * 32 + lane) * 4), r[j]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            for (int n = lane; n < cols; n += 32)
              bulk_store(out + static_cast<size_t>(c0 + n) * sg.M, stg + static_cast<uint32_t>(n * 128), 128);
            bulk_commit();
          }
        } else {
          for (int n0 = 0; n0 < nm; n0 += 16) {
            uint32_t r[16];
            tmem_ld16(taddr + n0, r);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (n0 + j < n_rows) out[static_cast<size_t>(n0 + j) * sg.M + lane] = __uint_as_float(r[j]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dempty + 8 * buf);
        ++tile;
      }
      c.next(a);
    }
    bulk_commit_wait_all();  // no copy still reads the staging when the CTA exits (also after an error)
  } else if (FMT == 1 && wid >= 8) {
    // ------------------------------------------------------------ int8 codes -> fp16 A operand in tensor memory
    const int cw = wid - 8;
    const int grp = cw / kConv;                 // this group converts the stages i with i mod NG == grp
    const int quarter = cw & 3;                 // = wid mod 4: the lane group this warp reaches
    const int r = quarter * 32 + lane;          // weight row within the block
    const int hk = (cw >> 2) % (kConv / 4);     // 64 K of the stage: one quantisation group, one atom
    Cur c;
    c.start(a);
    for (int g = 0; g < grp; ++g) c.next(a);
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
      for (int g = 0; g < NG && cn.valid; ++g) cn.next(a);
      uint16_t s_nx = s_cur, b_nx = b_cur;
      if (cn.valid) affine(cn, s_nx, b_nx);  // the next stage's scale and bias, loaded during this one
      if (!mbar_wait(wfull + 8 * sw, static_cast<uint32_t>((i / DW) & 1))) {
        ok = false;
        break;
      }
      // 128-byte code rows (128 K per copy) under the 128-byte swizzle: piece p (16 codes)
      // of row r at p ^ (r mod 8); this warp's 64 K are pieces 4 (hk mod 2) .. + 3 of copy hk / 2
      const uint32_t crow = ring + sw * Geo::kW + (hk >> 1) * (kTM * 128) + r * 128;
      uint4 w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = lds128(crow + (((4 * (hk & 1) + j) ^ (r & 7)) << 4));
      // the products that read this A slot last (stage i - DA) are done
      if (i >= DA && !mbar_wait(aempty + 8 * sa, static_cast<uint32_t>(((i / DA) + 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const __half2 sh = __float2half2_rn(bf16_to_f32(s_cur)), bh = __float2half2_rn(bf16_to_f32(b_cur));
      uint32_t hv[32];  // 64 fp16 values of K 64 hk .. 64 hk + 63 in K order, two per column
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t u[4] = {w[j].x ^ 0x80808080u, w[j].y ^ 0x80808080u, w[j].z ^ 0x80808080u,
                               w[j].w ^ 0x80808080u};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          hv[8 * j + 2 * m] = dequant_pair(u[m], 0x4140, sh, bh);
          hv[8 * j + 2 * m + 1] = dequant_pair(u[m], 0x4342, sh, bh);
        }
      }
      tmem_st32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                    static_cast<uint32_t>(sa * Geo::kACols + hk * (kAtomK / 2)),
                hv);
      // Every lane has used its codes (the stores above depend on them), so none of
      // its loads of the code slot is still in flight: the slot is free for the next
      // copy.  Releasing it before the values are used would let the copy overwrite
      // a slot a load is still reading.
      __syncwarp();
      if (lane == 0) mbar_arrive(wempty + 8 * sw);
      // the tensor-memory stores complete before the hand-over to the MMA thread
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(afull + 8 * sa);
      s_cur = s_nx;
      b_cur = b_nx;
      c = cn;
      i += NG;
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

int ks_of(int fmt, int nmax) {
  return fmt == 0 ? stage_k<0, 128>() : (nmax <= 128 ? stage_k<1, 128>() : stage_k<1, 256>());
}

}  // namespace

int wide_plan(GemvArgs& a, int num_sms, int fmt, int nmax) {
  a.stage_k = ks_of(fmt, nmax);
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
  const long long min_run = fmt == 1 ? kMinStages * 128 / a.stage_k : kMinStages;  // the same bytes per CTA
  const long long Cmin = (T + min_run - 1) / min_run;
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
  if (M % kTM || K % 128) return false;
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

int wide_nmax(const GemvArgs& a) {
  int nmax = 0;
  for (int i = 0; i < a.nseg; ++i) {
    const int nm = (a.seg[i].n_tiles * 8 + 15) & ~15;
    nmax = nm > nmax ? nm : nmax;
  }
  return nmax <= 128 ? 128 : 256;
}

cudaError_t launch_wide(GemvArgs& a, int fmt, int num_sms, bool pdl, cudaStream_t st) {
  const int ks = ks_of(fmt, wide_nmax(a));
  int nmax = 0;
  for (int i = 0; i < a.nseg; ++i) {
    const GemvSeg& sg = a.seg[i];
    if (sg.M % kTM || sg.K % ks || sg.n_tiles < 1 || sg.n_tiles * 8 > kMaxN) return cudaErrorInvalidValue;
    if (fmt == 1 && (sg.scale == nullptr || sg.bias == nullptr)) return cudaErrorInvalidValue;
    const int nm = (sg.n_tiles * 8 + 15) & ~15;
    if (sg.xt != nullptr && (sg.xt_rows < nm || (reinterpret_cast<uintptr_t>(sg.xt) & 15u))) return cudaErrorInvalidValue;
    nmax = nm > nmax ? nm : nmax;
  }
  const int C = wide_plan(a, num_sms, fmt, nmax <= 128 ? 128 : 256);
  if (a.total_stages < 1) return cudaErrorInvalidValue;
  if (fmt == 0) return nmax <= 128 ? launch_fmt<0, 128>(a, C, pdl, st) : launch_fmt<0, 256>(a, C, pdl, st);
  return nmax <= 128 ? launch_fmt<1, 128>(a, C, pdl, st) : launch_fmt<1, 256>(a, C, pdl, st);
}

}  // namespace df2
