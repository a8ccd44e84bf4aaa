// Building blocks of the weight-streaming pipelines (the projection GEMV and the
// LM head): bulk tensor copies into a ring of shared-memory stages handed over
// through mbarriers, and the bf16 tensor-core stage body.  A stage holds
// kBlockRows weight rows x kStageK of K and the matching 8-row activation boxes.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace df2 {
namespace pipe {

constexpr int kBlockRows = 64;                // weight rows per unit
constexpr int kStageK = kGemvStageK;          // K per stage of bf16 weights (16 KB of 64 rows)
// K per stage by weight format: int8 stages hold twice the K in the same 16 KB
// (the pipeline streams at a rate set by stages, not bytes).
template <int FMT>
constexpr int stage_k() { return FMT == 0 ? kStageK : 2 * kStageK; }
constexpr int kConsumers = kBlockRows / 16;   // consumer warps per CTA (16 weight rows each)
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kCtasPerSm = 2;
constexpr int kRingBudget = (kCtasPerSm == 1 ? 208 : 200 / kCtasPerSm) * 1024;
constexpr int kMaxDepth = 24;
// One weight copy: kBlockRows rows of 128 bytes (64 K of bf16, 128 K of int8 codes),
// 128-byte swizzle.
template <int FMT>
constexpr int wbox_k() { return FMT == 0 ? 64 : 128; }
template <int FMT>
constexpr int wbox_bytes() { return 128 * kBlockRows; }
constexpr long long kSpinLimit = 1ll << 22;

// Shared-memory geometry of one stage for a format and a number of 8-row activation tiles.
template <int FMT, int NT>
struct StageGeo {
  static constexpr int kWBytes = kBlockRows * stage_k<FMT>() * (FMT == 0 ? 2 : 1);
  static constexpr int kXPlane = 8 * NT * stage_k<FMT>() * 2;  // 8*NT rows x stage K x 2 B
  // activation planes: bf16 carries a low-order plane (hi + lo); fp16 (int8 weights)
  // rounds to 2^-12 relative and needs none
  static constexpr int kXPlanes = FMT == 0 ? 2 : 1;
  static constexpr int kBytes = kWBytes + kXPlanes * kXPlane;
  static constexpr int kDepthRaw = kRingBudget / kBytes;
  static constexpr int kDepth = kDepthRaw < 2 ? 2 : (kDepthRaw > kMaxDepth ? kMaxDepth : kDepthRaw);
  static constexpr int kSmem = kDepth * kBytes + 1024;  // + slack for 1 KB alignment
};

DF2_DEV uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

DF2_DEV void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

DF2_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for the phase of the given parity; false if it did not complete.
DF2_DEV bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (long long i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

DF2_DEV uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

DF2_DEV uint64_t evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

DF2_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

DF2_DEV uint4 lds128(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr));
  return r;
}

DF2_DEV void mbar_init_count(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

DF2_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// BF16 stage: weights kStageK/64 boxes [64 K][kBlockRows rows] (128-byte rows,
// 128-byte swizzle); activations per tile and plane kStageK/64 boxes [64 K][8 rows]
// (1 KB each, same swizzle).  A lane reads the two 16-byte pieces 2q and 2q + 1
// (K 16q .. 16q + 15 of the box) of weight rows g, g + 8 and activation row g.
// wa / xrow: row g of box 0 (weights of this warp / tile 0, hi plane).
// LO: the activations carry a low-order plane (kXPlane bytes after the high plane).
template <int NT, bool LO = true>
DF2_DEV void stage_bf16(int n_tiles, uint32_t wa, uint32_t xrow, int g, int q, float (&c0)[NT][4],
                        float (&c1)[NT][4], float (&c2)[NT][4], float (&c3)[NT][4]) {
  constexpr int kXPlane = 8 * NT * kStageK * 2;
  constexpr int kB = kStageK / 64;
  const uint32_t pa = static_cast<uint32_t>(((2 * q) ^ g) << 4), pc = static_cast<uint32_t>(((2 * q + 1) ^ g) << 4);
#pragma unroll
  for (int b = 0; b < kB; ++b) {
    const uint32_t wb = wa + b * wbox_bytes<0>();
    const uint4 a0 = lds128(wb + pa), a0b = lds128(wb + pc);                // row g
    const uint4 a1 = lds128(wb + 1024 + pa), a1b = lds128(wb + 1024 + pc);  // row g + 8
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < n_tiles) {
        const uint32_t xb = xrow + (t * kB + b) * 1024;
        const uint4 x0 = lds128(xb + pa), x1 = lds128(xb + pc);
        mma_bf16(c0[t], a0.x, a1.x, a0.y, a1.y, x0.x, x0.y);
        mma_bf16(c1[t], a0.z, a1.z, a0.w, a1.w, x0.z, x0.w);
        mma_bf16(c0[t], a0b.x, a1b.x, a0b.y, a1b.y, x1.x, x1.y);
        mma_bf16(c1[t], a0b.z, a1b.z, a0b.w, a1b.w, x1.z, x1.w);
        if (LO) {
          const uint4 y0 = lds128(xb + kXPlane + pa), y1 = lds128(xb + kXPlane + pc);
          mma_bf16(c2[t], a0.x, a1.x, a0.y, a1.y, y0.x, y0.y);
          mma_bf16(c3[t], a0.z, a1.z, a0.w, a1.w, y0.z, y0.w);
          mma_bf16(c2[t], a0b.x, a1b.x, a0b.y, a1b.y, y1.x, y1.y);
          mma_bf16(c3[t], a0b.z, a1b.z, a0b.w, a1b.w, y1.z, y1.w);
        }
      }
    }
  }
}

}  // namespace pipe
}  // namespace df2
