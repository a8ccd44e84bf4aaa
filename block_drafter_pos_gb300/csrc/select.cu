// Selector walk (step a10): the low-rank bigram selector of the vLLM PR #52816
// description ("Candidate selector"): score(p -> c) = <A[p] * gate_i, B[c]> +
// unary_i[c], with A, B the rank-256 codebooks, gate_i the projection of position
// i's hidden state and unary the candidate's drafter logit; the walk starts at the
// verified anchor, takes the argmax at T = 0 and an inverse-CDF draw from
// softmax(score / T) at T > 0, and returns q over the 16 candidates.
//
// One CTA per request.  The full 7 x 16 x 16 lattice is scored first (position 1
// from the anchor), one thread per (position, predecessor, candidate) pair over
// padded shared-memory rows, then one warp walks it (lane j = candidate j).  Any nonfinite candidate logit or
// score marks the request DFLASH2_E_NONFINITE ("LSE docs/DFLASH2.md": the
// selector rejects nonfinite scores).
#include <math.h>

#include "common.cuh"
#include "glue.h"
#include "internal.h"
#include "philox.cuh"

namespace df2 {

namespace {

constexpr int kP = 7, kK = 16, kRank = 256;

constexpr int kRowsA = 1 + (kP - 1) * kK;  // anchor + candidates of positions 1..6
constexpr int kRowsB = kP * kK;            // candidates of positions 1..7
constexpr int kRows = kRowsA + kRowsB;

// Codebook rows staged in shared memory in their stored format: bf16 (256 x 2 B) or
// Q8 codes (256 B) plus 4 groups of (scale, bias).
constexpr int kPadBf = kRank + 8;   // bf16 row stride: consecutive rows start 16 B apart mod 128 B
constexpr int kPadQ8 = kRank + 16;  // int8 row stride, same idea

struct SelSmem {
  uint16_t bf[kRows][kPadBf];  // BF16 rows (unused for Q8)
  int8_t q8[kRows][kPadQ8];    // Q8 codes (unused for BF16)
  uint16_t sb[kRows][8];       // Q8: scale[4], bias[4]
  float gate[kP][kRank];
  float lat[kP][kK][kK];       // scores [position][pred][cand]
  int cids[kP][kK];
  float cl[kP][kK];
  int bad;
};

constexpr int kThreads = 512;

DF2_DEV float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
DF2_DEV float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Edge score of predecessor row ra and candidate row rb at position i (without the unary term).
DF2_DEV float edge_dot(const SelSmem& sm, int fmt, int i, int ra, int rb) {
  const float* g = sm.gate[i];
  float s = 0.f;
  if (fmt == 0) {
    const uint4* A = reinterpret_cast<const uint4*>(sm.bf[ra]);
    const uint4* B = reinterpret_cast<const uint4*>(sm.bf[rb]);
#pragma unroll 4
    for (int k = 0; k < kRank / 8; ++k) {
      const uint4 av = A[k], bv = B[k];
      const float4 g0 = *reinterpret_cast<const float4*>(g + 8 * k);
      const float4 g1 = *reinterpret_cast<const float4*>(g + 8 * k + 4);
      s = fmaf(bf_lo(av.x), g0.x * bf_lo(bv.x), s);
      s = fmaf(bf_hi(av.x), g0.y * bf_hi(bv.x), s);
      s = fmaf(bf_lo(av.y), g0.z * bf_lo(bv.y), s);
      s = fmaf(bf_hi(av.y), g0.w * bf_hi(bv.y), s);
      s = fmaf(bf_lo(av.z), g1.x * bf_lo(bv.z), s);
      s = fmaf(bf_hi(av.z), g1.y * bf_hi(bv.z), s);
      s = fmaf(bf_lo(av.w), g1.z * bf_lo(bv.w), s);
      s = fmaf(bf_hi(av.w), g1.w * bf_hi(bv.w), s);
    }
  } else {
#pragma unroll
    for (int grp = 0; grp < kRank / 64; ++grp) {
      const float sa = bf16_to_f32(sm.sb[ra][grp]), ba = bf16_to_f32(sm.sb[ra][4 + grp]);
      const float sb = bf16_to_f32(sm.sb[rb][grp]), bb = bf16_to_f32(sm.sb[rb][4 + grp]);
      const int8_t* A = sm.q8[ra] + 64 * grp;
      const int8_t* B = sm.q8[rb] + 64 * grp;
      const float* gg = g + 64 * grp;
#pragma unroll 4
      for (int k = 0; k < 64; k += 4) {
        const char4 av = *reinterpret_cast<const char4*>(A + k), bv = *reinterpret_cast<const char4*>(B + k);
        const float4 g4 = *reinterpret_cast<const float4*>(gg + k);
        s = fmaf(fmaf(sa, static_cast<float>(av.x), ba), g4.x * fmaf(sb, static_cast<float>(bv.x), bb), s);
        s = fmaf(fmaf(sa, static_cast<float>(av.y), ba), g4.y * fmaf(sb, static_cast<float>(bv.y), bb), s);
        s = fmaf(fmaf(sa, static_cast<float>(av.z), ba), g4.z * fmaf(sb, static_cast<float>(bv.z), bb), s);
        s = fmaf(fmaf(sa, static_cast<float>(av.w), ba), g4.w * fmaf(sb, static_cast<float>(bv.w), bb), s);
      }
    }
  }
  return s;
}

__global__ void __launch_bounds__(kThreads) select_kernel(const SelectArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  pdl_begin();
  const int r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) sm.bad = 0;
  for (int e = tid; e < kP * kK; e += kThreads) {
    sm.cids[e / kK][e % kK] = min(max(a.cand_ids[static_cast<size_t>(r) * kP * kK + e], 0), a.V - 1);
    const float v = a.cand_logits[static_cast<size_t>(r) * kP * kK + e];
    sm.cl[e / kK][e % kK] = v;
    if (!isfinite(v)) atomicOr(&sm.bad, 1);
  }
  for (int e = tid; e < kP * kRank; e += kThreads) sm.gate[e / kRank][e % kRank] = a.gate[static_cast<size_t>(r) * kP * kRank + e];
  __syncthreads();
  const int anchor = min(max(a.anchor_ids[r], 0), a.V - 1);
  // stage every needed codebook row at once (one round trip): row k < kRowsA is the
  // predecessor row A[id], k >= kRowsA the successor row B[id]
  const int chunks = a.fmt == 0 ? kRank * 2 / 16 : kRank / 16;  // 16-byte pieces per row
  // every thread's pieces are loaded first (all in flight together), then stored
  constexpr int kPer = (kRows * kRank * 2 / 16 + kThreads - 1) / kThreads;
  uint4 piece[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int e = tid + kThreads * j;
    piece[j] = make_uint4(0, 0, 0, 0);
    if (e < kRows * chunks) {
      const int k = e / chunks, c = e % chunks;
      int id;
      const void* cb;
      if (k < kRowsA) {
        id = k == 0 ? anchor : sm.cids[(k - 1) / kK][(k - 1) % kK];
        cb = a.cb_a;
      } else {
        id = sm.cids[(k - kRowsA) / kK][(k - kRowsA) % kK];
        cb = a.cb_b;
      }
      piece[j] = a.fmt == 0 ? ld_cached(reinterpret_cast<const uint16_t*>(cb) + static_cast<size_t>(id) * kRank + c * 8)
                            : ld_cached(reinterpret_cast<const int8_t*>(cb) + static_cast<size_t>(id) * kRank + c * 16);
    }
  }
  if (a.fmt != 0) {  // Q8: 4 groups of (scale, bias) per row
    for (int e = tid; e < kRows * 4; e += kThreads) {
      const int k = e >> 2, c = e & 3;
      const int id = k < kRowsA ? (k == 0 ? anchor : sm.cids[(k - 1) / kK][(k - 1) % kK])
                                : sm.cids[(k - kRowsA) / kK][(k - kRowsA) % kK];
      const uint16_t* sc = k < kRowsA ? a.cb_a_scale : a.cb_b_scale;
      const uint16_t* bi = k < kRowsA ? a.cb_a_bias : a.cb_b_bias;
      sm.sb[k][c] = sc[static_cast<size_t>(id) * 4 + c];
      sm.sb[k][4 + c] = bi[static_cast<size_t>(id) * 4 + c];
    }
  }
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int e = tid + kThreads * j;
    if (e < kRows * chunks) {
      const int k = e / chunks, c = e % chunks;
      if (a.fmt == 0)
        *reinterpret_cast<uint4*>(&sm.bf[k][c * 8]) = piece[j];
      else
        *reinterpret_cast<uint4*>(&sm.q8[k][c * 16]) = piece[j];
    }
  }
  __syncthreads();
  // lattice: one thread per (position, pred, cand)
  const int n_pairs = kK + (kP - 1) * kK * kK;
  for (int pc = tid; pc < n_pairs; pc += kThreads) {
    int i, p, c;
    if (pc < kK) {
      i = 0;
      p = 0;
      c = pc;
    } else {
      const int e = pc - kK;
      i = 1 + e / (kK * kK);
      p = (e / kK) % kK;
      c = e % kK;
    }
    const int ra = i == 0 ? 0 : 1 + (i - 1) * kK + p;
    const int rb = kRowsA + i * kK + c;
    const float s = edge_dot(sm, a.fmt, i, ra, rb) + sm.cl[i][c];
    if (!isfinite(s)) atomicOr(&sm.bad, 1);
    if (i == 0) {
      for (int pp = 0; pp < kK; ++pp) sm.lat[0][pp][c] = s;
    } else {
      sm.lat[i][p][c] = s;
    }
  }
  __syncthreads();
  if (a.scores_out) {
    for (int e = tid; e < kP * kK * kK; e += kThreads)
      a.scores_out[static_cast<size_t>(r) * kP * kK * kK + e] = (&sm.lat[0][0][0])[e];
  }
  const int bad = sm.bad;
  auto& lat = sm.lat;
  auto& cids = sm.cids;
  if (wid != 0) return;
  // ---- the walk: one warp, lane j < 16 holds candidate j
  const float T = a.temperature[r];
  int32_t* path = a.path + static_cast<size_t>(r) * kP;
  float* qrow = a.q_rows + static_cast<size_t>(r) * kP * kK;
  if (!(T >= 0.f) || bad) {
    if (lane < kP) path[lane] = -1;
    for (int e = lane; e < kP * kK; e += 32) qrow[e] = 0.f;
    if (lane == 0) a.status[r] = (T >= 0.f) ? 2 : 1;
    return;
  }
  const uint64_t seed = a.seed[r], off = a.offset[r];
  const bool live = lane < kK;
  int prev = 0;
  for (int i = 0; i < kP; ++i) {
    const float sj = live ? lat[i][prev][lane] : -INFINITY;
    const int cid = live ? cids[i][lane] : 0x7FFFFFFF;
    int pick;
    float q;
    if (T == 0.f) {
      // argmax, equal scores -> smaller candidate id
      float bv = sj;
      int bi = lane, bc = cid;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o), oc = __shfl_xor_sync(0xffffffffu, bc, o);
        if (ov > bv || (ov == bv && oc < bc)) {
          bv = ov;
          bi = oi;
          bc = oc;
        }
      }
      pick = bi;
      q = (lane == pick) ? 1.f : 0.f;
    } else {
      const float m = warp_max(sj);
      const float e = live ? expf((sj - m) / T) : 0.f;
      const float tot = warp_sum(e);
      float cum = e;  // inclusive prefix sum over lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, cum, o);
        if (lane >= o) cum += t;
      }
      const float u = philox_uniform(seed, off, static_cast<uint32_t>(i), kPurposeWalk);
      const unsigned over = __ballot_sync(0xffffffffu, live && cum > u * tot);
      const unsigned pos = __ballot_sync(0xffffffffu, live && e > 0.f);
      pick = over ? __ffs(over) - 1 : (pos ? 31 - __clz(pos) : 0);
      q = e / tot;
    }
    if (live) qrow[i * kK + lane] = q;
    if (lane == 0) path[i] = cids[i][pick];
    prev = pick;
  }
  if (lane == 0) a.status[r] = 0;
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a, int n_req, bool pdl, cudaStream_t st) {
  static bool attr_set = false;  // set once, outside any later stream capture
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sizeof(SelSmem)));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(select_kernel, dim3(n_req), dim3(kThreads), sizeof(SelSmem), st, pdl, a);
}

}  // namespace df2
