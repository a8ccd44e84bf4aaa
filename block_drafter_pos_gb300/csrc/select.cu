// Selector walk (step a10): the low-rank bigram selector of the vLLM PR #52816
// description ("Candidate selector"): score(p -> c) = <A[p] * gate_i, B[c]> +
// unary_i[c], with A, B the rank-256 codebooks, gate_i the projection of position
// i's hidden state and unary the candidate's drafter logit; the walk starts at the
// verified anchor, takes the argmax at T = 0 and an inverse-CDF draw from
// softmax(score / T) at T > 0, and returns q over the 16 candidates.
//
// One CTA per request.  The full 7 x 16 x 16 lattice is scored first (position 1
// from the anchor), then one thread walks it.  Any nonfinite candidate logit or
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
struct SelSmem {
  uint16_t bf[kRows][kRank];   // BF16 rows (unused for Q8)
  int8_t q8[kRows][kRank];     // Q8 codes (unused for BF16)
  uint16_t sb[kRows][8];       // Q8: scale[4], bias[4]
  float gate[kP][kRank];
  float lat[kP][kK][kK];       // scores [position][pred][cand]
  int cids[kP][kK];
  float cl[kP][kK];
  int bad;
};

// Row `row` of the staged codebook rows, element r, as fp32.
DF2_DEV float cb_val(const SelSmem& sm, int fmt, int row, int r) {
  if (fmt == 0) return bf16_to_f32(sm.bf[row][r]);
  const int g = r >> 6;
  return bf16_to_f32(sm.sb[row][g]) * static_cast<float>(sm.q8[row][r]) + bf16_to_f32(sm.sb[row][4 + g]);
}

__global__ void __launch_bounds__(256) select_kernel(const SelectArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  pdl_begin();
  const int r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) sm.bad = 0;
  for (int e = tid; e < kP * kK; e += 256) {
    sm.cids[e / kK][e % kK] = min(max(a.cand_ids[static_cast<size_t>(r) * kP * kK + e], 0), a.V - 1);
    const float v = a.cand_logits[static_cast<size_t>(r) * kP * kK + e];
    sm.cl[e / kK][e % kK] = v;
    if (!isfinite(v)) atomicOr(&sm.bad, 1);
  }
  for (int e = tid; e < kP * kRank; e += 256) sm.gate[e / kRank][e % kRank] = a.gate[static_cast<size_t>(r) * kP * kRank + e];
  __syncthreads();
  const int anchor = min(max(a.anchor_ids[r], 0), a.V - 1);
  // stage every needed codebook row at once (one round trip): row k < kRowsA is the
  // predecessor row A[id], k >= kRowsA the successor row B[id]
  const int chunks = a.fmt == 0 ? kRank * 2 / 16 : kRank / 16;  // 16-byte pieces per row
  for (int e = tid; e < kRows * chunks; e += 256) {
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
    if (a.fmt == 0) {
      *reinterpret_cast<uint4*>(&sm.bf[k][c * 8]) =
          ld_cached(reinterpret_cast<const uint16_t*>(cb) + static_cast<size_t>(id) * kRank + c * 8);
    } else {
      *reinterpret_cast<uint4*>(&sm.q8[k][c * 16]) =
          ld_cached(reinterpret_cast<const int8_t*>(cb) + static_cast<size_t>(id) * kRank + c * 16);
      if (c < 4) {
        const uint16_t* sc = k < kRowsA ? a.cb_a_scale : a.cb_b_scale;
        const uint16_t* bi = k < kRowsA ? a.cb_a_bias : a.cb_b_bias;
        sm.sb[k][c] = sc[static_cast<size_t>(id) * 4 + c];
        sm.sb[k][4 + c] = bi[static_cast<size_t>(id) * 4 + c];
      }
    }
  }
  __syncthreads();
  // lattice: one warp per (position, pred, cand); lanes split the rank (fixed tree)
  const int n_pairs = kK + (kP - 1) * kK * kK;
  for (int pc = wid; pc < n_pairs; pc += 8) {
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
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kRank / 32; ++k) {
      const int rr = lane + 32 * k;
      s = fmaf(cb_val(sm, a.fmt, ra, rr), sm.gate[i][rr] * cb_val(sm, a.fmt, rb, rr), s);
    }
    s = warp_sum(s) + sm.cl[i][c];
    if (lane == 0) {
      if (!isfinite(s)) atomicOr(&sm.bad, 1);
      if (i == 0) {
        for (int pp = 0; pp < kK; ++pp) sm.lat[0][pp][c] = s;
      } else {
        sm.lat[i][p][c] = s;
      }
    }
  }
  __syncthreads();
  if (a.scores_out) {
    for (int e = tid; e < kP * kK * kK; e += 256)
      a.scores_out[static_cast<size_t>(r) * kP * kK * kK + e] = (&sm.lat[0][0][0])[e];
  }
  const int bad = sm.bad;
  auto& lat = sm.lat;
  auto& cids = sm.cids;
  if (tid != 0) return;
  const float T = a.temperature[r];
  int32_t* path = a.path + static_cast<size_t>(r) * kP;
  float* qrow = a.q_rows + static_cast<size_t>(r) * kP * kK;
  if (!(T >= 0.f) || bad) {
    for (int i = 0; i < kP; ++i) {
      path[i] = -1;
      for (int j = 0; j < kK; ++j) qrow[i * kK + j] = 0.f;
    }
    a.status[r] = (T >= 0.f) ? 2 : 1;
    return;
  }
  const uint64_t seed = a.seed[r], off = a.offset[r];
  int prev = 0;
  for (int i = 0; i < kP; ++i) {
    const float* s = lat[i][prev];
    int pick = 0;
    if (T == 0.f) {
      for (int j = 1; j < kK; ++j)
        if (s[j] > s[pick] || (s[j] == s[pick] && cids[i][j] < cids[i][pick])) pick = j;
      for (int j = 0; j < kK; ++j) qrow[i * kK + j] = (j == pick) ? 1.f : 0.f;
    } else {
      float m = s[0];
      for (int j = 1; j < kK; ++j) m = fmaxf(m, s[j]);
      float e[kK];
      float tot = 0.f;
      for (int j = 0; j < kK; ++j) {
        e[j] = expf((s[j] - m) / T);
        tot += e[j];
      }
      const float u = philox_uniform(seed, off, static_cast<uint32_t>(i), kPurposeWalk);
      const float target = u * tot;
      float cum = 0.f;
      pick = -1;
      int last_pos = 0;
      for (int j = 0; j < kK; ++j) {
        cum += e[j];
        if (e[j] > 0.f) last_pos = j;
        if (pick < 0 && cum > target) pick = j;
      }
      if (pick < 0) pick = last_pos;
      for (int j = 0; j < kK; ++j) qrow[i * kK + j] = e[j] / tot;
    }
    path[i] = cids[i][pick];
    prev = pick;
  }
  a.status[r] = 0;
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
  return launch_ex(select_kernel, dim3(n_req), dim3(256), sizeof(SelSmem), st, pdl, a);
}

}  // namespace df2
