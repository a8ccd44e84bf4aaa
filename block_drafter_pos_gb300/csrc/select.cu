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
#include "philox.cuh"

namespace df2 {

namespace {

constexpr int kP = 7, kK = 16, kRank = 256;

// Loads one codebook row (bf16 or Q8/g64) as fp32 into dst[kRank].
__device__ void load_cb_row(float* dst, const void* cb, const uint16_t* sc, const uint16_t* bi, int fmt, int id,
                            int lane) {
  for (int r = lane; r < kRank; r += 32) {
    float v;
    if (fmt == 0) {
      v = bf16_to_f32(reinterpret_cast<const uint16_t*>(cb)[static_cast<size_t>(id) * kRank + r]);
    } else {
      const int8_t c = reinterpret_cast<const int8_t*>(cb)[static_cast<size_t>(id) * kRank + r];
      const int gi = static_cast<size_t>(id) * (kRank / 64) + r / 64;
      v = bf16_to_f32(sc[gi]) * static_cast<float>(c) + bf16_to_f32(bi[gi]);
    }
    dst[r] = v;
  }
}

__global__ void __launch_bounds__(256) select_kernel(const SelectArgs a) {
  __shared__ float apred[kK][kRank];   // predecessor rows of A (16 KB)
  __shared__ float bg[kK][kRank];      // gate_i * B[c] rows (16 KB)
  __shared__ float lat[kP][kK][kK];    // scores [position][pred][cand]
  __shared__ int cids[kP][kK];
  __shared__ float cl[kP][kK];
  __shared__ int bad;
  const int r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) bad = 0;
  for (int e = tid; e < kP * kK; e += 256) {
    cids[e / kK][e % kK] = min(max(a.cand_ids[static_cast<size_t>(r) * kP * kK + e], 0), a.V - 1);
    const float v = a.cand_logits[static_cast<size_t>(r) * kP * kK + e];
    cl[e / kK][e % kK] = v;
    if (!isfinite(v)) atomicOr(&bad, 1);
  }
  __syncthreads();
  const int anchor = min(max(a.anchor_ids[r], 0), a.V - 1);
  for (int i = 0; i < kP; ++i) {
    // predecessor rows: the anchor for position 1, else the 16 candidates of position i-1
    for (int p = wid; p < kK; p += 8) {
      const int id = (i == 0) ? anchor : cids[i - 1][p];
      if (i == 0 && p > 0) continue;
      load_cb_row(apred[p], a.cb_a, a.cb_a_scale, a.cb_a_bias, a.fmt, id, lane);
    }
    const float* gi = a.gate + (static_cast<size_t>(r) * kP + i) * kRank;
    for (int c = wid; c < kK; c += 8) {
      load_cb_row(bg[c], a.cb_b, a.cb_b_scale, a.cb_b_bias, a.fmt, cids[i][c], lane);
      __syncwarp();
      for (int k = lane; k < kRank; k += 32) bg[c][k] *= gi[k];
    }
    __syncthreads();
    const int npred = (i == 0) ? 1 : kK;
    for (int pc = wid; pc < npred * kK; pc += 8) {
      const int p = pc / kK, c = pc % kK;
      float s = 0.f;
#pragma unroll
      for (int k = 0; k < kRank / 32; ++k) s = fmaf(apred[p][lane + 32 * k], bg[c][lane + 32 * k], s);
      s = warp_sum(s) + cl[i][c];
      if (lane == 0) {
        if (!isfinite(s)) atomicOr(&bad, 1);
        if (i == 0) {
          for (int pp = 0; pp < kK; ++pp) lat[0][pp][c] = s;
        } else {
          lat[i][p][c] = s;
        }
      }
    }
    __syncthreads();
  }
  if (a.scores_out) {
    for (int e = tid; e < kP * kK * kK; e += 256) a.scores_out[static_cast<size_t>(r) * kP * kK * kK + e] = (&lat[0][0][0])[e];
  }
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

cudaError_t launch_select(const SelectArgs& a, int n_req, cudaStream_t st) {
  select_kernel<<<n_req, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace df2
