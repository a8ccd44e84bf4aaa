// Selector walk (step a10): the low-rank bigram selector of the vLLM PR #52816
// description ("Candidate selector"): score(p -> c) = <A[p] * gate_i, B[c]> +
// unary_i[c], with A, B the rank-256 codebooks, gate_i the projection of position
// i's hidden state and unary the candidate's drafter logit; the walk starts at the
// verified anchor, takes the argmax at T = 0 and an inverse-CDF draw from
// softmax(score / T) at T > 0, and returns q over the 16 candidates.
//
// One CTA per (request, position): it stages the 16 predecessor rows of A (the
// anchor's row at position 1) and the 16 candidate rows of B in shared memory and
// scores its 16 x 16 edges, one thread per (predecessor, candidate), into a scratch
// lattice.  The CTA that completes a request's B - 1 positions (fenced atomic
// ticket, no waiting) walks the lattice with one warp (lane j = candidate j): all
// B - 1 positions, or the first width - 1 for a request narrowed to a block width
// below B (the positions past it get no proposal).  Any
// nonfinite candidate logit or score marks the request DFLASH2_E_NONFINITE ("LSE
// docs/DFLASH2.md": the selector rejects nonfinite scores).
#include <math.h>

#include "common.cuh"
#include "glue.h"
#include "internal.h"
#include "philox.cuh"

namespace df2 {

namespace {

constexpr int kMaxP = kMaxBlock - 1, kK = 16, kRank = 256;

// Codebook rows staged in shared memory in their stored format: bf16 (256 x 2 B) or
// Q8 codes (256 B) plus 4 groups of (scale, bias).  Rows 0..15: predecessors (A),
// 16..31: candidates (B).
constexpr int kPadBf = kRank + 8;   // bf16 row stride: consecutive rows start 16 B apart mod 128 B
constexpr int kPadQ8 = kRank + 16;  // int8 row stride, same idea

struct SelSmem {
  uint16_t bf[2 * kK][kPadBf];  // BF16 rows (unused for Q8)
  int8_t q8[2 * kK][kPadQ8];    // Q8 codes (unused for BF16)
  uint16_t sb[2 * kK][8];       // Q8: scale[4], bias[4]
  float gate[kRank];
  float cl[kK];
  int cids[kMaxP][kK];
  float lat[kMaxP][kK][kK];     // the walker's copy of the lattice
  uint8_t back[kMaxP][kK];      // Viterbi: best predecessor of each candidate
  // draft tree: node 0 is the root (the anchor), nodes 1..n the tree's
  float t_score[kTreeMaxNodes + 1];
  int t_cand[kTreeMaxNodes + 1], t_depth[kTreeMaxNodes + 1];
  uint32_t t_taken[kTreeMaxNodes + 1];  // children already in the tree (bit c)
  int bad;
  int last;
};

constexpr int kThreads = kK * kK;  // one thread per (predecessor, candidate)

DF2_DEV float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
DF2_DEV float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Edge score of predecessor row ra and candidate row rb (without the unary term).
DF2_DEV float edge_dot(const SelSmem& sm, int fmt, int ra, int rb) {
  const float* g = sm.gate;
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

// Draft tree of one request ("qwen35: DSpark speculative decoding ... #625", DDTree
// commit: each expansion scores the candidates as the draft log-prob plus the
// selector compatibility with the branch's actual parent, log-softmax-normalised per
// position, so best-first comparisons across depths are on a log-prob scale).  The
// lattice holds unary logit + compatibility; the vocabulary normaliser of the draft
// log-prob is a per-position constant and cancels in the per-parent log-softmax.
// One warp: each lattice row (position, parent candidate) is turned into log q in
// place, then the tree grows best-first: every step adds the highest-scoring child,
// over the root and every node already in, that is not in yet (equal scores: the
// earlier parent, then the smaller candidate index), until the budget is reached.
// FP32 throughout; node k of the output is tree node k + 1 (parent -1 = the root).
__device__ void tree_grow(const SelectArgs& a, SelSmem& sm, int r, int np) {
  const int lane = threadIdx.x & 31;
  for (int row = lane; row < np * kK; row += 32) {
    float* v = sm.lat[row / kK][row % kK];
    float m = v[0];
#pragma unroll
    for (int c = 1; c < kK; ++c) m = fmaxf(m, v[c]);
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kK; ++c) s += expf(v[c] - m);
    const float lse = m + logf(s);
#pragma unroll
    for (int c = 0; c < kK; ++c) v[c] -= lse;
  }
  if (lane == 0) {
    sm.t_score[0] = 0.f;
    sm.t_cand[0] = 0;  // position 1's rows all come from the anchor: row 0
    sm.t_depth[0] = 0;
    sm.t_taken[0] = 0u;
  }
  __syncwarp();
  const size_t o = static_cast<size_t>(r) * a.tree_budget;
  int n = 0;
  while (n < a.tree_budget) {
    // this lane's best option over parents lane, lane + 32 (node indices 0..n)
    float bv = -INFINITY;
    int bq = 0x7FFFFFFF, bc = 0x7FFFFFFF;
    for (int q = lane; q <= n; q += 32) {
      const int d = sm.t_depth[q];
      if (d >= np) continue;
      const float base = sm.t_score[q];
      const float* row = sm.lat[d][sm.t_cand[q]];
      const uint32_t taken = sm.t_taken[q];
      for (int c = 0; c < kK; ++c) {
        if (taken & (1u << c)) continue;
        const float v = base + row[c];
        if (v > bv || (v == bv && (q < bq || (q == bq && c < bc)))) {
          bv = v;
          bq = q;
          bc = c;
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oq = __shfl_xor_sync(0xffffffffu, bq, off), oc = __shfl_xor_sync(0xffffffffu, bc, off);
      if (ov > bv || (ov == bv && (oq < bq || (oq == bq && oc < bc)))) {
        bv = ov;
        bq = oq;
        bc = oc;
      }
    }
    if (bq == 0x7FFFFFFF) break;  // every node is at the last position and every child is in
    ++n;
    if (lane == 0) {
      const int d = sm.t_depth[bq] + 1;
      sm.t_score[n] = bv;
      sm.t_cand[n] = bc;
      sm.t_depth[n] = d;
      sm.t_taken[n] = 0u;
      sm.t_taken[bq] |= 1u << bc;
      a.t_token[o + n - 1] = sm.cids[d - 1][bc];
      a.t_parent[o + n - 1] = bq - 1;
      a.t_depth[o + n - 1] = d;
      a.t_score[o + n - 1] = bv;
    }
    __syncwarp();
  }
  if (lane == 0) {
    a.t_n[r] = n;
    a.status[r] = 0;
  }
}

__global__ void __launch_bounds__(kThreads) select_kernel(const SelectArgs a) {
  __shared__ __align__(16) SelSmem sm;
  pdl_begin();
  const int r = blockIdx.x, i = blockIdx.y;
  const int P = a.B - 1;  // positions of a request's rows of candidates, gate, lattice and path
  // positions walked: 1..width-1 (the request's block width; every position is scored)
  const int np = a.width != nullptr ? min(max(a.width[r], 2), a.B) - 1 : P;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) sm.bad = 0;
  // candidates of this position (and of the previous one: the predecessors)
  if (tid < 2 * kK) {
    const int pos = tid < kK ? i : i - 1;
    if (pos >= 0) {
      const int e = pos * kK + (tid % kK);
      sm.cids[pos][tid % kK] = min(max(a.cand_ids[static_cast<size_t>(r) * P * kK + e], 0), a.V - 1);
    }
  }
  if (tid < kK) {
    const float v = a.cand_logits[(static_cast<size_t>(r) * P + i) * kK + tid];
    sm.cl[tid] = v;
    if (!isfinite(v)) atomicOr(&sm.bad, 1);
  }
  sm.gate[tid] = a.gate[(static_cast<size_t>(r) * P + i) * kRank + tid];
  __syncthreads();
  const int anchor = min(max(a.anchor_ids[r], 0), a.V - 1);
  const int n_pred = i == 0 ? 1 : kK;
  // stage the rows (every thread's pieces loaded before any is stored): row k < 16
  // the predecessor A[id], k >= 16 the candidate B[id]
  const int chunks = a.fmt == 0 ? kRank * 2 / 16 : kRank / 16;  // 16-byte pieces per row
  constexpr int kPer = (2 * kK * kRank * 2 / 16 + kThreads - 1) / kThreads;
  uint4 piece[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int e = tid + kThreads * j;
    const int k = e / chunks, c = e % chunks;
    piece[j] = make_uint4(0, 0, 0, 0);
    if (k < 2 * kK && (k >= kK || k < n_pred)) {
      const int id = k < kK ? (i == 0 ? anchor : sm.cids[i - 1][k]) : sm.cids[i][k - kK];
      const void* cb = k < kK ? a.cb_a : a.cb_b;
      piece[j] = a.fmt == 0 ? ld_cached(reinterpret_cast<const uint16_t*>(cb) + static_cast<size_t>(id) * kRank + c * 8)
                            : ld_cached(reinterpret_cast<const int8_t*>(cb) + static_cast<size_t>(id) * kRank + c * 16);
    }
  }
  if (a.fmt != 0 && tid < 2 * kK * 4) {  // Q8: 4 groups of (scale, bias) per row
    const int k = tid >> 2, c = tid & 3;
    if (k >= kK || k < n_pred) {
      const int id = k < kK ? (i == 0 ? anchor : sm.cids[i - 1][k]) : sm.cids[i][k - kK];
      const uint16_t* sc = k < kK ? a.cb_a_scale : a.cb_b_scale;
      const uint16_t* bi = k < kK ? a.cb_a_bias : a.cb_b_bias;
      sm.sb[k][c] = sc[static_cast<size_t>(id) * 4 + c];
      sm.sb[k][4 + c] = bi[static_cast<size_t>(id) * 4 + c];
    }
  }
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int e = tid + kThreads * j;
    const int k = e / chunks, c = e % chunks;
    if (k < 2 * kK && (k >= kK || k < n_pred)) {
      if (a.fmt == 0)
        *reinterpret_cast<uint4*>(&sm.bf[k][c * 8]) = piece[j];
      else
        *reinterpret_cast<uint4*>(&sm.q8[k][c * 16]) = piece[j];
    }
  }
  __syncthreads();
  // edge (p, c): position 1 has the anchor as its only predecessor (the same row for every p)
  {
    const int p = tid / kK, c = tid % kK;
    const float s = edge_dot(sm, a.fmt, i == 0 ? 0 : p, kK + c) + sm.cl[c];
    if (!isfinite(s)) atomicOr(&sm.bad, 1);
    a.lat[((static_cast<size_t>(r) * P + i) * kK + p) * kK + c] = s;
  }
  __threadfence();  // every writer's lattice scores visible device-wide before the ticket
  __syncthreads();
  // the CTA completing this request's seven positions walks the lattice
  if (tid == 0) {
    a.bad[r * P + i] = sm.bad;
    __threadfence();
    const unsigned int done = atomicAdd(&a.counters[r], 1u);
    sm.last = done == P - 1;
    if (sm.last) {
      a.counters[r] = 0;  // zero for the next launch
      __threadfence();
    }
  }
  __syncthreads();
  if (!sm.last) return;
  int bad_any = 0;
  for (int e = tid; e < P * kK * kK; e += kThreads) {
    const float v = __ldcg(a.lat + static_cast<size_t>(r) * P * kK * kK + e);
    (&sm.lat[0][0][0])[e] = v;
    if (a.scores_out) a.scores_out[static_cast<size_t>(r) * P * kK * kK + e] = v;
  }
  if (tid < P * kK) sm.cids[tid / kK][tid % kK] =
      min(max(a.cand_ids[static_cast<size_t>(r) * P * kK + tid], 0), a.V - 1);
  if (tid < np) bad_any = __ldcg(a.bad + r * P + tid);
  bad_any = __syncthreads_or(bad_any);
  const int bad = bad_any;
  auto& lat = sm.lat;
  auto& cids = sm.cids;
  if (wid != 0) return;
  // ---- the walk: one warp, lane j < 16 holds candidate j
  const float T = a.tree_budget > 0 ? 0.f : a.temperature[r];  // the tree is built for greedy verification
  int32_t* path = a.tree_budget > 0 ? nullptr : a.path + static_cast<size_t>(r) * P;
  float* qrow = a.tree_budget > 0 ? nullptr : a.q_rows + static_cast<size_t>(r) * P * kK;
  // a weight-pipeline wait of this step's draft that gave up leaves its candidates undefined
  const bool pipe_bad = a.pipe_err != nullptr && __ldcg(a.pipe_err) != 0;
  if (!(T >= 0.f) || bad || pipe_bad) {
    if (a.tree_budget > 0) {
      if (lane == 0) a.t_n[r] = 0;
    } else {
      if (lane < P) path[lane] = -1;
      for (int e = lane; e < P * kK; e += 32) qrow[e] = 0.f;
    }
    if (lane == 0) a.status[r] = pipe_bad ? 3 : (T >= 0.f) ? 2 : 1;
    return;
  }
  const bool live = lane < kK;
  if (a.tree_budget > 0) {
    tree_grow(a, sm, r, np);
    return;
  }
  // positions past the width: no proposal
  if (lane >= np && lane < P) path[lane] = -1;
  for (int e = np * kK + lane; e < P * kK; e += 32) qrow[e] = 0.f;
  if (T == 0.f && a.mode == 1) {
    // globally best path: best_1(c) = s_1(c); best_i(c) = max_p best_{i-1}(p) + s_i(p, c)
    // (float32 sums; equal -> the predecessor with the smaller id), then read back
    float best = live ? lat[0][0][lane] : -INFINITY;
    for (int i = 1; i < np; ++i) {
      float nb = -INFINITY;
      int bp = 0, bid = 0x7FFFFFFF;
      for (int p = 0; p < kK; ++p) {
        const float bpv = __shfl_sync(0xffffffffu, best, p);
        if (live) {
          const float v = bpv + lat[i][p][lane];
          const int pid = cids[i - 1][p];
          if (v > nb || (v == nb && pid < bid)) {
            nb = v;
            bp = p;
            bid = pid;
          }
        }
      }
      if (live) sm.back[i][lane] = static_cast<uint8_t>(bp);
      best = live ? nb : -INFINITY;
    }
    // the end of the path: argmax over candidates, equal -> smaller id
    float bv = best;
    int bi = lane, bc = live ? cids[np - 1][lane] : 0x7FFFFFFF;
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
    __syncwarp();
    int c = bi;
    for (int i = np - 1; i >= 0; --i) {  // read back through the recorded predecessors
      if (live) qrow[i * kK + lane] = lane == c ? 1.f : 0.f;
      if (lane == 0) path[i] = cids[i][c];
      c = i > 0 ? sm.back[i][c] : 0;
    }
    if (lane == 0) a.status[r] = 0;
    return;
  }
  const uint64_t seed = a.seed[r], off = a.offset[r];
  int prev = 0;
  for (int i = 0; i < np; ++i) {
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
  if (a.rank != kRank || (a.B != 8 && a.B != 16)) return cudaErrorInvalidValue;
  return launch_ex(select_kernel, dim3(n_req, a.B - 1), dim3(kThreads), 0, st, pdl, a);
}

}  // namespace df2
