// Verification of the B - 1 proposals of a block of B positions (step a11): exact
// match against the target argmax for greedy requests; probability-ratio rejection
// with residual sampling for T > 0 ("LSE docs/DFLASH2.md", first paragraph: the
// target verifies all seven proposals of a block of 8 with probability-ratio
// rejection and residual sampling, greedy requests stay deterministic).  A request
// narrowed to width w < B verifies its first w - 1 proposals with rows 0..w-1
// (the long-context narrowing of "qwen35: DSpark speculative decoding ... #625").
//
// Pass 1 (grid vocab chunks x R x B rows, chunks fastest): per chunk max, argmax (smallest index on
// ties), sum of exp((z - m) / T), NaN / +inf flags; rows at or past a request's width
// are skipped but counted.  Pass 2 (one CTA per request):
// folds the chunk statistics in a fixed order and runs the sequential accept chain;
// a residual or bonus draw locates its vocabulary chunk from per-chunk masses and
// scans that one chunk with a block-wide prefix sum.
#include <math.h>

#include "common.cuh"
#include "glue.h"
#include "internal.h"
#include "philox.cuh"

namespace df2 {

namespace {

constexpr int kK = 16;

// Block width of request r: 2..B, B when no widths are given.
DF2_DEV int width_of(const int32_t* width, int r, int B) { return width != nullptr ? min(max(width[r], 2), B) : B; }

// One count on a request's device-wide counter, ordered after this thread's earlier
// writes (release) and before its later reads (acquire); returns the previous value.
DF2_DEV unsigned int count_acq_rel(unsigned int* counter) {
  unsigned int prev;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(counter) : "memory");
  return prev;
}

// Chunk statistics written by other CTAs of the launch, read from L2.
DF2_DEV VerifyStat ldst(const VerifyStat* p) {
  VerifyStat v;
  v.m = __ldcg(&p->m);
  v.s = __ldcg(&p->s);
  v.s_lo = __ldcg(&p->s_lo);
  v.arg = __ldcg(&p->arg);
  v.flags = __ldcg(&p->flags);
  return v;
}

// a + b = s + e exactly (Knuth's TwoSum; six float operations, no reassociation).
DF2_DEV void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bp = s - a;
  e = (a - (s - bp)) + (b - bp);
}

// Inverse-CDF draw over the vocabulary of row j from weights w(x) = p(x) - min(p(x),
// q(x)) (residual, use_q) or p(x) (bonus / zero residual).  Runs on the whole CTA.
// A draw lands within eps of an entry boundary with probability about 2 eps V, so
// at V = 248,320 the position of u * total among the cumulative masses must be far
// finer than FP32 gives (an FP32 fold of 61 chunk masses alone errs by ~1e-7): the
// chunk masses (compensated chunk sums, FP64 rescale), their fold, u * total and the
// in-chunk prefix sums are FP64; the per-entry weights stay the FP32 values of p
// that the accept test uses.
// *mass_out (thread 0) receives the drawn-from weights' total before any fallback:
// the residual mass sum_x max(0, p(x) - q(x)) when use_q, else the p-mass.
__device__ int draw_row(const VerifyArgs& a, const float* z, const VerifyStat* st, float M, float tot, float T,
                        const int* cid, const float* qv, bool use_q, float u, double* csum, double* red,
                        float* mass_out) {
  // chunk masses (fixed order): p-mass of chunk c = s_c * exp((m_c - M)/T) / tot,
  // minus the candidates' min(p, q) in that chunk when drawing from the residual.
  const int nc = a.n_chunks;
  const float inv_t = 1.f / T;
  const double dT = static_cast<double>(T), dtot = static_cast<double>(tot);
  auto p_mass = [&](const VerifyStat& sc) {
    return (sc.m > -INFINITY) ? (static_cast<double>(sc.s) + static_cast<double>(sc.s_lo)) *
                                    exp((static_cast<double>(sc.m) - static_cast<double>(M)) / dT) / dtot
                              : 0.0;
  };
  for (int c = threadIdx.x; c < nc; c += blockDim.x) {
    double mass = p_mass(ldst(st + c));
    if (use_q) {
      for (int k = 0; k < kK; ++k) {
        if (cid[k] / kVerifyChunk == c) {
          const float p = expf((z[cid[k]] - M) * inv_t) / tot;
          mass -= static_cast<double>(fminf(p, qv[k]));
        }
      }
      mass = fmax(mass, 0.0);
    }
    csum[c] = mass;
  }
  __syncthreads();
  __shared__ int sh_chunk, sh_fallback;
  __shared__ double sh_need;
  if (threadIdx.x == 0) {
    double total = 0.0;
    for (int c = 0; c < nc; ++c) total += csum[c];
    *mass_out = static_cast<float>(total);
    const bool fallback = use_q && !(total > 1e-30);
    if (fallback) {
      total = 0.0;
      for (int c = 0; c < nc; ++c) {
        csum[c] = p_mass(ldst(st + c));
        total += csum[c];
      }
    }
    const double target = static_cast<double>(u) * total;
    double acc = 0.0;
    int pick = -1, lastpos = 0;
    for (int c = 0; c < nc; ++c) {
      if (csum[c] > 0.0) lastpos = c;
      if (pick < 0 && acc + csum[c] > target) pick = c;
      if (pick < 0) acc += csum[c];
    }
    sh_need = target - acc;  // remaining mass to cover inside the chunk
    if (pick < 0) {
      pick = lastpos;             // rounding left u * total past the end:
      sh_need = INFINITY;         // take the last positive entry of the last chunk
    }
    sh_chunk = pick;
    sh_fallback = fallback;
  }
  __syncthreads();
  const int c = sh_chunk;
  const bool q_on = use_q && !sh_fallback;
  const double need = sh_need;
  const int v0 = c * kVerifyChunk;
  const int v1 = min(a.V, v0 + kVerifyChunk);
  // block-wide scan in id order: each thread owns a contiguous run of 16 ids
  const int per = kVerifyChunk / 256;
  const int b0 = v0 + threadIdx.x * per;
  float wv[kVerifyChunk / 256];
  double run = 0.0;
  for (int t = 0; t < per; ++t) {
    const int v = b0 + t;
    float w = 0.f;
    if (v < v1) {
      const float x = z[v];
      w = isnan(x) ? 0.f : expf((x - M) * inv_t) / tot;
      if (q_on) {
        for (int k = 0; k < kK; ++k)
          if (cid[k] == v) w = fmaxf(0.f, w - qv[k]);
      }
    }
    wv[t] = w;
    run += static_cast<double>(w);
  }
  // exclusive prefix of the per-thread runs
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  double incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) red[wid] = incl;
  __syncthreads();
  double wbase = 0.0;
  for (int w = 0; w < wid; ++w) wbase += red[w];
  double acc = wbase + incl - run;
  __shared__ int sh_pick, sh_last;
  if (threadIdx.x == 0) {
    sh_pick = 0x7FFFFFFF;
    sh_last = -1;
  }
  __syncthreads();
  int found = 0x7FFFFFFF, lastpos = -1;
  for (int t = 0; t < per; ++t) {
    if (wv[t] > 0.f) lastpos = b0 + t;
    acc += static_cast<double>(wv[t]);
    if (found == 0x7FFFFFFF && acc > need && wv[t] > 0.f) found = b0 + t;
  }
  if (found != 0x7FFFFFFF) atomicMin(&sh_pick, found);
  if (lastpos >= 0) atomicMax(&sh_last, lastpos);
  __syncthreads();
  int x = sh_pick != 0x7FFFFFFF ? sh_pick : sh_last;
  if (x < 0) x = ldst(st + c).arg;
  __syncthreads();
  return x;
}

// The accept / emit chain of request r (run by the statistics CTA that completes
// the request's set).
__device__ void chain_body(const VerifyArgs& a, int r) {
  extern __shared__ double csum[];  // [n_chunks]
  __shared__ double red[8];
  __shared__ float rowM[kMaxBlock], rowS[kMaxBlock];
  __shared__ int rowA[kMaxBlock], rowF[kMaxBlock], rowBad;
  __shared__ int cid[kK];
  __shared__ float qv[kK];
  const int B = a.B, P = B - 1;  // block positions, proposal slots of a row of path / q
  const int w = width_of(a.width, r, B), np = w - 1;  // rows verified, proposals tested (bonus row np)
  int32_t* emitted = a.emitted + static_cast<size_t>(r) * B;
  // debug output: NaN wherever this request gets no probability
  float* probs = a.probs != nullptr ? a.probs + static_cast<size_t>(r) * B * 2 : nullptr;
  if (probs != nullptr && threadIdx.x < 2 * B) probs[threadIdx.x] = __int_as_float(0x7FC00000);
  __shared__ float sh_mass;
  if (a.status[r] != 0) {
    if (threadIdx.x < B) emitted[threadIdx.x] = -1;
    if (threadIdx.x == 0) {
      a.n_accepted[r] = 0;
      a.n_emitted[r] = 0;
    }
    return;
  }
  const float T = a.temperature[r];
  const VerifyStat* st = a.stats + static_cast<size_t>(r) * B * a.n_chunks;
  // warp j folds the chunk statistics of rows j, j + 8 (lane-strided, fixed shuffle tree)
  for (int j = threadIdx.x >> 5; j < w; j += 8) {
    const int lane = threadIdx.x & 31;
    const VerifyStat* sj = st + static_cast<size_t>(j) * a.n_chunks;
    float M = -INFINITY;
    int A = 0x7FFFFFFF, F = 0;
    for (int c = lane; c < a.n_chunks; c += 32) {
      const VerifyStat sc = ldst(sj + c);
      F |= sc.flags;
      if (sc.m > M || (sc.m == M && sc.arg < A)) {
        M = sc.m;
        A = sc.arg;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, M, o);
      const int oa = __shfl_xor_sync(0xffffffffu, A, o);
      if (om > M || (om == M && oa < A)) {
        M = om;
        A = oa;
      }
      F |= __shfl_xor_sync(0xffffffffu, F, o);
    }
    float S = 0.f;
    if (T > 0.f && M > -INFINITY && M < INFINITY)
      for (int c = lane; c < a.n_chunks; c += 32)
        if (const VerifyStat sc = ldst(sj + c); sc.m > -INFINITY) S += (sc.s + sc.s_lo) * expf((sc.m - M) / T);
    S = warp_sum(S);
    if (lane == 0) {
      rowM[j] = M;
      rowS[j] = S;
      rowA[j] = A;
      rowF[j] = F != 0 || !(M > -INFINITY) || !(M < INFINITY);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int bad = 0;
    for (int j = 0; j < w; ++j) bad |= rowF[j];
    rowBad = bad;
  }
  __syncthreads();
  if (rowBad) {
    if (threadIdx.x < B) emitted[threadIdx.x] = -1;
    if (threadIdx.x == 0) {
      a.n_accepted[r] = 0;
      a.n_emitted[r] = 0;
      a.status[r] = 2;
    }
    return;
  }
  const int32_t* path = a.path + static_cast<size_t>(r) * P;
  if (!(T > 0.f)) {
    if (threadIdx.x == 0) {
      int n = 0;
      while (n < np && path[n] == rowA[n]) {
        emitted[n] = path[n];
        ++n;
      }
      emitted[n] = rowA[n];
      for (int j = n + 1; j < B; ++j) emitted[j] = -1;
      a.n_accepted[r] = n;
      a.n_emitted[r] = n + 1;
    }
    return;
  }
  const uint64_t seed = a.seed[r], off = a.offset[r];
  const float* zr = a.logits + static_cast<size_t>(r) * B * a.V;
  // The accept tests of the w - 1 rows depend only on the path, q and the target
  // row, not on each other: thread j < w - 1 takes row j (all loads of the rows in
  // flight together), then the chain stops at the first rejection.
  __shared__ int acc_row[kMaxBlock];
  __syncthreads();  // the NaN fill above is done before these entries are written
  if (threadIdx.x < np) {
    const int j = threadIdx.x;
    const int d = min(max(path[j], 0), a.V - 1);
    const int32_t* ci = a.cand_ids + (static_cast<size_t>(r) * P + j) * kK;
    const float* qj = a.q_rows + (static_cast<size_t>(r) * P + j) * kK;
    const float zd = zr[static_cast<size_t>(j) * a.V + d];
    float qd = 0.f;
    for (int k = 0; k < kK; ++k)
      if (min(max(ci[k], 0), a.V - 1) == d) qd = qj[k];
    const float pd = expf((zd - rowM[j]) / T) / rowS[j];
    const float u = philox_uniform(seed, off, static_cast<uint32_t>(j), kPurposeAccept);
    acc_row[j] = (qd > 0.f) ? (u * qd < pd) : 1;
    if (probs != nullptr) probs[2 * j] = pd;  // p_j at every row's proposal (the accept test's value)
  }
  __syncthreads();
  int n_acc = np;
  for (int j = 0; j < np; ++j)
    if (!acc_row[j]) {
      n_acc = j;
      break;
    }
  if (n_acc < np) {
    const int j = n_acc;
    if (threadIdx.x < kK) {
      cid[threadIdx.x] = min(max(a.cand_ids[(static_cast<size_t>(r) * P + j) * kK + threadIdx.x], 0), a.V - 1);
      qv[threadIdx.x] = a.q_rows[(static_cast<size_t>(r) * P + j) * kK + threadIdx.x];
    }
    __syncthreads();
    const float* z = zr + static_cast<size_t>(j) * a.V;
    const float u = philox_uniform(seed, off, static_cast<uint32_t>(j), kPurposeResample);
    const int x = draw_row(a, z, st + static_cast<size_t>(j) * a.n_chunks, rowM[j], rowS[j], T, cid, qv, true, u,
                           csum, red, &sh_mass);
    if (threadIdx.x == 0) {
      if (probs != nullptr) probs[2 * j + 1] = sh_mass;
      for (int t = 0; t < j; ++t) emitted[t] = path[t];
      emitted[j] = x;
      for (int t = j + 1; t < B; ++t) emitted[t] = -1;
      a.n_accepted[r] = j;
      a.n_emitted[r] = j + 1;
    }
    return;
  }
  const float u = philox_uniform(seed, off, static_cast<uint32_t>(np), kPurposeResample);
  const float* z = zr + static_cast<size_t>(np) * a.V;
  const int x = draw_row(a, z, st + static_cast<size_t>(np) * a.n_chunks, rowM[np], rowS[np], T, cid, qv, false, u,
                         csum, red, &sh_mass);
  if (threadIdx.x == 0) {
    if (probs != nullptr) probs[2 * np] = expf((z[x] - rowM[np]) / T) / rowS[np];
    for (int t = 0; t < np; ++t) emitted[t] = path[t];
    emitted[np] = x;
    for (int t = np + 1; t < B; ++t) emitted[t] = -1;
    a.n_accepted[r] = np;
    a.n_emitted[r] = np + 1;
  }
}

// Statistics of one (target row, vocabulary chunk): max, argmax, compensated sum of
// exp((z - max) / T), flags.
DF2_DEV void row_chunk_stats(const VerifyArgs& a, int rj, int r, int chunk) {
  __shared__ float sm_m[8], sm_s[8], sm_sl[8];
  __shared__ int sm_a[8], sm_f[8];
  const float T = a.temperature[r];
  const float* z = a.logits + static_cast<size_t>(rj) * a.V;
  const int v0 = chunk * kVerifyChunk;
  const int v1 = min(a.V, v0 + kVerifyChunk);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  constexpr int kPer = kVerifyChunk / 256;
  float xs[kPer];  // this thread's logits of the chunk, loaded once (all in flight)
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int v = v0 + threadIdx.x + 256 * j;
    xs[j] = v < v1 ? z[v] : -INFINITY;
  }
  float m = -INFINITY;
  int arg = 0x7FFFFFFF;
  int flags = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int v = v0 + threadIdx.x + 256 * j;
    const float x = xs[j];
    if (v >= v1) continue;
    if (isnan(x)) {
      flags |= 1;
      continue;
    }
    if (x == INFINITY) flags |= 2;
    if (x > m || (x == m && v < arg)) {
      m = x;
      arg = v;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const int oa = __shfl_xor_sync(0xffffffffu, arg, o);
    if (om > m || (om == m && oa < arg)) {
      m = om;
      arg = oa;
    }
    flags |= __shfl_xor_sync(0xffffffffu, flags, o);
  }
  if (lane == 0) {
    sm_m[wid] = m;
    sm_a[wid] = arg;
    sm_f[wid] = flags;
  }
  __syncthreads();
  float M = sm_m[0];
  int A = sm_a[0], F = 0;
  for (int w = 0; w < 8; ++w) {
    if (sm_m[w] > M || (sm_m[w] == M && sm_a[w] < A)) {
      M = sm_m[w];
      A = sm_a[w];
    }
    F |= sm_f[w];
  }
  // sum of exp((z - M) / T) over the chunk, compensated (sum + error term, both kept):
  // the draws of the chain need the chunk masses far finer than one FP32 rounding
  float s = 0.f, s_lo = 0.f;
  if (T > 0.f && M > -INFINITY && M < INFINITY) {
    const float inv_t = 1.f / T;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int v = v0 + threadIdx.x + 256 * j;
      if (v < v1 && !isnan(xs[j])) {
        float t, e;
        two_sum(s, expf((xs[j] - M) * inv_t), t, e);
        s = t;
        s_lo += e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float os = __shfl_xor_sync(0xffffffffu, s, o), ol = __shfl_xor_sync(0xffffffffu, s_lo, o);
      float t, e;
      two_sum(s, os, t, e);
      s = t;
      s_lo += ol + e;
    }
    __syncthreads();
    if (lane == 0) {
      sm_s[wid] = s;
      sm_sl[wid] = s_lo;
    }
    __syncthreads();
    s = sm_s[0];
    s_lo = sm_sl[0];
    for (int w = 1; w < 8; ++w) {
      float t, e;
      two_sum(s, sm_s[w], t, e);
      s = t;
      s_lo += sm_sl[w] + e;
    }
  }
  if (threadIdx.x == 0) {
    VerifyStat st;
    st.m = M;
    st.s = s;
    st.s_lo = s_lo;
    st.arg = A;
    st.flags = F;
    a.stats[static_cast<size_t>(rj) * a.n_chunks + chunk] = st;
  }
}

// The target logits and temperatures are caller inputs that the previous kernel may
// have written (the target model's), so the statistics wait for it.
__global__ void __launch_bounds__(256) verify_stats_kernel(const VerifyArgs a) {
  pdl_begin_early();
  // chunks vary fastest in launch order, so a request's set completes early and its
  // chain overlaps the statistics of the requests after it
  const int rj = blockIdx.y;  // r * B + j
  const int r = rj / a.B, j_row = rj % a.B;
  const int chunk = blockIdx.x;
  // rows at or past the request's width are not read, only counted
  if (j_row < width_of(a.width, r, a.B)) row_chunk_stats(a, rj, r, chunk);
  // count this chunk; the CTA that completes request r's B x n_chunks runs its chain.
  // Thread 0 wrote this chunk's statistics itself, so its count releases them (no fence
  // by every thread); the count also acquires the other chunks' statistics for the chain.
  __shared__ bool last;
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned int prev = count_acq_rel(a.counters + r);
    last = prev == static_cast<unsigned int>(a.B * a.n_chunks - 1);
    if (last) a.counters[r] = 0u;  // every CTA of the set has counted
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  chain_body(a, r);
}

// ------------------------------------------------------------------ draft tree, greedy
// Greedy verification of a draft tree ("qwen35: DSpark speculative decoding ...
// #625", DDTree commits: tree verification emits the text plain decoding emits).
// Pass 1: one CTA per (request, target row, 4096-id chunk): chunk max, argmax
// (smallest id on ties), NaN / +inf flags; rows past the request's tree are skipped
// but still counted.  The CTA completing a request's set folds each row's argmax and
// walks the tree from the root: move to the child carrying the current row's argmax
// while one exists; emit the path, then the last row's argmax.
__device__ void tree_chain(const TreeVerifyArgs& a, int r) {
  __shared__ int am[kTreeMaxNodes + 1], bad_row[kTreeMaxNodes + 1];
  const int n = min(max(a.n_nodes[r], 0), a.budget);
  const int kB = a.B;
  int32_t* emitted = a.emitted + static_cast<size_t>(r) * kB;
  if (a.status[r] != 0) {
    if (threadIdx.x < kB) emitted[threadIdx.x] = -1;
    if (threadIdx.x == 0) {
      a.n_accepted[r] = 0;
      a.n_emitted[r] = 0;
    }
    return;
  }
  // warp w folds rows w, w + 8, ... (lane-strided over chunks, fixed shuffle tree)
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int row = w; row <= n; row += 8) {
    const VerifyStat* sj = a.stats + (static_cast<size_t>(r) * (a.budget + 1) + row) * a.n_chunks;
    float M = -INFINITY;
    int A = 0x7FFFFFFF, F = 0;
    for (int c = lane; c < a.n_chunks; c += 32) {
      const VerifyStat sc = ldst(sj + c);
      F |= sc.flags;
      if (sc.m > M || (sc.m == M && sc.arg < A)) {
        M = sc.m;
        A = sc.arg;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, M, o);
      const int oa = __shfl_xor_sync(0xffffffffu, A, o);
      if (om > M || (om == M && oa < A)) {
        M = om;
        A = oa;
      }
      F |= __shfl_xor_sync(0xffffffffu, F, o);
    }
    if (lane == 0) {
      am[row] = A;
      bad_row[row] = F != 0 || !(M > -INFINITY) || !(M < INFINITY);
    }
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  int bad = 0;
  for (int row = 0; row <= n; ++row) bad |= bad_row[row];
  if (bad) {
    for (int j = 0; j < kB; ++j) emitted[j] = -1;
    a.n_accepted[r] = 0;
    a.n_emitted[r] = 0;
    a.status[r] = 2;
    return;
  }
  const int32_t* tok = a.token + static_cast<size_t>(r) * a.budget;
  const int32_t* par = a.parent + static_cast<size_t>(r) * a.budget;
  int cur = -1, acc = 0;
  while (acc < kB - 1) {
    const int t = am[cur + 1];
    int nxt = -1;
    for (int k = 0; k < n; ++k)
      if (par[k] == cur && tok[k] == t) {
        nxt = k;
        break;
      }
    if (nxt < 0) break;
    emitted[acc++] = t;
    cur = nxt;
  }
  emitted[acc] = am[cur + 1];
  for (int j = acc + 1; j < kB; ++j) emitted[j] = -1;
  a.n_accepted[r] = acc;
  a.n_emitted[r] = acc + 1;
}

__global__ void __launch_bounds__(256) tree_stats_kernel(const TreeVerifyArgs a) {
  __shared__ float sm_m[8];
  __shared__ int sm_a[8], sm_f[8];
  pdl_begin_early();
  const int r = blockIdx.y / (a.budget + 1), row = blockIdx.y % (a.budget + 1);
  const int chunk = blockIdx.x;
  const int n = min(max(a.n_nodes[r], 0), a.budget);
  if (row <= n) {
    const float* z = a.logits + (static_cast<size_t>(r) * (a.budget + 1) + row) * a.V;
    const int v0 = chunk * kVerifyChunk;
    const int v1 = min(a.V, v0 + kVerifyChunk);
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    constexpr int kPer = kVerifyChunk / 256;
    float xs[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int v = v0 + threadIdx.x + 256 * j;
      xs[j] = v < v1 ? z[v] : -INFINITY;
    }
    float m = -INFINITY;
    int arg = 0x7FFFFFFF, flags = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int v = v0 + threadIdx.x + 256 * j;
      const float x = xs[j];
      if (v >= v1) continue;
      if (isnan(x)) {
        flags |= 1;
        continue;
      }
      if (x == INFINITY) flags |= 2;
      if (x > m || (x == m && v < arg)) {
        m = x;
        arg = v;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, m, o);
      const int oa = __shfl_xor_sync(0xffffffffu, arg, o);
      if (om > m || (om == m && oa < arg)) {
        m = om;
        arg = oa;
      }
      flags |= __shfl_xor_sync(0xffffffffu, flags, o);
    }
    if (lane == 0) {
      sm_m[wid] = m;
      sm_a[wid] = arg;
      sm_f[wid] = flags;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float M = sm_m[0];
      int A = sm_a[0], F = 0;
      for (int w = 0; w < 8; ++w) {
        if (sm_m[w] > M || (sm_m[w] == M && sm_a[w] < A)) {
          M = sm_m[w];
          A = sm_a[w];
        }
        F |= sm_f[w];
      }
      VerifyStat st;
      st.m = M;
      st.s = 0.f;
      st.s_lo = 0.f;
      st.arg = A;
      st.flags = F;
      a.stats[(static_cast<size_t>(r) * (a.budget + 1) + row) * a.n_chunks + chunk] = st;
    }
  }
  // count this CTA; the one completing request r's rows x chunks walks its tree (thread
  // 0 wrote the statistics: its count releases them and acquires the others')
  __shared__ bool last;
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned int prev = count_acq_rel(a.counters + r);
    last = prev == static_cast<unsigned int>((a.budget + 1) * a.n_chunks - 1);
    if (last) a.counters[r] = 0u;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  tree_chain(a, r);
}

}  // namespace

cudaError_t launch_tree_verify(const TreeVerifyArgs& a, int n_req, bool pdl, cudaStream_t st) {
  if (a.budget < 1 || a.budget > kTreeMaxNodes || a.n_chunks < 1) return cudaErrorInvalidValue;
  if (static_cast<long long>(n_req) * (a.budget + 1) > 65535) return cudaErrorInvalidValue;  // grid rows
  if (a.B != 8 && a.B != 16) return cudaErrorInvalidValue;
  return launch_ex(tree_stats_kernel, dim3(a.n_chunks, n_req * (a.budget + 1)), dim3(256), 0, st, pdl, a);
}

cudaError_t launch_verify(const VerifyArgs& a, int n_req, bool pdl, cudaStream_t st) {
  if (a.B != 8 && a.B != 16) return cudaErrorInvalidValue;
  if (static_cast<long long>(n_req) * a.B > 65535) return cudaErrorInvalidValue;  // grid rows
  return launch_ex(verify_stats_kernel, dim3(a.n_chunks, n_req * a.B), dim3(256), a.n_chunks * sizeof(double), st, pdl,
                   a);
}

}  // namespace df2
