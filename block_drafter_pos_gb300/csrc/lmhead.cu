// Shared LM head fused with the vocabulary top-16 (step a8), plus the merge that
// also finishes the selector projection (step a9).
//
// The LM head [V][H] is the largest single weight stream of the step.  It runs
// on the same pipeline as the projections (pipeline.cuh): each CTA (two per SM)
// owns a contiguous range of 64-row vocabulary blocks; a producer warp streams
// the block's weights and the hidden state through a ring of shared-memory
// stages with bulk tensor copies, and four consumer warps run the MMAs (16 rows
// each).  When a block is done its 64 x N logits go to shared memory, are scaled
// by the row's 1/rms (final RMSNorm, applied after the projection), optionally
// written out, and folded into a running top-16 per block row.  Only the 16 best
// (value, index) keys per CTA and row leave the kernel; the merge kernel picks
// the global top-16.
//
// Ordering ("LSE docs/DFLASH2.md", top-k paragraph): NaN first (by index), then
// descending value with +/-inf in their usual places, equal values -> smaller
// index.  Encoded as one 64-bit key so every comparison is exact.
#include <math.h>

#include "common.cuh"
#include "glue.h"
#include "internal.h"
#include "pipeline.cuh"

namespace df2 {

namespace {

using namespace pipe;

constexpr int kTopK = 16;

DF2_DEV void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory"); }

template <int NT, bool LO>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) lmhead_kernel(const __grid_constant__ LmHeadArgs a) {
  using Geo = StageGeo<0, NT>;
  constexpr int D = Geo::kDepth;
  constexpr int kXBoxes = kStageK / 64;  // activation boxes per tile and plane
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[D], empty_bar[D];
  __shared__ float logit[NT * 8][kBlockRows + 1];
  __shared__ unsigned long long run[NT * 8][kTopK];
  __shared__ float rscale[NT * 8];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t full0 = smem_u32(&full_bar[0]), empty0 = smem_u32(&empty_bar[0]);
  const int n_rows = a.n_rows;
  const int nt = n_rows >> 3;
  for (int e = threadIdx.x; e < NT * 8 * kTopK; e += blockDim.x) (&run[0][0])[e] = 0ull;
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
  const int blocks = (a.V + kBlockRows - 1) / kBlockRows;
  const int b0 = static_cast<int>((static_cast<long long>(blocks) * blockIdx.x) / gridDim.x);
  const int b1 = static_cast<int>((static_cast<long long>(blocks) * (blockIdx.x + 1)) / gridDim.x);
  const int nst = a.H / kStageK;
  const int total = (b1 - b0) * nst;  // stages of this CTA: block b0 + it / nst, K (it % nst) * kStageK

  if (wid == kConsumers) {
    // ---------------------------------------------------------------- producer warp
    const uint64_t policy = evict_first_policy(), xpolicy = evict_last_policy();
    const int xbytes = nt * kXBoxes * 1024 * (LO ? 2 : 1);
    // the next stage whose weights get armed (K stage within the block, block)
    int w_st = 0, w_blk = b0;
    auto arm_w = [&](int it) {
      const int slot = it % D;
      if (lane == 0) mbar_expect_tx(full0 + 8 * slot, Geo::kWBytes + xbytes);
      __syncwarp();
      if (lane < kStageK / 64)
        tma_load_2d(ring + slot * Geo::kBytes + lane * wbox_bytes<0>(), &a.wmap, w_st * kStageK + lane * 64,
                    w_blk * kBlockRows, full0 + 8 * slot, policy);
      if (++w_st == nst) {
        w_st = 0;
        ++w_blk;
      }
    };
    // this lane's activation box (the same every stage): plane, tile, 64-K box
    const int n_x = nt * kXBoxes * (LO ? 2 : 1);
    const int x_plane = lane / (nt * kXBoxes), x_rem = lane % (nt * kXBoxes);
    const int x_t = x_rem / kXBoxes, x_b = x_rem % kXBoxes;
    const uint32_t x_dst = Geo::kWBytes + x_plane * Geo::kXPlane + (x_t * kXBoxes + x_b) * 1024;
    const int x_row = x_plane * a.x_lo_row + x_t * 8;
    int x_st = 0;
    auto issue_x = [&](int it) {
      if (lane < n_x)  // n_x <= 32 (nt <= 4, 2 boxes, 2 planes)
        tma_load_2d(ring + (it % D) * Geo::kBytes + x_dst, &a.xmap, x_st * kStageK + x_b * 64, x_row,
                    full0 + 8 * (it % D), xpolicy);
      if (++x_st == nst) x_st = 0;
    };
    const int np = total < D ? total : D;
    for (int it = 0; it < np; ++it) arm_w(it);  // weights first: they do not depend on the previous kernel
    pdl_wait();
    bool ok = true;
    int it = 0;
    for (; it < total; ++it) {
      if (it >= np) {
        if (!__all_sync(0xffffffffu, mbar_wait(empty0 + 8 * (it % D), static_cast<uint32_t>(((it / D) + 1) & 1)))) {
          ok = false;
          break;
        }
        arm_w(it);
      }
      issue_x(it);
    }
    if (!ok && lane == 0 && a.err != nullptr) atomicExch(a.err, 1);
    for (int j = it > D ? it - D : 0; j < it; ++j) mbar_wait(full0 + 8 * (j % D), static_cast<uint32_t>((j / D) & 1));
    return;
  }

  // ------------------------------------------------------------------ consumer warps
  pdl_wait();
  for (int n = wid; n < n_rows; n += kConsumers) {  // final-norm scale of each row (1: already normalised)
    const float rs = a.ss != nullptr ? warp_inv_rms(a.ss, n, a.nch, a.H, a.eps) : 1.f;
    if (lane == 0) rscale[n] = rs;
  }
  const int g = lane >> 2, q = lane & 3;
  const uint32_t wrow = static_cast<uint32_t>((wid * 16 + g) * 128);
  const uint32_t xrow = static_cast<uint32_t>(g * 128);
  float c0[NT][4], c1[NT][4], c2[NT][4], c3[NT][4];
  int st = -1, blk = b0 - 1;  // K stage within the block, block
  for (int it = 0; it < total; ++it) {
    if (++st == nst || it == 0) {
      st = 0;
      ++blk;
    }
    if (st == 0) {
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) c0[t][e] = c1[t][e] = c2[t][e] = c3[t][e] = 0.f;
    }
    const int slot = it % D;
    if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * slot, static_cast<uint32_t>((it / D) & 1)))) {
      if (lane == 0 && a.err != nullptr) atomicExch(a.err, 1);
      break;
    }
    const uint32_t base = ring + slot * Geo::kBytes;
    stage_bf16<NT, LO>(nt, base + wrow, base + Geo::kWBytes + xrow, g, q, c0, c1, c2, c3);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * slot);
    if (st + 1 < nst) continue;
    // ---- block done: logits to shared memory, then scale, write out and fold into the top-16
    const int lr = wid * 16 + g;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < nt) {
        const int n0 = t * 8 + 2 * q;
        logit[n0][lr] = (c0[t][0] + c1[t][0]) + (c2[t][0] + c3[t][0]);
        logit[n0 + 1][lr] = (c0[t][1] + c1[t][1]) + (c2[t][1] + c3[t][1]);
        logit[n0][lr + 8] = (c0[t][2] + c1[t][2]) + (c2[t][2] + c3[t][2]);
        logit[n0 + 1][lr + 8] = (c0[t][3] + c1[t][3]) + (c2[t][3] + c3[t][3]);
      }
    }
    consumer_sync();
    const int v0 = blk * kBlockRows;
    for (int n = wid; n < n_rows; n += kConsumers) {
      const int pos = n % a.B;
      if (pos == 0) continue;  // the anchor position is not sampled
      const float rs = rscale[n];
      unsigned long long* rn = run[n];
      const unsigned long long thr = rn[kTopK - 1];
      unsigned long long mine[2];
      bool any = false;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int idx = lane + 32 * j;
        const int v = v0 + idx;
        const float val = logit[n][idx] * rs;
        if (a.logits_out != nullptr && v < a.V)
          a.logits_out[(static_cast<size_t>(n / a.B) * (a.B - 1) + pos - 1) * a.V + v] = val;
        const unsigned long long key = v < a.V ? topk_key(val, static_cast<uint32_t>(v)) : 0ull;
        mine[j] = key > thr ? key : 0ull;
        any |= mine[j] != 0ull;
      }
      if (!__any_sync(0xffffffffu, any)) continue;
      // insert the passing candidates one by one into the sorted list held by lanes
      // 0..15 (descending): rank by ballot, shift the tail down one lane
      unsigned long long held = lane < kTopK ? rn[lane] : 0ull;
      unsigned long long cut = thr;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        unsigned m = __ballot_sync(0xffffffffu, mine[j] != 0ull);
        while (m != 0u) {
          const int src = __ffs(m) - 1;
          m &= m - 1u;
          const unsigned long long cand = __shfl_sync(0xffffffffu, mine[j], src);
          if (cand <= cut) continue;  // uniform: every lane holds the same cut
          const int p = __popc(__ballot_sync(0xffffffffu, lane < kTopK && held > cand));
          const unsigned long long up = __shfl_up_sync(0xffffffffu, held, 1);
          if (lane < kTopK && lane > p) held = up;
          if (lane == p) held = cand;
          cut = __shfl_sync(0xffffffffu, held, kTopK - 1);
        }
      }
      if (lane < kTopK) rn[lane] = held;
      __syncwarp();
    }
    consumer_sync();  // the logit tile is free for the next block
  }
  // ---- per-CTA top-16 out
  for (int e = threadIdx.x; e < n_rows * kTopK; e += kConsumers * 32) {
    const int n = e / kTopK, j = e % kTopK;
    a.part_keys[(static_cast<size_t>(n) * a.n_cta + blockIdx.x) * kTopK + j] = run[n][j];
  }
}

// grid (n_rows), 256 threads: global top-16 of one block row from the per-CTA lists,
// and the selector gate of that row (sum of split partials, times 1/rms).
__global__ void __launch_bounds__(256) topk_merge_kernel(const TopkMergeArgs a) {
  __shared__ unsigned long long wtop[8][kTopK];
  __shared__ float rs;
  pdl_begin();
  const int n = blockIdx.x;
  const int pos = n % a.B, rq = n / a.B;
  if (pos == 0) return;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (a.err != nullptr && __ldcg(a.err) != 0) {  // the per-CTA lists are incomplete: write the sentinel
    if (threadIdx.x < kTopK) {
      const size_t o = (static_cast<size_t>(rq) * (a.B - 1) + pos - 1) * kTopK + threadIdx.x;
      a.cand_ids[o] = -1;
      a.cand_logits[o] = __int_as_float(0x7FC00000);
    }
    return;
  }
  if (wid == 0) {
    const float v = a.ss != nullptr ? warp_inv_rms(a.ss, n, a.nch, a.H, a.eps) : 1.f;
    if (lane == 0) rs = v;
  }
  const int total = a.n_cta * kTopK;  // <= 256 * kPer (checked at launch)
  const unsigned long long* src = a.part_keys + static_cast<size_t>(n) * total;
  constexpr int kPer = 32;
  unsigned long long keys[kPer];  // every CTA's list, loaded once
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int e = threadIdx.x + 256 * j;
    keys[j] = e < total ? src[e] : 0ull;
  }
  // keys are unique (distinct indices) and picked in decreasing order, so the keys
  // still available in a round are exactly those below the previous winner.
  // Level 1: each warp's top-16 of its own keys (no block barrier).
  unsigned long long last = ~0ull, mine16 = 0ull;
  for (int round = 0; round < kTopK; ++round) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if (keys[j] < last && keys[j] > best) best = keys[j];
    last = warp_max_u64(best);
    if (lane == round) mine16 = last;
  }
  if (lane < kTopK) wtop[wid][lane] = mine16;
  __syncthreads();
  // Level 2: warp 0 merges the 8 lists (4 keys per lane).
  if (wid == 0) {
    unsigned long long k4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) k4[j] = (&wtop[0][0])[lane + 32 * j];
    last = ~0ull;
    for (int round = 0; round < kTopK; ++round) {
      unsigned long long best = 0ull;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (k4[j] < last && k4[j] > best) best = k4[j];
      const unsigned long long win = warp_max_u64(best);
      last = win;
      if (lane == 0) {
        const size_t o = (static_cast<size_t>(rq) * (a.B - 1) + pos - 1) * kTopK + round;
        a.cand_ids[o] = static_cast<int32_t>(key_index(win));
        a.cand_logits[o] = key_value(win);
      }
    }
  }
  __syncthreads();
  if (a.sel == nullptr) return;
  const size_t plane = static_cast<size_t>(a.n_rows) * a.rank;
  for (int j = threadIdx.x; j < a.rank; j += blockDim.x) {
    const float* p = a.sel + static_cast<size_t>(n) * a.rank + j;
    float v = 0.f;
    const int np = gemv_plane_count(a.psel, j);
    for (int s0 = 0; s0 < np; s0 += 16) {  // planes in order, 16 loads in flight
      float t[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) t[k] = (s0 + k < np) ? p[static_cast<size_t>(s0 + k) * plane] : 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) v += t[k];
    }
    a.gate[(static_cast<size_t>(rq) * (a.B - 1) + pos - 1) * a.rank + j] = v * rs;
  }
}

// The warp's 32 keys in decreasing order across the lanes (bitonic sorting network).
DF2_DEV unsigned long long warp_sort_desc(unsigned long long v, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, j);
      const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
      v = keep_max ? (o > v ? o : v) : (o < v ? o : v);
    }
  }
  return v;
}

// grid (n_chunks, (B - 1) R), 256 threads, 16 consecutive vocabulary entries per thread.
// The chunk's 16 largest keys are found without ranking all 4096: the 16th largest
// of a warp's 32 per-thread maxima (a bitonic sort across the warp) is a lower
// bound T of the chunk's 16th largest key (16 distinct entries reach it), so only
// the entries >= the largest such T are candidates; one warp ranks those.  If the
// candidates overflow the buffer (few distinct values, e.g. a chunk past the
// vocabulary's end), every warp ranks its own entries and warp 0 merges.  Up to 64
// candidates (the usual case) are ranked by sorting networks rather than by 16
// rounds of warp maxima.
__global__ void __launch_bounds__(256, 4) logits_topk_kernel(const LogitsTopkArgs a) {
  constexpr int kCap = 1024;
  __shared__ unsigned long long cand[kCap];
  __shared__ unsigned long long wthr[8];
  __shared__ unsigned long long wtop[8][kTopK];
  __shared__ int n_cand;
  __shared__ float rs_sh;
  __shared__ int np_sh[kLogitChunk / 16 / 8];  // plane counts of the chunk's 128-id blocks (at least 64 ids)
  // before the wait: shapes only (once per CTA, not per thread)
  if (threadIdx.x < kLogitChunk / 128)
    np_sh[threadIdx.x] = gemv_plane_count(a.pl, blockIdx.x * kLogitChunk + threadIdx.x * 128);
  pdl_begin();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int rq = blockIdx.y / (a.B - 1), pos = blockIdx.y % (a.B - 1) + 1, n = rq * a.B + pos;
  if (wid == 0) {
    const float v = a.ss != nullptr ? warp_inv_rms(a.ss, n, a.nch, a.H, a.eps) : 1.f;
    if (lane == 0) {
      rs_sh = v;
      n_cand = 0;
    }
  }
  __syncthreads();
  const float rs = rs_sh;
  const int v0 = blockIdx.x * kLogitChunk + threadIdx.x * 16;
  unsigned long long keys[16];
  if (v0 < a.V) {  // V is a multiple of 16: the thread's 16 entries are all in range, in one weight block
    const size_t plane = static_cast<size_t>(a.n_rows) * a.V;
    const float* src = a.part + static_cast<size_t>(n) * a.V + v0;
    const int np = np_sh[(threadIdx.x * 16) >> 7];  // v0's block within the chunk (blocks of 128 ids)
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
    for (int p = 0; p < np; ++p) {  // planes in order
      const float4* q = reinterpret_cast<const float4*>(src + static_cast<size_t>(p) * plane);
      float4 t[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) t[j] = __ldcs(q + j);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[4 * j] += t[j].x;
        acc[4 * j + 1] += t[j].y;
        acc[4 * j + 2] += t[j].z;
        acc[4 * j + 3] += t[j].w;
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      acc[j] *= rs;
      keys[j] = topk_key(acc[j], static_cast<uint32_t>(v0 + j));
    }
    if (a.logits_out != nullptr) {
      float4* o = reinterpret_cast<float4*>(a.logits_out + (static_cast<size_t>(rq) * (a.B - 1) + pos - 1) * a.V + v0);
#pragma unroll
      for (int j = 0; j < 4; ++j) o[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) keys[j] = 0ull;
  }
  // the warp's per-thread maxima sorted in decreasing order; lane 15 holds the 16th
  unsigned long long v = 0ull;
#pragma unroll
  for (int j = 0; j < 16; ++j) v = keys[j] > v ? keys[j] : v;
  v = warp_sort_desc(v, lane);
  if (lane == 15) wthr[wid] = v;
  __syncthreads();
  unsigned long long T = wthr[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) T = wthr[w] > T ? wthr[w] : T;
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (keys[j] >= T) {
      const int p = atomicAdd(&n_cand, 1);
      if (p < kCap) cand[p] = keys[j];
    }
  __syncthreads();
  const int nc = n_cand;
  unsigned long long last = ~0ull;
  if (nc <= kCap) {
    if (wid != 0) return;
    unsigned long long out = 0ull;
    if (nc <= 64) {
      // two sorted halves; the 32 largest of both, x[i] vs y[31 - i], form a bitonic
      // sequence that five merge stages put in decreasing order
      const unsigned long long x = warp_sort_desc(lane < nc ? cand[lane] : 0ull, lane);
      const unsigned long long y = warp_sort_desc(lane + 32 < nc ? cand[lane + 32] : 0ull, lane);
      const unsigned long long yr = __shfl_sync(0xffffffffu, y, 31 - lane);
      out = x > yr ? x : yr;
#pragma unroll
      for (int j = 16; j > 0; j >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, out, j);
        out = (lane & j) == 0 ? (o > out ? o : out) : (o < out ? o : out);
      }
    } else {
      for (int round = 0; round < kTopK; ++round) {
        unsigned long long best = 0ull;
        for (int i = lane; i < nc; i += 32) {
          const unsigned long long c = cand[i];
          if (c < last && c > best) best = c;
        }
        last = warp_max_u64(best);
        if (lane == round) out = last;
      }
    }
    if (lane < kTopK) a.part_keys[(static_cast<size_t>(n) * a.n_chunks + blockIdx.x) * kTopK + lane] = out;
    return;
  }
  // keys are unique, so the keys still available in a round are those below the last winner
  unsigned long long mine16 = 0ull;
  for (int round = 0; round < kTopK; ++round) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (keys[j] < last && keys[j] > best) best = keys[j];
    last = warp_max_u64(best);
    if (lane == round) mine16 = last;
  }
  if (lane < kTopK) wtop[wid][lane] = mine16;
  __syncthreads();
  if (wid == 0) {
    unsigned long long k4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) k4[j] = (&wtop[0][0])[lane + 32 * j];
    last = ~0ull;
    unsigned long long out = 0ull;
    for (int round = 0; round < kTopK; ++round) {
      unsigned long long best = 0ull;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (k4[j] < last && k4[j] > best) best = k4[j];
      last = warp_max_u64(best);
      if (lane == round) out = last;
    }
    if (lane < kTopK) a.part_keys[(static_cast<size_t>(n) * a.n_chunks + blockIdx.x) * kTopK + lane] = out;
  }
}

template <int NT, bool LO>
cudaError_t launch_nt(const LmHeadArgs& a, bool pdl, cudaStream_t st) {
  constexpr int smem = StageGeo<0, NT>::kSmem;
  static std::atomic<unsigned long long> attr_done{0};
  const cudaError_t e = set_smem_once(lmhead_kernel<NT, LO>, smem, attr_done);
  if (e != cudaSuccess) return e;
  return launch_ex(lmhead_kernel<NT, LO>, dim3(a.n_cta), dim3(kThreads), smem, st, pdl, a);
}

}  // namespace

int lmhead_ctas(int num_sms) { return num_sms * kCtasPerSm; }

cudaError_t launch_lmhead(const LmHeadArgs& a, bool pdl, cudaStream_t st) {
  const int nt = a.n_rows / 8;
  if (a.n_rows < 8 || a.n_rows % 8 || a.H % kStageK || a.n_cta < 1) return cudaErrorInvalidValue;
  if ((a.B != 8 && a.B != 16) || a.n_rows % a.B) return cudaErrorInvalidValue;
  const bool lo = a.x_lo_row >= 0;
  if (nt <= 1) return lo ? launch_nt<1, true>(a, pdl, st) : launch_nt<1, false>(a, pdl, st);
  if (nt <= 2) return lo ? launch_nt<2, true>(a, pdl, st) : launch_nt<2, false>(a, pdl, st);
  if (nt <= 4) return lo ? launch_nt<4, true>(a, pdl, st) : launch_nt<4, false>(a, pdl, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_topk_merge(const TopkMergeArgs& a, bool pdl, cudaStream_t st) {
  if (a.n_cta < 1 || a.n_cta * kTopK > 256 * 32) return cudaErrorInvalidValue;
  if ((a.B != 8 && a.B != 16) || a.n_rows % a.B) return cudaErrorInvalidValue;
  return launch_ex(topk_merge_kernel, dim3(a.n_rows), dim3(256), 0, st, pdl, a);
}

cudaError_t launch_logits_topk(const LogitsTopkArgs& a, int n_req, bool pdl, cudaStream_t st) {
  if (a.V % 16 || a.n_chunks < 1 || a.n_chunks * kTopK > 8192) return cudaErrorInvalidValue;
  if (a.B != 8 && a.B != 16) return cudaErrorInvalidValue;
  return launch_ex(logits_topk_kernel, dim3(a.n_chunks, (a.B - 1) * n_req), dim3(256), 0, st, pdl, a);
}

}  // namespace df2
