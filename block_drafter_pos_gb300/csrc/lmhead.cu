// Shared LM head fused with the vocabulary top-16 (step a8), plus the merge that
// also finishes the selector projection (step a9).
//
// The LM head [V][H] is the largest single weight stream of the step.  A
// persistent grid walks it once: each CTA owns a contiguous range of vocabulary
// rows and processes it in sub-blocks of 256 rows (one 16-row tile per warp,
// mma.sync m16n8k16 with the weights as the A operand, as in gemv.cu).  The
// sub-block's logits go to shared memory, are scaled by the row's 1/rms (final
// RMSNorm, applied after the projection), optionally written out, and folded into
// a running top-16 per block row.  Only the 16 best (value, index) keys per CTA
// and row leave the kernel; the merge kernel picks the global top-16.
//
// Ordering ("LSE docs/DFLASH2.md", top-k paragraph): NaN first (by index), then
// descending value with +/-inf in their usual places, equal values -> smaller
// index.  Encoded as one 64-bit key so every comparison is exact.
#include <math.h>

#include "common.cuh"
#include "glue.h"
#include "internal.h"

namespace df2 {

namespace {

constexpr int kWarps = 16;
constexpr int kSub = kWarps * 16;  // vocabulary rows per sub-block
constexpr int kMaxRows = 32;       // block rows (8 per request) handled by this kernel
constexpr int kTopK = 16;

template <int NT>
__global__ void __launch_bounds__(kWarps * 32, 1) lmhead_topk_kernel(const LmHeadArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* logit = reinterpret_cast<float*>(smem_raw);                                   // [NT*8][kSub]
  unsigned long long* run = reinterpret_cast<unsigned long long*>(logit + NT * 8 * kSub);  // [NT*8][16]
  __shared__ float rscale[kMaxRows];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int n_rows = a.n_rows;
  const int nt = n_rows >> 3;  // n-tiles actually present (<= NT)
  const int tiles_total = a.V / 16;
  const int t0 = static_cast<int>((static_cast<long long>(tiles_total) * blockIdx.x) / gridDim.x);
  const int t1 = static_cast<int>((static_cast<long long>(tiles_total) * (blockIdx.x + 1)) / gridDim.x);
  for (int e = threadIdx.x; e < NT * 8 * kTopK; e += blockDim.x) run[e] = 0ull;
  pdl_trigger();
  bool waited = false;
  for (int tb = t0; tb < t1; tb += kWarps) {
    const int tile = tb + wid;
    // ---- GEMV: one 16-row tile per warp
    if (tile < t1) {
      const int row0 = tile * 16;
      const __nv_bfloat16* w0 = reinterpret_cast<const __nv_bfloat16*>(a.w) + static_cast<size_t>(row0 + g) * a.H + 8 * q;
      const __nv_bfloat16* w1 = w0 + static_cast<size_t>(8) * a.H;
      const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(a.x) + static_cast<size_t>(g) * a.H + 8 * q;
      float acc[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
      uint4 ra[4], rb[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        ra[j] = ld_stream(w0 + 32 * j);
        rb[j] = ld_stream(w1 + 32 * j);
      }
      if (!waited) {  // weights first; the hidden state comes from the previous kernel
        pdl_wait();
        waited = true;
      }
      for (int k = 0; k < a.H; k += 128) {
        uint4 ca[4], cb[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          ca[j] = ra[j];
          cb[j] = rb[j];
        }
        if (k + 128 < a.H) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            ra[j] = ld_stream(w0 + k + 128 + 32 * j);
            rb[j] = ld_stream(w1 + k + 128 + 32 * j);
          }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t < nt) {
            const __nv_bfloat16* xt = xb + static_cast<size_t>(t * 8) * a.H + k;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 x = ld_cached(xt + 32 * j);
              mma_bf16(acc[t], ca[j].x, cb[j].x, ca[j].y, cb[j].y, x.x, x.y);
              mma_bf16(acc[t], ca[j].z, cb[j].z, ca[j].w, cb[j].w, x.z, x.w);
              if (a.x_lo) {  // low-order part of the hidden state: x = hi + lo
                const uint4 y = ld_cached(xt + a.x_lo + 32 * j);
                mma_bf16(acc[t], ca[j].x, cb[j].x, ca[j].y, cb[j].y, y.x, y.y);
                mma_bf16(acc[t], ca[j].z, cb[j].z, ca[j].w, cb[j].w, y.z, y.w);
              }
            }
          }
        }
      }
      const int lr = wid * 16 + g;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t >= nt) break;
        const int n0 = t * 8 + 2 * q;
        logit[(n0)*kSub + lr] = acc[t][0];
        logit[(n0 + 1) * kSub + lr] = acc[t][1];
        logit[(n0)*kSub + lr + 8] = acc[t][2];
        logit[(n0 + 1) * kSub + lr + 8] = acc[t][3];
      }
    }
    if (!waited) {  // warps without a tile in this sub-block
      pdl_wait();
      waited = true;
    }
    if (tb == t0) {  // final-norm scale of each row (1 when the input is already normalised)
      for (int n = wid; n < n_rows; n += kWarps) {
        const float rs = a.ss != nullptr ? warp_inv_rms(a.ss, n, a.nch, a.H, a.eps) : 1.f;
        if (lane == 0) rscale[n] = rs;
      }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n_rows * kSub; e += blockDim.x) logit[e] *= rscale[e / kSub];
    __syncthreads();
    const int v0 = tb * 16;
    const int nv = min(kSub, (t1 - tb) * 16);
    // ---- optional full logits (positions 1..7 only)
    if (a.logits_out) {
      for (int e = threadIdx.x; e < n_rows * kSub; e += blockDim.x) {
        const int n = e / kSub, j = e % kSub;
        const int pos = n & 7;
        if (pos != 0 && j < nv) {
          const int rq = n >> 3;
          a.logits_out[(static_cast<size_t>(rq) * 7 + pos - 1) * a.V + v0 + j] = logit[n * kSub + j];
        }
      }
    }
    // ---- running top-16 per row: warp w handles rows w, w + 16, ...
    for (int n = wid; n < n_rows; n += kWarps) {
      if ((n & 7) == 0) continue;  // the anchor position is not sampled
      unsigned long long* rn = run + n * kTopK;
      const unsigned long long thr = rn[kTopK - 1];
      unsigned long long mine[kSub / 32];
      bool any = false;
#pragma unroll
      for (int j = 0; j < kSub / 32; ++j) {
        const int idx = lane + 32 * j;
        const unsigned long long key = idx < nv ? topk_key(logit[n * kSub + idx], static_cast<uint32_t>(v0 + idx)) : 0ull;
        mine[j] = key > thr ? key : 0ull;
        any |= mine[j] != 0ull;
      }
      if (!__any_sync(0xffffffffu, any)) continue;
      unsigned long long held = lane < kTopK ? rn[lane] : 0ull;
      unsigned long long result = 0ull;
      for (int round = 0; round < kTopK; ++round) {
        unsigned long long best = held;
#pragma unroll
        for (int j = 0; j < kSub / 32; ++j) best = mine[j] > best ? mine[j] : best;
        const unsigned long long win = warp_max_u64(best);
        if (lane == round) result = win;
        if (win != 0ull) {
          if (held == win) held = 0ull;
#pragma unroll
          for (int j = 0; j < kSub / 32; ++j)
            if (mine[j] == win) mine[j] = 0ull;
        }
      }
      __syncwarp();
      if (lane < kTopK) rn[lane] = result;
      __syncwarp();
    }
    __syncthreads();
  }
  // ---- per-CTA top-16 out
  for (int e = threadIdx.x; e < n_rows * kTopK; e += blockDim.x) {
    const int n = e / kTopK, j = e % kTopK;
    a.part_keys[(static_cast<size_t>(n) * a.n_cta + blockIdx.x) * kTopK + j] = run[n * kTopK + j];
  }
}

// grid (n_rows), 256 threads: global top-16 of one block row from the per-CTA lists,
// and the selector gate of that row (sum of split partials, times 1/rms).
__global__ void __launch_bounds__(256) topk_merge_kernel(const TopkMergeArgs a) {
  __shared__ unsigned long long wbest[8];
  __shared__ float rs;
  pdl_begin();
  const int n = blockIdx.x;
  const int pos = n & 7, rq = n >> 3;
  if (pos == 0) return;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (wid == 0) {
    const float v = a.ss != nullptr ? warp_inv_rms(a.ss, n, a.nch, a.H, a.eps) : 1.f;
    if (lane == 0) rs = v;
  }
  const int total = a.n_cta * kTopK;
  const unsigned long long* src = a.part_keys + static_cast<size_t>(n) * total;
  // keys are unique (distinct indices) and picked in decreasing order, so the keys
  // still available in a round are exactly those below the previous winner.
  unsigned long long last = ~0ull;
  for (int round = 0; round < kTopK; ++round) {
    unsigned long long best = 0ull;
    for (int e = threadIdx.x; e < total; e += blockDim.x) {
      const unsigned long long k = src[e];
      if (k < last && k > best) best = k;
    }
    best = warp_max_u64(best);
    if (lane == 0) wbest[wid] = best;
    __syncthreads();
    unsigned long long win = 0ull;
    for (int w = 0; w < 8; ++w) win = wbest[w] > win ? wbest[w] : win;
    __syncthreads();
    last = win;
    if (threadIdx.x == 0) {
      const size_t o = (static_cast<size_t>(rq) * 7 + pos - 1) * kTopK + round;
      a.cand_ids[o] = static_cast<int32_t>(key_index(win));
      a.cand_logits[o] = key_value(win);
    }
  }
  __syncthreads();
  if (a.sel == nullptr) return;
  const size_t plane = static_cast<size_t>(a.n_rows) * a.rank;
  for (int j = threadIdx.x; j < a.rank; j += blockDim.x) {
    const float* p = a.sel + static_cast<size_t>(n) * a.rank + j;
    float v = 0.f;
    for (int s0 = 0; s0 < a.sel_splits; s0 += 16) {  // split planes in order, 16 loads in flight
      float t[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) t[k] = (s0 + k < a.sel_splits) ? p[static_cast<size_t>(s0 + k) * plane] : 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) v += t[k];
    }
    a.gate[(static_cast<size_t>(rq) * 7 + pos - 1) * a.rank + j] = v * rs;
  }
}

template <int NT>
cudaError_t launch_nt(const LmHeadArgs& a, bool pdl, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(NT) * 8 * kSub * sizeof(float) + static_cast<size_t>(NT) * 8 * kTopK * 8;
  static bool attr_set = false;  // set once, outside any later stream capture
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(lmhead_topk_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(lmhead_topk_kernel<NT>, dim3(a.n_cta), dim3(kWarps * 32), smem, st, pdl, a);
}

}  // namespace

cudaError_t launch_lmhead(const LmHeadArgs& a, bool pdl, cudaStream_t st) {
  const int nt = a.n_rows / 8;
  if (nt <= 1) return launch_nt<1>(a, pdl, st);
  if (nt <= 2) return launch_nt<2>(a, pdl, st);
  if (nt <= 4) return launch_nt<4>(a, pdl, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_topk_merge(const TopkMergeArgs& a, bool pdl, cudaStream_t st) {
  return launch_ex(topk_merge_kernel, dim3(a.n_rows), dim3(256), 0, st, pdl, a);
}

}  // namespace df2
