// Block attention of the drafter (step a5): 8 block queries per request attend,
// noncausally, to all 8 block keys and to the context keys inside the sliding
// window ("LSE docs/DFLASH2.md", block paragraph: noncausal within the block,
// context keys obey the 2048-position sliding window).  Query i sits at absolute
// position L + i (L = keys in the cache); it sees context key k iff
// L + i - k < window.  GQA: the 4 query heads of one KV head share its keys.
//
// Split over keys (flash-decoding style): one CTA per (request, KV head, chunk of
// 128 context keys), plus one CTA for the 8 block keys; all 32 queries of the KV
// head group (4 heads x 8 positions) are handled together so every key is read
// once.  Keys outside the window are never read.  A combine kernel merges the
// chunk partials (max, sum, unnormalised output) in a fixed order.
#include <math.h>

#include "common.cuh"
#include "glue.h"

namespace df2 {

namespace {

constexpr int kHd = 128;
constexpr int kQ = 32;        // queries per KV head group (4 heads x 8 positions)
constexpr int kKeys = kAttnChunk;
constexpr int kPad = kHd + 1;
constexpr int kPartStride = kHd + 2;

struct AttnSmem {
  float q[kQ][kHd];
  float kv[kKeys][kPad];
  float p[kQ][kKeys];
};

__global__ void __launch_bounds__(256) attn_chunk_kernel(const AttnArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>(smem_raw);
  const int nkv = a.n_kv_heads;
  const int r = blockIdx.x / nkv, kvh = blockIdx.x % nkv;
  const int chunk = blockIdx.y;
  const int tid = threadIdx.x;
  const int nn = min(max(a.n_new[r], 0), 8);
  const int L = min(max(a.ctx_len[r], 0), a.kv_capacity - nn) + nn;  // same clamping as the cache append
  const int lo0 = max(0, L - (a.window - 1));
  const int n_ctx = L - lo0;
  const int n_ctx_chunks = (n_ctx + kKeys - 1) / kKeys;
  const bool block_chunk = chunk == a.n_chunks - 1;
  float* out = a.part + ((static_cast<size_t>(r) * nkv + kvh) * a.n_chunks + chunk) * kQ * kPartStride;
  int k_begin = 0, nk = 0;
  if (block_chunk) {
    nk = 8;
  } else if (chunk < n_ctx_chunks) {
    k_begin = lo0 + chunk * kKeys;
    nk = min(kKeys, L - k_begin);
  }
  if (nk == 0) {
    if (tid < kQ) {
      out[tid * kPartStride + 0] = -INFINITY;
      out[tid * kPartStride + 1] = 0.f;
    }
    return;
  }
  const int rep = a.n_q_heads / nkv;  // 4
  const float qscale = rsqrtf(static_cast<float>(kHd)) * 1.4426950408889634f;  // log2(e)/sqrt(hd)
  // queries: qi = hr * 8 + i  ->  head kvh*rep + hr, block row r*8 + i
  for (int e = tid; e < kQ * kHd; e += 256) {
    const int qi = e / kHd, d = e % kHd;
    const int hr = qi >> 3, i = qi & 7;
    sm.q[qi][d] = a.q[((static_cast<size_t>(r) * 8 + i) * a.n_q_heads + kvh * rep + hr) * kHd + d] * qscale;
  }
  // keys
  if (block_chunk) {
    for (int e = tid; e < 8 * kHd; e += 256) {
      const int k = e / kHd, d = e % kHd;
      sm.kv[k][d] = a.kb[((static_cast<size_t>(r) * 8 + k) * nkv + kvh) * kHd + d];
    }
  } else {
    const uint16_t* kc = a.k_cache + (static_cast<size_t>(r) * a.kv_capacity + k_begin) * nkv * kHd + kvh * kHd;
    for (int e = tid; e < nk * (kHd / 8); e += 256) {
      const int k = e / (kHd / 8), d8 = (e % (kHd / 8)) * 8;
      const uint4 v = ld_stream(kc + static_cast<size_t>(k) * nkv * kHd + d8);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        sm.kv[k][d8 + 2 * j] = __uint_as_float(w[j] << 16);
        sm.kv[k][d8 + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
  }
  __syncthreads();
  // scores: thread -> 4 queries (warp id) x 4 keys (lane + 32 j)
  {
    const int qg = tid >> 5, kg = tid & 31;
    float s[4][4] = {};
    for (int d = 0; d < kHd; ++d) {
      float qv[4], kv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) qv[i] = sm.q[qg * 4 + i][d];
#pragma unroll
      for (int j = 0; j < 4; ++j) kv[j] = sm.kv[kg + 32 * j][d];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[i][j] = fmaf(qv[i], kv[j], s[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int qi = qg * 4 + i;
      const int pos_i = qi & 7;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int k = kg + 32 * j;
        bool ok = k < nk;
        if (!block_chunk) ok = ok && (k_begin + k >= L + pos_i - (a.window - 1));
        sm.p[qi][k] = ok ? s[i][j] : -INFINITY;
      }
    }
  }
  __syncthreads();
  // softmax statistics per query: warp w handles queries 4w..4w+3
  {
    const int w = tid >> 5, lane = tid & 31;
    for (int i = 0; i < 4; ++i) {
      const int qi = w * 4 + i;
      float v[4];
      float m = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[j] = sm.p[qi][lane + 32 * j];
        m = fmaxf(m, v[j]);
      }
      m = warp_max(m);
      float l = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float p = (m == -INFINITY) ? 0.f : exp2f(v[j] - m);
        sm.p[qi][lane + 32 * j] = p;
        l += p;
      }
      l = warp_sum(l);
      if (lane == 0) {
        out[qi * kPartStride + 0] = m;
        out[qi * kPartStride + 1] = l;
      }
    }
  }
  __syncthreads();
  // values
  if (block_chunk) {
    for (int e = tid; e < 8 * kHd; e += 256) {
      const int k = e / kHd, d = e % kHd;
      sm.kv[k][d] = a.vb[((static_cast<size_t>(r) * 8 + k) * nkv + kvh) * kHd + d];
    }
  } else {
    const uint16_t* vc = a.v_cache + (static_cast<size_t>(r) * a.kv_capacity + k_begin) * nkv * kHd + kvh * kHd;
    for (int e = tid; e < nk * (kHd / 8); e += 256) {
      const int k = e / (kHd / 8), d8 = (e % (kHd / 8)) * 8;
      const uint4 v = ld_stream(vc + static_cast<size_t>(k) * nkv * kHd + d8);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        sm.kv[k][d8 + 2 * j] = __uint_as_float(w[j] << 16);
        sm.kv[k][d8 + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
  }
  __syncthreads();
  // out[q][d] = sum_k p[q][k] v[k][d]: thread -> 4 queries (warp id) x 4 dims (lane + 32 j)
  {
    const int qg = tid >> 5, dg = tid & 31;
    float o[4][4] = {};
    for (int k = 0; k < nk; ++k) {
      float pv[4], vv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pv[i] = sm.p[qg * 4 + i][k];
#pragma unroll
      for (int j = 0; j < 4; ++j) vv[j] = sm.kv[k][dg + 32 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) o[i][j] = fmaf(pv[i], vv[j], o[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) out[(qg * 4 + i) * kPartStride + 2 + dg + 32 * j] = o[i][j];
  }
}

// grid (R, nq), 128 threads: merge chunk partials of one query head for the 8 positions.
__global__ void __launch_bounds__(128) attn_combine_kernel(const AttnArgs a) {
  __shared__ float sm[4 * 8];
  const int r = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  const int nkv = a.n_kv_heads;
  const int rep = a.n_q_heads / nkv;
  const int kvh = h / rep, hr = h % rep;
  const float* base = a.part + (static_cast<size_t>(r) * nkv + kvh) * a.n_chunks * kQ * kPartStride;
  float ov[8];
  for (int i = 0; i < 8; ++i) {
    const int qi = hr * 8 + i;
    float M = -INFINITY;
    for (int c = 0; c < a.n_chunks; ++c) {
      const float* pc = base + (static_cast<size_t>(c) * kQ + qi) * kPartStride;
      if (pc[1] > 0.f) M = fmaxf(M, pc[0]);
    }
    float acc = 0.f, den = 0.f;
    for (int c = 0; c < a.n_chunks; ++c) {
      const float* pc = base + (static_cast<size_t>(c) * kQ + qi) * kPartStride;
      if (pc[1] > 0.f) {
        const float f = exp2f(pc[0] - M);
        den += f * pc[1];
        acc += f * pc[2 + d];
      }
    }
    ov[i] = acc / den;
  }
  const int ld = a.n_q_heads * kHd;
  const int c = h * kHd + d;
  if (a.fmt == 0) {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(a.act_o);
    for (int i = 0; i < 8; ++i) o[(static_cast<size_t>(r) * 8 + i) * ld + c] = __float2bfloat16_rn(ov[i]);
  } else {
    __half* o = reinterpret_cast<__half*>(a.act_o);
    const int lane = d & 31, wid = d >> 5;
    float rs[8];
    for (int i = 0; i < 8; ++i) {
      const __half hv = __float2half_rn(ov[i]);
      o[(static_cast<size_t>(r) * 8 + i) * ld + c] = hv;
      rs[i] = warp_sum(__half2float(hv));
    }
    if (lane == 0)
      for (int i = 0; i < 8; ++i) sm[wid * 8 + i] = rs[i];
    __syncthreads();
    if (d < 16) {
      const int gq = d / 8, i = d % 8;
      const int KG = ld / 64;
      a.xsum_o[(static_cast<size_t>(r) * 8 + i) * KG + h * 2 + gq] = sm[(2 * gq) * 8 + i] + sm[(2 * gq + 1) * 8 + i];
    }
  }
}

}  // namespace

cudaError_t launch_attention(const AttnArgs& a, int n_req, cudaStream_t st) {
  static bool attr_set = false;
  const size_t smem = sizeof(AttnSmem);
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  attn_chunk_kernel<<<dim3(n_req * a.n_kv_heads, a.n_chunks), 256, smem, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_combine_kernel<<<dim3(n_req, a.n_q_heads), 128, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace df2
