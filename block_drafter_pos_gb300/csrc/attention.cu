// Block attention of the drafter (step a5): B block queries per request (B = 8 or
// 16) attend, noncausally, to all B block keys and to the context keys inside the sliding
// window ("LSE docs/DFLASH2.md", block paragraph: noncausal within the block,
// context keys obey the 2048-position sliding window).  Query i sits at absolute
// position L + i (L = keys in the cache); it sees context key k iff
// L + i - k < window.  GQA: the 4 query heads of one KV head share its keys.
//
// Split over keys (flash-decoding style): one CTA per (request, KV head, chunk of
// 64 context keys), plus one CTA for the B block keys; all 4 B queries of a KV
// head group (4 heads x B positions) are handled together so every key is read
// once.  A request narrowed to a block width w < B masks its block keys at
// positions >= w, so its first w rows are exactly a block-w forward.  Keys outside
// the window are never read.  Context chunks run on the tensor cores (mma.sync
// m16n8k16 in fp16, fp32 accumulators; fragments by ldmatrix): the bf16 K/V rows
// convert to fp16 exactly inside fp16's normal range (saturated at +-65504 beyond
// it), queries and probabilities round to fp16 (2^-11 relative).  One product per
// MMA: a bf16 hi + lo split of queries and probabilities doubled the shared-memory
// fragment loads, which bound the kernel, and bf16 alone (2^-8) is too coarse.
// The block chunk uses FFMA on the fp32 block keys.  A combine kernel merges the
// chunk partials (max, sum, unnormalised output) in a fixed order.
#include <math.h>

#include "common.cuh"
#include "glue.h"
#include "internal.h"

namespace df2 {

namespace {

constexpr int kHd = 128;
constexpr int kKeys = kAttnChunk;
constexpr int kPartStride = kHd + 2;
constexpr int kLd = kHd + 8;    // bf16 row pitch (272 B): conflict-free fragment loads
constexpr int kPLd = kKeys + 8;

// B block positions: kQ = 4 B queries per KV head group (4 heads x B positions),
// query qi = hr * B + i is head kvh * 4 + hr at block position i.
template <int B>
struct CtxSmem {
  static constexpr int kQ = 4 * B;
  __half q[kQ][kLd];              // scaled queries
  __half k[kKeys][kLd];
  __half v[kKeys][kLd];
  float s[kQ][kKeys + 4];         // scores (log2 units), then probabilities
  __half p[kQ][kPLd];
  float alpha[kQ];                // rescale of the running output, per query
};

template <int B>
struct BlkSmem {
  static constexpr int kQ = 4 * B;
  float q[kQ][kHd];
  float kv[B][kHd + 1];
  float p[kQ][B];
};

// Eight bf16 values -> eight fp16 values (exact inside fp16's normal range; saturated
// at +-65504 beyond it, so no infinity enters the softmax).
DF2_DEV uint4 bf16x8_to_f16x8(uint4 v) {
  auto cv = [](uint32_t w) {
    const float a = fminf(fmaxf(__uint_as_float(w << 16), -65504.f), 65504.f);
    const float b = fminf(fmaxf(__uint_as_float(w & 0xFFFF0000u), -65504.f), 65504.f);
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  };
  return make_uint4(cv(v.x), cv(v.y), cv(v.z), cv(v.w));
}

// A fragment of mma m16n8k16 (rows 0..15 x K 0..15 of an fp16 tile whose rows are 16-byte
// aligned): lane L supplies row (L mod 8) + 8 ((L / 8) mod 2), K offset 8 (L / 16), so
// the registers are {rows 0-7 K 0-7, rows 8-15 K 0-7, rows 0-7 K 8-15, rows 8-15 K 8-15}.
DF2_DEV void ldmatrix_a(uint32_t (&r)[4], const __half* row0, int pitch, int lane) {
  const __half* p = row0 + ((lane & 7) + ((lane >> 3) & 1) * 8) * pitch + (lane >> 4) * 8;
  const unsigned addr = static_cast<unsigned>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// B fragment (K 0..15 x n 0..7) from an fp16 tile stored n-major ([n][K], rows 16-byte
// aligned): lane L < 16 supplies row L mod 8, K offset 8 (L / 8).
DF2_DEV void ldmatrix_b(uint32_t& b0, uint32_t& b1, const __half* row0, int pitch, int lane) {
  const __half* p = row0 + (lane & 7) * pitch + ((lane >> 3) & 1) * 8;
  const unsigned addr = static_cast<unsigned>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(b0), "=r"(b1) : "r"(addr));
}

DF2_DEV void ldmatrix_x2_trans(uint32_t& r0, uint32_t& r1, const void* smem_row) {
  const unsigned addr = static_cast<unsigned>(__cvta_generic_to_shared(smem_row));
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// ------------------------------------------------------------------ context chunk (tensor cores)
// Every thread's K/V loads of the chunk, issued together: 4 rows x 16 bytes of K and of V.
struct KvRegs {
  uint4 k[4], v[4];
};

DF2_DEV KvRegs load_kv(const AttnArgs& a, int r, int kvh, int k_begin, int nk) {
  const int tid = threadIdx.x, nkv = a.n_kv_heads;
  const uint16_t* kc = a.k_cache + (static_cast<size_t>(r) * a.kv_capacity + k_begin) * nkv * kHd + kvh * kHd;
  const uint16_t* vc = a.v_cache + (static_cast<size_t>(r) * a.kv_capacity + k_begin) * nkv * kHd + kvh * kHd;
  KvRegs x;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = tid + 256 * j;
    const int k = e / (kHd / 8), d8 = (e % (kHd / 8)) * 8;
    x.k[j] = x.v[j] = make_uint4(0, 0, 0, 0);
    if (k < nk) {
      x.k[j] = ld_stream(kc + static_cast<size_t>(k) * nkv * kHd + d8);
      x.v[j] = ld_stream(vc + static_cast<size_t>(k) * nkv * kHd + d8);
    }
  }
  return x;
}

// Context chunks c0 .. c1 - 1 of one (request, KV head), 64 keys each, with a
// running (online) softmax: per query the running maximum m and sum l, and the
// unnormalised output O, rescaled by 2^(m_old - m_new) whenever the maximum
// grows.  The next chunk's K/V loads are issued before the current chunk is
// computed.  The first chunk's K/V are loaded before the wait on the previous
// kernel when none of its rows is appended by it.  Writes the part's (m, l, O).
template <int B>
DF2_DEV void ctx_part(const AttnArgs& a, unsigned char* smem_raw, int r, int kvh, int lo0, int c0, int c1, int L,
                      int nn, float* out) {
  constexpr int kQ = 4 * B, kMT = kQ / 16, kQW = kQ / 8;  // queries, query tiles, queries per warp
  CtxSmem<B>& sm = *reinterpret_cast<CtxSmem<B>*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int rep = a.n_q_heads / a.n_kv_heads;
  const float qscale = rsqrtf(static_cast<float>(kHd)) * 1.4426950408889634f;  // log2(e)/sqrt(hd)
  auto kbeg = [&](int c) { return lo0 + c * kKeys; };
  auto nkeys = [&](int c) { return min(kKeys, L - kbeg(c)); };
  KvRegs kv;
  const bool early = kbeg(c0) + nkeys(c0) <= L - nn;  // rows L - nn .. L - 1 are appended by the previous kernel
  if (early) kv = load_kv(a, r, kvh, kbeg(c0), nkeys(c0));
  pdl_wait();
  pdl_trigger();
  if (!early) kv = load_kv(a, r, kvh, kbeg(c0), nkeys(c0));
  // queries -> fp16 (qi = hr * B + i: head kvh*rep + hr, block row r*B + i); loads first
  float qv[kQ * kHd / 256];
#pragma unroll
  for (int j = 0; j < kQ * kHd / 256; ++j) {
    const int e = tid + 256 * j;
    const int qi = e / kHd, d = e % kHd;
    const int hr = qi / B, i = qi % B;
    qv[j] = a.q[((static_cast<size_t>(r) * B + i) * a.n_q_heads + kvh * rep + hr) * kHd + d];
  }
#pragma unroll
  for (int j = 0; j < kQ * kHd / 256; ++j) {
    const int e = tid + 256 * j;
    const int qi = e / kHd, d = e % kHd;
    sm.q[qi][d] = __float2half_rn(qv[j] * qscale);
  }
  float m_run[kQW], l_run[kQW];  // queries kQW wid .. kQW wid + kQW - 1 (the same in every lane)
#pragma unroll
  for (int i = 0; i < kQW; ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.f;
  }
  float o[2][kMT][4] = {};  // dim tiles 2 wid + dn, query tiles mt
  for (int c = c0; c < c1; ++c) {
    const int k_begin = kbeg(c), nk = nkeys(c);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = tid + 256 * j;
      const int k = e / (kHd / 8), d8 = (e % (kHd / 8)) * 8;
      *reinterpret_cast<uint4*>(&sm.k[k][d8]) = bf16x8_to_f16x8(kv.k[j]);
      *reinterpret_cast<uint4*>(&sm.v[k][d8]) = bf16x8_to_f16x8(kv.v[j]);
    }
    if (c + 1 < c1) kv = load_kv(a, r, kvh, kbeg(c + 1), nkeys(c + 1));  // in flight during this chunk
    __syncthreads();
    // S = Q K^T: kMT query tiles x 8 key tiles; warp w takes key tile w for every query tile
    {
      const int nt = wid;
      float cs[kMT][4] = {};
#pragma unroll
      for (int ks = 0; ks < kHd / 16; ++ks) {
        uint32_t b0, b1;
        ldmatrix_b(b0, b1, &sm.k[nt * 8][ks * 16], kLd, lane);
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          uint32_t af[4];
          ldmatrix_a(af, &sm.q[mt * 16][ks * 16], kLd, lane);
          mma_f16(cs[mt], af[0], af[1], af[2], af[3], b0, b1);
        }
      }
      const int lim = L - (a.window - 1) - k_begin;  // query i sees chunk key k iff k >= lim + i
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int qi = mt * 16 + g + 8 * h2;
          const int pos_i = qi % B;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int k = nt * 8 + 2 * q + e;
            const bool ok = k < nk && k >= lim + pos_i;
            sm.s[qi][k] = ok ? cs[mt][2 * h2 + e] : -INFINITY;
          }
        }
      }
    }
    __syncthreads();
    // running softmax statistics: warp w handles queries kQW w .. kQW w + kQW - 1, lane keys
    // lane, lane + 32
#pragma unroll
    for (int i = 0; i < kQW; ++i) {
      const int qi = wid * kQW + i;
      const float v0 = sm.s[qi][lane], v1 = sm.s[qi][lane + 32];
      const float m_new = fmaxf(m_run[i], warp_max(fmaxf(v0, v1)));
      const bool none = m_new == -INFINITY;  // no visible key yet
      const float alpha = none ? 1.f : exp2f(m_run[i] - m_new);
      const float p0 = none ? 0.f : exp2f(v0 - m_new);
      const float p1 = none ? 0.f : exp2f(v1 - m_new);
      l_run[i] = l_run[i] * alpha + warp_sum(p0 + p1);
      m_run[i] = m_new;
      sm.p[qi][lane] = __float2half_rn(p0);
      sm.p[qi][lane + 32] = __float2half_rn(p1);
      if (lane == 0) sm.alpha[qi] = alpha;
    }
    __syncthreads();
    // O = alpha O + P V: kMT query tiles x 16 dim tiles; warp w takes dim tiles 2w, 2w+1
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
      const float a0 = sm.alpha[mt * 16 + g], a1 = sm.alpha[mt * 16 + g + 8];
#pragma unroll
      for (int dn = 0; dn < 2; ++dn) {
        o[dn][mt][0] *= a0;
        o[dn][mt][1] *= a0;
        o[dn][mt][2] *= a1;
        o[dn][mt][3] *= a1;
      }
    }
#pragma unroll
    for (int ks = 0; ks < kKeys / 16; ++ks) {
      uint32_t bv[2][2];
#pragma unroll
      for (int dn = 0; dn < 2; ++dn) ldmatrix_x2_trans(bv[dn][0], bv[dn][1], &sm.v[ks * 16 + (lane & 15)][(wid * 2 + dn) * 8]);
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {  // one probability fragment serves both dimension tiles
        uint32_t af[4];
        ldmatrix_a(af, &sm.p[mt * 16][ks * 16], kPLd, lane);
#pragma unroll
        for (int dn = 0; dn < 2; ++dn) mma_f16(o[dn][mt], af[0], af[1], af[2], af[3], bv[dn][0], bv[dn][1]);
      }
    }
    __syncthreads();  // k, v, p and alpha are rewritten by the next chunk
  }
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < kQW; ++i) {
      out[(wid * kQW + i) * kPartStride + 0] = m_run[i];
      out[(wid * kQW + i) * kPartStride + 1] = l_run[i];
    }
  }
#pragma unroll
  for (int dn = 0; dn < 2; ++dn) {
    const int nt = wid * 2 + dn;
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
      const int q0 = mt * 16 + g, d0 = nt * 8 + 2 * q;
      out[q0 * kPartStride + 2 + d0] = o[dn][mt][0];
      out[q0 * kPartStride + 2 + d0 + 1] = o[dn][mt][1];
      out[(q0 + 8) * kPartStride + 2 + d0] = o[dn][mt][2];
      out[(q0 + 8) * kPartStride + 2 + d0 + 1] = o[dn][mt][3];
    }
  }
}

// ------------------------------------------------------------------ block chunk (B fp32 keys, FFMA)
// Keys at block positions >= the request's width are masked (p = 0).
template <int B>
DF2_DEV void blk_chunk(const AttnArgs& a, unsigned char* smem_raw, int r, int kvh, float* out) {
  constexpr int kQ = 4 * B;
  BlkSmem<B>& sm = *reinterpret_cast<BlkSmem<B>*>(smem_raw);
  const int tid = threadIdx.x;
  const int nkv = a.n_kv_heads, rep = a.n_q_heads / nkv;
  const int w = a.width != nullptr ? min(max(a.width[r], 2), B) : B;
  const float qscale = rsqrtf(static_cast<float>(kHd)) * 1.4426950408889634f;
  for (int e = tid; e < kQ * kHd; e += 256) {
    const int qi = e / kHd, d = e % kHd;
    sm.q[qi][d] = a.q[((static_cast<size_t>(r) * B + (qi % B)) * a.n_q_heads + kvh * rep + (qi / B)) * kHd + d] * qscale;
  }
  for (int e = tid; e < B * kHd; e += 256) {
    const int k = e / kHd, d = e % kHd;
    sm.kv[k][d] = a.kb[((static_cast<size_t>(r) * B + k) * nkv + kvh) * kHd + d];
  }
  __syncthreads();
  // kQ queries x B keys: B * B / 64 dot products per thread (1 at B = 8)
  for (int e = tid; e < kQ * B; e += 256) {
    const int qi = e / B, k = e % B;
    float s = 0.f;
    for (int d = 0; d < kHd; ++d) s = fmaf(sm.q[qi][d], sm.kv[k][d], s);
    sm.p[qi][k] = s;
  }
  __syncthreads();
  if (tid < kQ) {
    float m = -INFINITY;
    for (int k = 0; k < w; ++k) m = fmaxf(m, sm.p[tid][k]);
    float l = 0.f;
    for (int k = 0; k < B; ++k) {
      const float p = k < w ? exp2f(sm.p[tid][k] - m) : 0.f;
      sm.p[tid][k] = p;
      l += p;
    }
    out[tid * kPartStride + 0] = m;
    out[tid * kPartStride + 1] = l;
  }
  for (int e = tid; e < B * kHd; e += 256) {
    const int k = e / kHd, d = e % kHd;
    sm.kv[k][d] = a.vb[((static_cast<size_t>(r) * B + k) * nkv + kvh) * kHd + d];
  }
  __syncthreads();
  for (int e = tid; e < kQ * kHd; e += 256) {
    const int qi = e / kHd, d = e % kHd;
    float o = 0.f;
#pragma unroll
    for (int k = 0; k < B; ++k) o = fmaf(sm.p[qi][k], sm.kv[k][d], o);
    out[qi * kPartStride + 2 + d] = o;
  }
}

// grid (R * nkv, n_chunks): part p < n_chunks - 1 takes context chunks
// p cpc .. p cpc + cpc - 1 (those that exist); the last part the B block keys.
// Three CTAs per SM at B = 8, two at B = 16 (the context chunk's shared memory).
template <int B>
__global__ void __launch_bounds__(256, B == 8 ? 3 : 2) attn_chunk_kernel(const AttnArgs a) {
  constexpr int kQ = 4 * B;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int nkv = a.n_kv_heads;
  const int r = blockIdx.x / nkv, kvh = blockIdx.x % nkv;
  const int part = blockIdx.y;
  const int nn = min(max(a.n_new[r], 0), B);
  const int L = min(max(a.ctx_len[r], 0), a.kv_capacity - nn) + nn;  // same clamping as the cache append
  const int lo0 = max(0, L - (a.window - 1));
  const int n_ctx_chunks = (L - lo0 + kKeys - 1) / kKeys;
  const int c0 = part * a.cpc, c1 = min(c0 + a.cpc, n_ctx_chunks);
  float* out = a.part + ((static_cast<size_t>(r) * nkv + kvh) * a.n_chunks + part) * kQ * kPartStride;
  if (part == a.n_chunks - 1) {
    pdl_begin();
    blk_chunk<B>(a, smem_raw, r, kvh, out);
  } else if (c0 < c1) {
    ctx_part<B>(a, smem_raw, r, kvh, lo0, c0, c1, L, nn, out);
  } else {
    pdl_begin();
    if (threadIdx.x < kQ) {  // no keys in this part
      out[threadIdx.x * kPartStride + 0] = -INFINITY;
      out[threadIdx.x * kPartStride + 1] = 0.f;
    }
  }
}

// One warp per (request, query head, block position, 128 / DW of the dimensions):
// merges the parts' partials in part order; lane holds dimensions
// (128 / DW) quarter + lane + 32 j.  DW = 4 spreads a request over more warps when
// there are few requests.
template <int B, int DW>
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnArgs a) {
  constexpr int kQ = 4 * B;
  constexpr int kJ = 4 / DW;  // dimensions per lane
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x;
  const int item = blockIdx.y * 8 + (threadIdx.x >> 5);  // (head * B + position) * DW + quarter
  if (item >= a.n_q_heads * B * DW) return;
  const int quarter = item % DW, h = item / (B * DW), i = (item / DW) % B;
  const int nkv = a.n_kv_heads;
  const int rep = a.n_q_heads / nkv;
  const int kvh = h / rep, hr = h % rep;
  const int qi = hr * B + i;
  const int d0 = quarter * (kHd / DW) + lane;
  const float* base = a.part + (static_cast<size_t>(r) * nkv + kvh) * a.n_chunks * kQ * kPartStride;
  // part statistics: lane c holds parts c and c + 32 (n_chunks <= 64)
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int c = lane + 32 * u;
    if (c < a.n_chunks) {
      const float* pc = base + (static_cast<size_t>(c) * kQ + qi) * kPartStride;
      l[u] = pc[1];
      if (l[u] > 0.f) m[u] = pc[0];
    }
  }
  const float M = warp_max(fmaxf(m[0], m[1]));
  float f[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) f[u] = (l[u] > 0.f) ? exp2f(m[u] - M) : 0.f;
  const float den = warp_sum(f[0] * l[0] + f[1] * l[1]);
  float o[kJ];
#pragma unroll
  for (int j = 0; j < kJ; ++j) o[j] = 0.f;
  constexpr int kP = 32 / kJ;  // parts whose loads are in flight together
  for (int c0 = 0; c0 < a.n_chunks; c0 += kP) {  // added in part order
    float fc[kP], t[kP][kJ];
#pragma unroll
    for (int u = 0; u < kP; ++u) {
      const int c = c0 + u;
      fc[u] = c < a.n_chunks ? __shfl_sync(0xffffffffu, f[(c >> 5) & 1], c & 31) : 0.f;
      const float* pc = base + (static_cast<size_t>(c) * kQ + qi) * kPartStride + 2 + d0;
#pragma unroll
      for (int j = 0; j < kJ; ++j) t[u][j] = fc[u] != 0.f ? pc[32 * j] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kP; ++u)
#pragma unroll
      for (int j = 0; j < kJ; ++j)
        if (fc[u] != 0.f) o[j] += fc[u] * t[u][j];
  }
  const int ld = a.n_q_heads * kHd;
#pragma unroll
  for (int j = 0; j < kJ; ++j) {
    const size_t idx = act_offset(r * B + i, h * kHd + d0 + 32 * j, ld, a.tiled_o);
    const float v = o[j] / den;
    if (a.fmt == 0) {
      __nv_bfloat16* p = reinterpret_cast<__nv_bfloat16*>(a.act_o);
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      p[idx] = hi;
      if (a.act_o_lo) p[a.act_o_lo + idx] = __float2bfloat16_rn(v - __bfloat162float(hi));
    } else {
      __half* p = reinterpret_cast<__half*>(a.act_o);
      const __half hi = __float2half_rn(v);
      p[idx] = hi;
      if (a.act_o_lo) p[a.act_o_lo + idx] = __float2half_rn(v - __half2float(hi));
    }
  }
}

template <int B>
cudaError_t launch_attention_b(const AttnArgs& a, int n_req, bool pdl, cudaStream_t st) {
  static std::atomic<unsigned long long> attr_done{0};
  const size_t smem = sizeof(CtxSmem<B>) > sizeof(BlkSmem<B>) ? sizeof(CtxSmem<B>) : sizeof(BlkSmem<B>);
  {
    const cudaError_t e = set_smem_once(attn_chunk_kernel<B>, static_cast<int>(smem), attr_done);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch_ex(attn_chunk_kernel<B>, dim3(n_req * a.n_kv_heads, a.n_chunks), dim3(256), smem, st, pdl, a);
  if (e != cudaSuccess) return e;
  if (n_req * B < 32)  // few block rows: four warps per (head, position), 32 dimensions each
    return launch_ex(attn_combine_kernel<B, 4>, dim3(n_req, (a.n_q_heads * B * 4 + 7) / 8), dim3(256), 0, st, pdl, a);
  return launch_ex(attn_combine_kernel<B, 1>, dim3(n_req, (a.n_q_heads * B + 7) / 8), dim3(256), 0, st, pdl, a);
}

}  // namespace

cudaError_t launch_attention(const AttnArgs& a, int n_req, bool pdl, cudaStream_t st) {
  if (a.B == 8) return launch_attention_b<8>(a, n_req, pdl, st);
  if (a.B == 16) return launch_attention_b<16>(a, n_req, pdl, st);
  return cudaErrorInvalidValue;
}

}  // namespace df2
