// Block attention of the drafter (step a5): B block queries per request (B = 8 or
// 16) attend, noncausally, to all B block keys and to the context keys inside the sliding
// window ("LSE docs/DFLASH2.md", block paragraph: noncausal within the block,
// context keys obey the 2048-position sliding window).  Query i sits at absolute
// position L + i (L = keys in the cache); it sees context key k iff
// L + i - k < window.  GQA: the 4 query heads of one KV head share its keys.
//
// Split over keys (flash-decoding style): one CTA per (request, KV head, part of
// cpc chunks of 64 context keys), plus one CTA for the B block keys; all 4 B queries
// of a KV head group (4 heads x B positions) are handled together so every key is
// read once.  A request narrowed to a block width w < B masks its block keys at
// positions >= w, so its first w rows are exactly a block-w forward.  Keys outside
// the window are never read.  Context chunks run on the tensor cores (mma.sync
// m16n8k16 in bf16, fp32 accumulators; fragments by ldmatrix): K and V are used as
// stored (bf16, exact), queries and probabilities as bf16 hi + lo pairs (two products
// each, ~2^-16 relative), and each warp keeps its scores, probabilities and running
// softmax in registers.  An earlier version converted every K/V chunk to fp16 so
// queries and probabilities could be single fp16 products; the conversion was most of
// its instructions.  The block part uses FFMA on the fp32 block keys.  A combine
// kernel merges the parts' (max, sum, unnormalised output) in a fixed order.
#include <math.h>

#include "common.cuh"
#include "glue.h"
#include "internal.h"

namespace df2 {

namespace {

constexpr int kHd = 128;
constexpr int kKeys = kAttnChunk;
constexpr int kPartStride = kHd + 2;
// Query and K/V tiles: rows of 128 bf16 (256 bytes, 16 pieces of 16 bytes), piece p of
// row r stored at p ^ (r mod 8): the eight rows of every 8 x 8 fragment load fall on
// distinct banks without padding.
DF2_DEV int swz_off(int r, int piece) { return r * 256 + ((piece ^ (r & 7)) << 4); }

// B block positions: kQ = 4 B queries per KV head group (4 heads x B positions),
// query qi = hr * B + i is head kvh * 4 + hr at block position i.
template <int B>
struct CtxSmem {
  static constexpr int kQ = 4 * B;
  // K/V buffers: three at B = 8 (112 KB: two CTAs per SM), two at B = 16
  static constexpr int kNB = B == 8 ? 3 : 2;
  uint16_t qh[kQ][kHd], ql[kQ][kHd];  // scaled queries, bf16 hi and lo parts (swizzled rows)
  union {
    struct {
      uint16_t k[kNB][kKeys][kHd];  // bf16 K and V of a chunk (swizzled rows)
      uint16_t v[kNB][kKeys][kHd];
    };
    struct {  // after the last chunk
      float so[kQ][kHd + 4];        // the merged output of the part
      float mw[8][16], lw[8][16];   // per warp: running maximum and sum of its 16 query rows
    };
  };
};

template <int B>
struct BlkSmem {
  static constexpr int kQ = 4 * B;
  float q[kQ][kHd];
  float kv[B][kHd + 1];
  float p[kQ][B];
};

// A fragment of mma m16n8k16 (rows 0..15 x K 0..15 of a 16-bit tile whose rows are 16-byte
// aligned): lane L supplies row (L mod 8) + 8 ((L / 8) mod 2), K offset 8 (L / 16), so
// the registers are {rows 0-7 K 0-7, rows 8-15 K 0-7, rows 0-7 K 8-15, rows 8-15 K 8-15}.
DF2_DEV void ldmatrix_a(uint32_t (&r)[4], const void* tile, int row0, int piece0, int lane) {
  const unsigned addr = static_cast<unsigned>(__cvta_generic_to_shared(tile)) +
                        swz_off(row0 + (lane & 7) + ((lane >> 3) & 1) * 8, piece0 + (lane >> 4));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// B fragment (K 0..15 x n 0..7) from a 16-bit tile stored n-major ([n][K], rows 16-byte
// aligned): lane L < 16 supplies row L mod 8, K offset 8 (L / 8).
DF2_DEV void ldmatrix_b(uint32_t& b0, uint32_t& b1, const void* tile, int row0, int piece0, int lane) {
  const unsigned addr =
      static_cast<unsigned>(__cvta_generic_to_shared(tile)) + swz_off(row0 + (lane & 7), piece0 + ((lane >> 3) & 1));
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(b0), "=r"(b1) : "r"(addr));
}

DF2_DEV void ldmatrix_x2_trans(uint32_t& r0, uint32_t& r1, const void* tile, int row, int piece) {
  const unsigned addr = static_cast<unsigned>(__cvta_generic_to_shared(tile)) + swz_off(row, piece);
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// 16-byte asynchronous copy global -> shared; bytes = 0 fills the 16 bytes with zeros.
DF2_DEV void cp_async16(void* smem_dst, const void* src, uint32_t bytes) {
  const unsigned dst = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}

// Two floats -> bf16x2 hi and lo parts (x = hi + lo to ~2^-16 relative).
DF2_DEV void split_bf16(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const float2 f = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x - f.x, y - f.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// ------------------------------------------------------------------ context chunk (tensor cores)
// The bf16 K/V rows of one chunk straight into buffer `buf` of the K/V tiles by
// asynchronous copies (cp.async, 16 bytes each; rows at or past nk are zero-filled).
template <int B>
DF2_DEV void stage_kv(const AttnArgs& a, CtxSmem<B>& sm, int buf, int r, int kvh, int k_begin, int nk) {
  const int tid = threadIdx.x, nkv = a.n_kv_heads;
  const uint16_t* kc = a.k_cache + (static_cast<size_t>(r) * a.kv_capacity + k_begin) * nkv * kHd + kvh * kHd;
  const uint16_t* vc = a.v_cache + (static_cast<size_t>(r) * a.kv_capacity + k_begin) * nkv * kHd + kvh * kHd;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = tid + 256 * j;
    const int k = e / (kHd / 8), d8 = (e % (kHd / 8)) * 8;
    const int kk = k < nk ? k : 0;  // a valid address; the copy reads nothing then
    const uint32_t bytes = k < nk ? 16u : 0u;
    const int off = swz_off(k, d8 / 8);
    cp_async16(reinterpret_cast<unsigned char*>(&sm.k[buf][0][0]) + off, kc + static_cast<size_t>(kk) * nkv * kHd + d8,
               bytes);
    cp_async16(reinterpret_cast<unsigned char*>(&sm.v[buf][0][0]) + off, vc + static_cast<size_t>(kk) * nkv * kHd + d8,
               bytes);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Context chunks c0 .. c1 - 1 of one (request, KV head), 64 keys each.  Warp w takes
// query tile w / WPM (16 queries) and keys (w mod WPM) KW .. + KW - 1 of every chunk
// (WPM = 8 / query tiles warps share a tile, KW = 64 / WPM keys each), and keeps its
// scores, probabilities and running softmax in registers: per query row the running
// maximum m and sum l (over the lanes of a quad) and the unnormalised output O
// (16 x 128, rescaled by 2^(m_old - m_new) when the maximum grows); the score
// accumulators become the probability operand of the next product.  K and V stay
// bf16 (exact); queries and probabilities enter the products as bf16 hi + lo pairs
// (two products each, ~2^-16 relative).  The chunks' K/V tiles are triple-buffered
// at B = 8 (the copies of the next two chunks run while a chunk is computed; 112 KB,
// two CTAs per SM with unpadded, swizzled rows) and double-buffered at B = 16; one
// barrier per chunk.  At
// the end the WPM warps of a query tile merge their (m, l, O) in warp order through
// shared memory and the part's (m, l, O) is written.
template <int B>
DF2_DEV void ctx_part(const AttnArgs& a, unsigned char* smem_raw, int r, int kvh, int lo0, int c0, int c1, int L,
                      int nn, float* out) {
  constexpr int kQ = 4 * B, kMT = kQ / 16;
  constexpr int WPM = 8 / kMT, KW = kKeys / WPM, NTW = KW / 8, KSP = KW / 16;
  CtxSmem<B>& sm = *reinterpret_cast<CtxSmem<B>*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int mt = wid / WPM, wp = wid % WPM;
  const int rep = a.n_q_heads / a.n_kv_heads;
  const float qscale = rsqrtf(static_cast<float>(kHd)) * 1.4426950408889634f;  // log2(e)/sqrt(hd)
  auto kbeg = [&](int c) { return lo0 + c * kKeys; };
  auto nkeys = [&](int c) { return min(kKeys, L - kbeg(c)); };
  const bool early = kbeg(c0) + nkeys(c0) <= L - nn;  // rows L - nn .. L - 1 are appended by the previous kernel
  if (early) stage_kv<B>(a, sm, 0, r, kvh, kbeg(c0), nkeys(c0));
  pdl_wait();
  pdl_trigger();
  if (!early) stage_kv<B>(a, sm, 0, r, kvh, kbeg(c0), nkeys(c0));
  constexpr int NB = CtxSmem<B>::kNB;
  for (int j = 1; j < NB - 1; ++j) {  // the first NB - 1 chunks in flight (one group each, empty past the part)
    if (c0 + j < c1)
      stage_kv<B>(a, sm, j, r, kvh, kbeg(c0 + j), nkeys(c0 + j));
    else
      asm volatile("cp.async.commit_group;" ::: "memory");
  }
  // queries -> bf16 hi + lo (qi = hr * B + i: head kvh*rep + hr, block row r*B + i)
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
    const float x = qv[j] * qscale;
    const __nv_bfloat16 hi = __float2bfloat16_rn(x), lo = __float2bfloat16_rn(x - __bfloat162float(hi));
    const int qi = e / kHd, d = e % kHd;
    const int off = swz_off(qi, d >> 3) / 2 + (d & 7);  // in bf16 elements
    (&sm.qh[0][0])[off] = *reinterpret_cast<const uint16_t*>(&hi);
    (&sm.ql[0][0])[off] = *reinterpret_cast<const uint16_t*>(&lo);
  }
  const int qi0 = mt * 16 + g, qi1 = qi0 + 8;  // this lane's two query rows
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[kHd / 8][4];
#pragma unroll
  for (int dt = 0; dt < kHd / 8; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
  for (int c = c0; c < c1; ++c) {
    const int buf = (c - c0) % NB;
    const int k_begin = kbeg(c), nk = nkeys(c);
    // this chunk's group has completed (NB - 2 later groups may still be in flight)
    if (NB == 3)
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    else
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    // every thread's copies of this chunk have landed, every warp is done with the
    // buffer of the previous chunk, and the queries are in place
    __syncthreads();
    if (c + NB - 1 < c1)  // in flight during the next NB - 1 chunks
      stage_kv<B>(a, sm, (buf + NB - 1) % NB, r, kvh, kbeg(c + NB - 1), nkeys(c + NB - 1));
    else
      asm volatile("cp.async.commit_group;" ::: "memory");
    // S = Q K^T for the warp's 16 queries x KW keys
    float s[NTW][4];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < kHd / 16; ++ks) {
      uint32_t ah[4], al[4];
      ldmatrix_a(ah, &sm.qh[0][0], mt * 16, ks * 2, lane);
      ldmatrix_a(al, &sm.ql[0][0], mt * 16, ks * 2, lane);
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) {
        uint32_t b0, b1;
        ldmatrix_b(b0, b1, &sm.k[buf][0][0], wp * KW + nt * 8, ks * 2, lane);
        mma_bf16(s[nt], ah[0], ah[1], ah[2], ah[3], b0, b1);
        mma_bf16(s[nt], al[0], al[1], al[2], al[3], b0, b1);
      }
    }
    // window and chunk-end masks; row maxima over the quad's lanes
    const int lim = L - (a.window - 1) - k_begin;  // query i sees chunk key k iff k >= lim + i
    const int p0 = qi0 % B, p1 = qi1 % B;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int k = wp * KW + nt * 8 + 2 * q + e;
        if (!(k < nk && k >= lim + p0)) s[nt][e] = -INFINITY;
        if (!(k < nk && k >= lim + p1)) s[nt][2 + e] = -INFINITY;
        mx0 = fmaxf(mx0, s[nt][e]);
        mx1 = fmaxf(mx1, s[nt][2 + e]);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const bool none0 = mn0 == -INFINITY, none1 = mn1 == -INFINITY;  // no visible key yet
    const float al0 = none0 ? 1.f : exp2f(m0 - mn0), al1 = none1 ? 1.f : exp2f(m1 - mn1);
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        s[nt][e] = none0 ? 0.f : exp2f(s[nt][e] - mn0);
        s[nt][2 + e] = none1 ? 0.f : exp2f(s[nt][2 + e] - mn1);
        ps0 += s[nt][e];
        ps1 += s[nt][2 + e];
      }
    }
    ps0 += __shfl_xor_sync(0xffffffffu, ps0, 1);
    ps0 += __shfl_xor_sync(0xffffffffu, ps0, 2);
    ps1 += __shfl_xor_sync(0xffffffffu, ps1, 1);
    ps1 += __shfl_xor_sync(0xffffffffu, ps1, 2);
    l0 = l0 * al0 + ps0;
    l1 = l1 * al1 + ps1;
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int dt = 0; dt < kHd / 8; ++dt) {
      o[dt][0] *= al0;
      o[dt][1] *= al0;
      o[dt][2] *= al1;
      o[dt][3] *= al1;
    }
    // O += P V: the probabilities of key tiles 2j, 2j + 1 (bf16 hi + lo) are the A
    // fragments of the j-th 16 keys
#pragma unroll
    for (int j = 0; j < KSP; ++j) {
      uint32_t ph[4], pl[4];
      split_bf16(s[2 * j][0], s[2 * j][1], ph[0], pl[0]);
      split_bf16(s[2 * j][2], s[2 * j][3], ph[1], pl[1]);
      split_bf16(s[2 * j + 1][0], s[2 * j + 1][1], ph[2], pl[2]);
      split_bf16(s[2 * j + 1][2], s[2 * j + 1][3], ph[3], pl[3]);
#pragma unroll
      for (int dt = 0; dt < kHd / 8; ++dt) {
        uint32_t b0, b1;
        ldmatrix_x2_trans(b0, b1, &sm.v[buf][0][0], wp * KW + j * 16 + (lane & 15), dt);
        mma_bf16(o[dt], ph[0], ph[1], ph[2], ph[3], b0, b1);
        mma_bf16(o[dt], pl[0], pl[1], pl[2], pl[3], b0, b1);
      }
    }
  }
  __syncthreads();  // every warp is done with the K/V tiles: the merge area overlays them
  // merge the WPM warps of each query tile, in warp order
  if (q == 0) {
    sm.mw[wid][g] = m0;
    sm.mw[wid][g + 8] = m1;
    sm.lw[wid][g] = l0;
    sm.lw[wid][g + 8] = l1;
  }
  __syncthreads();
  float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
  for (int u = 0; u < WPM; ++u) {
    M0 = fmaxf(M0, sm.mw[mt * WPM + u][g]);
    M1 = fmaxf(M1, sm.mw[mt * WPM + u][g + 8]);
  }
  const float f0 = (m0 == -INFINITY) ? 0.f : exp2f(m0 - M0), f1 = (m1 == -INFINITY) ? 0.f : exp2f(m1 - M1);
  float(*so)[kHd + 4] = sm.so;  // overlays the K/V tiles, free now
#pragma unroll
  for (int u = 0; u < WPM; ++u) {
    if (wp == u) {
#pragma unroll
      for (int dt = 0; dt < kHd / 8; ++dt) {
        const int d = dt * 8 + 2 * q;
        if (u == 0) {
          so[qi0][d] = o[dt][0] * f0;
          so[qi0][d + 1] = o[dt][1] * f0;
          so[qi1][d] = o[dt][2] * f1;
          so[qi1][d + 1] = o[dt][3] * f1;
        } else {
          so[qi0][d] += o[dt][0] * f0;
          so[qi0][d + 1] += o[dt][1] * f0;
          so[qi1][d] += o[dt][2] * f1;
          so[qi1][d + 1] += o[dt][3] * f1;
        }
      }
      if (u == 0 && q == 0) {
        float L0 = 0.f, L1 = 0.f;
        for (int v = 0; v < WPM; ++v) {
          const float mv0 = sm.mw[mt * WPM + v][g], mv1 = sm.mw[mt * WPM + v][g + 8];
          if (mv0 > -INFINITY) L0 += sm.lw[mt * WPM + v][g] * exp2f(mv0 - M0);
          if (mv1 > -INFINITY) L1 += sm.lw[mt * WPM + v][g + 8] * exp2f(mv1 - M1);
        }
        out[qi0 * kPartStride + 0] = M0;
        out[qi0 * kPartStride + 1] = L0;
        out[qi1 * kPartStride + 0] = M1;
        out[qi1 * kPartStride + 1] = L1;
      }
    }
    __syncthreads();
  }
  for (int e = tid; e < kQ * kHd; e += 256) {
    const int qi = e / kHd, d = e % kHd;
    out[qi * kPartStride + 2 + d] = so[qi][d];
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
// Two CTAs per SM (the context part's registers: a 16 x 128 output tile per warp).
template <int B>
__global__ void __launch_bounds__(256, 2) attn_chunk_kernel(const AttnArgs a) {
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
