// Element-wise stages between the weight-streaming projections: block embedding
// and taps packing (start), the taps-projection norm input (fc_finish), the
// dynamic convolution before a sublayer (conv_in) and after it with the residual
// add (conv_out), SwiGLU, and q/k norm + RoPE + context cache append after the QKV
// projection (qkv_finish).  Each consumer adds the producer GEMV's split planes in
// split order.
//
// RMSNorm is deferred: producers write x * w and per-chunk sums of squares, and
// the consumer applies 1/rms (the scale commutes with the projections).
//
// A CTA takes one tile of 8 rows (warp i = row i of the tile).  Rows are request-
// major, B block positions per request (8 or 16): row n is position n % B of
// request n / B, so a block of 16 spans two tiles and the convolutions read the
// row before a tile's first from global memory when it belongs to the same block.  Row
// statistics cross CTAs only through those partial sums, read in a fixed order
// (bit-reproducible).
#include "common.cuh"
#include "elementwise.cuh"
#include "glue.h"
#include "internal.h"

namespace df2 {

namespace {

using namespace ew;

constexpr int kB = 8;       // rows per tile (one CTA of the channel kernels)
constexpr int kCw = 32;     // channels per CTA of the channel kernels: warp i = tile row i, lane = channel
constexpr int kThreads = kB * kCw;

// Sum of the split planes p[s * plane], s = 0..S-1, added in split order.  The
// loads of up to B planes are issued together so their latency is paid once.
template <int B>
DF2_DEV float plane_sum_b(const float* p, size_t plane, int S) {
  float y = 0.f;
  for (int s0 = 0; s0 < S; s0 += B) {
    float t[B];
#pragma unroll
    for (int j = 0; j < B; ++j) t[j] = (s0 + j < S) ? p[static_cast<size_t>(s0 + j) * plane] : 0.f;
#pragma unroll
    for (int j = 0; j < B; ++j) y += t[j];
  }
  return y;
}

DF2_DEV float plane_sum(const float* p, size_t plane, int S) {
  return S <= 8 ? plane_sum_b<8>(p, plane, S) : plane_sum_b<32>(p, plane, S);
}

// Per-row sum of squares of this CTA's 32 channels -> ss[row][blockIdx.y] (one warp = one row).
DF2_DEV void emit_ss(float v, int row, float* ss, int nch) {
  const float s = warp_sum(v * v);
  if ((threadIdx.x & 31) == 0) ss[static_cast<size_t>(row) * nch + blockIdx.y] = s;
}

// The channel kernels after the projections take 4 channels per thread, 128 per CTA
// (one row per warp), with 16-byte loads and 8-byte stores: at many requests these
// kernels are bound by instruction issue, not by their bytes.
constexpr int kV = 4;
constexpr int kCv = kCw * kV;

// V = 2 or 4 consecutive values (16- or 8-byte aligned).
template <int V>
DF2_DEV void ld_f32v(const float* p, float (&v)[V]) {
  if constexpr (V == 4) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
  } else {
    const float2 t = *reinterpret_cast<const float2*>(p);
    v[0] = t.x, v[1] = t.y;
  }
}
template <int V>
DF2_DEV void st_f32v(float* p, const float (&v)[V]) {
  if constexpr (V == 4)
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  else
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
}
template <int V>
DF2_DEV void ld_bf16v(const uint16_t* p, float (&v)[V]) {
  if constexpr (V == 4) {
    const float4 t = ld_bf16x4(p);
    v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    v[0] = __uint_as_float(u << 16), v[1] = __uint_as_float(u & 0xFFFF0000u);
  }
}
template <int V>
DF2_DEV void put_actv(void* act, size_t lo, int fmt, size_t idx, const float (&v)[V]) {
  if constexpr (V == 4) {
    put_act4(act, lo, fmt, idx, make_float4(v[0], v[1], v[2], v[3]));
  } else {
    put_act(act, lo, fmt, idx, v[0]);
    put_act(act, lo, fmt, idx + 1, v[1]);
  }
}

// ------------------------------------------------------------------ start of the step
// blockIdx.y < H/32: block embedding, first norm input and its sums of squares;
// above: taps of the new context rows packed into the fc projection's input.
// It reads caller inputs (ids, lengths, taps) that the previous kernel may have
// written (the serving loop's state update, or the caller's own kernel), so it waits
// for that kernel first; its successor, the taps projection, starts its weight copies
// meanwhile.
__global__ void __launch_bounds__(kThreads) start_kernel(const StartArgs a) {
  pdl_begin_early();
  // a new step: the previous step's select has read the error word by now (it ran
  // before the previous verify, whose completion the wait above implies)
  if (a.pipe_err != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *a.pipe_err = 0;
  const int i = threadIdx.x >> 5;
  const int row = blockIdx.x * kB + i;
  const int r = row / a.B, pos = row % a.B;
  const int ny = a.H / kCw;
  if (static_cast<int>(blockIdx.y) < ny) {
    const int c = blockIdx.y * kCw + (threadIdx.x & 31);
    const int anchor = min(max(a.anchor_ids[r], 0), a.V - 1);  // ids are clamped into the table
    const int id = (pos == 0) ? anchor : a.mask_id;
    const float xv = bf16_to_f32(a.embed[static_cast<size_t>(id) * a.H + c]);
    const size_t idx = static_cast<size_t>(row) * a.H + c;
    a.x[idx] = xv;
    put_act(a.act_a, a.act_a_lo, a.fmt, act_offset(row, c, a.H, a.tiled_a), xv * bf16_to_f32(a.norm_w[c]));
    emit_ss(xv, row, a.ss_x, a.nch);
  } else {
    const int c = (blockIdx.y - ny) * kCw + (threadIdx.x & 31);
    const int nn = min(max(a.n_new[r], 0), a.B);  // rows >= n_new are zero
    const size_t idx = static_cast<size_t>(row) * (a.n_taps * a.H) + c;
    put_act(a.act_taps, a.act_taps_lo, a.fmt, act_offset(row, c, a.n_taps * a.H, a.tiled_taps),
            (pos < nn) ? a.taps[idx] : 0.f);
  }
}

// ------------------------------------------------------------------ taps projection finish
// c = y * w_hidden_norm into the context rows of the QKV input (1/rms of y is
// applied after the K/V projection); ss of y.
DF2_DEV void fc_finish_body(const FcFinishArgs& a) {
  __shared__ int np_sh[2];
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kB + (threadIdx.x >> 5);
  const int c = blockIdx.y * kCv + kV * lane;
  if (threadIdx.x < 2) np_sh[threadIdx.x] = gemv_plane_count(a.pl, blockIdx.y * kCv + 64 * threadIdx.x);
  __syncthreads();
  const float4 w = ld_bf16x4(a.norm_w + c);
  const float4 y =
      plane_sum4(a.y + static_cast<size_t>(row) * a.H + c, static_cast<size_t>(a.n_rows) * a.H, np_sh[lane >> 4]);
  put_act4(a.act, a.act_lo, a.fmt, act_offset(a.act_row0 + row, c, a.H, a.tiled), mul4(y, w));
  emit_ss4(y, row, a.ss, a.nch, c);
}

// ------------------------------------------------------------------ conv before a sublayer
// r_i = 1/rms(x_i); delta = r_i * (W_delta (x_i * w)) for all four (io, tap) rows;
// a_i = r_i x_i w;  a'_i = (b0 + d0_i) a_i + (b1 + d1_i) a_{i-1}.
// 32 V channels per CTA (V per thread): a row's 8 V dynamic coefficients of the CTA's
// 2 V groups are summed over their split planes by 4 / V lanes each (planes split by
// residue), so with few block rows (V = 2, about 15 planes a coefficient at one
// request) one round of plane loads suffices, and with many (V = 4) the kernel issues
// a quarter of the one-channel kernel's instructions.
template <int V>
DF2_DEV void conv_in_body(const ConvInArgs& a) {
  constexpr int kCta = kCw * V;     // channels per CTA
  constexpr int kVals = 8 * V;      // coefficients per row: (io, tap) x local group
  constexpr int kSplit = 32 / kVals;  // lanes per coefficient
  __shared__ __align__(16) float ash[kB][kCta];
  __shared__ int np_sh[4];
  const int i = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kB + i;
  const int c = blockIdx.y * kCta + V * lane;
  const int G = a.H / 16;
  // plane counts of the (io, tap) rows of the CTA's groups (2 V consecutive rows each,
  // inside one weight block), once per CTA
  if (threadIdx.x < 4) np_sh[threadIdx.x] = gemv_plane_count(a.pl, threadIdx.x * G + blockIdx.y * 2 * V);
  __syncthreads();
  // loads independent of the planes and of 1/rms first: one round of latency
  const size_t idx = static_cast<size_t>(row) * a.H + c;
  float x0[V], w[V], b0[V], b1[V];
  ld_f32v<V>(a.x + idx, x0);
  ld_bf16v<V>(a.norm_w + c, w);
  ld_bf16v<V>(a.base + c, b0);
  ld_bf16v<V>(a.base + a.H + c, b1);
  float dv, rr;
  {
    const int e = lane % kVals, part_id = lane / kVals;
    const int it = e / (2 * V), gl = e % (2 * V);
    const int gidx = it * G + blockIdx.y * 2 * V + gl;
    const size_t plane = static_cast<size_t>(a.n_rows) * (4 * G);
    const float* p = a.dproj + static_cast<size_t>(row) * (4 * G) + gidx;
    const int np = np_sh[it];
    float part = 0.f;
    for (int s0 = part_id; s0 < np; s0 += 16 * kSplit) {  // 16 planes' loads in flight, added in order
      float t[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        t[j] = (s0 + kSplit * j < np) ? p[static_cast<size_t>(s0 + kSplit * j) * plane] : 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) part += t[j];
    }
#pragma unroll
    for (int o = kVals; o < 32; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    rr = warp_inv_rms(a.ss, row, a.nch, a.H, a.eps);
    dv = part * rr;
    if (part_id == 0) a.delta[static_cast<size_t>(row) * (4 * G) + gidx] = dv;
  }
  const int gl = (V * lane) >> 4;  // local group of this lane's channels
  const float d0 = __shfl_sync(0xffffffffu, dv, gl), d1 = __shfl_sync(0xffffffffu, dv, 2 * V + gl);
  float ai[V];
#pragma unroll
  for (int k = 0; k < V; ++k) ai[k] = x0[k] * rr * w[k];
  st_f32v<V>(&ash[i][V * lane], ai);
  // a tile that starts inside a block (B = 16): its first row's predecessor, from global
  float prev0[V];
#pragma unroll
  for (int k = 0; k < V; ++k) prev0[k] = 0.f;
  if (i == 0 && row % a.B != 0) {
    const float rp = warp_inv_rms(a.ss, row - 1, a.nch, a.H, a.eps);
    float xp[V];
    ld_f32v<V>(a.x + idx - a.H, xp);
#pragma unroll
    for (int k = 0; k < V; ++k) prev0[k] = xp[k] * rp * w[k];
  }
  __syncthreads();
  float prev[V], o[V];
  if (i > 0) ld_f32v<V>(&ash[i - 1][V * lane], prev);
#pragma unroll
  for (int k = 0; k < V; ++k) {
    if (i == 0) prev[k] = prev0[k];
    o[k] = (b0[k] + d0) * ai[k] + (b1[k] + d1) * prev[k];
  }
  put_actv<V>(a.act, a.act_lo, a.fmt, act_offset(row, c, a.H, a.tiled), o);
}

template <int V>
__global__ void __launch_bounds__(kThreads) conv_in_kernel(const ConvInArgs a) {
  pdl_begin_early();  // followed by a weight launch
  conv_in_body<V>(a);
}

// First layer: the taps-projection finish and the conv before the attention
// sublayer read different inputs and write different outputs, so they share one
// launch (blockIdx.z selects the role; the grid is the conv's, 32 V channels per
// CTA, of which the finish's 128-channel CTAs take the first H / 128).
template <int V>
__global__ void __launch_bounds__(kThreads) fc_finish_conv_in_kernel(const FcFinishArgs f, const ConvInArgs c) {
  pdl_begin_early();  // followed by a weight launch
  if (blockIdx.z == 0) {
    if (static_cast<int>(blockIdx.y) < f.H / kCv) fc_finish_body(f);
  } else {
    conv_in_body<V>(c);
  }
}

// ------------------------------------------------------------------ conv after a sublayer + residual
// y = sum of split planes; x_i += (b2 + d2_i) y_i + (b3 + d3_i) y_{i-1} (the
// convolution wrapping the sublayer's output); act = x * w_next; ss of x.
__global__ void __launch_bounds__(kThreads) conv_out_kernel(const ConvOutArgs a) {
  __shared__ float4 ysh[kB][kCw];
  __shared__ int np_sh[2];
  if (threadIdx.x < 2) np_sh[threadIdx.x] = gemv_plane_count(a.pl, blockIdx.y * kCv + 64 * threadIdx.x);  // shapes only
  __syncthreads();
  pdl_begin_early();  // followed by a weight launch
  const int i = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kB + i;
  const int c = blockIdx.y * kCv + kV * lane;
  const int G = a.H / 16;
  const int g = c >> 4;
  const size_t idx = static_cast<size_t>(row) * a.H + c;
  // every load independent of the planes is issued first: one round of latency
  const float* d = a.delta + static_cast<size_t>(row) * (4 * G);
  const float d2 = d[2 * G + g], d3 = d[3 * G + g];
  const float4 b2 = ld_bf16x4(a.base + 2 * a.H + c), b3 = ld_bf16x4(a.base + 3 * a.H + c);
  const float4 x0 = ld4(a.x + idx);
  const float4 w = ld_bf16x4(a.norm_w + c);
  const size_t plane = static_cast<size_t>(a.n_rows) * a.H;
  const int np = np_sh[lane >> 4];
  const float4 y = plane_sum4(a.part + idx, plane, np);
  ysh[i][lane] = y;
  // a tile that starts inside a block (B = 16): its first row's predecessor, from global
  float4 yp0 = make_float4(0.f, 0.f, 0.f, 0.f);
  if (i == 0 && row % a.B != 0) yp0 = plane_sum4(a.part + idx - a.H, plane, np);
  __syncthreads();
  const float4 yp = i > 0 ? ysh[i - 1][lane] : yp0;
  const float4 xv = conv_out4(x0, y, yp, b2, b3, d2, d3);
  *reinterpret_cast<float4*>(a.x + idx) = xv;
  const float4 act = mul4(xv, w);
  put_act4(a.act, a.act_lo, a.fmt, act_offset(row, c, a.H, a.tiled), act);
  if (a.act2 != nullptr) put_act4(a.act2, a.act2_lo, 0, act_offset(row, c, a.H, a.tiled2), act);
  emit_ss4(xv, row, a.ss, a.nch, c);
}

// ------------------------------------------------------------------ SwiGLU
// h = silu(gate) * up from the split planes of the two projections.
__global__ void __launch_bounds__(kThreads) swiglu_kernel(const SwigluArgs a) {
  __shared__ int np_sh[4];
  if (threadIdx.x < 4)  // before the wait: shapes only (gate, up) x (channel halves: 64-row GEMV blocks)
    np_sh[threadIdx.x] = gemv_plane_count(threadIdx.x < 2 ? a.pg : a.pu, blockIdx.y * kCv + 64 * (threadIdx.x & 1));
  __syncthreads();
  pdl_begin_early();  // followed by a weight launch
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kB + (threadIdx.x >> 5);
  const int c = blockIdx.y * kCv + kV * lane;
  const size_t idx = static_cast<size_t>(row) * a.F + c;
  const size_t plane = static_cast<size_t>(a.n_rows) * a.F;
  // the gate and up planes' loads all in flight together, each added in split order
  const int ng = np_sh[lane >> 4], nu = np_sh[2 + (lane >> 4)];
  float4 gs = make_float4(0.f, 0.f, 0.f, 0.f), us = gs;
  for (int s0 = 0; s0 < (ng > nu ? ng : nu); s0 += 4) {
    float4 tg[4], tu[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      tg[j] = (s0 + j < ng) ? ld4(a.part_g + idx + static_cast<size_t>(s0 + j) * plane) : make_float4(0.f, 0.f, 0.f, 0.f);
      tu[j] = (s0 + j < nu) ? ld4(a.part_u + idx + static_cast<size_t>(s0 + j) * plane) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      gs = add4(gs, tg[j]);
      us = add4(us, tu[j]);
    }
  }
  put_act4(a.act, a.act_lo, a.fmt, act_offset(row, c, a.F, a.tiled), swiglu4(gs, us));
}

// ------------------------------------------------------------------ q/k norm, RoPE, cache append
// One warp per (row, head); lane holds dims lane + 32 c (c = 0..3), so the NEOX
// pair (d, d + 64) is (c, c + 2) of the same lane.  Items per request: B query rows
// x nq heads, then 2 B key rows (B block + B context) x nkv, then 2 B value rows x nkv.
// The eight items of a CTA are consecutive heads of one row whenever the head counts
// allow (the usual case), so the rotation angles (FP64 reduction, the costly part on
// a part with few FP64 units) are computed once per CTA into shared memory; a CTA
// whose items sit at different positions computes them per lane, the same way.

// cos and sin of position pos x inverse frequency f: the angle in FP64, reduced by 2 pi
// in FP64 (Cody-Waite, with 2 pi split into a double and its remainder); only the
// reduced angle in [-pi, pi] goes through single-precision sincos.
DF2_DEV void rope_angle(int pos, double f, float& sn, float& cs) {
  const double ang = static_cast<double>(pos) * f;
  const double turns = rint(ang * 0.15915494309189535);  // 1 / (2 pi)
  const double red = fma(-turns, 6.283185307179586, ang) - turns * 2.4492935982947064e-16;
  sincosf(static_cast<float>(red), &sn, &cs);
}

__global__ void __launch_bounds__(256) qkv_finish_kernel(const QkvFinishArgs a) {
  __shared__ int pos_sh[8];
  __shared__ float sn_sh[64], cs_sh[64];
  pdl_begin();
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int item = blockIdx.y * 8 + wid;
  const int nq = a.n_q_heads, nkv = a.n_kv_heads, B = a.B;
  const int n_items = B * nq + 2 * 2 * B * nkv;
  // lengths are clamped so a bad length can never address outside the cache
  const int nn = min(max(a.n_new[r], 0), B);
  const int ctx = min(max(a.ctx_len[r], 0), a.kv_capacity - nn);
  const int L = ctx + nn;
  int kind = 2, j = 0, hh = 0;
  if (item < B * nq) {
    kind = 0;
    j = item / nq;
    hh = item % nq;
  } else if (item < n_items) {
    const int e = item - B * nq;
    kind = 1 + e / (2 * B * nkv);
    const int e2 = e % (2 * B * nkv);
    j = e2 / nkv;
    hh = e2 % nkv;
  }
  const bool ctx_row = j >= B;
  const int jj = ctx_row ? j - B : j;
  const bool valid = item < n_items && !(ctx_row && jj >= nn);
  const int pos = ctx_row ? ctx + jj : L + jj;
  // the CTA's rotated positions: one shared angle table when they agree
  if (lane == 0) pos_sh[wid] = (valid && kind != 2) ? pos : -1;
  __syncthreads();
  int upos = -1;
  bool uniform = true;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const int p = pos_sh[w];
    if (p >= 0) {
      if (upos < 0) upos = p;
      else if (p != upos) uniform = false;
    }
  }
  uniform = uniform && upos >= 0;
  if (uniform && threadIdx.x < 64) rope_angle(upos, a.inv_freq[threadIdx.x], sn_sh[threadIdx.x], cs_sh[threadIdx.x]);
  __syncthreads();
  if (!valid) return;
  const int row0 = r * B;
  const float* src;
  size_t plane;
  const GemvPlanes& pm = kind == 0 ? a.pq : (kind == 1 ? a.pk : a.pv);
  if (kind == 0) {
    src = a.q_out + (static_cast<size_t>(row0 + jj) * nq + hh) * 128;
    plane = static_cast<size_t>(a.n_rows) * nq * 128;
  } else {
    const size_t prow = ctx_row ? static_cast<size_t>(a.n_rows) + row0 + jj : static_cast<size_t>(row0 + jj);
    src = (kind == 1 ? a.k_out : a.v_out) + (prow * nkv + hh) * 128;
    plane = static_cast<size_t>(2 * a.n_rows) * nkv * 128;
  }
  // dims lane + 32 c: c = 0, 1 in the head's first 64-row block, c = 2, 3 in its second
  const int np0 = gemv_plane_count(pm, hh * 128), np1 = gemv_plane_count(pm, hh * 128 + 64);
  const int npx = np0 > np1 ? np0 : np1;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  for (int s0 = 0; s0 < npx; s0 += 8) {  // planes in order, 8 planes' loads in flight
    float t[8][4];
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        t[u][c] = (s0 + u < (c < 2 ? np0 : np1)) ? src[(s0 + u) * plane + lane + 32 * c] : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int c = 0; c < 4; ++c) v[c] += t[u][c];
  }
  if (ctx_row) {
    const float rc = warp_inv_rms(a.ss_c, row0 + jj, a.nch, a.H, a.eps);
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] *= rc;
  }
  if (kind != 2) {
    const uint16_t* nw = kind == 0 ? a.q_norm : a.k_norm;
    const float ms = warp_sum(v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3]) / 128.f;
    const float rs = rsqrtf(ms + a.eps);
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] = v[c] * rs * bf16_to_f32(nw[lane + 32 * c]);
    // NEOX: out[j] = x[j] cos - x[j+64] sin; out[j+64] = x[j+64] cos + x[j] sin
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float sn, cs;
      if (uniform) {
        sn = sn_sh[lane + 32 * c];
        cs = cs_sh[lane + 32 * c];
      } else {
        rope_angle(pos, a.inv_freq[lane + 32 * c], sn, cs);
      }
      const float x1 = v[c], x2 = v[c + 2];
      v[c] = x1 * cs - x2 * sn;
      v[c + 2] = x2 * cs + x1 * sn;
    }
  }
  if (!ctx_row) {
    float* dst = kind == 0 ? a.q : (kind == 1 ? a.kb : a.vb);
    const int nh = kind == 0 ? nq : nkv;
#pragma unroll
    for (int c = 0; c < 4; ++c) dst[(static_cast<size_t>(row0 + jj) * nh + hh) * 128 + lane + 32 * c] = v[c];
  } else {
    uint16_t* cache = kind == 1 ? a.k_cache : a.v_cache;
    const size_t base = ((static_cast<size_t>(r) * a.kv_capacity + pos) * nkv + hh) * 128;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const __nv_bfloat16 b = __float2bfloat16_rn(v[c]);
      cache[base + lane + 32 * c] = *reinterpret_cast<const uint16_t*>(&b);
    }
  }
}

// ------------------------------------------------------------------ serving-loop state update
// One thread per request: the rows appended this step become context, the last
// emitted token the next anchor, the emitted tokens the next new rows.
__global__ void __launch_bounds__(32) advance_kernel(const AdvanceArgs a, int n_req) {
  pdl_begin();
  const int r = blockIdx.x * 32 + threadIdx.x;
  if (r >= n_req) return;
  const int ne = min(max(a.n_emitted[r], 0), a.B);
  a.ctx_len[r] += min(max(a.n_new[r], 0), a.B);
  if (ne > 0) a.anchor_ids[r] = a.emitted[r * a.B + ne - 1];
  a.n_new[r] = ne;
  a.offset[r] += 1;
}

// ------------------------------------------------------------------ block width by context length
// The long-context narrowing of "qwen35: DSpark speculative decoding ... #625" (its
// long-context commits): verify cost grows with the block's rows times the context, so
// a request whose context passes a threshold drafts and verifies a narrower block.
// The rule reads the context length only.  One thread per request; the lengths may
// come from the previous kernel (the loop's state update), so it waits for it.
__global__ void __launch_bounds__(32) block_width_kernel(const BlockWidthArgs a, int n_req) {
  pdl_begin();
  const int r = blockIdx.x * 32 + threadIdx.x;
  if (r >= n_req) return;
  const long long L = static_cast<long long>(max(a.ctx_len[r], 0)) + max(a.n_new[r], 0);
  a.width[r] = (a.threshold > 0 && L > a.threshold) ? a.narrow : a.B;
}

}  // namespace

// Channels per thread of the conv-in: 2 with few block rows (one round of coefficient
// plane loads; measured 18 us a step faster at one request), 4 with many (fewer
// instructions; 34 us faster at 16 requests).
int conv_in_v(int n_rows) { return n_rows >= 32 ? 4 : 2; }

cudaError_t launch_block_width(const BlockWidthArgs& a, int n_req, bool pdl, cudaStream_t st) {
  if ((a.B != 8 && a.B != 16) || a.narrow < 2 || a.narrow > a.B) return cudaErrorInvalidValue;
  return launch_ex(block_width_kernel, dim3((n_req + 31) / 32), dim3(32), 0, st, pdl, a, n_req);
}

cudaError_t launch_advance(const AdvanceArgs& a, int n_req, bool pdl, cudaStream_t st) {
  if (a.B != 8 && a.B != 16) return cudaErrorInvalidValue;
  return launch_ex(advance_kernel, dim3((n_req + 31) / 32), dim3(32), 0, st, pdl, a, n_req);
}

// The channel kernels' grids: one CTA per (8-row tile, 32-channel chunk); n_rows =
// B n_req is a multiple of 8.
cudaError_t launch_start(const StartArgs& a, int n_req, bool pdl, cudaStream_t st) {
  if ((a.B != 8 && a.B != 16)) return cudaErrorInvalidValue;
  return launch_ex(start_kernel, dim3(n_req * a.B / kB, (a.H + a.n_taps * a.H) / kCw), dim3(kThreads), 0, st, pdl, a);
}
cudaError_t launch_fc_finish_conv_in(const FcFinishArgs& f, const ConvInArgs& c, int n_req, bool pdl, cudaStream_t st) {
  if (f.H != c.H || f.n_rows != c.n_rows || f.n_rows % kB) return cudaErrorInvalidValue;
  if (f.H % kCv) return cudaErrorInvalidValue;
  if (conv_in_v(c.n_rows) == 4)
    return launch_ex(fc_finish_conv_in_kernel<4>, dim3(f.n_rows / kB, f.H / kCv, 2), dim3(kThreads), 0, st, pdl, f, c);
  return launch_ex(fc_finish_conv_in_kernel<2>, dim3(f.n_rows / kB, f.H / 64, 2), dim3(kThreads), 0, st, pdl, f, c);
}
cudaError_t launch_conv_in(const ConvInArgs& a, int n_req, bool pdl, cudaStream_t st) {
  if (a.n_rows % kB || a.H % kCv) return cudaErrorInvalidValue;
  if (conv_in_v(a.n_rows) == 4)
    return launch_ex(conv_in_kernel<4>, dim3(a.n_rows / kB, a.H / kCv), dim3(kThreads), 0, st, pdl, a);
  return launch_ex(conv_in_kernel<2>, dim3(a.n_rows / kB, a.H / 64), dim3(kThreads), 0, st, pdl, a);
}
cudaError_t launch_conv_out(const ConvOutArgs& a, int n_req, bool pdl, cudaStream_t st) {
  if (a.n_rows % kB || a.H % kCv) return cudaErrorInvalidValue;
  return launch_ex(conv_out_kernel, dim3(a.n_rows / kB, a.H / kCv), dim3(kThreads), 0, st, pdl, a);
}
cudaError_t launch_swiglu(const SwigluArgs& a, int n_req, bool pdl, cudaStream_t st) {
  if (a.n_rows % kB || a.F % kCv) return cudaErrorInvalidValue;
  return launch_ex(swiglu_kernel, dim3(a.n_rows / kB, a.F / kCv), dim3(kThreads), 0, st, pdl, a);
}
cudaError_t launch_qkv_finish(const QkvFinishArgs& a, int n_req, bool pdl, cudaStream_t st) {
  if ((a.B != 8 && a.B != 16) || a.n_rows != a.B * n_req) return cudaErrorInvalidValue;
  const int n_items = a.B * a.n_q_heads + 4 * a.B * a.n_kv_heads;
  return launch_ex(qkv_finish_kernel, dim3(n_req, (n_items + 7) / 8), dim3(256), 0, st, pdl, a);
}

}  // namespace df2
