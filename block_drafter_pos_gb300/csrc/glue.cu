// Element-wise stages between the weight-streaming projections: block embedding
// and taps packing (start), the taps-projection norm input (fc_finish), the
// dynamic convolution before a sublayer (conv_in) and after it with the residual
// add (conv_out), SwiGLU, and q/k norm + RoPE + context cache append after the QKV
// projection (qkv_finish).  Each consumer adds the producer GEMV's split planes in
// split order.
//
// RMSNorm is deferred: producers write x * w and per-chunk sums of squares, and
// the consumer applies 1/rms (the scale commutes with the projections).  Row
// statistics cross CTAs only through those partial sums, read in a fixed order
// (bit-reproducible).
#include "common.cuh"
#include "glue.h"
#include "internal.h"

namespace df2 {

namespace {

constexpr int kB = 8;       // block positions
constexpr int kCh = 128;    // channels per CTA (one thread per channel, all 8 rows)

DF2_DEV void put_act(void* act, size_t lo, int fmt, size_t idx, float v) {
  if (fmt == 0) {
    __nv_bfloat16* p = reinterpret_cast<__nv_bfloat16*>(act);
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    p[idx] = h;
    if (lo) p[lo + idx] = __float2bfloat16_rn(v - __bfloat162float(h));
  } else {
    __half* p = reinterpret_cast<__half*>(act);
    const __half h = __float2half_rn(v);
    p[idx] = h;
    if (lo) p[lo + idx] = __float2half_rn(v - __half2float(h));
  }
}

// Per-row sum of squares of this CTA's 128 channels -> ss[row][blockIdx.y].
__device__ void emit_ss(const float (&v)[kB], int row0, float* ss, int nch, float* sm) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  float r[kB];
#pragma unroll
  for (int i = 0; i < kB; ++i) r[i] = warp_sum(v[i] * v[i]);
  __syncthreads();
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < kB; ++i) sm[wid * kB + i] = r[i];
  }
  __syncthreads();
  if (threadIdx.x < kB) {
    const int i = threadIdx.x;
    ss[static_cast<size_t>(row0 + i) * nch + blockIdx.y] = ((sm[i] + sm[kB + i]) + sm[2 * kB + i]) + sm[3 * kB + i];
  }
}

// ------------------------------------------------------------------ start of the step
__global__ void __launch_bounds__(kCh) start_kernel(const StartArgs a) {
  __shared__ float sm[4 * kB];
  pdl_begin();
  const int r = blockIdx.x;
  const int c = blockIdx.y * kCh + threadIdx.x;
  const int row0 = r * kB;
  if (blockIdx.y * kCh < a.H) {
    const int anchor = min(max(a.anchor_ids[r], 0), a.V - 1);  // ids are clamped into the table
    const float w = bf16_to_f32(a.norm_w[c]);
    float xv[kB];
#pragma unroll
    for (int i = 0; i < kB; ++i) {
      const int id = (i == 0) ? anchor : a.mask_id;
      xv[i] = bf16_to_f32(a.embed[static_cast<size_t>(id) * a.H + c]);
      const size_t idx = static_cast<size_t>(row0 + i) * a.H + c;
      a.x[idx] = xv[i];
      put_act(a.act_a, a.act_a_lo, a.fmt, idx, xv[i] * w);
    }
    emit_ss(xv, row0, a.ss_x, a.nch, sm);
  }
  // taps of the new context rows (rows >= n_new are zero)
  const int nn = min(max(a.n_new[r], 0), kB);
  const int KT = a.n_taps * a.H;
#pragma unroll
  for (int j = 0; j < kB; ++j) {
    const size_t idx = static_cast<size_t>(row0 + j) * KT + c;
    put_act(a.act_taps, a.act_taps_lo, a.fmt, idx, (j < nn) ? a.taps[idx] : 0.f);
  }
}

// ------------------------------------------------------------------ taps projection finish
// c = y * w_hidden_norm into the context rows of the QKV input (1/rms of y is
// applied after the K/V projection); ss of y.
__global__ void __launch_bounds__(kCh) fc_finish_kernel(const FcFinishArgs a) {
  __shared__ float sm[4 * kB];
  pdl_begin();
  const int r = blockIdx.x;
  const int c = blockIdx.y * kCh + threadIdx.x;
  const int row0 = r * kB;
  const float w = bf16_to_f32(a.norm_w[c]);
  float yv[kB];
  const size_t plane = static_cast<size_t>(a.n_rows) * a.H;
#pragma unroll
  for (int j = 0; j < kB; ++j) {
    float y = 0.f;
    for (int sp = 0; sp < a.splits; ++sp) y += a.y[sp * plane + static_cast<size_t>(row0 + j) * a.H + c];
    yv[j] = y;
    put_act(a.act, a.act_lo, a.fmt, static_cast<size_t>(a.act_row0 + row0 + j) * a.H + c, yv[j] * w);
  }
  emit_ss(yv, row0, a.ss, a.nch, sm);
}

// ------------------------------------------------------------------ conv before a sublayer
// r_i = 1/rms(x_i); delta = r_i * (W_delta (x_i * w)) for all four (io, tap) rows;
// a_i = r_i x_i w;  a'_i = (b0 + d0_i) a_i + (b1 + d1_i) a_{i-1}.
__global__ void __launch_bounds__(kCh) conv_in_kernel(const ConvInArgs a) {
  __shared__ float dsh[kB][2][kCh / 16];  // [row][tap][local group] of the conv before the sublayer
  __shared__ float rr[kB];
  pdl_begin();
  const int r = blockIdx.x;
  const int c = blockIdx.y * kCh + threadIdx.x;
  const int row0 = r * kB;
  const int G = a.H / 16;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int i = wid; i < kB; i += kCh / 32) {
    const float v = warp_inv_rms(a.ss, row0 + i, a.nch, a.H, a.eps);
    if (lane == 0) rr[i] = v;
  }
  __syncthreads();
  // 8 rows x 4 (io, tap) x 8 local groups = 256 delta values, 2 per thread
  for (int e = threadIdx.x; e < kB * 32; e += kCh) {
    const int i = e >> 5, io = (e >> 4) & 1, t = (e >> 3) & 1, gl = e & 7;
    const int gidx = (io * 2 + t) * G + blockIdx.y * (kCh / 16) + gl;
    const size_t plane = static_cast<size_t>(a.n_rows) * (4 * G);
    float dsum = 0.f;
#pragma unroll 4
    for (int sp = 0; sp < a.splits; ++sp) dsum += a.dproj[sp * plane + static_cast<size_t>(row0 + i) * (4 * G) + gidx];
    const float d = dsum * rr[i];
    if (io == 0) dsh[i][t][gl] = d;
    a.delta[static_cast<size_t>(row0 + i) * (4 * G) + gidx] = d;
  }
  __syncthreads();
  const int gl = threadIdx.x >> 4;
  const float w = bf16_to_f32(a.norm_w[c]);
  const float b0 = bf16_to_f32(a.base[c]), b1 = bf16_to_f32(a.base[a.H + c]);
  float prev = 0.f;
#pragma unroll
  for (int i = 0; i < kB; ++i) {
    const size_t idx = static_cast<size_t>(row0 + i) * a.H + c;
    const float ai = a.x[idx] * rr[i] * w;
    put_act(a.act, a.act_lo, a.fmt, idx, (b0 + dsh[i][0][gl]) * ai + (b1 + dsh[i][1][gl]) * prev);
    prev = ai;
  }
}

// ------------------------------------------------------------------ conv after a sublayer + residual
// y = sum of split planes; x_i += (b2 + d2_i) y_i + (b3 + d3_i) y_{i-1} (the
// convolution wrapping the sublayer's output); act = x * w_next; ss of x.
__global__ void __launch_bounds__(kCh) conv_out_kernel(const ConvOutArgs a) {
  __shared__ float sm[4 * kB];
  pdl_begin();
  const int r = blockIdx.x;
  const int c = blockIdx.y * kCh + threadIdx.x;
  const int row0 = r * kB;
  const int G = a.H / 16;
  const int g = c >> 4;
  const size_t plane = static_cast<size_t>(a.n_rows) * a.H;
  const float b2 = bf16_to_f32(a.base[2 * a.H + c]), b3 = bf16_to_f32(a.base[3 * a.H + c]);
  const float w = bf16_to_f32(a.norm_w[c]);
  float y[kB];
#pragma unroll
  for (int i = 0; i < kB; ++i) y[i] = 0.f;
  for (int sp = 0; sp < a.splits; ++sp) {  // split planes in order; the 8 rows' loads are independent
#pragma unroll
    for (int i = 0; i < kB; ++i) y[i] += a.part[sp * plane + static_cast<size_t>(row0 + i) * a.H + c];
  }
  float xv[kB];
#pragma unroll
  for (int i = 0; i < kB; ++i) {
    const float* d = a.delta + static_cast<size_t>(row0 + i) * (4 * G);
    const float yprev = i > 0 ? y[i - 1] : 0.f;
    const size_t idx = static_cast<size_t>(row0 + i) * a.H + c;
    xv[i] = a.x[idx] + (b2 + d[2 * G + g]) * y[i] + (b3 + d[3 * G + g]) * yprev;
    a.x[idx] = xv[i];
    put_act(a.act, a.act_lo, a.fmt, idx, xv[i] * w);
    if (a.act2 != nullptr) put_act(a.act2, a.act2_lo, 0, idx, xv[i] * w);
  }
  emit_ss(xv, row0, a.ss, a.nch, sm);
}

// ------------------------------------------------------------------ SwiGLU
// h = silu(gate) * up from the split planes of the two projections.
__global__ void __launch_bounds__(kCh) swiglu_kernel(const SwigluArgs a) {
  pdl_begin();
  const int r = blockIdx.x;
  const int c = blockIdx.y * kCh + threadIdx.x;
  const int row0 = r * kB;
  const size_t plane = static_cast<size_t>(a.n_rows) * a.F;
  float gs[kB], us[kB];
#pragma unroll
  for (int i = 0; i < kB; ++i) gs[i] = us[i] = 0.f;
  for (int sp = 0; sp < a.splits; ++sp) {
#pragma unroll
    for (int i = 0; i < kB; ++i) {
      gs[i] += a.part_g[sp * plane + static_cast<size_t>(row0 + i) * a.F + c];
      us[i] += a.part_u[sp * plane + static_cast<size_t>(row0 + i) * a.F + c];
    }
  }
#pragma unroll
  for (int i = 0; i < kB; ++i)
    put_act(a.act, a.act_lo, a.fmt, static_cast<size_t>(row0 + i) * a.F + c, gs[i] / (1.f + __expf(-gs[i])) * us[i]);
}

// ------------------------------------------------------------------ q/k norm, RoPE, cache append
// One warp per (row, head); lane holds dims lane + 32 c (c = 0..3), so the NEOX
// pair (d, d + 64) is (c, c + 2) of the same lane.  Items: 8 query rows x nq heads,
// then 16 key rows (8 block + 8 context) x nkv, then 16 value rows x nkv.
__global__ void __launch_bounds__(256) qkv_finish_kernel(const QkvFinishArgs a) {
  pdl_begin();
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.y * 8 + (threadIdx.x >> 5);
  const int nq = a.n_q_heads, nkv = a.n_kv_heads;
  const int n_items = kB * nq + 2 * 2 * kB * nkv;
  if (item >= n_items) return;
  // lengths are clamped so a bad length can never address outside the cache
  const int nn = min(max(a.n_new[r], 0), kB);
  const int ctx = min(max(a.ctx_len[r], 0), a.kv_capacity - nn);
  const int L = ctx + nn;
  int kind, j, hh;
  if (item < kB * nq) {
    kind = 0;
    j = item / nq;
    hh = item % nq;
  } else {
    const int e = item - kB * nq;
    kind = 1 + e / (2 * kB * nkv);
    const int e2 = e % (2 * kB * nkv);
    j = e2 / nkv;
    hh = e2 % nkv;
  }
  const bool ctx_row = j >= kB;
  const int jj = ctx_row ? j - kB : j;
  if (ctx_row && jj >= nn) return;
  const int row0 = r * kB;
  const float* src;
  size_t plane;
  if (kind == 0) {
    src = a.q_out + (static_cast<size_t>(row0 + jj) * nq + hh) * 128;
    plane = static_cast<size_t>(a.n_rows) * nq * 128;
  } else {
    const size_t prow = ctx_row ? static_cast<size_t>(a.n_rows) + row0 + jj : static_cast<size_t>(row0 + jj);
    src = (kind == 1 ? a.k_out : a.v_out) + (prow * nkv + hh) * 128;
    plane = static_cast<size_t>(2 * a.n_rows) * nkv * 128;
  }
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  for (int sp = 0; sp < a.splits; ++sp)  // split planes in order
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] += src[sp * plane + lane + 32 * c];
  if (ctx_row) {
    const float rc = warp_inv_rms(a.ss_c, row0 + jj, a.nch, a.H, a.eps);
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] *= rc;
  }
  const int pos = ctx_row ? ctx + jj : L + jj;
  if (kind != 2) {
    const uint16_t* nw = kind == 0 ? a.q_norm : a.k_norm;
    const float ms = warp_sum(v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3]) / 128.f;
    const float rs = rsqrtf(ms + a.eps);
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] = v[c] * rs * bf16_to_f32(nw[lane + 32 * c]);
    // NEOX: out[j] = x[j] cos - x[j+64] sin; out[j+64] = x[j+64] cos + x[j] sin
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      double sn, cs;
      sincos(static_cast<double>(pos) * a.inv_freq[lane + 32 * c], &sn, &cs);
      const float x1 = v[c], x2 = v[c + 2];
      v[c] = static_cast<float>(x1 * cs - x2 * sn);
      v[c + 2] = static_cast<float>(x2 * cs + x1 * sn);
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

}  // namespace

cudaError_t launch_start(const StartArgs& a, int n_req, bool pdl, cudaStream_t st) {
  return launch_ex(start_kernel, dim3(n_req, (a.n_taps * a.H) / kCh), dim3(kCh), 0, st, pdl, a);
}
cudaError_t launch_fc_finish(const FcFinishArgs& a, int n_req, bool pdl, cudaStream_t st) {
  return launch_ex(fc_finish_kernel, dim3(n_req, a.H / kCh), dim3(kCh), 0, st, pdl, a);
}
cudaError_t launch_conv_in(const ConvInArgs& a, int n_req, bool pdl, cudaStream_t st) {
  return launch_ex(conv_in_kernel, dim3(n_req, a.H / kCh), dim3(kCh), 0, st, pdl, a);
}
cudaError_t launch_conv_out(const ConvOutArgs& a, int n_req, bool pdl, cudaStream_t st) {
  return launch_ex(conv_out_kernel, dim3(n_req, a.H / kCh), dim3(kCh), 0, st, pdl, a);
}
cudaError_t launch_swiglu(const SwigluArgs& a, int n_req, bool pdl, cudaStream_t st) {
  return launch_ex(swiglu_kernel, dim3(n_req, a.F / kCh), dim3(kCh), 0, st, pdl, a);
}
cudaError_t launch_qkv_finish(const QkvFinishArgs& a, int n_req, bool pdl, cudaStream_t st) {
  const int n_items = kB * a.n_q_heads + 4 * kB * a.n_kv_heads;
  return launch_ex(qkv_finish_kernel, dim3(n_req, (n_items + 7) / 8), dim3(256), 0, st, pdl, a);
}

}  // namespace df2
