// Element-wise stages between the weight-streaming projections: block embedding,
// taps packing, RMSNorm (deferred: each stage writes x * w and per-chunk sums of
// squares; the consumer applies 1/rms), the grouped dynamic convolution before and
// after each sublayer, the residual add, SwiGLU, and the q/k norm + RoPE + context
// cache append after the QKV projection.
//
// Layout: one CTA = 128 channels of all 8 block rows of one request, one thread =
// one channel, so the 2-tap convolution along the block (rows i and i-1) stays in
// registers.  Row statistics cross CTAs only through per-chunk partial sums read
// back in a fixed order (bit-reproducible).
#include "common.cuh"
#include "glue.h"

namespace df2 {

namespace {

constexpr int kB = 8;       // block positions
constexpr int kCh = 128;    // channels per CTA

// Writes the 8 rows' activations (bf16, or fp16 + per-64 group sums) of this CTA's
// channel chunk.  sm: >= 4*8 floats of shared memory.
__device__ void emit_act(const float (&v)[kB], int row0, void* act, float* xsum, int ld, int fmt, float* sm) {
  const int c = blockIdx.y * kCh + threadIdx.x;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (fmt == 0) {
    __nv_bfloat16* a = reinterpret_cast<__nv_bfloat16*>(act);
#pragma unroll
    for (int i = 0; i < kB; ++i) a[static_cast<size_t>(row0 + i) * ld + c] = __float2bfloat16_rn(v[i]);
    return;
  }
  __half* a = reinterpret_cast<__half*>(act);
  float r[kB];
#pragma unroll
  for (int i = 0; i < kB; ++i) {
    const __half h = __float2half_rn(v[i]);
    a[static_cast<size_t>(row0 + i) * ld + c] = h;
    r[i] = warp_sum(__half2float(h));
  }
  __syncthreads();
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < kB; ++i) sm[wid * kB + i] = r[i];
  }
  __syncthreads();
  if (threadIdx.x < 2 * kB) {
    const int gq = threadIdx.x / kB, i = threadIdx.x % kB;
    const int KG = ld >> 6;
    xsum[static_cast<size_t>(row0 + i) * KG + blockIdx.y * 2 + gq] = sm[(2 * gq) * kB + i] + sm[(2 * gq + 1) * kB + i];
  }
  __syncthreads();
}

// Per-row sum of squares of this CTA's channels -> ss[row][blockIdx.y].
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
  __syncthreads();
}

// 1/rms of row `row` from its chunk partials.
__device__ __forceinline__ float inv_rms(const float* ss, int row, int nch, int H, float eps) {
  float s = 0.f;
  for (int j = 0; j < nch; ++j) s += ss[static_cast<size_t>(row) * nch + j];
  return rsqrtf(s / static_cast<float>(H) + eps);
}

// ------------------------------------------------------------------ start of the step
__global__ void __launch_bounds__(kCh) start_kernel(const StartArgs a) {
  __shared__ float sm[4 * kB];
  const int r = blockIdx.x;
  const int c = blockIdx.y * kCh + threadIdx.x;
  const int row0 = r * kB;
  if (blockIdx.y * kCh < a.H) {
    const int anchor = min(max(a.anchor_ids[r], 0), a.V - 1);  // ids are clamped into the table
    float xv[kB], av[kB];
#pragma unroll
    for (int i = 0; i < kB; ++i) {
      const int id = (i == 0) ? anchor : a.mask_id;
      xv[i] = bf16_to_f32(a.embed[static_cast<size_t>(id) * a.H + c]);
      a.x[static_cast<size_t>(row0 + i) * a.H + c] = xv[i];
      av[i] = xv[i] * bf16_to_f32(a.norm_w[c]);
    }
    emit_act(av, row0, a.act_a, a.xsum_a, a.H, a.fmt, sm);
    emit_ss(xv, row0, a.ss_x, a.nch, sm);
  }
  // taps of the new context rows (rows >= n_new are zero)
  const int nn = min(max(a.n_new[r], 0), kB);
  const int KT = a.n_taps * a.H;
  float tv[kB];
#pragma unroll
  for (int j = 0; j < kB; ++j) tv[j] = (j < nn) ? a.taps[(static_cast<size_t>(row0 + j)) * KT + c] : 0.f;
  emit_act(tv, row0, a.act_taps, a.xsum_taps, KT, a.fmt, sm);
}

// ------------------------------------------------------------------ taps projection finish
// c = y * w_hidden_norm (the 1/rms of y is applied by the K/V finish); ss of y.
__global__ void __launch_bounds__(kCh) fc_finish_kernel(const FcFinishArgs a) {
  __shared__ float sm[4 * kB];
  const int r = blockIdx.x;
  const int c = blockIdx.y * kCh + threadIdx.x;
  const int row0 = r * kB;
  const size_t plane = static_cast<size_t>(a.n_rows) * a.H;
  float yv[kB], cv[kB];
  const float w = bf16_to_f32(a.norm_w[c]);
#pragma unroll
  for (int j = 0; j < kB; ++j) {
    float s = 0.f;
    for (int sp = 0; sp < a.splits; ++sp) s += a.part[sp * plane + static_cast<size_t>(row0 + j) * a.H + c];
    yv[j] = s;
    cv[j] = s * w;
  }
  emit_act(cv, a.act_row0 + row0, a.act, a.xsum, a.H, a.fmt, sm);
  emit_ss(yv, row0, a.ss, a.nch, sm);
}

// ------------------------------------------------------------------ conv before a sublayer
// delta = r_i * sum_s P; a_i = r_i * x_i * w; a'_i = (b0 + d0_i) a_i + (b1 + d1_i) a_{i-1}
__global__ void __launch_bounds__(kCh) conv_in_kernel(const ConvInArgs a) {
  __shared__ float sm[4 * kB];
  __shared__ float dsh[kB][2][2][kCh / 16];  // [row][io][tap][local group]
  __shared__ float rr[kB];
  const int r = blockIdx.x;
  const int c = blockIdx.y * kCh + threadIdx.x;
  const int row0 = r * kB;
  const int G = a.H / 16;
  if (threadIdx.x < kB) rr[threadIdx.x] = inv_rms(a.ss, row0 + threadIdx.x, a.nch, a.H, a.eps);
  __syncthreads();
  if (threadIdx.x < 32) {
    const int io = threadIdx.x >> 4, t = (threadIdx.x >> 3) & 1, gl = threadIdx.x & 7;
    const int gidx = (io * 2 + t) * G + blockIdx.y * (kCh / 16) + gl;
    const size_t plane = static_cast<size_t>(a.n_rows) * (4 * G);
    for (int i = 0; i < kB; ++i) {
      float s = 0.f;
      for (int sp = 0; sp < a.splits; ++sp) s += a.part[sp * plane + static_cast<size_t>(row0 + i) * (4 * G) + gidx];
      s *= rr[i];
      dsh[i][io][t][gl] = s;
      a.delta[static_cast<size_t>(row0 + i) * (4 * G) + gidx] = s;
    }
  }
  __syncthreads();
  const int gl = threadIdx.x >> 4;
  const float w = bf16_to_f32(a.norm_w[c]);
  const float b0 = bf16_to_f32(a.base[c]), b1 = bf16_to_f32(a.base[a.H + c]);
  float out[kB];
  float prev = 0.f;
#pragma unroll
  for (int i = 0; i < kB; ++i) {
    const float ai = a.x[static_cast<size_t>(row0 + i) * a.H + c] * rr[i] * w;
    out[i] = (b0 + dsh[i][0][0][gl]) * ai + (b1 + dsh[i][0][1][gl]) * prev;
    prev = ai;
  }
  emit_act(out, row0, a.act, a.xsum, a.H, a.fmt, sm);
}

// ------------------------------------------------------------------ conv after a sublayer + residual
// y = sum_s P; x_i += (b2 + d2_i) y_i + (b3 + d3_i) y_{i-1}; act = x * w_next; ss of x.
__global__ void __launch_bounds__(kCh) conv_out_kernel(const ConvOutArgs a) {
  __shared__ float sm[4 * kB];
  const int r = blockIdx.x;
  const int c = blockIdx.y * kCh + threadIdx.x;
  const int row0 = r * kB;
  const int G = a.H / 16;
  const int g = c >> 4;
  const size_t plane = static_cast<size_t>(a.n_rows) * a.H;
  const float b2 = bf16_to_f32(a.base[2 * a.H + c]), b3 = bf16_to_f32(a.base[3 * a.H + c]);
  const float w = bf16_to_f32(a.norm_w[c]);
  float xv[kB], av[kB];
  float yprev = 0.f;
#pragma unroll
  for (int i = 0; i < kB; ++i) {
    float y = 0.f;
    for (int sp = 0; sp < a.splits; ++sp) y += a.part[sp * plane + static_cast<size_t>(row0 + i) * a.H + c];
    const float* d = a.delta + static_cast<size_t>(row0 + i) * (4 * G);
    const float conv = (b2 + d[2 * G + g]) * y + (b3 + d[3 * G + g]) * yprev;
    yprev = y;
    const size_t xi = static_cast<size_t>(row0 + i) * a.H + c;
    xv[i] = a.x[xi] + conv;
    a.x[xi] = xv[i];
    av[i] = xv[i] * w;
  }
  emit_act(av, row0, a.act, a.xsum, a.H, a.fmt, sm);
  if (a.act_bf16 != nullptr) emit_act(av, row0, a.act_bf16, nullptr, a.H, 0, sm);
  emit_ss(xv, row0, a.ss, a.nch, sm);
}

// ------------------------------------------------------------------ SwiGLU
__global__ void __launch_bounds__(kCh) swiglu_kernel(const SwigluArgs a) {
  __shared__ float sm[4 * kB];
  const int r = blockIdx.x;
  const int c = blockIdx.y * kCh + threadIdx.x;
  const int row0 = r * kB;
  const size_t plane = static_cast<size_t>(a.n_rows) * a.F;
  float hv[kB];
#pragma unroll
  for (int i = 0; i < kB; ++i) {
    float gs = 0.f, us = 0.f;
    for (int sp = 0; sp < a.splits; ++sp) {
      gs += a.part_g[sp * plane + static_cast<size_t>(row0 + i) * a.F + c];
      us += a.part_u[sp * plane + static_cast<size_t>(row0 + i) * a.F + c];
    }
    hv[i] = gs / (1.f + __expf(-gs)) * us;
  }
  emit_act(hv, row0, a.act, a.xsum, a.F, a.fmt, sm);
}

// ------------------------------------------------------------------ q/k norm, RoPE, cache append
// grid (R, nq + 2 nkv), 128 threads = head_dim.  Head h < nq: queries of the block;
// nq <= h < nq+nkv: keys (block rows, and new context rows into the cache);
// the rest: values.
__global__ void __launch_bounds__(128) qkv_finish_kernel(const QkvFinishArgs a) {
  __shared__ float red[32];
  __shared__ float buf[128];
  const int r = blockIdx.x;
  const int h = blockIdx.y;
  const int d = threadIdx.x;
  const int row0 = r * kB;
  const int nq = a.n_q_heads, nkv = a.n_kv_heads;
  // lengths are clamped so a bad length can never address outside the cache
  const int nn = min(max(a.n_new[r], 0), kB);
  const int ctx = min(max(a.ctx_len[r], 0), a.kv_capacity - nn);
  const int L = ctx + nn;
  int kind, hh;
  if (h < nq) {
    kind = 0;
    hh = h;
  } else if (h < nq + nkv) {
    kind = 1;
    hh = h - nq;
  } else {
    kind = 2;
    hh = h - nq - nkv;
  }
  const float* part = kind == 0 ? a.part_q : (kind == 1 ? a.part_k : a.part_v);
  const int M = kind == 0 ? nq * 128 : nkv * 128;
  const int rows_out = kind == 0 ? a.n_rows : 2 * a.n_rows;  // k/v segments hold block + context rows
  const size_t plane = static_cast<size_t>(rows_out) * M;
  const float nw = kind == 0 ? bf16_to_f32(a.q_norm[d]) : (kind == 1 ? bf16_to_f32(a.k_norm[d]) : 1.f);
  const int half = d & 63;
  const double inv_freq = a.inv_freq[half];
  const int nrows = (kind == 0) ? kB : 2 * kB;
  for (int j = 0; j < nrows; ++j) {
    const bool ctx_row = j >= kB;
    const int jj = ctx_row ? j - kB : j;
    if (ctx_row && jj >= nn) break;                              // uniform across the CTA
    const int prow = ctx_row ? a.n_rows + row0 + jj : row0 + jj;  // row in the GEMV output
    float v = 0.f;
    for (int sp = 0; sp < a.splits; ++sp) v += part[sp * plane + static_cast<size_t>(prow) * M + hh * 128 + d];
    if (ctx_row) v *= inv_rms(a.ss_c, row0 + jj, a.nch, a.H, a.eps);
    const int pos = ctx_row ? ctx + jj : L + jj;
    if (kind != 2) {
      const float ms = block_sum(v * v, red) / 128.f;
      v = v * rsqrtf(ms + a.eps) * nw;
      buf[d] = v;
      __syncthreads();
      const float other = buf[d ^ 64];
      __syncthreads();
      double sn, cs;
      sincos(static_cast<double>(pos) * inv_freq, &sn, &cs);
      // NEOX: out[j] = x[j] cos - x[j+64] sin; out[j+64] = x[j+64] cos + x[j] sin
      v = (d < 64) ? static_cast<float>(v * cs - other * sn) : static_cast<float>(v * cs + other * sn);
    }
    if (!ctx_row) {
      float* dst = kind == 0 ? a.q : (kind == 1 ? a.kb : a.vb);
      const int nh = kind == 0 ? nq : nkv;
      dst[(static_cast<size_t>(row0 + jj) * nh + hh) * 128 + d] = v;
    } else {
      uint16_t* cache = kind == 1 ? a.k_cache : a.v_cache;
      const size_t idx = ((static_cast<size_t>(r) * a.kv_capacity + pos) * nkv + hh) * 128 + d;
      const __nv_bfloat16 b = __float2bfloat16_rn(v);
      cache[idx] = *reinterpret_cast<const uint16_t*>(&b);
    }
  }
}

}  // namespace

cudaError_t launch_start(const StartArgs& a, int n_req, cudaStream_t st) {
  const int chunks = (a.n_taps * a.H) / kCh;
  start_kernel<<<dim3(n_req, chunks), kCh, 0, st>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_fc_finish(const FcFinishArgs& a, int n_req, cudaStream_t st) {
  fc_finish_kernel<<<dim3(n_req, a.H / kCh), kCh, 0, st>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_conv_in(const ConvInArgs& a, int n_req, cudaStream_t st) {
  conv_in_kernel<<<dim3(n_req, a.H / kCh), kCh, 0, st>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_conv_out(const ConvOutArgs& a, int n_req, cudaStream_t st) {
  conv_out_kernel<<<dim3(n_req, a.H / kCh), kCh, 0, st>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_swiglu(const SwigluArgs& a, int n_req, cudaStream_t st) {
  swiglu_kernel<<<dim3(n_req, a.F / kCh), kCh, 0, st>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_qkv_finish(const QkvFinishArgs& a, int n_req, cudaStream_t st) {
  qkv_finish_kernel<<<dim3(n_req, a.n_q_heads + 2 * a.n_kv_heads), 128, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace df2
