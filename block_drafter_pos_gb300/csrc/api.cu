// Host side of the C ABI: argument validation, scratch layout, and the launch
// sequence of one draft block (a1-a9), the selector (a10) and the verify (a11).
// No allocation after dflash2_create; no host synchronisation in the step calls.
//
// Per layer the draft block launches: delta projection, conv-in, QKV projection,
// q/k norm + RoPE + cache append, block attention (+ combine), output projection
// (epilogue: conv-out + residual + post-norm input), delta projection, conv-in,
// gate/up projection (epilogue: SwiGLU), down projection (epilogue: conv-out +
// residual + next norm input).  Every kernel is launched with programmatic
// dependent launch so its prologue overlaps the previous kernel's tail.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <new>

#include "../../include/dflash2.h"
#include "glue.h"
#include "internal.h"

using namespace df2;

struct dflash2_handle {
  dflash2_config cfg;
  dflash2_weights w;
  int max_req, kv_cap, num_sms, fmt;
  bool pdl;
  int H, G, F, V, nq, nkv, qd, kvd, KT;
  int nch128, nch16;  // chunks of the two kinds of sums-of-squares partials
  int n_attn_chunks, n_verify_chunks, lm_ctas;
  // scratch
  char* arena;
  size_t arena_bytes;
  float *x, *ss128, *ss16, *ss_c, *dproj, *delta_a, *delta_m, *fc_out, *q_out, *k_out, *v_out, *sel_out;
  float *q, *kb, *vb, *attn_part, *part;
  int* counters;
  void *act_a, *act_qkv, *act_taps, *act_o, *act_h;
  uint16_t* act_fin;
  // element offsets of the low-order activation planes (x = hi + lo)
  size_t lo_a, lo_qkv, lo_taps, lo_o, lo_h, lo_fin;
  unsigned long long* topk_keys;
  VerifyStat* vstats;
  double* inv_freq;
  int64_t launches;
  cudaEvent_t ev_lm0, ev_lm1;
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define DF2_CHECK(expr)                           \
  do {                                            \
    cudaError_t e_ = (expr);                      \
    if (e_ != cudaSuccess) return DFLASH2_E_CUDA; \
  } while (0)

GemvSeg seg_base(const dflash2_matrix& m, const void* x, size_t xlo, int ldx, int n_tiles, int rows, int K) {
  GemvSeg s;
  memset(&s, 0, sizeof(s));
  s.w = m.w;
  s.scale = static_cast<const uint16_t*>(m.scale);
  s.bias = static_cast<const uint16_t*>(m.bias);
  s.x = x;
  s.xlo_off = xlo;
  s.ldx = ldx;
  s.K = K;
  s.n_tiles = n_tiles;
  s.tiles = rows / 16;
  s.epi = kEpiStore;
  return s;
}

GemvSeg seg_store(const dflash2_matrix& m, const void* x, size_t xlo, int ldx, int n_tiles, int M, int K, float* out) {
  GemvSeg s = seg_base(m, x, xlo, ldx, n_tiles, M, K);
  s.out = out;
  s.ldo = M;
  return s;
}

dflash2_status run_gemv(dflash2_handle* h, std::initializer_list<GemvSeg> segs, cudaStream_t st) {
  GemvArgs a;
  memset(&a, 0, sizeof(a));
  int max_tiles = 0;
  for (const GemvSeg& s : segs) {
    a.seg[a.nseg++] = s;
    max_tiles = std::max(max_tiles, s.n_tiles);
  }
  a.part = h->part;
  a.counters = h->counters;
  DF2_CHECK(launch_gemv(a, h->fmt, max_tiles, h->num_sms, h->pdl, st));
  h->launches += 1;
  return DFLASH2_OK;
}

bool valid_matrix(const dflash2_matrix& m, int fmt) {
  if (!m.w || !aligned16(m.w)) return false;
  if (fmt == DFLASH2_WEIGHTS_Q8G64 && (!m.scale || !m.bias)) return false;
  return true;
}

// Scratch of the largest GEMV launch of a step (partial slots, tile counters).
void gemv_scratch(const dflash2_handle* h, int R, size_t* part_floats, int* counters) {
  const int N = 8 * R;
  const dflash2_matrix dummy = {nullptr, nullptr, nullptr};
  GemvSeg list[][3] = {
      {seg_base(dummy, nullptr, 0, h->KT, R, h->H, h->KT)},
      {seg_base(dummy, nullptr, 0, h->H, R, 4 * h->G, h->H)},
      {seg_base(dummy, nullptr, 0, h->H, R, h->qd, h->H), seg_base(dummy, nullptr, 0, h->H, 2 * R, h->kvd, h->H),
       seg_base(dummy, nullptr, 0, h->H, 2 * R, h->kvd, h->H)},
      {seg_base(dummy, nullptr, 0, h->qd, R, h->H, h->qd)},
      {seg_base(dummy, nullptr, 0, h->H, R, 2 * h->F, h->H)},
      {seg_base(dummy, nullptr, 0, h->F, R, h->H, h->F)},
      {seg_base(dummy, nullptr, 0, h->H, R, h->cfg.rank, h->H)},
  };
  const int nsegs[] = {1, 1, 3, 1, 1, 1, 1};
  (void)N;
  *part_floats = 0;
  *counters = 0;
  for (int i = 0; i < 7; ++i) {
    GemvArgs a;
    memset(&a, 0, sizeof(a));
    for (int j = 0; j < nsegs[i]; ++j) a.seg[a.nseg++] = list[i][j];
    size_t pf = 0;
    int nc = 0;
    gemv_plan(a, h->fmt, h->num_sms, &pf, &nc);
    *part_floats = std::max(*part_floats, pf);
    *counters = std::max(*counters, nc);
  }
}

}  // namespace

extern "C" {

const char* dflash2_status_string(dflash2_status s) {
  switch (s) {
    case DFLASH2_OK: return "ok";
    case DFLASH2_E_INVAL: return "invalid argument";
    case DFLASH2_E_NONFINITE: return "nonfinite logit or selector score";
    case DFLASH2_E_CUDA: return "CUDA error";
    case DFLASH2_E_UNSUPPORTED: return "unsupported geometry";
    default: return "unknown status";
  }
}

dflash2_status dflash2_create(const dflash2_config* cfg, const dflash2_weights* w, int32_t max_requests,
                              int32_t kv_capacity, dflash2_handle** out) {
  if (!cfg || !w || !out || max_requests < 1 || kv_capacity < 1) return DFLASH2_E_INVAL;
  *out = nullptr;
  const dflash2_config& c = *cfg;
  if (c.hidden <= 0 || c.n_layers <= 0 || c.n_q_heads <= 0 || c.n_kv_heads <= 0 || c.ffn <= 0 || c.vocab <= 0 ||
      c.n_taps <= 0 || c.window <= 1 || c.rms_eps < 0.f || c.rope_theta <= 0.0)
    return DFLASH2_E_INVAL;
  if (c.mask_token_id < 0 || c.mask_token_id >= c.vocab) return DFLASH2_E_INVAL;
  if (c.weight_format != DFLASH2_WEIGHTS_BF16 && c.weight_format != DFLASH2_WEIGHTS_Q8G64) return DFLASH2_E_INVAL;
  if (c.head_dim != 128 || c.block != 8 || c.top_k != 16 || c.rank != 256 || c.conv_taps != 2 ||
      c.conv_group != 16 || c.n_layers > DFLASH2_MAX_LAYERS || c.n_q_heads != 4 * c.n_kv_heads ||
      c.hidden % 128 || c.ffn % 128 || c.vocab % 16 || max_requests > 4 ||
      (c.window - 1 + kAttnChunk - 1) / kAttnChunk + 1 > 64)
    return DFLASH2_E_UNSUPPORTED;
  const int fmt = c.weight_format;
  if (!w->embed || !w->lm_head || !w->hidden_norm || !w->final_norm || !aligned16(w->lm_head)) return DFLASH2_E_INVAL;
  if (!valid_matrix(w->fc, fmt) || !valid_matrix(w->sel_proj, fmt) || !valid_matrix(w->cb_a, fmt) ||
      !valid_matrix(w->cb_b, fmt))
    return DFLASH2_E_INVAL;
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash2_layer_weights& L = w->layers[l];
    if (!L.input_norm || !L.post_norm || !L.q_norm || !L.k_norm || !L.attn_base || !L.mlp_base) return DFLASH2_E_INVAL;
    const dflash2_matrix* ms[] = {&L.q, &L.k, &L.v, &L.o, &L.gate, &L.up, &L.down, &L.attn_delta, &L.mlp_delta};
    for (const dflash2_matrix* m : ms)
      if (!valid_matrix(*m, fmt)) return DFLASH2_E_INVAL;
  }
  dflash2_handle* h = new (std::nothrow) dflash2_handle;
  if (!h) return DFLASH2_E_CUDA;
  memset(h, 0, sizeof(*h));
  h->cfg = c;
  h->w = *w;
  h->max_req = max_requests;
  h->kv_cap = kv_capacity;
  h->fmt = fmt;
  h->pdl = true;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    delete h;
    return DFLASH2_E_CUDA;
  }
  h->H = c.hidden;
  h->G = c.hidden / 16;
  h->F = c.ffn;
  h->V = c.vocab;
  h->nq = c.n_q_heads;
  h->nkv = c.n_kv_heads;
  h->qd = c.n_q_heads * 128;
  h->kvd = c.n_kv_heads * 128;
  h->KT = c.n_taps * c.hidden;
  h->nch128 = c.hidden / 128;
  h->nch16 = c.hidden / 16;
  h->n_attn_chunks = (c.window - 1 + kAttnChunk - 1) / kAttnChunk + 1;
  h->n_verify_chunks = (c.vocab + kVerifyChunk - 1) / kVerifyChunk;
  h->lm_ctas = h->num_sms;  // one 16-warp CTA per SM (the kernel needs 128 registers a thread)
  const size_t N = 8 * static_cast<size_t>(max_requests);
  const size_t esz = 2;  // bf16 / fp16 activations
  size_t part_floats = 0;
  int n_counters = 0;
  gemv_scratch(h, max_requests, &part_floats, &n_counters);
  struct Buf {
    void** p;
    size_t bytes;
  };
  const Buf bufs[] = {
      {reinterpret_cast<void**>(&h->x), N * h->H * 4},
      {reinterpret_cast<void**>(&h->ss128), N * h->nch128 * 4},
      {reinterpret_cast<void**>(&h->ss16), N * h->nch16 * 4},
      {reinterpret_cast<void**>(&h->ss_c), N * h->nch128 * 4},
      {reinterpret_cast<void**>(&h->dproj), N * 4 * h->G * 4},
      {reinterpret_cast<void**>(&h->delta_a), N * 4 * h->G * 4},
      {reinterpret_cast<void**>(&h->delta_m), N * 4 * h->G * 4},
      {reinterpret_cast<void**>(&h->fc_out), N * h->H * 4},
      {reinterpret_cast<void**>(&h->q_out), N * h->qd * 4},
      {reinterpret_cast<void**>(&h->k_out), 2 * N * h->kvd * 4},
      {reinterpret_cast<void**>(&h->v_out), 2 * N * h->kvd * 4},
      {reinterpret_cast<void**>(&h->sel_out), N * c.rank * 4},
      {reinterpret_cast<void**>(&h->q), N * h->qd * 4},
      {reinterpret_cast<void**>(&h->kb), N * h->kvd * 4},
      {reinterpret_cast<void**>(&h->vb), N * h->kvd * 4},
      {reinterpret_cast<void**>(&h->attn_part),
       static_cast<size_t>(max_requests) * h->nkv * h->n_attn_chunks * 32 * 130 * 4},
      {reinterpret_cast<void**>(&h->part), part_floats * 4},
      {reinterpret_cast<void**>(&h->counters), static_cast<size_t>(n_counters) * 4},
      {reinterpret_cast<void**>(&h->act_a), 2 * N * h->H * esz},  // hi and lo planes
      {reinterpret_cast<void**>(&h->act_qkv), 2 * 2 * N * h->H * esz},
      {reinterpret_cast<void**>(&h->act_taps), 2 * N * h->KT * esz},
      {reinterpret_cast<void**>(&h->act_o), 2 * N * h->qd * esz},
      {reinterpret_cast<void**>(&h->act_h), 2 * N * h->F * esz},
      {reinterpret_cast<void**>(&h->act_fin), 2 * N * h->H * 2},
      {reinterpret_cast<void**>(&h->topk_keys), N * h->lm_ctas * 16 * 8},
      {reinterpret_cast<void**>(&h->vstats),
       static_cast<size_t>(max_requests) * 8 * h->n_verify_chunks * sizeof(VerifyStat)},
      {reinterpret_cast<void**>(&h->inv_freq), 64 * 8},
  };
  h->lo_a = N * h->H;
  h->lo_qkv = 2 * N * h->H;
  h->lo_taps = N * h->KT;
  h->lo_o = N * h->qd;
  h->lo_h = N * h->F;
  h->lo_fin = N * h->H;
  size_t total = 0;
  for (const Buf& b : bufs) total += (b.bytes + 255) & ~static_cast<size_t>(255);
  if (cudaMalloc(&h->arena, total) != cudaSuccess) {
    delete h;
    return DFLASH2_E_CUDA;
  }
  h->arena_bytes = total;
  size_t off = 0;
  for (const Buf& b : bufs) {
    *b.p = h->arena + off;
    off += (b.bytes + 255) & ~static_cast<size_t>(255);
  }
  double invf[64];
  for (int j = 0; j < 64; ++j) invf[j] = pow(c.rope_theta, -2.0 * j / 128.0);
  if (cudaMemset(h->arena, 0, total) != cudaSuccess ||
      cudaMemcpy(h->inv_freq, invf, sizeof(invf), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(h->arena);
    delete h;
    return DFLASH2_E_CUDA;
  }
  *out = h;
  return DFLASH2_OK;
}

dflash2_status dflash2_destroy(dflash2_handle* h) {
  if (!h) return DFLASH2_E_INVAL;
  cudaFree(h->arena);
  delete h;
  return DFLASH2_OK;
}

int64_t dflash2_launch_count(const dflash2_handle* h) { return h ? h->launches : -1; }

dflash2_status dflash2_set_lmhead_events(dflash2_handle* h, void* start, void* stop) {
  if (!h || ((start == nullptr) != (stop == nullptr))) return DFLASH2_E_INVAL;
  h->ev_lm0 = static_cast<cudaEvent_t>(start);
  h->ev_lm1 = static_cast<cudaEvent_t>(stop);
  return DFLASH2_OK;
}

int64_t dflash2_lmhead_bytes(const dflash2_handle* h, int32_t n_req) {
  if (!h || n_req < 1) return -1;
  const int64_t N = 8 * static_cast<int64_t>(n_req);
  return static_cast<int64_t>(h->V) * h->H * 2  // LM-head weights, read once
         + 2 * N * h->H * 2                      // bf16 hidden state, hi and lo planes
         + N * h->lm_ctas * 16 * 8;              // per-CTA top-16 keys written
}

dflash2_status dflash2_draft_block(dflash2_handle* h, int32_t n_req, const int32_t* anchor_ids,
                                   const int32_t* ctx_len, const int32_t* n_new, const float* taps, void* k_cache,
                                   void* v_cache, int32_t* cand_ids, float* cand_logits, float* gate,
                                   float* logits_out, void* stream) {
  if (!h || n_req < 1 || n_req > h->max_req) return DFLASH2_E_INVAL;
  if (!anchor_ids || !ctx_len || !n_new || !taps || !k_cache || !v_cache || !cand_ids || !cand_logits || !gate)
    return DFLASH2_E_INVAL;
  if (!aligned16(taps) || !aligned16(k_cache) || !aligned16(v_cache)) return DFLASH2_E_INVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dflash2_config& c = h->cfg;
  const int fmt = h->fmt;
  const bool pdl = h->pdl;
  const int R = n_req;
  const int N = 8 * R;
  const int H = h->H, G = h->G;
  const size_t layer_stride = static_cast<size_t>(h->max_req) * h->kv_cap * h->kvd;  // elements
  // ---- a2: block embedding, first norm input, taps packing
  {
    StartArgs a;
    a.anchor_ids = anchor_ids;
    a.n_new = n_new;
    a.embed = static_cast<const uint16_t*>(h->w.embed);
    a.norm_w = static_cast<const uint16_t*>(h->w.layers[0].input_norm);
    a.taps = taps;
    a.x = h->x;
    a.act_a = h->act_a;
    a.act_a_lo = h->lo_a;
    a.ss_x = h->ss128;
    a.act_taps = h->act_taps;
    a.act_taps_lo = h->lo_taps;
    a.H = H;
    a.n_taps = c.n_taps;
    a.mask_id = c.mask_token_id;
    a.nch = h->nch128;
    a.fmt = fmt;
    a.V = h->V;
    DF2_CHECK(launch_start(a, R, pdl, st));
    h->launches++;
  }
  // ---- a1: taps projection fc [H][n_taps H], then hidden_norm input of the context rows
  {
    dflash2_status s = run_gemv(h, {seg_store(h->w.fc, h->act_taps, h->lo_taps, h->KT, R, H, h->KT, h->fc_out)}, st);
    if (s) return s;
    FcFinishArgs a;
    a.y = h->fc_out;
    a.norm_w = static_cast<const uint16_t*>(h->w.hidden_norm);
    a.act = h->act_qkv;
    a.act_lo = h->lo_qkv;
    a.ss = h->ss_c;
    a.H = H;
    a.act_row0 = N;
    a.nch = h->nch128;
    a.fmt = fmt;
    DF2_CHECK(launch_fc_finish(a, R, pdl, st));
    h->launches++;
  }
  const float* ss_in = h->ss128;  // sums of squares of the current x and their chunk count
  int nch_in = h->nch128;
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash2_layer_weights& L = h->w.layers[l];
    uint16_t* kc = static_cast<uint16_t*>(k_cache) + l * layer_stride;
    uint16_t* vc = static_cast<uint16_t*>(v_cache) + l * layer_stride;
    // ---- a3: delta projection of the normed input, conv-in
    dflash2_status s =
        run_gemv(h, {seg_store(L.attn_delta, h->act_a, h->lo_a, H, R, 4 * G, H, h->dproj)}, st);
    if (s) return s;
    {
      ConvInArgs a;
      a.dproj = h->dproj;
      a.ss = ss_in;
      a.x = h->x;
      a.norm_w = static_cast<const uint16_t*>(L.input_norm);
      a.base = static_cast<const uint16_t*>(L.attn_base);
      a.delta = h->delta_a;
      a.act = h->act_qkv;
      a.act_lo = h->lo_qkv;
      a.H = H;
      a.nch = nch_in;
      a.fmt = fmt;
      a.eps = c.rms_eps;
      DF2_CHECK(launch_conv_in(a, R, pdl, st));
      h->launches++;
    }
    // ---- a4: q (block rows), k and v (block + new context rows)
    s = run_gemv(h,
                 {seg_store(L.q, h->act_qkv, h->lo_qkv, H, R, h->qd, H, h->q_out),
                  seg_store(L.k, h->act_qkv, h->lo_qkv, H, 2 * R, h->kvd, H, h->k_out),
                  seg_store(L.v, h->act_qkv, h->lo_qkv, H, 2 * R, h->kvd, H, h->v_out)},
                 st);
    if (s) return s;
    {
      QkvFinishArgs a;
      a.q_out = h->q_out;
      a.k_out = h->k_out;
      a.v_out = h->v_out;
      a.ss_c = h->ss_c;
      a.q_norm = static_cast<const uint16_t*>(L.q_norm);
      a.k_norm = static_cast<const uint16_t*>(L.k_norm);
      a.inv_freq = h->inv_freq;
      a.ctx_len = ctx_len;
      a.n_new = n_new;
      a.q = h->q;
      a.kb = h->kb;
      a.vb = h->vb;
      a.k_cache = kc;
      a.v_cache = vc;
      a.n_q_heads = h->nq;
      a.n_kv_heads = h->nkv;
      a.n_rows = N;
      a.kv_capacity = h->kv_cap;
      a.H = H;
      a.nch = h->nch128;
      a.eps = c.rms_eps;
      DF2_CHECK(launch_qkv_finish(a, R, pdl, st));
      h->launches++;
    }
    // ---- a5: block attention over the window
    {
      AttnArgs a;
      a.q = h->q;
      a.kb = h->kb;
      a.vb = h->vb;
      a.k_cache = kc;
      a.v_cache = vc;
      a.ctx_len = ctx_len;
      a.n_new = n_new;
      a.part = h->attn_part;
      a.act_o = h->act_o;
      a.act_o_lo = h->lo_o;
      a.n_q_heads = h->nq;
      a.n_kv_heads = h->nkv;
      a.kv_capacity = h->kv_cap;
      a.window = c.window;
      a.n_chunks = h->n_attn_chunks;
      a.fmt = fmt;
      DF2_CHECK(launch_attention(a, R, pdl, st));
      h->launches += 2;
    }
    // ---- a6: output projection; epilogue: conv-out, residual, post-attention norm input
    {
      GemvSeg sg = seg_base(L.o, h->act_o, h->lo_o, h->qd, R, H, h->qd);
      sg.epi = kEpiConvOut;
      sg.act = h->act_a;
      sg.act_lo = h->lo_a;
      sg.ld_act = H;
      sg.act_fmt = fmt;
      sg.xres = h->x;
      sg.delta = h->delta_a;
      sg.base = static_cast<const uint16_t*>(L.attn_base);
      sg.norm_w = static_cast<const uint16_t*>(L.post_norm);
      sg.ss = h->ss16;
      sg.G = G;
      s = run_gemv(h, {sg}, st);
      if (s) return s;
    }
    ss_in = h->ss16;
    nch_in = h->nch16;
    // ---- a7: MLP sublayer
    s = run_gemv(h, {seg_store(L.mlp_delta, h->act_a, h->lo_a, H, R, 4 * G, H, h->dproj)}, st);
    if (s) return s;
    {
      ConvInArgs a;
      a.dproj = h->dproj;
      a.ss = ss_in;
      a.x = h->x;
      a.norm_w = static_cast<const uint16_t*>(L.post_norm);
      a.base = static_cast<const uint16_t*>(L.mlp_base);
      a.delta = h->delta_m;
      a.act = h->act_qkv;
      a.act_lo = h->lo_qkv;
      a.H = H;
      a.nch = nch_in;
      a.fmt = fmt;
      a.eps = c.rms_eps;
      DF2_CHECK(launch_conv_in(a, R, pdl, st));
      h->launches++;
    }
    {
      GemvSeg sg = seg_base(L.gate, h->act_qkv, h->lo_qkv, H, R, 2 * h->F, H);  // tile = 8 gate + 8 up rows
      sg.w2 = L.up.w;
      sg.scale2 = static_cast<const uint16_t*>(L.up.scale);
      sg.bias2 = static_cast<const uint16_t*>(L.up.bias);
      sg.epi = kEpiSwiglu;
      sg.act = h->act_h;
      sg.act_lo = h->lo_h;
      sg.ld_act = h->F;
      sg.act_fmt = fmt;
      s = run_gemv(h, {sg}, st);
      if (s) return s;
    }
    {
      const bool last = l == c.n_layers - 1;
      GemvSeg sg = seg_base(L.down, h->act_h, h->lo_h, h->F, R, H, h->F);
      sg.epi = kEpiConvOut;
      sg.act = (last && fmt == 0) ? static_cast<void*>(h->act_fin) : h->act_a;
      sg.act_lo = (last && fmt == 0) ? h->lo_fin : h->lo_a;
      sg.ld_act = H;
      sg.act_fmt = fmt;
      sg.act2 = (last && fmt != 0) ? h->act_fin : nullptr;  // LM-head input is bf16 in both formats
      sg.act2_lo = h->lo_fin;
      sg.xres = h->x;
      sg.delta = h->delta_m;
      sg.base = static_cast<const uint16_t*>(L.mlp_base);
      sg.norm_w = static_cast<const uint16_t*>(last ? h->w.final_norm : h->w.layers[l + 1].input_norm);
      sg.ss = h->ss16;
      sg.G = G;
      s = run_gemv(h, {sg}, st);
      if (s) return s;
    }
  }
  // ---- a8: LM head + top-16
  {
    LmHeadArgs a;
    a.w = static_cast<const uint16_t*>(h->w.lm_head);
    a.x = h->act_fin;
    a.x_lo = h->lo_fin;
    a.ss = h->ss16;
    a.logits_out = logits_out;
    a.part_keys = h->topk_keys;
    a.V = h->V;
    a.H = H;
    a.n_rows = N;
    a.nch = h->nch16;
    a.n_cta = h->lm_ctas;
    a.eps = c.rms_eps;
    // external records: inside a stream capture they become event-record nodes the host can time
    if (h->ev_lm0) DF2_CHECK(cudaEventRecordWithFlags(h->ev_lm0, st, cudaEventRecordExternal));
    DF2_CHECK(launch_lmhead(a, pdl, st));
    if (h->ev_lm1) DF2_CHECK(cudaEventRecordWithFlags(h->ev_lm1, st, cudaEventRecordExternal));
    h->launches++;
  }
  // ---- a9: selector projection (same final hidden, in the matrix's format), merge top-16
  {
    const void* xin = fmt == 0 ? static_cast<const void*>(h->act_fin) : h->act_a;
    const size_t xlo = fmt == 0 ? h->lo_fin : h->lo_a;
    dflash2_status s = run_gemv(h, {seg_store(h->w.sel_proj, xin, xlo, H, R, c.rank, H, h->sel_out)}, st);
    if (s) return s;
    TopkMergeArgs a;
    a.part_keys = h->topk_keys;
    a.sel = h->sel_out;
    a.ss = h->ss16;
    a.cand_ids = cand_ids;
    a.cand_logits = cand_logits;
    a.gate = gate;
    a.n_rows = N;
    a.n_cta = h->lm_ctas;
    a.rank = c.rank;
    a.nch = h->nch16;
    a.H = H;
    a.eps = c.rms_eps;
    DF2_CHECK(launch_topk_merge(a, pdl, st));
    h->launches++;
  }
  return DFLASH2_OK;
}

dflash2_status dflash2_head_topk(dflash2_handle* h, int32_t n_rows, const void* hidden, int32_t* cand_ids,
                                 float* cand_logits, float* logits_out, void* stream) {
  if (!h || n_rows < 8 || n_rows % 8 || n_rows > 8 * h->max_req) return DFLASH2_E_INVAL;
  if (!hidden || !cand_ids || !cand_logits || !aligned16(hidden)) return DFLASH2_E_INVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LmHeadArgs a;
  a.w = static_cast<const uint16_t*>(h->w.lm_head);
  a.x = static_cast<const uint16_t*>(hidden);
  a.x_lo = 0;
  a.ss = nullptr;
  a.logits_out = logits_out;
  a.part_keys = h->topk_keys;
  a.V = h->V;
  a.H = h->H;
  a.n_rows = n_rows;
  a.nch = h->nch16;
  a.n_cta = h->lm_ctas;
  a.eps = h->cfg.rms_eps;
  DF2_CHECK(launch_lmhead(a, h->pdl, st));
  TopkMergeArgs m;
  m.part_keys = h->topk_keys;
  m.sel = nullptr;
  m.ss = nullptr;
  m.cand_ids = cand_ids;
  m.cand_logits = cand_logits;
  m.gate = nullptr;
  m.n_rows = n_rows;
  m.n_cta = h->lm_ctas;
  m.rank = h->cfg.rank;
  m.nch = h->nch16;
  m.H = h->H;
  m.eps = h->cfg.rms_eps;
  DF2_CHECK(launch_topk_merge(m, h->pdl, st));
  h->launches += 2;
  return DFLASH2_OK;
}

dflash2_status dflash2_select(dflash2_handle* h, int32_t n_req, const int32_t* anchor_ids, const int32_t* cand_ids,
                              const float* cand_logits, const float* gate, const float* temperature,
                              const uint64_t* seed, const uint64_t* philox_offset, int32_t* path, float* q_rows,
                              float* scores_out, int32_t* status, void* stream) {
  if (!h || n_req < 1 || n_req > h->max_req) return DFLASH2_E_INVAL;
  if (!anchor_ids || !cand_ids || !cand_logits || !gate || !temperature || !seed || !philox_offset || !path ||
      !q_rows || !status)
    return DFLASH2_E_INVAL;
  SelectArgs a;
  a.anchor_ids = anchor_ids;
  a.cand_ids = cand_ids;
  a.cand_logits = cand_logits;
  a.gate = gate;
  a.temperature = temperature;
  a.seed = seed;
  a.offset = philox_offset;
  a.cb_a = h->w.cb_a.w;
  a.cb_a_scale = static_cast<const uint16_t*>(h->w.cb_a.scale);
  a.cb_a_bias = static_cast<const uint16_t*>(h->w.cb_a.bias);
  a.cb_b = h->w.cb_b.w;
  a.cb_b_scale = static_cast<const uint16_t*>(h->w.cb_b.scale);
  a.cb_b_bias = static_cast<const uint16_t*>(h->w.cb_b.bias);
  a.path = path;
  a.q_rows = q_rows;
  a.scores_out = scores_out;
  a.status = status;
  a.rank = h->cfg.rank;
  a.fmt = h->fmt;
  a.V = h->V;
  DF2_CHECK(launch_select(a, n_req, h->pdl, static_cast<cudaStream_t>(stream)));
  h->launches++;
  return DFLASH2_OK;
}

dflash2_status dflash2_verify(dflash2_handle* h, int32_t n_req, const float* target_logits, const int32_t* path,
                              const int32_t* cand_ids, const float* q_rows, const float* temperature,
                              const uint64_t* seed, const uint64_t* philox_offset, int32_t* n_accepted,
                              int32_t* emitted, int32_t* n_emitted, int32_t* status, void* stream) {
  if (!h || n_req < 1 || n_req > h->max_req) return DFLASH2_E_INVAL;
  if (!target_logits || !path || !cand_ids || !q_rows || !temperature || !seed || !philox_offset || !n_accepted ||
      !emitted || !n_emitted || !status)
    return DFLASH2_E_INVAL;
  VerifyArgs a;
  a.logits = target_logits;
  a.path = path;
  a.cand_ids = cand_ids;
  a.q_rows = q_rows;
  a.temperature = temperature;
  a.seed = seed;
  a.offset = philox_offset;
  a.stats = h->vstats;
  a.n_accepted = n_accepted;
  a.emitted = emitted;
  a.n_emitted = n_emitted;
  a.status = status;
  a.V = h->V;
  a.n_chunks = h->n_verify_chunks;
  DF2_CHECK(launch_verify(a, n_req, h->pdl, static_cast<cudaStream_t>(stream)));
  h->launches += 2;
  return DFLASH2_OK;
}

}  // extern "C"
