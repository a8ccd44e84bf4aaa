// Host side of the C ABI: argument validation, scratch layout, and the launch
// sequence of one draft block (a1-a9), the selector (a10) and the verify (a11).
// No allocation after dflash2_create; no host synchronisation in the step calls.
//
// Per layer the draft block launches: delta projection, conv-in, QKV projection,
// q/k norm + RoPE + cache append, block attention (+ combine), output projection,
// conv-out + residual, delta projection, conv-in, gate/up projection, SwiGLU,
// down projection, conv-out + residual.  Each projection writes one fp32 plane per
// K split; the kernel after it adds the planes in split order (deterministic, no
// atomics, no inter-CTA signalling).  Every kernel is launched with programmatic
// dependent launch so its prologue overlaps the previous kernel's tail.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <initializer_list>
#include <new>

#include "../../include/dflash2.h"
#include "glue.h"
#include "internal.h"

using namespace df2;

static_assert(DFLASH2_TREE_MAX_NODES == kTreeMaxNodes, "draft-tree bound of the header and the kernels");

struct dflash2_handle {
  dflash2_config cfg;
  dflash2_weights w;
  int max_req, kv_cap, num_sms, fmt;
  int B;  // block positions per request (8 or 16); rows are request-major, B per request
  bool pdl;
  int H, G, F, V, nq, nkv, qd, kvd, KT;
  int nch_ss;  // 32-channel chunks of the sums-of-squares partials
  int n_attn_chunks, n_verify_chunks, lm_ctas;
  // where each projection's partial planes are (the launches' shapes are fixed at create)
  // plane maps of every projection launch: the GEMV (up to 4 requests) and the
  // tensor-core GEMM (calls with at least wide_min_rows block rows; set up when
  // max_requests reaches that)
  struct PlaneSet {
    GemvPlanes fc, d0, d, q, k, v, o, g, u, down, sel, lm;
    GemvPlanes q2, k2, v2;  // the GEMM's q/k/v launch with more than 128 key/value rows
  } pn, pw;
  bool wide;  // the tensor-core path is set up
  CUtensorMap wmap_fc, wmap_sel, wmap_lm, wmap_layer[DFLASH2_MAX_LAYERS][9];  // its weight maps
  float* lm_part;  // [p][N][V] LM-head partial planes of the GEMM path
  int lm_chunks;   // vocabulary chunks of its top-16
  // tensor maps of the projection matrices (bulk-copy descriptors, encoded at create)
  CUtensorMap map_fc, map_sel;
  CUtensorMap map_layer[DFLASH2_MAX_LAYERS][9];  // q k v o gate up down attn_delta mlp_delta
  // activation-buffer maps (hi rows then lo rows), encoded once the scratch exists
  CUtensorMap xm_taps, xm_a, xm_qkv, xm_o, xm_h, xm_fin;
  CUtensorMap map_lm, xm_lm;  // LM head weights; final hidden (bf16 in both formats) for the LM head
  int* gemv_err;  // device word set by a GEMV whose pipeline wait gave up
  unsigned int* verify_cnt;  // [max_req] verify chunk counters (zero between launches)
  float* sel_lat;            // [max_req][B-1][16][16] selector lattice scratch
  int32_t* sel_bad;          // [max_req][B-1] nonfinite flags per position
  unsigned int* sel_cnt;     // [max_req] selector position counters (zero between launches)
  VerifyStat* tstats;        // [max_req][kTreeMaxNodes + 1][n_verify_chunks] draft-tree row statistics
  unsigned int* tree_cnt;    // [max_req] draft-tree verify counters (zero between launches)
  int select_mode;           // 0: sequential walk, 1: Viterbi for greedy requests
  // scratch
  char* arena;
  size_t arena_bytes;
  float *x, *ss, *ss_c, *dproj, *delta_a, *delta_m, *fc_out, *q_out, *k_out, *v_out, *sel_out;
  float *q, *kb, *vb, *attn_part, *ypart, *gpart, *upart;
  void *act_a, *act_qkv, *act_taps, *act_o, *act_h;
  uint16_t* act_fin;
  // element offsets of the low-order activation planes (x = hi + lo)
  size_t lo_a, lo_qkv, lo_taps, lo_o, lo_h, lo_fin;
  unsigned long long* topk_keys;
  VerifyStat* vstats;
  double* inv_freq;
  int64_t launches;
  cudaEvent_t ev_lm0, ev_lm1;
  // profiling: event pairs around the weight-projection launches of draft_block calls
  cudaEvent_t* proj_ev;
  int proj_pairs, proj_next;
  bool in_draft;
  // dflash2_step: graphs of the argument sets seen, least recently used replaced
  struct StepGraph {
    dflash2_step_args key;
    int select_mode;  // the handle's selector mode when captured (a graph keeps its kernels' arguments)
    cudaGraphExec_t exec;
    int64_t launches;  // kernels in the graph
    uint64_t used;
  };
  StepGraph step_graph[DFLASH2_STEP_GRAPHS] = {};
  int n_step_graphs = 0;
  uint64_t step_clock = 0;
  cudaStream_t cap_stream = nullptr;  // the handle's own stream for the captures
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define DF2_CHECK(expr)                           \
  do {                                            \
    cudaError_t e_ = (expr);                      \
    if (e_ != cudaSuccess) return DFLASH2_E_CUDA; \
  } while (0)

// One projection segment: out[s] = W[:, split s] X[:, split s]^T for the
// 8 * n_tiles activation rows starting at x (tiles of 8 rows; B / 8 tiles per request).
enum { kQ, kK, kV, kO, kGate, kUp, kDown, kAttnDelta, kMlpDelta };

// One projection segment of either path.  x_rows: rows of one plane of the
// activation buffer behind xmap (its lo plane starts there); x: that buffer, from
// which the GEMM path encodes its own activation map; wide_map: the weight map of
// the GEMM path.
struct SegSpec {
  GemvSeg g;
  const CUtensorMap* wide_map;
  const void* x;
  bool x_tiled;  // the GEMM path finds x in its operand layout (written so by this library's kernels)
};

SegSpec seg(const CUtensorMap& wmap, const CUtensorMap& wide_map, const dflash2_matrix& m, const CUtensorMap& xmap,
            const void* x, int x_rows, int n_tiles, int M, int K, float* out) {
  SegSpec r;
  GemvSeg& s = r.g;
  memset(&s, 0, sizeof(s));
  s.wmap = wmap;
  s.xmap = xmap;
  s.x_lo_row = x_rows;
  s.scale = static_cast<const uint16_t*>(m.scale);
  s.bias = static_cast<const uint16_t*>(m.bias);
  s.M = M;
  s.K = K;
  s.n_tiles = n_tiles;
  s.out = out;
  r.wide_map = &wide_map;
  r.x = x;
  r.x_tiled = true;
  return r;
}

// Launches the segments on the GEMV (wide == false) or on the tensor-core GEMM.
// proj: a drafter weight projection (not the LM head), bracketed by the profiling
// events when they are set.
dflash2_status run_gemv(dflash2_handle* h, bool wide, std::initializer_list<SegSpec> segs, cudaStream_t st,
                        int fmt = -1, bool proj = true) {
  if (fmt < 0) fmt = h->fmt;
  const bool timed = proj && h->in_draft && h->proj_ev != nullptr && h->proj_next < h->proj_pairs;
  if (timed) DF2_CHECK(cudaEventRecordWithFlags(h->proj_ev[2 * h->proj_next], st, cudaEventRecordExternal));
  GemvArgs a;
  memset(&a, 0, sizeof(a));
  int max_tiles = 0;
  for (const SegSpec& s : segs) {
    GemvSeg& g = a.seg[a.nseg++];
    g = s.g;
    max_tiles = std::max(max_tiles, g.n_tiles);
    if (wide) {
      g.wmap = *s.wide_map;
      if (s.x_tiled) {
        g.xt = s.x;
        g.xt_rows = (g.x_lo_row + 15) & ~15;  // the rows of one plane, rounded up to 16: the rows of one slice
      } else if (!wide_encode_xmap(&g.xmap, s.x, 8 * g.n_tiles, g.K, fmt)) {
        return DFLASH2_E_CUDA;
      }
    }
  }
  a.err = h->gemv_err;
  if (wide)
    DF2_CHECK(launch_wide(a, fmt, h->num_sms, h->pdl, st));
  else
    DF2_CHECK(launch_gemv(a, fmt, max_tiles, h->num_sms, h->pdl, st));
  h->launches += 1;
  if (timed) {
    DF2_CHECK(cudaEventRecordWithFlags(h->proj_ev[2 * h->proj_next + 1], st, cudaEventRecordExternal));
    ++h->proj_next;
  }
  return DFLASH2_OK;
}

// Marks the span of one draft_block call (the projection events count from its start).
struct DraftScope {
  dflash2_handle* h;
  explicit DraftScope(dflash2_handle* hh) : h(hh) {
    h->in_draft = true;
    h->proj_next = 0;
  }
  ~DraftScope() { h->in_draft = false; }
};

// Calls with at least this many block rows run every projection on the tensor-core
// GEMM (measured with blocks of 8: with int8 weights it overtakes the GEMV at 32 rows,
// whose key/value launch needs the GEMV's 8-tile variant; with bf16 at 40).
int wide_min_rows(int fmt) { return fmt == DFLASH2_WEIGHTS_BF16 ? 40 : 32; }
bool wide_call(const dflash2_handle* h, int n_req) { return n_req * h->B >= wide_min_rows(h->fmt); }

bool valid_matrix(const dflash2_matrix& m, int fmt) {
  if (!m.w || !aligned16(m.w)) return false;
  // Q8 scale/bias rows are read 8 groups (16 bytes) at a time
  if (fmt == DFLASH2_WEIGHTS_Q8G64 && (!m.scale || !m.bias || !aligned16(m.scale) || !aligned16(m.bias))) return false;
  return true;
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
  if (c.head_dim != 128 || (c.block != 8 && c.block != 16) || c.top_k != 16 || c.rank != 256 || c.conv_taps != 2 ||
      c.conv_group != 16 || c.n_layers > DFLASH2_MAX_LAYERS || c.n_q_heads != 4 * c.n_kv_heads ||
      c.hidden % 256 || c.ffn % (c.weight_format == DFLASH2_WEIGHTS_BF16 ? 128 : 256) || c.vocab % 16 ||
      max_requests * c.block > 8 * DFLASH2_MAX_REQUESTS ||
      (c.window - 1 + kAttnChunk - 1) / kAttnChunk + 1 > 64)
    return DFLASH2_E_UNSUPPORTED;
  const int fmt = c.weight_format;
  // the tensor-core GEMM (handles of wide_min_rows or more block rows) takes weight
  // blocks of 128 rows: the delta projections' hidden/4 and the vocabulary
  if (max_requests * c.block >= wide_min_rows(fmt) && ((c.hidden / 4) % 128 || c.vocab % 128))
    return DFLASH2_E_UNSUPPORTED;
  // norm weights and convolution bases are read 4 channels (8 bytes) at a time
  if (!w->embed || !w->lm_head || !w->hidden_norm || !w->final_norm || !aligned16(w->lm_head) ||
      !aligned16(w->hidden_norm) || !aligned16(w->final_norm))
    return DFLASH2_E_INVAL;
  if (!valid_matrix(w->fc, fmt) || !valid_matrix(w->sel_proj, fmt) || !valid_matrix(w->cb_a, fmt) ||
      !valid_matrix(w->cb_b, fmt))
    return DFLASH2_E_INVAL;
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash2_layer_weights& L = w->layers[l];
    if (!L.input_norm || !L.post_norm || !L.q_norm || !L.k_norm || !L.attn_base || !L.mlp_base) return DFLASH2_E_INVAL;
    if (!aligned16(L.input_norm) || !aligned16(L.post_norm) || !aligned16(L.attn_base) || !aligned16(L.mlp_base))
      return DFLASH2_E_INVAL;
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
  h->B = c.block;
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
  h->nch_ss = c.hidden / 32;
  h->n_attn_chunks = (c.window - 1 + kAttnChunk - 1) / kAttnChunk + 1;
  h->n_verify_chunks = (c.vocab + kVerifyChunk - 1) / kVerifyChunk;
  h->lm_ctas = lmhead_ctas(h->num_sms);
  // plane maps of every projection launch (shapes only; the same plans as launch_gemv's
  // and launch_wide's), and the largest plane count of each output buffer over both
  h->wide = max_requests * h->B >= wide_min_rows(fmt);
  h->lm_chunks = (c.vocab + kLogitChunk - 1) / kLogitChunk;
  int maxp_fc = 0, maxp_d = 0, maxp_q = 0, maxp_k = 0, maxp_v = 0, maxp_y = 0, maxp_g = 0, maxp_u = 0, maxp_sel = 0,
      maxp_lm = 0;
  {
    auto shape = [](int M, int K) {
      GemvSeg g;
      memset(&g, 0, sizeof(g));
      g.M = M;
      g.K = K;
      g.n_tiles = 1;
      return g;
    };
    for (int path = 0; path < (h->wide ? 2 : 1); ++path) {
      dflash2_handle::PlaneSet& P = path == 0 ? h->pn : h->pw;
      auto plan = [&](std::initializer_list<GemvSeg> segs, std::initializer_list<GemvPlanes*> pls,
                      std::initializer_list<int*> maxes, int f, int nmax = 128) {
        GemvArgs a;
        memset(&a, 0, sizeof(a));
        for (const GemvSeg& g : segs) a.seg[a.nseg++] = g;
        const int C = path == 0 ? gemv_plan(a, h->num_sms, fmt) : wide_plan(a, h->num_sms, f, nmax);
        int i = 0;
        for (GemvPlanes* p : pls) *p = path == 0 ? gemv_planes(a, i++, C) : wide_planes(a, i++, C);
        i = 0;
        for (int* mx : maxes) {
          const int n = path == 0 ? gemv_max_planes(a, i, C) : wide_max_planes(a, i, C);
          *mx = std::max(*mx, n);
          ++i;
        }
      };
      plan({shape(h->H, h->KT), shape(4 * h->G, h->H)}, {&P.fc, &P.d0}, {&maxp_fc, &maxp_d}, fmt);
      plan({shape(4 * h->G, h->H)}, {&P.d}, {&maxp_d}, fmt);
      plan({shape(h->qd, h->H), shape(h->kvd, h->H), shape(h->kvd, h->H)}, {&P.q, &P.k, &P.v},
           {&maxp_q, &maxp_k, &maxp_v}, fmt);
      // the GEMM's launch with more than 128 key/value rows runs shorter int8 stages
      if (path == 1)
        plan({shape(h->qd, h->H), shape(h->kvd, h->H), shape(h->kvd, h->H)}, {&P.q2, &P.k2, &P.v2},
             {&maxp_q, &maxp_k, &maxp_v}, fmt, 256);
      plan({shape(h->H, h->qd)}, {&P.o}, {&maxp_y}, fmt);
      plan({shape(h->F, h->H), shape(h->F, h->H)}, {&P.g, &P.u}, {&maxp_g, &maxp_u}, fmt);
      plan({shape(h->H, h->F)}, {&P.down}, {&maxp_y}, fmt);
      plan({shape(c.rank, h->H)}, {&P.sel}, {&maxp_sel}, fmt);
      if (path == 1) plan({shape(h->V, h->H)}, {&P.lm}, {&maxp_lm}, 0);
    }
  }
  bool maps_ok = gemv_encode_wmap(&h->map_fc, w->fc.w, h->H, h->KT, fmt) &&
            gemv_encode_wmap(&h->map_sel, w->sel_proj.w, c.rank, h->H, fmt);
  for (int l = 0; l < c.n_layers && maps_ok; ++l) {
    const dflash2_layer_weights& L = w->layers[l];
    const struct {
      const dflash2_matrix* m;
      int M, K;
    } mats[9] = {{&L.q, h->qd, h->H},        {&L.k, h->kvd, h->H},     {&L.v, h->kvd, h->H},
                 {&L.o, h->H, h->qd},        {&L.gate, h->F, h->H},    {&L.up, h->F, h->H},
                 {&L.down, h->H, h->F},      {&L.attn_delta, 4 * h->G, h->H}, {&L.mlp_delta, 4 * h->G, h->H}};
    for (int i = 0; i < 9 && maps_ok; ++i) maps_ok = gemv_encode_wmap(&h->map_layer[l][i], mats[i].m->w, mats[i].M, mats[i].K, fmt);
  }
  if (h->wide) {
    // the tensor-core GEMM: 128-row weight blocks (every output width a multiple of 128)
    maps_ok = maps_ok && (4 * h->G) % 128 == 0 && h->V % 128 == 0 &&
              wide_encode_wmap(&h->wmap_fc, w->fc.w, h->H, h->KT, fmt) &&
              wide_encode_wmap(&h->wmap_sel, w->sel_proj.w, c.rank, h->H, fmt) &&
              wide_encode_wmap(&h->wmap_lm, w->lm_head, h->V, h->H, 0);
    for (int l = 0; l < c.n_layers && maps_ok; ++l) {
      const dflash2_layer_weights& L = w->layers[l];
      const dflash2_matrix* ms[9] = {&L.q, &L.k, &L.v, &L.o, &L.gate, &L.up, &L.down, &L.attn_delta, &L.mlp_delta};
      const int MK[9][2] = {{h->qd, h->H}, {h->kvd, h->H}, {h->kvd, h->H}, {h->H, h->qd}, {h->F, h->H},
                            {h->F, h->H}, {h->H, h->F}, {4 * h->G, h->H}, {4 * h->G, h->H}};
      for (int i = 0; i < 9 && maps_ok; ++i)
        maps_ok = wide_encode_wmap(&h->wmap_layer[l][i], ms[i]->w, MK[i][0], MK[i][1], fmt);
    }
  }
  if (!maps_ok) {
    delete h;
    return DFLASH2_E_UNSUPPORTED;
  }
  const size_t N = static_cast<size_t>(h->B) * max_requests;  // block rows
  const size_t esz = 2;  // bf16 / fp16 activations
  struct Buf {
    void** p;
    size_t bytes;
  };
  const Buf bufs[] = {
      {reinterpret_cast<void**>(&h->x), N * h->H * 4},
      {reinterpret_cast<void**>(&h->ss), N * h->nch_ss * 4},
      {reinterpret_cast<void**>(&h->ss_c), N * h->nch_ss * 4},
      {reinterpret_cast<void**>(&h->dproj), maxp_d * N * 4 * h->G * 4},
      {reinterpret_cast<void**>(&h->delta_a), N * 4 * h->G * 4},
      {reinterpret_cast<void**>(&h->delta_m), N * 4 * h->G * 4},
      {reinterpret_cast<void**>(&h->fc_out), maxp_fc * N * h->H * 4},
      {reinterpret_cast<void**>(&h->q_out), maxp_q * N * h->qd * 4},
      {reinterpret_cast<void**>(&h->k_out), maxp_k * 2 * N * h->kvd * 4},
      {reinterpret_cast<void**>(&h->v_out), maxp_v * 2 * N * h->kvd * 4},
      {reinterpret_cast<void**>(&h->sel_out), maxp_sel * N * c.rank * 4},
      {reinterpret_cast<void**>(&h->q), N * h->qd * 4},
      {reinterpret_cast<void**>(&h->kb), N * h->kvd * 4},
      {reinterpret_cast<void**>(&h->vb), N * h->kvd * 4},
      // per (request, KV head, part): 4 B queries x (max, sum, 128 outputs)
      {reinterpret_cast<void**>(&h->attn_part), 4 * N * h->nkv * h->n_attn_chunks * 130 * 4},
      {reinterpret_cast<void**>(&h->ypart), maxp_y * N * h->H * 4},
      {reinterpret_cast<void**>(&h->gpart), maxp_g * N * h->F * 4},
      {reinterpret_cast<void**>(&h->upart), maxp_u * N * h->F * 4},
      {reinterpret_cast<void**>(&h->act_a), 2 * N * h->H * esz},  // hi and lo planes
      {reinterpret_cast<void**>(&h->act_qkv), 2 * 2 * N * h->H * esz},
      {reinterpret_cast<void**>(&h->act_taps), 2 * N * h->KT * esz},
      {reinterpret_cast<void**>(&h->act_o), 2 * N * h->qd * esz},
      {reinterpret_cast<void**>(&h->act_h), 2 * N * h->F * esz},
      {reinterpret_cast<void**>(&h->act_fin), 2 * N * h->H * 2},
      {reinterpret_cast<void**>(&h->topk_keys), N * std::max(h->lm_ctas, h->wide ? h->lm_chunks : 0) * 16 * 8},
      {reinterpret_cast<void**>(&h->lm_part), static_cast<size_t>(maxp_lm) * N * h->V * 4},
      {reinterpret_cast<void**>(&h->vstats),
       N * h->n_verify_chunks * sizeof(VerifyStat)},
      {reinterpret_cast<void**>(&h->inv_freq), 64 * 8},
      {reinterpret_cast<void**>(&h->gemv_err), 4},
      {reinterpret_cast<void**>(&h->verify_cnt), static_cast<size_t>(max_requests) * 4},
      {reinterpret_cast<void**>(&h->sel_lat), static_cast<size_t>(max_requests) * (h->B - 1) * 16 * 16 * 4},
      {reinterpret_cast<void**>(&h->sel_bad), static_cast<size_t>(max_requests) * (h->B - 1) * 4},
      {reinterpret_cast<void**>(&h->sel_cnt), static_cast<size_t>(max_requests) * 4},
      {reinterpret_cast<void**>(&h->tstats),
       static_cast<size_t>(max_requests) * (kTreeMaxNodes + 1) * h->n_verify_chunks * sizeof(VerifyStat)},
      {reinterpret_cast<void**>(&h->tree_cnt), static_cast<size_t>(max_requests) * 4},
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
  // activation maps: one per GEMV input buffer (rows of one plane; the lo plane follows)
  const bool xok = gemv_encode_xmap(&h->xm_taps, h->act_taps, static_cast<int>(N), h->KT, fmt) &&
                   gemv_encode_xmap(&h->xm_a, h->act_a, static_cast<int>(N), h->H, fmt) &&
                   gemv_encode_xmap(&h->xm_qkv, h->act_qkv, static_cast<int>(2 * N), h->H, fmt) &&
                   gemv_encode_xmap(&h->xm_o, h->act_o, static_cast<int>(N), h->qd, fmt) &&
                   gemv_encode_xmap(&h->xm_h, h->act_h, static_cast<int>(N), h->F, fmt) &&
                   (fmt != 0 || gemv_encode_xmap(&h->xm_fin, h->act_fin, static_cast<int>(N), h->H, 0)) &&
                   lm_encode_map(&h->map_lm, w->lm_head, h->H, h->V, 64) &&
                   lm_encode_map(&h->xm_lm, h->act_fin, h->H, static_cast<int>(2 * N), 8);
  if (!xok) {
    cudaFree(h->arena);
    delete h;
    return DFLASH2_E_UNSUPPORTED;
  }
  *out = h;
  return DFLASH2_OK;
}

dflash2_status dflash2_destroy(dflash2_handle* h) {
  if (!h) return DFLASH2_E_INVAL;
  dflash2_step_graphs_clear(h);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
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

dflash2_status dflash2_set_projection_events(dflash2_handle* h, void* const* events, int32_t n_pairs) {
  if (!h || (events == nullptr) != (n_pairs == 0) || n_pairs < 0) return DFLASH2_E_INVAL;
  h->proj_ev = reinterpret_cast<cudaEvent_t*>(const_cast<void**>(events));
  h->proj_pairs = n_pairs;
  return DFLASH2_OK;
}

int32_t dflash2_projection_launches(const dflash2_handle* h) {
  if (!h) return -1;
  // fc + first delta; per layer: q/k/v, o, mlp delta, gate/up, down, and the attention
  // delta from the second layer on; the selector projection
  return 1 + h->cfg.n_layers * 5 + (h->cfg.n_layers - 1) + 1;
}

int64_t dflash2_projection_bytes(const dflash2_handle* h) {
  if (!h) return -1;
  const int64_t H = h->H, G4 = 4 * h->G;
  const int64_t per_layer = static_cast<int64_t>(h->qd) * H + 2 * static_cast<int64_t>(h->kvd) * H +
                            H * h->qd + 3 * static_cast<int64_t>(h->F) * H + 2 * G4 * H;
  const int64_t elems = per_layer * h->cfg.n_layers + H * h->KT + static_cast<int64_t>(h->cfg.rank) * H;
  // bf16: 2 bytes per weight; Q8/g64: one code byte plus a bf16 scale and bias per 64
  return h->fmt == DFLASH2_WEIGHTS_BF16 ? 2 * elems : elems + elems / 64 * 4;
}

dflash2_status dflash2_debug_set_pipeline_error(dflash2_handle* h, void* stream) {
  if (!h) return DFLASH2_E_INVAL;
  DF2_CHECK(cudaMemsetAsync(h->gemv_err, 1, sizeof(int), static_cast<cudaStream_t>(stream)));
  return DFLASH2_OK;
}

int64_t dflash2_lmhead_bytes(const dflash2_handle* h, int32_t n_req) {
  if (!h || n_req < 1) return -1;
  const int64_t N = static_cast<int64_t>(h->B) * n_req;
  if (wide_call(h, n_req))                         // tensor-core GEMM + chunked top-16
    return static_cast<int64_t>(h->V) * h->H * 2   // LM-head weights, read once
           + N * h->H * 2                          // bf16 hidden state, one plane
           + 2 * N * h->V * 4                      // logits written, then read by the top-16
           + N * h->lm_chunks * 16 * 8;            // per-chunk top-16 keys written
  return static_cast<int64_t>(h->V) * h->H * 2  // LM-head weights, read once
         + 2 * N * h->H * 2                      // bf16 hidden state, hi and lo planes
         + N * h->lm_ctas * 16 * 8;              // per-CTA top-16 keys written
}

dflash2_status dflash2_draft_block(dflash2_handle* h, int32_t n_req, const int32_t* anchor_ids,
                                   const int32_t* ctx_len, const int32_t* n_new, const float* taps, void* k_cache,
                                   void* v_cache, int32_t* cand_ids, float* cand_logits, float* gate,
                                   float* logits_out, const int32_t* width, void* stream) {
  if (!h || n_req < 1 || n_req > h->max_req) return DFLASH2_E_INVAL;
  if (!anchor_ids || !ctx_len || !n_new || !taps || !k_cache || !v_cache || !cand_ids || !cand_logits || !gate)
    return DFLASH2_E_INVAL;
  if (!aligned16(taps) || !aligned16(k_cache) || !aligned16(v_cache)) return DFLASH2_E_INVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DraftScope scope(h);
  const dflash2_config& c = h->cfg;
  const int fmt = h->fmt;
  const bool pdl = h->pdl;
  const int R = n_req, B = h->B;
  const int N = B * R;    // block rows
  const int NT = N / 8;   // 8-row tiles of the projections
  const int H = h->H, G = h->G;
  const size_t layer_stride = static_cast<size_t>(h->max_req) * h->kv_cap * h->kvd;  // elements
  const int N8 = B * h->max_req;  // rows of one plane of each activation buffer
  // many block rows: every projection on the tensor-core GEMM
  const bool wide = wide_call(h, R);
  const dflash2_handle::PlaneSet& P = wide ? h->pw : h->pn;
  // the tensor-core path reads its activations as one plane in the GEMM's operand
  // layout, slices of B max_requests rows rounded up to 16 (2 B max_requests for the
  // QKV input): a slice holds every row the MMA reads (rows rounded up to 16)
  const int tA = wide ? (N8 + 15) & ~15 : 0, tQ = wide ? 2 * N8 : 0;
  // the projections' inputs carry a low-order plane only on the GEMV path with bf16
  // weights (fp16 rounds to 2^-12 relative; the GEMM reads one plane)
  auto lo_of = [&](size_t lo) { return (wide || fmt != 0) ? static_cast<size_t>(0) : lo; };
  // ---- a2: block embedding, first norm input, taps packing
  {
    StartArgs a = {};
    a.anchor_ids = anchor_ids;
    a.n_new = n_new;
    a.embed = static_cast<const uint16_t*>(h->w.embed);
    a.norm_w = static_cast<const uint16_t*>(h->w.layers[0].input_norm);
    a.taps = taps;
    a.x = h->x;
    a.act_a = h->act_a;
    a.act_a_lo = lo_of(h->lo_a);
    a.tiled_a = tA;
    a.ss_x = h->ss;
    a.act_taps = h->act_taps;
    a.act_taps_lo = lo_of(h->lo_taps);
    a.tiled_taps = tA;
    a.H = H;
    a.n_taps = c.n_taps;
    a.mask_id = c.mask_token_id;
    a.nch = h->nch_ss;
    a.fmt = fmt;
    a.V = h->V;
    a.pipe_err = h->gemv_err;
    a.B = h->B;
    DF2_CHECK(launch_start(a, R, pdl, st));
    h->launches++;
  }
  // conv before the attention sublayer of layer l (delta projection already in dproj)
  auto conv_in_attn = [&](int l) {
    const dflash2_layer_weights& L = h->w.layers[l];
    ConvInArgs a = {};
    a.dproj = h->dproj;
    a.ss = h->ss;
    a.x = h->x;
    a.norm_w = static_cast<const uint16_t*>(L.input_norm);
    a.base = static_cast<const uint16_t*>(L.attn_base);
    a.delta = h->delta_a;
    a.act = h->act_qkv;
    a.act_lo = lo_of(h->lo_qkv);
    a.tiled = tQ;
    a.H = H;
    a.nch = h->nch_ss;
    a.fmt = fmt;
    a.pl = l == 0 ? P.d0 : P.d;
    a.n_rows = N;
    a.B = B;
    a.eps = c.rms_eps;
    return a;
  };
  // ---- a1 and layer 0's a3: the taps projection fc [H][n_taps H] and the first
  // delta projection read only what the start kernel wrote, so they share a launch;
  // so do the hidden_norm input of the context rows and the first conv-in.
  {
    dflash2_status s =
        run_gemv(h, wide,
                 {seg(h->map_fc, h->wmap_fc, h->w.fc, h->xm_taps, h->act_taps, N8, NT, H, h->KT, h->fc_out),
                  seg(h->map_layer[0][kAttnDelta], h->wmap_layer[0][kAttnDelta], h->w.layers[0].attn_delta, h->xm_a, h->act_a, N8, NT, 4 * G, H,
                      h->dproj)},
                 st);
    if (s) return s;
    FcFinishArgs a = {};
    a.y = h->fc_out;
    a.norm_w = static_cast<const uint16_t*>(h->w.hidden_norm);
    a.act = h->act_qkv;
    a.act_lo = lo_of(h->lo_qkv);
    a.tiled = tQ;
    a.ss = h->ss_c;
    a.H = H;
    a.act_row0 = N;
    a.nch = h->nch_ss;
    a.fmt = fmt;
    a.pl = P.fc;
    a.n_rows = N;
    DF2_CHECK(launch_fc_finish_conv_in(a, conv_in_attn(0), R, pdl, st));
    h->launches++;
  }
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash2_layer_weights& L = h->w.layers[l];
    uint16_t* kc = static_cast<uint16_t*>(k_cache) + l * layer_stride;
    uint16_t* vc = static_cast<uint16_t*>(v_cache) + l * layer_stride;
    dflash2_status s = DFLASH2_OK;
    if (l > 0) {
      // ---- a3: delta projection of the normed input, conv-in
      s = run_gemv(h, wide, {seg(h->map_layer[l][kAttnDelta], h->wmap_layer[l][kAttnDelta], L.attn_delta, h->xm_a, h->act_a, N8, NT, 4 * G, H, h->dproj)},
                   st);
      if (s) return s;
      DF2_CHECK(launch_conv_in(conv_in_attn(l), R, pdl, st));
      h->launches++;
    }
    // ---- a4: q (block rows), k and v (block + new context rows)
    s = run_gemv(h, wide,
                 {seg(h->map_layer[l][kQ], h->wmap_layer[l][kQ], L.q, h->xm_qkv, h->act_qkv, 2 * N8, NT, h->qd, H, h->q_out),
                  seg(h->map_layer[l][kK], h->wmap_layer[l][kK], L.k, h->xm_qkv, h->act_qkv, 2 * N8, 2 * NT, h->kvd, H, h->k_out),
                  seg(h->map_layer[l][kV], h->wmap_layer[l][kV], L.v, h->xm_qkv, h->act_qkv, 2 * N8, 2 * NT, h->kvd, H, h->v_out)},
                 st);
    if (s) return s;
    {
      QkvFinishArgs a = {};
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
      a.nch = h->nch_ss;
      const bool kv256 = wide && 2 * N > 128;  // the launch's plan (wide_nmax of its segments)
      a.pq = kv256 ? P.q2 : P.q;
      a.pk = kv256 ? P.k2 : P.k;
      a.pv = kv256 ? P.v2 : P.v;
      a.eps = c.rms_eps;
      a.B = h->B;
      DF2_CHECK(launch_qkv_finish(a, R, pdl, st));
      h->launches++;
    }
  // ---- a5: block attention over the window
    {
      AttnArgs a = {};
      a.q = h->q;
      a.kb = h->kb;
      a.vb = h->vb;
      a.k_cache = kc;
      a.v_cache = vc;
      a.ctx_len = ctx_len;
      a.n_new = n_new;
      a.part = h->attn_part;
      a.act_o = h->act_o;
      a.act_o_lo = lo_of(h->lo_o);
      a.tiled_o = tA;
      a.n_q_heads = h->nq;
      a.n_kv_heads = h->nkv;
      a.kv_capacity = h->kv_cap;
      a.window = c.window;
      a.cpc = attn_chunks_per_part(R, h->nkv, h->n_attn_chunks - 1, h->num_sms);
      a.n_chunks = (h->n_attn_chunks - 1 + a.cpc - 1) / a.cpc + 1;
      a.fmt = fmt;
      a.B = h->B;
      a.width = width;
      DF2_CHECK(launch_attention(a, R, pdl, st));
      h->launches += 2;
    }
    // ---- a6: output projection, conv-out + residual, post-attention norm input
    s = run_gemv(h, wide, {seg(h->map_layer[l][kO], h->wmap_layer[l][kO], L.o, h->xm_o, h->act_o, N8, NT, H, h->qd, h->ypart)}, st);
    if (s) return s;
    {
      ConvOutArgs a = {};
      a.part = h->ypart;
      a.delta = h->delta_a;
      a.base = static_cast<const uint16_t*>(L.attn_base);
      a.norm_w = static_cast<const uint16_t*>(L.post_norm);
      a.x = h->x;
      a.act = h->act_a;
      a.act_lo = lo_of(h->lo_a);
      a.tiled = tA;
      a.act2 = nullptr;
      a.act2_lo = 0;
      a.ss = h->ss;
      a.H = H;
      a.nch = h->nch_ss;
      a.fmt = fmt;
      a.pl = P.o;
      a.n_rows = N;
      a.B = h->B;
      DF2_CHECK(launch_conv_out(a, R, pdl, st));
      h->launches++;
    }
    // ---- a7: MLP sublayer
    s = run_gemv(h, wide, {seg(h->map_layer[l][kMlpDelta], h->wmap_layer[l][kMlpDelta], L.mlp_delta, h->xm_a, h->act_a, N8, NT, 4 * G, H, h->dproj)}, st);
    if (s) return s;
    {
      ConvInArgs a = {};
      a.dproj = h->dproj;
      a.ss = h->ss;
      a.x = h->x;
      a.norm_w = static_cast<const uint16_t*>(L.post_norm);
      a.base = static_cast<const uint16_t*>(L.mlp_base);
      a.delta = h->delta_m;
      a.act = h->act_qkv;
      a.act_lo = lo_of(h->lo_qkv);
      a.tiled = tQ;
      a.H = H;
      a.nch = h->nch_ss;
      a.fmt = fmt;
      a.pl = P.d;
      a.n_rows = N;
      a.eps = c.rms_eps;
      a.B = h->B;
      DF2_CHECK(launch_conv_in(a, R, pdl, st));
      h->launches++;
    }
    s = run_gemv(h, wide,
                 {seg(h->map_layer[l][kGate], h->wmap_layer[l][kGate], L.gate, h->xm_qkv, h->act_qkv, 2 * N8, NT, h->F, H, h->gpart),
                  seg(h->map_layer[l][kUp], h->wmap_layer[l][kUp], L.up, h->xm_qkv, h->act_qkv, 2 * N8, NT, h->F, H, h->upart)},
                 st);
    if (s) return s;
    {
      SwigluArgs a = {};
      a.part_g = h->gpart;
      a.part_u = h->upart;
      a.act = h->act_h;
      a.act_lo = lo_of(h->lo_h);
      a.tiled = tA;
      a.F = h->F;
      a.fmt = fmt;
      a.pg = P.g;
      a.pu = P.u;
      a.n_rows = N;
      DF2_CHECK(launch_swiglu(a, R, pdl, st));
      h->launches++;
    }
    s = run_gemv(h, wide, {seg(h->map_layer[l][kDown], h->wmap_layer[l][kDown], L.down, h->xm_h, h->act_h, N8, NT, H, h->F, h->ypart)}, st);
    if (s) return s;
    {
      const bool last = l == c.n_layers - 1;
      ConvOutArgs a = {};
      a.part = h->ypart;
      a.delta = h->delta_m;
      a.base = static_cast<const uint16_t*>(L.mlp_base);
      a.norm_w = static_cast<const uint16_t*>(last ? h->w.final_norm : h->w.layers[l + 1].input_norm);
      a.x = h->x;
      // LM-head input is bf16 in both formats; the next layer's input is in the matrices' format
      a.act = (last && fmt == 0) ? static_cast<void*>(h->act_fin) : h->act_a;
      a.act_lo = (last && fmt == 0) ? (wide ? 0 : h->lo_fin) : lo_of(h->lo_a);
      a.tiled = tA;
      a.act2 = (last && fmt != 0) ? h->act_fin : nullptr;
      a.act2_lo = wide ? 0 : h->lo_fin;
      a.tiled2 = tA;
      a.ss = h->ss;
      a.H = H;
      a.nch = h->nch_ss;
      a.fmt = fmt;
      a.pl = P.down;
      a.n_rows = N;
      a.B = h->B;
      DF2_CHECK(launch_conv_out(a, R, pdl, st));
      h->launches++;
    }
  }
  // ---- a8: LM head + top-16
  // external records: inside a stream capture they become event-record nodes the host can time
  if (h->ev_lm0) DF2_CHECK(cudaEventRecordWithFlags(h->ev_lm0, st, cudaEventRecordExternal));
  if (!wide) {
    LmHeadArgs a = {};
    a.wmap = h->map_lm;
    a.xmap = h->xm_lm;
    a.x_lo_row = N8;
    a.ss = h->ss;
    a.logits_out = logits_out;
    a.part_keys = h->topk_keys;
    a.V = h->V;
    a.H = H;
    a.n_rows = N;
    a.nch = h->nch_ss;
    a.n_cta = h->lm_ctas;
    a.eps = c.rms_eps;
    a.err = h->gemv_err;
    a.B = h->B;
    DF2_CHECK(launch_lmhead(a, pdl, st));
    h->launches++;
  } else {
    // logits of every block row as partial planes (tensor-core GEMM, bf16 hidden state),
    // then the top-16 of each vocabulary chunk of each sampled row
    dflash2_status s = run_gemv(
        h, true, {seg(h->map_lm, h->wmap_lm, dflash2_matrix{h->w.lm_head, nullptr, nullptr}, h->xm_lm, h->act_fin,
                      N8, NT, h->V, H, h->lm_part)},
        st, 0, false);
    if (s) return s;
    LogitsTopkArgs a = {};
    a.part = h->lm_part;
    a.ss = h->ss;
    a.logits_out = logits_out;
    a.part_keys = h->topk_keys;
    a.V = h->V;
    a.H = H;
    a.n_rows = N;
    a.nch = h->nch_ss;
    a.n_chunks = h->lm_chunks;
    a.eps = c.rms_eps;
    a.pl = P.lm;
    a.B = h->B;
    DF2_CHECK(launch_logits_topk(a, R, pdl, st));
    h->launches++;
  }
  if (h->ev_lm1) DF2_CHECK(cudaEventRecordWithFlags(h->ev_lm1, st, cudaEventRecordExternal));
  // ---- a9: selector projection (same final hidden, in the matrix's format), merge top-16
  {
    const CUtensorMap& xin = fmt == 0 ? h->xm_fin : h->xm_a;  // same final hidden, in the matrix's format
    const void* xin_p = fmt == 0 ? static_cast<const void*>(h->act_fin) : h->act_a;
    dflash2_status s = run_gemv(h, wide, {seg(h->map_sel, h->wmap_sel, h->w.sel_proj, xin, xin_p, N8, NT, c.rank, H, h->sel_out)}, st);
    if (s) return s;
    TopkMergeArgs a = {};
    a.part_keys = h->topk_keys;
    a.sel = h->sel_out;
    a.ss = h->ss;
    a.cand_ids = cand_ids;
    a.cand_logits = cand_logits;
    a.gate = gate;
    a.n_rows = N;
    a.n_cta = wide ? h->lm_chunks : h->lm_ctas;
    a.rank = c.rank;
    a.nch = h->nch_ss;
    a.psel = P.sel;
    a.H = H;
    a.eps = c.rms_eps;
    a.B = h->B;
    DF2_CHECK(launch_topk_merge(a, pdl, st));
    h->launches++;
  }
  return DFLASH2_OK;
}

dflash2_status dflash2_set_select_mode(dflash2_handle* h, int32_t mode) {
  if (!h || mode < 0 || mode > 1) return DFLASH2_E_INVAL;
  h->select_mode = mode;
  return DFLASH2_OK;
}

dflash2_status dflash2_advance(dflash2_handle* h, int32_t n_req, const int32_t* emitted, const int32_t* n_emitted,
                               int32_t* anchor_ids, int32_t* ctx_len, int32_t* n_new, uint64_t* philox_offset,
                               void* stream) {
  if (!h || n_req < 1 || n_req > h->max_req) return DFLASH2_E_INVAL;
  if (!emitted || !n_emitted || !anchor_ids || !ctx_len || !n_new || !philox_offset) return DFLASH2_E_INVAL;
  AdvanceArgs a = {};
  a.emitted = emitted;
  a.n_emitted = n_emitted;
  a.anchor_ids = anchor_ids;
  a.ctx_len = ctx_len;
  a.n_new = n_new;
  a.offset = philox_offset;
  a.B = h->B;
  DF2_CHECK(launch_advance(a, n_req, h->pdl, static_cast<cudaStream_t>(stream)));
  h->launches++;
  return DFLASH2_OK;
}

dflash2_status dflash2_block_width(dflash2_handle* h, int32_t n_req, const int32_t* ctx_len, const int32_t* n_new,
                                  int32_t ctx_threshold, int32_t narrow_width, int32_t* width, void* stream) {
  if (!h || n_req < 1 || n_req > h->max_req || !ctx_len || !n_new || !width) return DFLASH2_E_INVAL;
  if (ctx_threshold < 0 || narrow_width < 2 || narrow_width > h->B) return DFLASH2_E_INVAL;
  BlockWidthArgs a = {};
  a.ctx_len = ctx_len;
  a.n_new = n_new;
  a.width = width;
  a.B = h->B;
  a.threshold = ctx_threshold;
  a.narrow = narrow_width;
  DF2_CHECK(launch_block_width(a, n_req, h->pdl, static_cast<cudaStream_t>(stream)));
  h->launches++;
  return DFLASH2_OK;
}

dflash2_status dflash2_head_topk(dflash2_handle* h, int32_t n_rows, const void* hidden, int32_t* cand_ids,
                                 float* cand_logits, float* logits_out, void* stream) {
  if (!h || n_rows < h->B || n_rows % h->B || n_rows > h->B * h->max_req) return DFLASH2_E_INVAL;
  if (!hidden || !cand_ids || !cand_logits || !aligned16(hidden)) return DFLASH2_E_INVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (n_rows > 32) {  // more rows than the LM-head kernel holds: tensor-core GEMM, chunked top-16
    if (!h->wide) return DFLASH2_E_UNSUPPORTED;
    SegSpec sp = seg(h->map_lm, h->wmap_lm, dflash2_matrix{h->w.lm_head, nullptr, nullptr}, h->xm_lm, hidden, n_rows,
                     n_rows / 8, h->V, h->H, h->lm_part);
    sp.x_tiled = false;  // the caller's row-major hidden state: bulk tensor copies
    dflash2_status s = run_gemv(h, true, {sp}, st, 0, false);
    if (s) return s;
    LogitsTopkArgs a = {};
    a.part = h->lm_part;
    a.ss = nullptr;
    a.logits_out = logits_out;
    a.part_keys = h->topk_keys;
    a.V = h->V;
    a.H = h->H;
    a.n_rows = n_rows;
    a.nch = h->nch_ss;
    a.n_chunks = h->lm_chunks;
    a.eps = h->cfg.rms_eps;
    a.pl = h->pw.lm;
    a.B = h->B;
    DF2_CHECK(launch_logits_topk(a, n_rows / h->B, h->pdl, st));
    TopkMergeArgs m = {};
    m.part_keys = h->topk_keys;
    m.cand_ids = cand_ids;
    m.cand_logits = cand_logits;
    m.n_rows = n_rows;
    m.n_cta = h->lm_chunks;
    m.rank = h->cfg.rank;
    m.nch = h->nch_ss;
    m.H = h->H;
    m.eps = h->cfg.rms_eps;
    m.B = h->B;
    DF2_CHECK(launch_topk_merge(m, h->pdl, st));
    h->launches += 2;
    return DFLASH2_OK;
  }
  LmHeadArgs a = {};
  a.wmap = h->map_lm;
  if (!lm_encode_map(&a.xmap, hidden, h->H, n_rows, 8)) return DFLASH2_E_CUDA;
  a.x_lo_row = -1;
  a.ss = nullptr;
  a.logits_out = logits_out;
  a.part_keys = h->topk_keys;
  a.V = h->V;
  a.H = h->H;
  a.n_rows = n_rows;
  a.nch = h->nch_ss;
  a.n_cta = h->lm_ctas;
  a.eps = h->cfg.rms_eps;
  a.err = h->gemv_err;
  a.B = h->B;
  DF2_CHECK(launch_lmhead(a, h->pdl, st));
  TopkMergeArgs m = {};
  m.part_keys = h->topk_keys;
  m.sel = nullptr;
  m.ss = nullptr;
  m.cand_ids = cand_ids;
  m.cand_logits = cand_logits;
  m.gate = nullptr;
  m.n_rows = n_rows;
  m.n_cta = h->lm_ctas;
  m.rank = h->cfg.rank;
  m.nch = h->nch_ss;
  m.H = h->H;
  m.eps = h->cfg.rms_eps;
  m.B = h->B;
  DF2_CHECK(launch_topk_merge(m, h->pdl, st));
  h->launches += 2;
  return DFLASH2_OK;
}

dflash2_status dflash2_select(dflash2_handle* h, int32_t n_req, const int32_t* anchor_ids, const int32_t* cand_ids,
                              const float* cand_logits, const float* gate, const float* temperature,
                              const uint64_t* seed, const uint64_t* philox_offset, int32_t* path, float* q_rows,
                              float* scores_out, int32_t* status, const int32_t* width, void* stream) {
  if (!h || n_req < 1 || n_req > h->max_req) return DFLASH2_E_INVAL;
  if (!anchor_ids || !cand_ids || !cand_logits || !gate || !temperature || !seed || !philox_offset || !path ||
      !q_rows || !status)
    return DFLASH2_E_INVAL;
  SelectArgs a = {};
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
  a.lat = h->sel_lat;
  a.bad = h->sel_bad;
  a.counters = h->sel_cnt;
  a.mode = h->select_mode;
  a.width = width;
  a.pipe_err = h->gemv_err;
  a.rank = h->cfg.rank;
  a.fmt = h->fmt;
  a.V = h->V;
  a.B = h->B;
  DF2_CHECK(launch_select(a, n_req, h->pdl, static_cast<cudaStream_t>(stream)));
  h->launches++;
  return DFLASH2_OK;
}

dflash2_status dflash2_tree_build(dflash2_handle* h, int32_t n_req, int32_t budget, const int32_t* anchor_ids,
                                  const int32_t* cand_ids, const float* cand_logits, const float* gate,
                                  int32_t* node_token, int32_t* node_parent, int32_t* node_depth, float* node_score,
                                  int32_t* n_nodes, float* scores_out, int32_t* status, void* stream) {
  if (!h || n_req < 1 || n_req > h->max_req) return DFLASH2_E_INVAL;
  if (budget < 1 || budget > DFLASH2_TREE_MAX_NODES) return DFLASH2_E_INVAL;
  if (!anchor_ids || !cand_ids || !cand_logits || !gate || !node_token || !node_parent || !node_depth ||
      !node_score || !n_nodes || !status)
    return DFLASH2_E_INVAL;
  SelectArgs a = {};
  a.anchor_ids = anchor_ids;
  a.cand_ids = cand_ids;
  a.cand_logits = cand_logits;
  a.gate = gate;
  a.cb_a = h->w.cb_a.w;
  a.cb_a_scale = static_cast<const uint16_t*>(h->w.cb_a.scale);
  a.cb_a_bias = static_cast<const uint16_t*>(h->w.cb_a.bias);
  a.cb_b = h->w.cb_b.w;
  a.cb_b_scale = static_cast<const uint16_t*>(h->w.cb_b.scale);
  a.cb_b_bias = static_cast<const uint16_t*>(h->w.cb_b.bias);
  a.scores_out = scores_out;
  a.status = status;
  a.lat = h->sel_lat;
  a.bad = h->sel_bad;
  a.counters = h->sel_cnt;
  a.pipe_err = h->gemv_err;
  a.rank = h->cfg.rank;
  a.fmt = h->fmt;
  a.V = h->V;
  a.tree_budget = budget;
  a.t_token = node_token;
  a.t_parent = node_parent;
  a.t_depth = node_depth;
  a.t_score = node_score;
  a.t_n = n_nodes;
  a.B = h->B;
  DF2_CHECK(launch_select(a, n_req, h->pdl, static_cast<cudaStream_t>(stream)));
  h->launches++;
  return DFLASH2_OK;
}

dflash2_status dflash2_tree_verify(dflash2_handle* h, int32_t n_req, int32_t budget, const float* target_logits,
                                   const int32_t* node_token, const int32_t* node_parent, const int32_t* n_nodes,
                                   int32_t* n_accepted, int32_t* emitted, int32_t* n_emitted, int32_t* status,
                                   void* stream) {
  if (!h || n_req < 1 || n_req > h->max_req) return DFLASH2_E_INVAL;
  if (budget < 1 || budget > DFLASH2_TREE_MAX_NODES) return DFLASH2_E_INVAL;
  if (!target_logits || !node_token || !node_parent || !n_nodes || !n_accepted || !emitted || !n_emitted || !status)
    return DFLASH2_E_INVAL;
  TreeVerifyArgs a = {};
  a.logits = target_logits;
  a.token = node_token;
  a.parent = node_parent;
  a.n_nodes = n_nodes;
  a.stats = h->tstats;
  a.counters = h->tree_cnt;
  a.n_accepted = n_accepted;
  a.emitted = emitted;
  a.n_emitted = n_emitted;
  a.status = status;
  a.V = h->V;
  a.n_chunks = h->n_verify_chunks;
  a.budget = budget;
  a.B = h->B;
  DF2_CHECK(launch_tree_verify(a, n_req, h->pdl, static_cast<cudaStream_t>(stream)));
  h->launches++;
  return DFLASH2_OK;
}

dflash2_status dflash2_verify(dflash2_handle* h, int32_t n_req, const float* target_logits, const int32_t* path,
                              const int32_t* cand_ids, const float* q_rows, const float* temperature,
                              const uint64_t* seed, const uint64_t* philox_offset, int32_t* n_accepted,
                              int32_t* emitted, int32_t* n_emitted, float* probs_out, int32_t* status,
                              const int32_t* width, void* stream) {
  if (!h || n_req < 1 || n_req > h->max_req) return DFLASH2_E_INVAL;
  if (!target_logits || !path || !cand_ids || !q_rows || !temperature || !seed || !philox_offset || !n_accepted ||
      !emitted || !n_emitted || !status)
    return DFLASH2_E_INVAL;
  VerifyArgs a = {};
  a.logits = target_logits;
  a.path = path;
  a.cand_ids = cand_ids;
  a.q_rows = q_rows;
  a.temperature = temperature;
  a.seed = seed;
  a.offset = philox_offset;
  a.stats = h->vstats;
  a.counters = h->verify_cnt;
  a.n_accepted = n_accepted;
  a.emitted = emitted;
  a.n_emitted = n_emitted;
  a.status = status;
  a.probs = probs_out;
  a.width = width;
  a.V = h->V;
  a.n_chunks = h->n_verify_chunks;
  a.B = h->B;
  DF2_CHECK(launch_verify(a, n_req, h->pdl, static_cast<cudaStream_t>(stream)));
  h->launches += 1;
  return DFLASH2_OK;
}

dflash2_status dflash2_step_graphs_clear(dflash2_handle* h) {
  if (!h) return DFLASH2_E_INVAL;
  for (int i = 0; i < h->n_step_graphs; ++i)
    if (h->step_graph[i].exec) cudaGraphExecDestroy(h->step_graph[i].exec);
  h->n_step_graphs = 0;
  return DFLASH2_OK;
}

dflash2_status dflash2_step(dflash2_handle* h, const dflash2_step_args* args, void* stream) {
  if (!h || !args) return DFLASH2_E_INVAL;
  // the key: the fields only (a zeroed copy, so padding never differs)
  dflash2_step_args k;
  memset(&k, 0, sizeof(k));
  k.n_req = args->n_req;
  k.anchor_ids = args->anchor_ids;
  k.ctx_len = args->ctx_len;
  k.n_new = args->n_new;
  k.taps = args->taps;
  k.k_cache = args->k_cache;
  k.v_cache = args->v_cache;
  k.cand_ids = args->cand_ids;
  k.cand_logits = args->cand_logits;
  k.gate = args->gate;
  k.temperature = args->temperature;
  k.seed = args->seed;
  k.philox_offset = args->philox_offset;
  k.path = args->path;
  k.q_rows = args->q_rows;
  k.status = args->status;
  k.target_logits = args->target_logits;
  k.n_accepted = args->n_accepted;
  k.emitted = args->emitted;
  k.n_emitted = args->n_emitted;
  k.width = args->width;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // with profiling events set, the calls run as they are (a graph would keep recording
  // the events after the caller has cleared them)
  const bool profiling = h->ev_lm0 != nullptr || h->proj_ev != nullptr;
  for (int i = 0; i < h->n_step_graphs && !profiling; ++i) {
    dflash2_handle::StepGraph& g = h->step_graph[i];
    if (g.select_mode == h->select_mode && memcmp(&g.key, &k, sizeof(k)) == 0) {
      DF2_CHECK(cudaGraphLaunch(g.exec, st));
      h->launches += g.launches;
      g.used = ++h->step_clock;
      return DFLASH2_OK;
    }
  }
  // a new set: the three calls as they are, on the caller's stream
  auto run = [&](cudaStream_t s) {
    dflash2_status r = dflash2_draft_block(h, k.n_req, k.anchor_ids, k.ctx_len, k.n_new, k.taps, k.k_cache, k.v_cache,
                                           k.cand_ids, k.cand_logits, k.gate, nullptr, k.width, s);
    if (r == DFLASH2_OK)
      r = dflash2_select(h, k.n_req, k.anchor_ids, k.cand_ids, k.cand_logits, k.gate, k.temperature, k.seed,
                         k.philox_offset, k.path, k.q_rows, nullptr, k.status, k.width, s);
    if (r == DFLASH2_OK)
      r = dflash2_verify(h, k.n_req, k.target_logits, k.path, k.cand_ids, k.q_rows, k.temperature, k.seed,
                         k.philox_offset, k.n_accepted, k.emitted, k.n_emitted, nullptr, k.status, k.width, s);
    return r;
  };
  const dflash2_status r = run(st);
  if (r != DFLASH2_OK || profiling) return r;
  // then its graph, captured on the handle's own stream (nothing runs)
  if (!h->cap_stream && cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking) != cudaSuccess) {
    h->cap_stream = nullptr;
    cudaGetLastError();
    return DFLASH2_OK;
  }
  const int64_t n0 = h->launches;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  bool ok = cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
  if (ok) {
    const dflash2_status rc = run(h->cap_stream);
    ok = cudaStreamEndCapture(h->cap_stream, &graph) == cudaSuccess && rc == DFLASH2_OK && graph != nullptr;
  }
  const int64_t n_graph = h->launches - n0;
  h->launches = n0;  // the capture launched nothing
  if (ok) ok = cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess;
  if (graph) cudaGraphDestroy(graph);
  if (!ok) {
    cudaGetLastError();  // the set stays uncached; the step itself has run
    return DFLASH2_OK;
  }
  int slot = h->n_step_graphs;
  if (slot == DFLASH2_STEP_GRAPHS) {  // replace the least recently used
    slot = 0;
    for (int i = 1; i < DFLASH2_STEP_GRAPHS; ++i)
      if (h->step_graph[i].used < h->step_graph[slot].used) slot = i;
    cudaGraphExecDestroy(h->step_graph[slot].exec);
  } else {
    ++h->n_step_graphs;
  }
  h->step_graph[slot].key = k;
  h->step_graph[slot].select_mode = h->select_mode;
  h->step_graph[slot].exec = exec;
  h->step_graph[slot].launches = n_graph;
  h->step_graph[slot].used = ++h->step_clock;
  return DFLASH2_OK;
}

}  // extern "C"
