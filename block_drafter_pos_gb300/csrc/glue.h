// Argument blocks of the element-wise stages (glue.cu) and of the attention,
// LM-head, selector and verify kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace df2 {

// Activation buffers hold a high plane and, at element offset *_lo, a low-order
// plane (value = hi + lo); bf16 for BF16 weights (fmt 0), fp16 for Q8 (fmt 1).

struct StartArgs {
  const int32_t* anchor_ids;
  const int32_t* n_new;
  const uint16_t* embed;   // bf16 [V][H]
  const uint16_t* norm_w;  // input_norm of layer 0
  const float* taps;       // [R][8][n_taps*H]
  float* x;                // residual stream [N][H]
  void* act_a;             // x * w: input of layer 0's delta projection [N][H]
  size_t act_a_lo;
  float* ss_x;             // [N][H/32]
  void* act_taps;          // [N][n_taps*H]
  size_t act_taps_lo;
  int H, n_taps, mask_id, nch, fmt, V;
  int B;                    // block positions per request (8 or 16); rows are request-major
  int tiled_a, tiled_taps;  // > 0: tensor-core operand layout with that many rows per slice (act_offset)
  int* pipe_err;            // the step's weight-pipeline error word, cleared here (may be NULL)
};

struct FcFinishArgs {
  const float* y;          // taps projection partial planes [p][N][H]
  const uint16_t* norm_w;  // hidden_norm
  void* act;               // QKV input; context rows start at act_row0
  size_t act_lo;
  float* ss;               // [N][H/32] sums of squares of y
  int H, act_row0, nch, fmt, n_rows;
  GemvPlanes pl;           // planes of y
  int tiled;               // > 0: act in the tensor-core operand layout (act_offset)
};

struct ConvInArgs {
  const float* dproj;      // delta projection partial planes of x * w, [p][N][4G] (not yet scaled by 1/rms)
  const float* ss;         // [N][nch] sums of squares of x
  const float* x;          // residual stream
  const uint16_t* norm_w;
  const uint16_t* base;    // [4][H]
  float* delta;            // out: [N][4G] scaled by 1/rms
  void* act;               // out: conv-in'd sublayer input [N][H]
  size_t act_lo;
  int H, nch, fmt, n_rows;
  float eps;
  GemvPlanes pl;           // planes of dproj
  int tiled;               // > 0: act in the tensor-core operand layout (act_offset)
  int B;                   // block positions per request (the convolution stops at a block's start)
};

// Dynamic convolution after a sublayer, residual add, next norm's input.
struct ConvOutArgs {
  const float* part;       // sublayer output partial planes [p][N][H]
  const float* delta;      // [N][4G] (io 1 = conv after the sublayer)
  const uint16_t* base;    // [4][H]
  const uint16_t* norm_w;  // norm weight of the next sublayer
  float* x;                // residual stream [N][H], updated in place
  void* act;               // x * w_next in the next projection's format, plus low plane at act + act_lo
  size_t act_lo;
  uint16_t* act2;          // optional bf16 copy (LM-head input), or null
  size_t act2_lo;
  float* ss;               // [N][H/32] sums of squares of the updated x
  int H, nch, fmt, n_rows;
  GemvPlanes pl;           // planes of part
  int tiled, tiled2;       // > 0: act / act2 in the tensor-core operand layout (act_offset)
  int B;                   // block positions per request (the convolution stops at a block's start)
};

// SwiGLU of the gate and up projections: act = silu(gate) * up.
struct SwigluArgs {
  const float* part_g;     // gate partial planes [p][N][F]
  const float* part_u;     // up partial planes [p][N][F]
  void* act;               // [N][F] plus low plane at act + act_lo
  size_t act_lo;
  int F, fmt, n_rows;
  GemvPlanes pg, pu;       // planes of the two projections
  int tiled;               // > 0: act in the tensor-core operand layout (act_offset)
};

struct QkvFinishArgs {
  const float* q_out;      // partial planes [p][N][nq*128]
  const float* k_out;      // partial planes [p][2N][nkv*128]: block rows, then context rows
  const float* v_out;
  const float* ss_c;       // [N][nch] of the projected taps
  const uint16_t* q_norm;
  const uint16_t* k_norm;
  const double* inv_freq;  // [64]
  const int32_t* ctx_len;
  const int32_t* n_new;
  float* q;                // [N][nq][128]
  float* kb;               // [N][nkv][128]
  float* vb;
  uint16_t* k_cache;       // this layer's slice: [max_req][cap][nkv][128]
  uint16_t* v_cache;
  int n_q_heads, n_kv_heads, n_rows, kv_capacity, H, nch;
  float eps;
  GemvPlanes pq, pk, pv;   // planes of the three projections
  int B;                   // block positions per request; new context rows per request <= B
};

cudaError_t launch_start(const StartArgs& a, int n_req, bool pdl, cudaStream_t st);
cudaError_t launch_conv_in(const ConvInArgs& a, int n_req, bool pdl, cudaStream_t st);
cudaError_t launch_fc_finish_conv_in(const FcFinishArgs& f, const ConvInArgs& c, int n_req, bool pdl, cudaStream_t st);
cudaError_t launch_qkv_finish(const QkvFinishArgs& a, int n_req, bool pdl, cudaStream_t st);
cudaError_t launch_conv_out(const ConvOutArgs& a, int n_req, bool pdl, cudaStream_t st);
cudaError_t launch_swiglu(const SwigluArgs& a, int n_req, bool pdl, cudaStream_t st);

// ---------------------------------------------------------------- attention
struct AttnArgs {
  const float* q;          // [N][nq][128]
  const float* kb;         // [N][nkv][128]
  const float* vb;
  const uint16_t* k_cache; // this layer's slice [max_req][cap][nkv][128]
  const uint16_t* v_cache;
  const int32_t* ctx_len;
  const int32_t* n_new;
  float* part;             // [R][nkv][n_chunks][32][130] per part: (m, l, unnormalised output) of 32 queries
  void* act_o;             // [N][nq*128]
  size_t act_o_lo;
  int n_q_heads, n_kv_heads, kv_capacity, window, fmt;
  int n_chunks;            // parts: ceil(context chunks / cpc) + 1 (the block keys)
  int cpc;                 // context chunks of 64 keys per part
  int tiled_o;             // > 0: act_o in the tensor-core operand layout (act_offset)
  int B;                   // block positions per request (8 or 16): 4 B queries per KV head group
  const int32_t* width;    // [R] block width of each request (2..B; keys at positions >= width are
                           // masked, so its first width rows are a block-width forward), or null: B
};
constexpr int kAttnChunk = 64;
cudaError_t launch_attention(const AttnArgs& a, int n_req, bool pdl, cudaStream_t st);

// ---------------------------------------------------------------- LM head + top-k
struct LmHeadArgs {
  CUtensorMap wmap;        // LM head bf16 [V][H] (lm_encode_map, 64-row boxes)
  CUtensorMap xmap;        // hidden bf16 [rows][H], hi plane rows then lo plane rows (8-row boxes)
  int x_lo_row;            // first row of the low-order plane in xmap, or -1 (none)
  const float* ss;         // [N][nch] sums of squares of x, or null (x already normalised)
  float* logits_out;       // [R][7][V] or null
  unsigned long long* part_keys;  // [N][n_cta][16]
  int V, H, n_rows, nch, n_cta;
  float eps;
  int* err;                // set nonzero if a pipeline wait gave up, or null
  int B;                   // block positions per request: row n is position n % B of request n / B
};
// Bulk-copy map of a bf16 matrix [rows][inner] in boxes of box_rows x 64 elements
// (128-byte rows, 128-byte swizzle); rows past the end read as zero.
bool lm_encode_map(CUtensorMap* map, const void* p, int inner, int rows, int box_rows);
// CTAs of the LM-head launch (the per-CTA candidate lists the merge reads).
int lmhead_ctas(int num_sms);
cudaError_t launch_lmhead(const LmHeadArgs& a, bool pdl, cudaStream_t st);

// Top-16 of the LM head's logits when they come from the tensor-core GEMM as partial
// planes: grid (n_chunks, 7 R), one non-anchor row x kLogitChunk vocabulary entries
// per CTA; writes that chunk's 16 largest keys to part_keys[n][chunk] (the layout of
// the LM-head kernel's per-CTA lists, so the same merge follows) and, if asked, the
// logits.
constexpr int kLogitChunk = 4096;
struct LogitsTopkArgs {
  const float* part;       // [p][N][V] partial planes of W_lm h (h not yet scaled by 1/rms)
  const float* ss;         // [N][nch] sums of squares of the final hidden state
  float* logits_out;       // [R][7][V] or null
  unsigned long long* part_keys;  // [N][n_chunks][16]
  int V, H, n_rows, nch, n_chunks;
  float eps;
  GemvPlanes pl;           // planes of part
  int B;                   // block positions per request
};
cudaError_t launch_logits_topk(const LogitsTopkArgs& a, int n_req, bool pdl, cudaStream_t st);

struct TopkMergeArgs {
  const unsigned long long* part_keys;  // [N][n_cta][16]
  const float* sel;        // selector projection partial planes [p][N][rank], or null
  const float* ss;
  int32_t* cand_ids;       // [R][7][16]
  float* cand_logits;
  float* gate;             // [R][7][rank]
  int n_rows, n_cta, rank, nch, H;
  float eps;
  GemvPlanes psel;         // planes of sel
  const int* err;          // or null: when nonzero, every row gets the sentinel (ids -1, logits NaN)
  int B;                   // block positions per request
};
cudaError_t launch_topk_merge(const TopkMergeArgs& a, bool pdl, cudaStream_t st);

// ---------------------------------------------------------------- selector
struct SelectArgs {
  const int32_t* anchor_ids;
  const int32_t* cand_ids;     // [R][7][16]
  const float* cand_logits;
  const float* gate;           // [R][7][rank]
  const float* temperature;
  const uint64_t* seed;
  const uint64_t* offset;
  const void* cb_a;            // bf16 [V][rank] or int8 codes
  const uint16_t* cb_a_scale;
  const uint16_t* cb_a_bias;
  const void* cb_b;
  const uint16_t* cb_b_scale;
  const uint16_t* cb_b_bias;
  int32_t* path;
  float* q_rows;
  float* scores_out;           // [R][7][16][16] or null
  int32_t* status;
  float* lat;                  // scratch [R][7][16][16]: the lattice's scores, one position per CTA
  int32_t* bad;                // scratch [R][7]: nonfinite logit or score seen at that position
  unsigned int* counters;      // [R] finished positions of the launch; zero before and after it
  int rank, fmt, V;
  int mode;                    // 0: sequential walk; 1: globally best path (Viterbi) for greedy requests
  const int* pipe_err;         // nonzero: a pipeline wait of the step's draft gave up (may be NULL)
  // draft tree instead of a path (tree_budget > 0): best-first growth over the lattice
  int tree_budget;
  int32_t* t_token;            // [R][tree_budget]
  int32_t* t_parent;           // [R][tree_budget]: -1 = the root (anchor), else an earlier node
  int32_t* t_depth;            // [R][tree_budget]: block position 1..7
  float* t_score;              // [R][tree_budget]: cumulative log-probability
  int32_t* t_n;                // [R]: nodes built
  int B;                       // block positions per request: B - 1 proposal positions
  const int32_t* width;        // [R] block width (2..B): positions 1..width-1 are walked; null: B
};
constexpr int kTreeMaxNodes = 32;
constexpr int kMaxBlock = 16;  // block positions per request: 8 or 16
cudaError_t launch_select(const SelectArgs& a, int n_req, bool pdl, cudaStream_t st);



// ---------------------------------------------------------------- verify
constexpr int kVerifyChunk = 4096;
struct VerifyStat {
  float m;       // chunk max (of z)
  float s;       // sum exp((z - m) / T) over the chunk (T > 0), compensated: the sum is s + s_lo
  float s_lo;
  int32_t arg;   // argmax (smallest index among equal maxima)
  int32_t flags; // bit 0: NaN seen, bit 1: +inf seen
};
struct VerifyArgs {
  const float* logits;         // [R][8][V]
  const int32_t* path;         // [R][7]
  const int32_t* cand_ids;     // [R][7][16]
  const float* q_rows;         // [R][7][16]
  const float* temperature;
  const uint64_t* seed;
  const uint64_t* offset;
  VerifyStat* stats;           // [R][8][n_chunks]
  int32_t* n_accepted;
  int32_t* emitted;            // [R][8]
  int32_t* n_emitted;
  int32_t* status;
  float* probs;                // [R][8][2] or null: p_j at the proposal / bonus, residual mass (debug output)
  unsigned int* counters;      // [R] finished chunk statistics of the launch; zero before and after it
  int V, n_chunks;
  int B;                       // block positions per request: B target rows, B - 1 proposals
  const int32_t* width;        // [R] block width (2..B): rows 0..width-1 are verified; null: B
};
cudaError_t launch_verify(const VerifyArgs& a, int n_req, bool pdl, cudaStream_t st);

// ---------------------------------------------------------------- draft-tree verification (greedy)
struct TreeVerifyArgs {
  const float* logits;         // [R][budget + 1][V]: row 0 the root, row 1 + k node k
  const int32_t* token;        // [R][budget]
  const int32_t* parent;       // [R][budget]
  const int32_t* n_nodes;      // [R]
  VerifyStat* stats;           // [R][budget + 1][n_chunks]
  unsigned int* counters;      // [R] (zero between launches)
  int32_t* n_accepted;
  int32_t* emitted;            // [R][8]
  int32_t* n_emitted;
  int32_t* status;
  int V, n_chunks, budget;
  int B;                       // block positions per request (emitted rows)
};
cudaError_t launch_tree_verify(const TreeVerifyArgs& a, int n_req, bool pdl, cudaStream_t st);

// ---------------------------------------------------------------- serving-loop state update
struct AdvanceArgs {
  const int32_t* emitted;   // [R][8]
  const int32_t* n_emitted; // [R]
  int32_t* anchor_ids;      // [R] in/out
  int32_t* ctx_len;         // [R] in/out
  int32_t* n_new;           // [R] in/out
  uint64_t* offset;         // [R] in/out
  int B;                    // block positions per request
};
cudaError_t launch_advance(const AdvanceArgs& a, int n_req, bool pdl, cudaStream_t st);

// Block width of each request by context length: width[r] = narrow if threshold > 0
// and ctx_len[r] + n_new[r] > threshold, else B.
struct BlockWidthArgs {
  const int32_t* ctx_len;
  const int32_t* n_new;
  int32_t* width;
  int B, threshold, narrow;
};
cudaError_t launch_block_width(const BlockWidthArgs& a, int n_req, bool pdl, cudaStream_t st);

}  // namespace df2
