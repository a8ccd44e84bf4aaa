/*
 * dflash2.h - C ABI of one DFlash2 draft + select + verify step on an sm_103a GPU.
 *
 * The step is the one described by the DFlash2 pages:
 *   - "LSE docs/DFLASH2.md": drafter geometry (5 layers, width 5120, 32 query /
 *     8 KV heads, head dim 128, FFN 17408, RoPE theta 1e7), the 8-position block
 *     (anchor + 7 mask tokens, noncausal, 2048-key sliding window over context
 *     K/V), 2-tap dynamic convolution over groups of 16 channels, top-16
 *     candidates with rank-256 selector codebooks, probability-ratio rejection
 *     with residual sampling, the top-k ordering policy and the affine Q8/g64
 *     weight format;
 *   - "[Spec Decode] DFlash2: local convolution + candidate selector - #52816"
 *     (vLLM PR description): the convolution formula, the selector edge score,
 *     the walk from the verified anchor and the q returned for the verify;
 *   - "qwen35: DSpark speculative decoding (Qwen3.8-27B drafters) - #625": the
 *     wider draft block (16 positions; greedy chains stay those of plain decoding
 *     at any width), the long-context narrowing of the block, and the draft tree.
 *
 * Blocks: a handle drafts blocks of B = cfg.block positions (8 or 16): position 0
 * is the anchor, 1..B-1 are mask tokens, so a request has B - 1 proposals and B
 * target rows.  Rows of per-position tensors are request-major.  A request may be
 * narrowed to a block width w (2..B) for a step (`width` arguments; see
 * dflash2_block_width): it is then drafted, walked and verified exactly as a block
 * of w positions of the same drafter, and entries for its positions w..B-1 are
 * unspecified (drafter outputs) or padding (path -1, q 0, emitted -1).
 *
 * Conventions (all entry points):
 *   - Every tensor argument is a DEVICE pointer owned by the caller, unless the
 *     argument says "host".  The handle owns only its scratch.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL =
 *     the legacy default stream).  They do not synchronise, and allocate nothing
 *     after dflash2_create.
 *   - Errors the host can see (bad sizes, NULL pointers, misalignment) return
 *     DFLASH2_E_INVAL before anything is launched.  A launch failure returns
 *     DFLASH2_E_CUDA.  Errors found on the device (a NaN or +inf logit or
 *     selector score; a bounded wait of a weight-streaming pipeline that gave up)
 *     go to the per-request `status` words; such a request gets
 *     n_accepted = n_emitted = 0.
 *   - Stream order holds for every input: a call's first kernel waits for the
 *     stream's earlier work before it reads one, even when that work is a kernel
 *     launched just before.  Weight copies may start earlier (overlapping the
 *     previous kernel), so the weights given to dflash2_create must not change
 *     while the handle is in use.
 *   - One handle serves one stream at a time (its scratch is shared by calls).
 *   - Integers are int32 unless stated; BF16 is stored as 16-bit patterns.
 */
#ifndef DFLASH2_H
#define DFLASH2_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t dflash2_status;
enum {
  DFLASH2_OK = 0,
  DFLASH2_E_INVAL = 1,        /* bad argument: size, NULL pointer, alignment            */
  DFLASH2_E_NONFINITE = 2,    /* device status word: NaN/+inf logit or selector score   */
  DFLASH2_E_CUDA = 3,         /* CUDA launch or runtime error                           */
  DFLASH2_E_UNSUPPORTED = 4   /* geometry or request count with no instantiated kernel  */
};

enum { DFLASH2_WEIGHTS_BF16 = 0, DFLASH2_WEIGHTS_Q8G64 = 1 };

#define DFLASH2_MAX_LAYERS 8
/* Largest max_requests of dflash2_create with blocks of 8; max_requests * block
 * <= 8 * DFLASH2_MAX_REQUESTS (128 block rows per step). */
#define DFLASH2_MAX_REQUESTS 16

/* Drafter geometry ("LSE docs/DFLASH2.md", compatible-drafter paragraph). */
typedef struct dflash2_config {
  int32_t hidden;         /* H: 5120                                              */
  int32_t n_layers;       /* 5 (<= DFLASH2_MAX_LAYERS)                            */
  int32_t n_q_heads;      /* 32                                                   */
  int32_t n_kv_heads;     /* 8                                                    */
  int32_t head_dim;       /* 128 (the only value with kernels)                    */
  int32_t ffn;            /* F: 17408                                             */
  int32_t vocab;          /* V: 248320                                            */
  int32_t n_taps;         /* target feature taps: 5                               */
  int32_t block;          /* positions per draft block: 8 (anchor + 7 masks) or 16 */
  int32_t top_k;          /* candidates per position: 16                          */
  int32_t rank;           /* selector codebook rank: 256                          */
  int32_t window;         /* sliding window over context keys: 2048               */
  int32_t conv_taps;      /* dynamic convolution taps: 2                          */
  int32_t conv_group;     /* channels per dynamic coefficient: 16                 */
  int32_t mask_token_id;  /* id of the mask token (embedding row)                 */
  int32_t weight_format;  /* DFLASH2_WEIGHTS_BF16 or DFLASH2_WEIGHTS_Q8G64        */
  double rope_theta;      /* 1e7                                                  */
  float rms_eps;          /* RMSNorm epsilon: 1e-6                                */
} dflash2_config;

/* One weight matrix W [out][in], row-major.
 * BF16 format: w = bf16[out][in]; scale = bias = NULL.
 * Q8G64 format ("LSE docs/DFLASH2.md", Q8 paragraph): w = int8 codes [out][in],
 * scale and bias = bf16 [out][in/64]; the weight is scale * code + bias. */
typedef struct dflash2_matrix {
  const void* w;
  const void* scale;
  const void* bias;
} dflash2_matrix;

/* Per-layer weights.  Norm weights and convolution bases are BF16 in both formats.
 *   input_norm, post_norm [H]; q_norm, k_norm [head_dim]
 *   q [nq*hd][H], k [nkv*hd][H], v [nkv*hd][H], o [H][nq*hd]
 *   gate, up [F][H], down [H][F]
 *   attn_delta, mlp_delta [2*conv_taps*H/conv_group][H]: row (io*taps + t)*G + g,
 *     io 0 = the convolution before the sublayer, 1 = after it, G = H/conv_group
 *   attn_base, mlp_base [2*conv_taps][H]: row io*taps + t */
typedef struct dflash2_layer_weights {
  const void* input_norm;
  const void* post_norm;
  const void* q_norm;
  const void* k_norm;
  const void* attn_base;
  const void* mlp_base;
  dflash2_matrix q, k, v, o, gate, up, down, attn_delta, mlp_delta;
} dflash2_layer_weights;

/* All weights.  embed and lm_head [V][H] are BF16 (shared with the target);
 * fc [H][n_taps*H]; hidden_norm, final_norm [H]; sel_proj [rank][H];
 * cb_a, cb_b [V][rank] (selector codebooks, predecessor and successor). */
typedef struct dflash2_weights {
  const void* embed;
  const void* lm_head;
  const void* hidden_norm;
  const void* final_norm;
  dflash2_matrix fc, sel_proj, cb_a, cb_b;
  dflash2_layer_weights layers[DFLASH2_MAX_LAYERS];
} dflash2_weights;

typedef struct dflash2_handle dflash2_handle;

/* Creates a handle: validates the geometry, copies the weight pointers (the
 * weights stay caller-owned and must outlive the handle) and allocates the
 * scratch for up to `max_requests` requests.  `kv_capacity` is the number of
 * positions per request in the caller's K/V caches.  Must be called with the
 * target device current.  Returns DFLASH2_E_UNSUPPORTED for a geometry the
 * kernels do not cover: head_dim != 128, block not 8 or 16, top_k != 16, rank !=
 * 256, conv taps != 2 or group != 16, n_q_heads != 4 * n_kv_heads, hidden not a
 * multiple of 256, ffn not a multiple of 128 (BF16) or 256 (Q8G64), vocab not a
 * multiple of 16, more than DFLASH2_MAX_LAYERS layers, max_requests * block over
 * 8 * DFLASH2_MAX_REQUESTS, or a window over 64 attention chunks of 64 keys; and,
 * when max_requests * block reaches 40 (BF16) or 32 (Q8G64) rows, hidden / 4 or
 * vocab not a multiple of 128: calls with that many block rows run every
 * projection on the tensor-core GEMM, in 128-row weight blocks.  Every weight
 * matrix, Q8 scale and Q8 bias, and every norm weight and convolution base except
 * q_norm and k_norm, must start on a 16-byte boundary (DFLASH2_E_INVAL
 * otherwise).  Encodes one bulk-copy descriptor per projection matrix, so the
 * weights must not move while the handle lives. */
dflash2_status dflash2_create(const dflash2_config* cfg, const dflash2_weights* w, int32_t max_requests,
                              int32_t kv_capacity, dflash2_handle** out);

dflash2_status dflash2_destroy(dflash2_handle* h);

/* Draft block: steps a1-a9 of the method for n_req requests.
 *   anchor_ids [R]       verified anchor token of each request
 *   ctx_len [R]          keys already in the cache before this call
 *   n_new [R]            new context rows to append (0..block; at most the previous
 *                        step's width)
 *   taps [R][block][n_taps*H] float32: target feature taps of the new rows
 *                        (rows >= n_new[r] are ignored)
 *   k_cache, v_cache     bf16 [n_layers][max_requests][kv_capacity][nkv][hd]; rows
 *                        ctx_len..ctx_len+n_new-1 of each request are written (the
 *                        new context rows' K after k_norm and RoPE, and V), then
 *                        rows max(0, L-window+1)..L-1 are read, L = ctx_len+n_new
 *   cand_ids [R][block-1][top_k]     top-16 vocabulary ids of positions 1..block-1, in
 *                        order: NaN first (by id), then value descending, ties to
 *                        the smaller id ("LSE docs/DFLASH2.md", top-k paragraph)
 *   cand_logits [R][block-1][top_k] float32 drafter logits of those ids
 *   gate [R][block-1][rank] float32  selector projection of the final hidden state
 *   logits_out [R][block-1][V] float32 or NULL: full drafter logits (debugging,
 *                        test harness)
 *   width [R] or NULL    block width of each request (clamped into 2..block; NULL:
 *                        block): the block keys at positions >= width are masked
 *                        in the attention, so positions 0..width-1 are a block of
 *                        width positions
 * Requires ctx_len + n_new <= kv_capacity.  Every wait in the weight-streaming
 * pipelines is bounded; one that gives up sets the handle's error word (cleared at
 * the start of each call), which the following dflash2_select reports per request. */
dflash2_status dflash2_draft_block(dflash2_handle* h, int32_t n_req, const int32_t* anchor_ids,
                                   const int32_t* ctx_len, const int32_t* n_new, const float* taps,
                                   void* k_cache, void* v_cache, int32_t* cand_ids, float* cand_logits,
                                   float* gate, float* logits_out, const int32_t* width, void* stream);

/* Selector walk (step a10; vLLM PR #52816 description, candidate selector):
 * score(p -> c) = <A[p] * gate_i, B[c]> + cand_logit_i[c]; the walk starts at the
 * anchor.  temperature[r] == 0: greedy, argmax with ties to the smaller id, q row
 * one-hot.  temperature[r] > 0: q_i = softmax(score / T) over the 16 candidates, the
 * choice is the first j with cumsum_j > u * sum, u from Philox4x32-10 with key =
 * seed[r], counter = (philox_offset[r] lo32, hi32, slot = i-1, purpose 0).
 *   path [R][block-1] chosen ids; q_rows [R][block-1][top_k] float32
 *   scores_out [R][block-1][top_k][top_k] float32 or NULL: the score lattice
 *   status [R] written: DFLASH2_OK, DFLASH2_E_NONFINITE (nonfinite logit/score),
 *   DFLASH2_E_INVAL (negative temperature) or DFLASH2_E_CUDA (a pipeline wait of the
 *   handle's last dflash2_draft_block gave up: its candidates and gate are undefined;
 *   the handle's error word is cleared by the next dflash2_draft_block)
 *   temperature [R] float32 (negative -> status DFLASH2_E_INVAL); seed, philox_offset [R] uint64
 *   width [R] or NULL: the walk takes positions 1..width-1 (clamped into 2..block;
 *   NULL: block); path entries past them are -1 and their q rows 0.  Every
 *   position's lattice is still scored (scores_out). */
dflash2_status dflash2_select(dflash2_handle* h, int32_t n_req, const int32_t* anchor_ids,
                              const int32_t* cand_ids, const float* cand_logits, const float* gate,
                              const float* temperature, const uint64_t* seed, const uint64_t* philox_offset,
                              int32_t* path, float* q_rows, float* scores_out, int32_t* status,
                              const int32_t* width, void* stream);

/* Selector mode of the handle's later dflash2_select calls (an ablation of the
 * walk; vLLM PR #52816 description: "walk the best path from the verified anchor").
 *   0 (default): the sequential walk above.
 *   1: for greedy requests (temperature 0) the globally best path instead, the
 *      path of highest total edge score over the 16^(width-1) candidate sequences, by
 *      dynamic programming with float32 sums (equal sums -> the predecessor with
 *      the smaller id; equal ends -> the smaller id); q rows one-hot.  Requests with
 *      temperature > 0 still walk and sample.
 * Returns DFLASH2_E_INVAL for another mode. */
dflash2_status dflash2_set_select_mode(dflash2_handle* h, int32_t mode);

/* Verification (step a11; "LSE docs/DFLASH2.md", first paragraph).
 *   target_logits [R][block][V] float32: row j is the target's distribution for
 *   block position j+1 (row block-1 = the bonus position).
 *   Greedy (T == 0): accept while path[j] == argmax row j (ties -> smaller id);
 *   emit the argmax at the first mismatch, or of the last row if all accepted.
 *   T > 0: p_j = softmax(row j / T); accept if u < p_j(d)/q_j(d) (purpose 1, slot
 *   j); on rejection draw from max(0, p_j - q_j) normalised by inverse CDF in id
 *   order (purpose 2, slot j; from p_j if that mass <= 1e-30); if all accepted draw
 *   the bonus from the last row (purpose 2, slot block-1).
 *   width [R] or NULL: a request of width w (clamped into 2..block; NULL: block)
 *   tests proposals 0..w-2 against rows 0..w-2, takes its bonus from row w-1
 *   (slot w-1), and its rows w..block-1 are not read.
 *   n_accepted [R]; emitted [R][block] (-1 padded); n_emitted [R] = n_accepted+1.
 *   probs_out [R][block][2] float32 or NULL (debugging, test harness): for a request
 *   with T > 0, [j][0] = p_j(path[j]) for j < block-1 and [block-1][0] = p of the
 *   bonus token when all proposals were accepted; [j][1] = the residual mass
 *   sum_x max(0, p_j(x) - q_j(x)) of the rejected row j.  Every other entry (and
 *   every entry of a greedy, skipped or nonfinite request) is NaN.
 *   status [R] in/out: a request whose status is nonzero on entry is skipped
 *   (n_accepted = n_emitted = 0); a NaN or +inf in a row, or a row whose maximum
 *   is -inf, sets DFLASH2_E_NONFINITE. */
dflash2_status dflash2_verify(dflash2_handle* h, int32_t n_req, const float* target_logits, const int32_t* path,
                              const int32_t* cand_ids, const float* q_rows, const float* temperature,
                              const uint64_t* seed, const uint64_t* philox_offset, int32_t* n_accepted,
                              int32_t* emitted, int32_t* n_emitted, float* probs_out, int32_t* status,
                              const int32_t* width, void* stream);

/* ---- Draft tree (DDTree) ----
 * "qwen35: DSpark speculative decoding (Qwen3.8-27B drafters) - #625", DDTree
 * commit: a draft tree whose branches are chosen by the draft log-prob plus the
 * selector compatibility with the branch's actual parent, log-softmax-normalised per
 * position, grown best-first under a node budget.
 * dflash2_tree_build: from one draft block's candidates (the outputs of
 * dflash2_draft_block), for each request a tree rooted at the anchor.  A node at
 * depth d (1..block-1) carries one of the top_k candidates of block position d; the
 * children of a node are the candidates of the next position.  Child c of a parent
 * whose own candidate is p scores log q(c | p) = s(p -> c) - logsumexp_c' s(p -> c'),
 * s the selector score of dflash2_select; a node's score is the sum along its path.
 * The tree grows by adding, one at a time, the highest-scoring child (over the root
 * and every node already in) not yet in it, until `budget` nodes (1..
 * DFLASH2_TREE_MAX_NODES; the root not counted) are in; equal scores go to the
 * child of the earlier-added parent (the root first), then to the smaller candidate
 * index.  FP32.
 *   node_token, node_parent, node_depth [R][budget] int32, node_score [R][budget]
 *   float32, in the order the nodes were added: node k's parent is -1 (the root) or
 *   a node j < k; n_nodes [R]; scores_out: the selector lattice as in dflash2_select,
 *   or NULL.  status [R] written as by dflash2_select (no temperature: the tree is
 *   verified greedily).
 * dflash2_tree_verify: greedy verification of the trees.  target_logits
 *   [R][budget + 1][V] float32: row 0 is the target's distribution after the anchor,
 *   row 1 + k after tree node k (rows past n_nodes are not read).  From the root,
 *   move to the child whose token is the argmax of the current row (ties -> smaller
 *   id) while one exists; emitted [R][block] holds the path's tokens, then the argmax
 *   of the last row (-1 padded); n_accepted = the path's length, n_emitted =
 *   n_accepted + 1.  status in/out as in dflash2_verify (nonzero on entry: skipped;
 *   a NaN or +inf in a read row, or a row whose maximum is -inf: E_NONFINITE).
 * Both return DFLASH2_E_INVAL for a NULL pointer, n_req outside 1..max_requests or a
 * budget outside 1..DFLASH2_TREE_MAX_NODES (nothing is launched). */
#define DFLASH2_TREE_MAX_NODES 32
dflash2_status dflash2_tree_build(dflash2_handle* h, int32_t n_req, int32_t budget, const int32_t* anchor_ids,
                                  const int32_t* cand_ids, const float* cand_logits, const float* gate,
                                  int32_t* node_token, int32_t* node_parent, int32_t* node_depth, float* node_score,
                                  int32_t* n_nodes, float* scores_out, int32_t* status, void* stream);
dflash2_status dflash2_tree_verify(dflash2_handle* h, int32_t n_req, int32_t budget, const float* target_logits,
                                   const int32_t* node_token, const int32_t* node_parent, const int32_t* n_nodes,
                                   int32_t* n_accepted, int32_t* emitted, int32_t* n_emitted, int32_t* status,
                                   void* stream);

/* Serving-loop state update after dflash2_verify, on the device (so a multi-step
 * loop can be captured in one graph; "LSE docs/DFLASH2.md", block paragraph: each
 * draft is an anchor plus block-1 masks; vLLM PR #52816 description, candidate
 * selector: the walk starts at the verified anchor).  For each request r:
 *   ctx_len[r] += n_new[r]          the rows this step appended are now context
 *   if n_emitted[r] > 0: anchor_ids[r] = emitted[r][n_emitted[r] - 1]
 *   n_new[r] = n_emitted[r]          the emitted tokens are the next step's new rows
 *   philox_offset[r] += 1            a fresh Philox counter range for the next step
 * A request that verify skipped or rejected (n_emitted = 0) keeps its anchor and
 * appends nothing next step.  The caller supplies the next step's taps for the new
 * rows and keeps ctx_len + block <= kv_capacity.
 *   anchor_ids, ctx_len, n_new [R] int32 in/out; philox_offset [R] uint64 in/out;
 *   emitted [R][block], n_emitted [R] int32 (dflash2_verify's outputs).
 * All device pointers, caller-owned; asynchronous on `stream`.  Returns
 * DFLASH2_E_INVAL for a null pointer or n_req outside 1..max_requests (nothing is
 * launched), DFLASH2_E_CUDA if the launch fails. */
dflash2_status dflash2_advance(dflash2_handle* h, int32_t n_req, const int32_t* emitted, const int32_t* n_emitted,
                               int32_t* anchor_ids, int32_t* ctx_len, int32_t* n_new, uint64_t* philox_offset,
                               void* stream);

/* ---- One step from a captured CUDA graph ----
 * The arguments of one draft + select + verify step: the fields of
 * dflash2_draft_block, dflash2_select and dflash2_verify of the same names and
 * meanings (logits_out, scores_out and probs_out are NULL in a step).  width is
 * shared by the three calls (NULL: block). */
typedef struct dflash2_step_args {
  int32_t n_req;
  const int32_t* anchor_ids;    /* [R] */
  const int32_t* ctx_len;       /* [R] */
  const int32_t* n_new;         /* [R] */
  const float* taps;            /* [R][block][n_taps*H] */
  void* k_cache;                /* bf16 [n_layers][max_requests][kv_capacity][nkv][hd] */
  void* v_cache;
  int32_t* cand_ids;            /* [R][block-1][top_k] */
  float* cand_logits;           /* [R][block-1][top_k] */
  float* gate;                  /* [R][block-1][rank] */
  const float* temperature;     /* [R] */
  const uint64_t* seed;         /* [R] */
  const uint64_t* philox_offset; /* [R] */
  int32_t* path;                /* [R][block-1] */
  float* q_rows;                /* [R][block-1][top_k] */
  int32_t* status;              /* [R] written by the select, read and written by the verify */
  const float* target_logits;   /* [R][block][V] */
  int32_t* n_accepted;          /* [R] */
  int32_t* emitted;             /* [R][block] */
  int32_t* n_emitted;           /* [R] */
  const int32_t* width;         /* [R] or NULL */
} dflash2_step_args;

/* Number of argument sets whose step graphs a handle keeps (least recently used
 * replaced). */
#define DFLASH2_STEP_GRAPHS 4

/* One step: dflash2_draft_block, dflash2_select and dflash2_verify on `args`, in
 * that order on `stream`, with the same results.  The first call with a given
 * argument set (the same values in every field, under the same selector mode) runs
 * the three calls as they are and then captures them into a CUDA graph on a stream
 * of the handle's own (the capture launches nothing); later calls with that set
 * launch the graph on `stream`, one launch instead of about seventy.  The graph
 * reads the buffers each time it runs, so a serving loop changes their contents
 * between steps, not their addresses (dflash2_advance keeps them).  A handle keeps DFLASH2_STEP_GRAPHS sets;
 * their graphs are freed by dflash2_step_graphs_clear or dflash2_destroy, and must
 * be cleared before a buffer they name is freed.  While the handle has profiling
 * events set (dflash2_set_lmhead_events, dflash2_set_projection_events) the calls
 * run as they are, nothing captured or replayed.  Not for concurrent use of one
 * handle from several threads.  Returns what the three calls return (their checks
 * run on the first call with a set; nothing is cached when one fails) or
 * DFLASH2_E_CUDA if a launch fails; a failed capture leaves the set uncached, and
 * the next call with it runs the three calls again. */
dflash2_status dflash2_step(dflash2_handle* h, const dflash2_step_args* args, void* stream);

/* Frees the handle's step graphs (waits for none of their launches: the caller
 * orders this after them, e.g. by synchronising the streams they ran on). */
dflash2_status dflash2_step_graphs_clear(dflash2_handle* h);

/* Block width of each request by context length ("qwen35: DSpark speculative
 * decoding ... #625", long-context commits: the verify's cost grows with the
 * block's rows times the context, so past a context threshold the block narrows;
 * the rule reads the context length only, so a prompt's width is reproducible):
 *   width[r] = narrow_width  if ctx_threshold > 0 and ctx_len[r] + n_new[r] > ctx_threshold
 *              block         otherwise
 * ctx_len + n_new is the context the step's block attends to (the keys after this
 * step's append).  The pages' default is ctx_threshold 8192, narrow_width 8 for a
 * drafter of block 16; ctx_threshold 0 disables narrowing.
 *   ctx_len, n_new [R] int32 (dflash2_draft_block's inputs); width [R] int32 out.
 * Returns DFLASH2_E_INVAL for a null pointer, n_req outside 1..max_requests, a
 * negative threshold or narrow_width outside 2..block (nothing is launched). */
dflash2_status dflash2_block_width(dflash2_handle* h, int32_t n_req, const int32_t* ctx_len, const int32_t* n_new,
                                  int32_t ctx_threshold, int32_t narrow_width, int32_t* width, void* stream);

/* LM head + top-16 alone (step a8 on given final hidden states): logits of block
 * positions 1..B-1 = W_lm . hidden (hidden already normalised, BF16), top-16 with
 * the ordering of dflash2_draft_block.  Row n of `hidden` is request n/B, block
 * position n%B (position 0 is not projected), B = the handle's block.  n_rows: a
 * multiple of B, <= B*max_requests.  Up to 32 rows run on the LM-head kernel; more
 * rows (a handle whose calls reach the tensor-core GEMM, see dflash2_create, else
 * DFLASH2_E_UNSUPPORTED) on the tensor-core GEMM, with the logits in handle
 * scratch, then a chunked top-16.
 *   hidden [n_rows][H] bf16; cand_ids, cand_logits [n_rows/B][B-1][top_k];
 *   logits_out [n_rows/B][B-1][V] float32 or NULL. */
dflash2_status dflash2_head_topk(dflash2_handle* h, int32_t n_rows, const void* hidden, int32_t* cand_ids,
                                 float* cand_logits, float* logits_out, void* stream);

/* Number of kernel launches the handle has issued since it was created (all
 * entry points).  Host-side counter; no device work. */
int64_t dflash2_launch_count(const dflash2_handle* h);

/* Profiling hook: when both events are non-NULL (cudaEvent_t passed as void*),
 * dflash2_draft_block records `start` right before and `stop` right after its
 * LM-head + top-16 kernel (the GEMM and the chunked top-16 on the tensor-core
 * path) on the call's stream.  NULL, NULL turns it off. */
dflash2_status dflash2_set_lmhead_events(dflash2_handle* h, void* start, void* stop);

/* Profiling hook: when `events` is non-NULL (an array of 2 * n_pairs cudaEvent_t
 * passed as void*, kept alive by the caller while set), each dflash2_draft_block
 * call records events[2i] right before and events[2i+1] right after its i-th
 * drafter weight-projection launch (the taps projection with the first delta, then
 * per layer q/k/v, o, delta, gate/up, down and, from the second layer on, the
 * attention delta, and finally the selector projection; not the LM head), for
 * i < n_pairs, on the call's stream.  An event record between two launches keeps the
 * later one from overlapping the earlier one's tail, so the pairs time each launch
 * alone.  NULL, 0 turns it off. */
dflash2_status dflash2_set_projection_events(dflash2_handle* h, void* const* events, int32_t n_pairs);

/* Number of drafter weight-projection launches of one dflash2_draft_block call, and
 * the weight bytes they stream together (every drafter matrix once, Q8 scale and
 * bias included), for roofline reports. */
int32_t dflash2_projection_launches(const dflash2_handle* h);
int64_t dflash2_projection_bytes(const dflash2_handle* h);

/* Algorithmic bytes the LM-head + top-16 kernel of one draft_block call streams
 * (LM-head weights + activations + candidate outputs; on the tensor-core path
 * also the logits the GEMM writes and the top-16 kernel reads), for
 * roofline reports. */
int64_t dflash2_lmhead_bytes(const dflash2_handle* h, int32_t n_req);

/* ---- LM head + top-16 without any device allocation ----
 * The paper has no counterpart of this call: it exists for users of this
 * library that cannot allocate device memory.  Some run inside a runtime whose
 * allocator owns all of HBM, or as a plug-in of another framework's memory pool.
 * Others must not risk a cudaMalloc on their path, because one can synchronise
 * the device or fail for lack of memory in the middle of a step.  It computes
 * what dflash2_head_topk computes (logits of block positions 1..7 of each
 * request and their top-16, with hidden already normalised), but needs no
 * handle.  Its scratch (the per-CTA candidate lists, 640 KiB) is one fixed
 * device array inside this library (1.25 MiB), plus one error word, held on every
 * GPU that uses it until the process exits.
 *   lm_head  [vocab][hidden_dim] bf16, 16-byte aligned, caller-owned.
 *   hidden   [n_rows][hidden_dim] bf16, 16-byte aligned; row n is block position
 *            n%8 of request n/8 (position 0 is not projected).
 *   cand_ids, cand_logits  [n_rows/8][7][16]; logits_out [n_rows/8][7][vocab] or NULL.
 * Returns DFLASH2_E_INVAL for null or misaligned pointers, n_rows not a positive
 * multiple of 8, vocab < 16 or hidden_dim < 128, and DFLASH2_E_UNSUPPORTED for
 * n_rows > DFLASH2_NOALLOC_MAX_ROWS, vocab not a multiple of 16 or hidden_dim not
 * a multiple of 128; nothing is launched then.  CTAs: two per SM (as the handle's
 * LM head) when that is <= DFLASH2_NOALLOC_MAX_CTAS, else one per SM (at most
 * DFLASH2_NOALLOC_MAX_CTAS), so every SM streams an equal share of the vocabulary.
 * Failure on the device: every wait of the LM head's weight pipeline is bounded;
 * one that gives up sets the call's error word (cleared at the start of each call)
 * and the call then writes the sentinel cand_ids = -1, cand_logits = NaN for every
 * row (its logits_out are undefined).  The return value cannot report it: the
 * call does not synchronise.
 * The first call on each device looks up the arrays' device addresses (with that
 * device current); make that first call before any stream capture.  It calls no
 * cudaMalloc or cudaFree and no allocating library routine.  All calls share the
 * one array: calls whose kernels overlap on the GPU (other streams, other
 * threads) race on it and must be serialised by the caller.  Every entry a call
 * reads is written earlier in the same call (the error word is cleared by an
 * asynchronous memset on `stream`), so nothing needs clearing between calls. */
#define DFLASH2_NOALLOC_MAX_ROWS 32
#define DFLASH2_NOALLOC_MAX_CTAS 320
dflash2_status dflash2_head_topk_noalloc(const void* lm_head, int32_t vocab, int32_t hidden_dim, int32_t n_rows,
                                         const void* hidden, int32_t* cand_ids, float* cand_logits,
                                         float* logits_out, void* stream);

/* ---- Test hooks (failure paths driven from the host; no kernel waits out a
 * limit or faults) ----
 * dflash2_debug_set_pipeline_error: marks the handle's pipeline error word on
 * `stream`, as a bounded weight-pipeline wait of the last dflash2_draft_block
 * that gave up would.  The next dflash2_select then reports DFLASH2_E_CUDA for
 * every request (path -1, q rows 0) and dflash2_verify emits nothing for them;
 * the next dflash2_draft_block clears the word.
 * dflash2_debug_noalloc_inject_error(1): until called with 0, every
 * dflash2_head_topk_noalloc call starts with its error word set instead of
 * clear, as if its LM head's pipeline wait had given up (process-wide). */
dflash2_status dflash2_debug_set_pipeline_error(dflash2_handle* h, void* stream);
dflash2_status dflash2_debug_noalloc_inject_error(int32_t on);

/* Human-readable text of a status code (static string). */
const char* dflash2_status_string(dflash2_status s);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH2_H */
