"""FP64 oracle of one DFlash2 step: draft block (taps projection, drafter layers,
LM head, top-16, selector gate), selector walk, and verification.

Test infrastructure only (see oracle/__init__.py).  Every function states the
page passage it follows and the reading taken where the pages leave a step open.

Pages cited:
  [LSE]  "LSE docs/DFLASH2.md" (Geramy/LSE) - drafter geometry paragraph; block,
         mask, window, conv and selector paragraph; Q8 conversion paragraph;
         test paragraphs (attention, selector rounding bound, top-k policy).
  [LUCE] "qwen35: DSpark speculative decoding (Qwen3.8-27B drafters) - #625"
         (lucebox) - DFlash 2 commit (conv prepare/finish, selector chain),
         fp64 RoPE commit, greedy-width commit.
  [VLLM] "[Spec Decode] DFlash2: local convolution + candidate selector -
         #52816" (vLLM) - PR description: conv formula, selector edge score,
         walk and q for the lossless verify.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np

from . import philox

STATUS_OK = 0
STATUS_INVAL = 1
STATUS_NONFINITE = 2


# ----------------------------------------------------------------------------- numbers

def bf16_to_f64(bits) -> np.ndarray:
    """BF16 bit patterns -> exact float64 values."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """Round float64 to the nearest bfloat16 value (8 significant bits, ties to even);
    returns float64.  Used where the method stores BF16 (the context K/V cache)."""
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)                      # x = m * 2^e, |m| in [0.5, 1)
    return np.ldexp(np.round(m * 256.0), e - 8)


def matrix_f64(m, rows: Optional[slice] = None) -> np.ndarray:
    """Dense float64 copy of a weight matrix (rows optional).

    BF16: exact.  Q8/group64: w = scale * q + bias per group of 64 along the
    input dimension, scale and bias BF16 ([LSE] Q8 conversion paragraph: affine
    Q8, group 64, BF16 scale and bias).  Both products are exact in float64.
    """
    sl = rows if rows is not None else slice(None)
    if m["kind"] == "bf16":
        return bf16_to_f64(m["w"][sl])
    codes = np.asarray(m["codes"][sl], np.float64)
    M, K = codes.shape
    s = bf16_to_f64(m["scale"][sl])[:, :, None]
    b = bf16_to_f64(m["bias"][sl])[:, :, None]
    return (codes.reshape(M, K // 64, 64) * s + b).reshape(M, K)


def matmul_rows(m, X: np.ndarray, row_chunk: int = 8192) -> np.ndarray:
    """Y[n][o] = sum_k W[o][k] X[n][k] in float64, W decoded in row chunks."""
    M = (m["w"] if m["kind"] == "bf16" else m["codes"]).shape[0]
    Y = np.empty((X.shape[0], M), np.float64)
    for r0 in range(0, M, row_chunk):
        W = matrix_f64(m, slice(r0, r0 + row_chunk))
        Y[:, r0:r0 + W.shape[0]] = X @ W.T
    return Y


def rmsnorm(x: np.ndarray, w_bits, eps: float) -> np.ndarray:
    """y = x / sqrt(mean(x^2) + eps) * w over the last axis (Qwen-style RMSNorm;
    the pages name the norms but not their form - reading: the Qwen3 convention
    of the target family, eps 1e-6)."""
    w = bf16_to_f64(w_bits)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * w


def silu(x):
    return x / (1.0 + np.exp(-x))


# ----------------------------------------------------------------------------- RoPE

def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """inv_freq_j = theta^(-2j/head_dim), j < head_dim/2, in float64 ([LUCE] fp64
    RoPE commit: theta = 1e7 needs double precision frequencies)."""
    j = np.arange(head_dim // 2, dtype=np.float64)
    return theta ** (-2.0 * j / head_dim)


def rope_neox(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """NEOX (half-split) rotary embedding ([LUCE] description: plain NEOX rope;
    [LSE] geometry: theta 10,000,000).  x [..., n, hd] with positions broadcast
    over the leading axis: out[j] = x[j] cos - x[j+hd/2] sin,
    out[j+hd/2] = x[j+hd/2] cos + x[j] sin, angle = pos * inv_freq_j."""
    hd = x.shape[-1]
    half = hd // 2
    ang = np.asarray(pos, np.float64)[:, None] * rope_inv_freq(hd, theta)[None, :]   # [n_pos][half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# ----------------------------------------------------------------------------- dynamic conv

def dyn_conv(x: np.ndarray, base: np.ndarray, delta: np.ndarray, group: int) -> np.ndarray:
    """Grouped dynamic causal convolution over the block ([VLLM] PR description,
    "Grouped dynamic depthwise convolution": out[i,c] = sum_t (base[t,c] +
    delta[i,t,g(c)]) * x[i-t,c], taps zero across the block boundary; [LUCE]
    DFlash 2 commit: per-element base plus per-group dynamic coefficient).

    x [B][H]; base [taps][H] (float64); delta [B][taps][G]; g(c) = c // group.
    Reading: x[i-t] = 0 for i-t < 0, so the anchor (i = 0) never sees another block.
    """
    B, H = x.shape
    taps = base.shape[0]
    out = np.zeros_like(x)
    for t in range(taps):
        coef = base[t][None, :] + np.repeat(delta[:, t, :], group, axis=1)     # [B][H]
        shifted = np.zeros_like(x)
        if t < B:
            shifted[t:] = x[:B - t]
        out += coef * shifted
    return out


# ----------------------------------------------------------------------------- attention

def visible_context_range(L: int, i: int, window: int):
    """Context keys visible to block query i ([LSE] block paragraph: context keys obey
    the 2048-position sliding window).  Reading: the query sits at absolute position
    L + i, key k (< L) is visible iff (L + i) - k < window."""
    return max(0, L + i - window + 1), L


def block_attention(q, k_blk, v_blk, k_ctx, v_ctx, L: int, window: int) -> np.ndarray:
    """Block attention: noncausal inside the 8-position block, sliding window over the
    context ([LSE] block paragraph; vLLM PR discussion: sliding_attention with
    is_causal false).  GQA: query head h uses KV head h // (nq / nkv); scale 1/sqrt(hd).

    q [B][nq][hd]; k_blk, v_blk [B][nkv][hd]; k_ctx, v_ctx [L][nkv][hd] (positions
    0..L-1, rows outside the window are never read).  Returns [B][nq*hd].
    """
    B, nq, hd = q.shape
    nkv = k_blk.shape[1]
    rep = nq // nkv
    out = np.zeros((B, nq, hd))
    for i in range(B):
        lo, hi = visible_context_range(L, i, window)
        for h in range(nq):
            kv = h // rep
            keys = np.concatenate([k_ctx[lo:hi, kv, :], k_blk[:, kv, :]], axis=0)
            vals = np.concatenate([v_ctx[lo:hi, kv, :], v_blk[:, kv, :]], axis=0)
            s = keys @ q[i, h] / math.sqrt(hd)
            p = np.exp(s - s.max())
            p /= p.sum()
            out[i, h] = p @ vals
    return out.reshape(B, nq * hd)


# ----------------------------------------------------------------------------- drafter

def _heads(x, n, hd):
    return x.reshape(x.shape[0], n, hd)


def draft_block(g, W: Dict, anchor: int, ctx_len: int, n_new: int, taps: np.ndarray,
                k_cache: List[np.ndarray], v_cache: List[np.ndarray]) -> Dict[str, np.ndarray]:
    """One request's draft block: a1..a9.

    g: geometry; W: weights (see workloads.gen); taps [n_new][n_taps*H] float32
    for context positions ctx_len..ctx_len+n_new-1; k_cache/v_cache: per layer
    [cap][nkv][hd] BF16 bits (positions below ctx_len already filled).  The new
    context rows are written into the caches (BF16) in place.

    Readings (the pages leave the wiring open):
      * taps -> c = RMSNorm_hidden(W_fc . concat(taps)) ([LSE] geometry paragraph:
        five post-block target states; tensor inventory has fc and hidden_norm);
        a new context row's K/V in every layer are RoPE(k_norm(W_k c)) and W_v c at
        its absolute position, stored BF16.
      * block rows: x_0 = E[anchor], x_i = E[mask] (i = 1..7) at positions L + i,
        L = ctx_len + n_new ([LSE] block paragraph: one anchor and seven masks).
      * each sublayer: a = RMSNorm(x); delta = W_delta a; a' = conv_in(a); sublayer
        on a'; y' = conv_out(y); x += y' ([VLLM]: wraps each sublayer in and out from
        one projection of its input).
      * attention: Qwen3 layer with q_norm/k_norm before NEOX RoPE; MLP: SwiGLU.
      * h = RMSNorm_final(x); logits = W_lm h and gate = W_sel h at positions 1..7.
    """
    H, hd, nq, nkv = g.hidden, g.head_dim, g.n_q_heads, g.n_kv_heads
    B, G, T = g.block, g.groups, g.conv_taps
    eps = g.rms_eps
    L = ctx_len + n_new
    # a1: taps projection
    c = rmsnorm(matmul_rows(W["fc"], np.asarray(taps, np.float64)), W["hidden_norm"], eps)
    pos_new = np.arange(ctx_len, ctx_len + n_new)
    # a2: block embedding
    ids = [anchor] + [g.mask_id] * (B - 1)
    x = bf16_to_f64(W["embed"][ids])
    pos_blk = np.arange(L, L + B)
    trace = {"c": c}
    for l in range(g.n_layers):
        p = f"l{l}."
        # a3: attention sublayer input, delta, conv-in
        a = rmsnorm(x, W[p + "input_norm"], eps)
        d = matmul_rows(W[p + "attn_delta"], a).reshape(B, 2, T, G)
        base = bf16_to_f64(W[p + "attn_base"]).reshape(2, T, H)
        a1 = dyn_conv(a, base[0], d[:, 0], g.conv_group)
        # a4: q, k, v of the block; k, v of the new context rows
        q = rope_neox(rmsnorm(_heads(matmul_rows(W[p + "q"], a1), nq, hd), W[p + "q_norm"], eps), pos_blk, g.rope_theta)
        kb = rope_neox(rmsnorm(_heads(matmul_rows(W[p + "k"], a1), nkv, hd), W[p + "k_norm"], eps), pos_blk, g.rope_theta)
        vb = _heads(matmul_rows(W[p + "v"], a1), nkv, hd)
        if n_new > 0:
            kc = rope_neox(rmsnorm(_heads(matmul_rows(W[p + "k"], c), nkv, hd), W[p + "k_norm"], eps), pos_new, g.rope_theta)
            vc = _heads(matmul_rows(W[p + "v"], c), nkv, hd)
            k_cache[l][ctx_len:L] = _bf16_bits(kc)
            v_cache[l][ctx_len:L] = _bf16_bits(vc)
        lo = max(0, L - g.window + 1)
        kctx = np.zeros((L, nkv, hd))
        vctx = np.zeros((L, nkv, hd))
        kctx[lo:L] = bf16_to_f64(k_cache[l][lo:L])
        vctx[lo:L] = bf16_to_f64(v_cache[l][lo:L])
        # a5: block attention
        o = block_attention(q, kb, vb, kctx, vctx, L, g.window)
        # a6: output projection, conv-out, residual
        y = matmul_rows(W[p + "o"], o)
        x = x + dyn_conv(y, base[1], d[:, 1], g.conv_group)
        # a7: MLP sublayer
        m = rmsnorm(x, W[p + "post_norm"], eps)
        dm = matmul_rows(W[p + "mlp_delta"], m).reshape(B, 2, T, G)
        mbase = bf16_to_f64(W[p + "mlp_base"]).reshape(2, T, H)
        m1 = dyn_conv(m, mbase[0], dm[:, 0], g.conv_group)
        hmid = silu(matmul_rows(W[p + "gate"], m1)) * matmul_rows(W[p + "up"], m1)
        f = matmul_rows(W[p + "down"], hmid)
        x = x + dyn_conv(f, mbase[1], dm[:, 1], g.conv_group)
        trace[f"x{l}"] = x.copy()
    # a8, a9: final norm, LM head and selector gate at block positions 1..7
    h = rmsnorm(x, W["final_norm"], eps)
    logits = matmul_rows({"kind": "bf16", "w": W["lm_head"]}, h[1:])
    gate = matmul_rows(W["sel_proj"], h[1:])
    trace.update({"h": h, "logits": logits, "gate": gate})
    return trace


def _bf16_bits(x) -> np.ndarray:
    v = round_to_bf16(x).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------- top-k

def topk(row: np.ndarray, k: int):
    """Top-k of one logits row with the policy of [LSE] (top-k paragraphs): equal
    scores select the smaller original index, +inf and -inf keep their normal
    order, NaNs come first ordered by index (so a nonfinite row stays visible and
    the selector rejects it).  Returns (ids int32[k], values float64[k])."""
    row = np.asarray(row)
    idx = np.arange(row.size)
    nan = np.isnan(row)
    neg = np.where(nan, 0.0, -row.astype(np.float64))
    order = np.lexsort((idx, neg, ~nan))
    sel = order[:k]
    return sel.astype(np.int32), row[sel].astype(np.float64)


# ----------------------------------------------------------------------------- selector

def codebook_rows(m, ids) -> np.ndarray:
    ids = np.asarray(ids, np.int64)
    if m["kind"] == "bf16":
        return bf16_to_f64(m["w"][ids])
    sub = {"kind": "q8", "codes": m["codes"][ids], "scale": m["scale"][ids], "bias": m["bias"][ids]}
    return matrix_f64(sub)


def selector_scores(A_pred: np.ndarray, gate: np.ndarray, B_cand: np.ndarray, unary: np.ndarray) -> np.ndarray:
    """Edge scores s(p -> c) = <A[p] * gate, B[c]> + unary[c] ([VLLM] PR description,
    candidate selector; [LSE] selector paragraph: rank-256 codebooks, each choice
    conditioned on its predecessor).  gate = W_sel h is the projection of the
    position's hidden state; unary is the candidate's drafter logit (the checkpoint
    has no learned unary tensor, so the LM-head score is the unary term).

    A_pred [P][r], gate [r], B_cand [C][r], unary [C] -> [P][C], written out as the
    explicit rank-r triple product."""
    P, r = A_pred.shape
    C = B_cand.shape[0]
    s = np.zeros((P, C))
    for pi in range(P):
        for ci in range(C):
            s[pi, ci] = float(np.sum(A_pred[pi] * gate * B_cand[ci])) + float(unary[ci])
    return s


def selector_lattice(cb_a, cb_b, anchor: int, cand_ids: np.ndarray, cand_logits: np.ndarray,
                     gate: np.ndarray) -> np.ndarray:
    """Every edge score of the block ([VLLM] PR description, candidate selector):
    position 1 from the anchor, positions 2..7 from every candidate of the previous
    position.  Returns [P][K][K]: scores[i][p][c] = s_{i+1}(pred p -> cand c), where
    the predecessor of position 1 is the anchor for every p (its row repeats)."""
    P, K = cand_ids.shape
    scores = np.zeros((P, K, K))
    Bc = [codebook_rows(cb_b, cand_ids[i]) for i in range(P)]
    a_anchor = codebook_rows(cb_a, [anchor])
    scores[0] = np.repeat(selector_scores(a_anchor, gate[0], Bc[0], cand_logits[0]), K, axis=0)
    for i in range(1, P):
        scores[i] = selector_scores(codebook_rows(cb_a, cand_ids[i - 1]), gate[i], Bc[i], cand_logits[i])
    return scores


def walk(g, cb_a, cb_b, anchor: int, cand_ids: np.ndarray, cand_logits: np.ndarray, gate: np.ndarray,
         temperature: float, seed: int, offset: int, uniform_fn=None):
    """Selector path from the verified anchor over the top-16 candidates of block
    positions 1..7 ([VLLM] PR description: walk the best path from the verified
    anchor; at T > 0 walk by inverse CDF and return q over the K candidates;
    [LSE]: greedy requests keep deterministic selection).

    Greedy (T == 0): c_i = argmax_c s_i(c_{i-1}, c), c_0 = anchor; the decision is
    taken on float32-rounded scores, ties -> smaller vocabulary id; q row one-hot.
    Sampled: q_i = softmax(s_i(c_{i-1}, .) / T) over the candidates in top-k order;
    u from Philox (slot i-1, purpose 0); pick the first j with cumsum_j > u * sum.

    Returns dict(path int32[7], q_rows [7][K], scores [7][K][K] (row p of position 1
    repeats the anchor row), status, margins [7]) where a margin is the distance of
    the decision from its boundary (score gap, or |u*sum - nearest cumsum| / sum).
    """
    P, K = cand_ids.shape
    status = STATUS_OK
    uni = uniform_fn or (lambda slot, purpose: philox.uniform(seed, offset, slot, purpose))
    scores = selector_lattice(cb_a, cb_b, anchor, cand_ids, cand_logits, gate)
    if not np.all(np.isfinite(scores)) or not np.all(np.isfinite(cand_logits)):
        return {"path": np.full(P, -1, np.int32), "q_rows": np.zeros((P, K)), "scores": scores,
                "status": STATUS_NONFINITE, "margins": np.zeros(P)}
    path = np.zeros(P, np.int32)
    q_rows = np.zeros((P, K))
    margins = np.zeros(P)
    prev = 0
    for i in range(P):
        s = scores[i, prev] if i > 0 else scores[0, 0]
        if temperature == 0.0:
            s32 = s.astype(np.float32)
            best = max(s32)
            tied = [j for j in range(K) if s32[j] == best]
            j = min(tied, key=lambda jj: cand_ids[i, jj])
            srt = np.sort(s)[::-1]
            margins[i] = srt[0] - srt[1]
            q_rows[i, j] = 1.0
        else:
            e = np.exp((s - s.max()) / temperature)
            tot = e.sum()
            u = uni(i, philox.PURPOSE_WALK)
            cum = np.cumsum(e)
            hit = np.nonzero(cum > u * tot)[0]
            j = int(hit[0]) if hit.size else int(np.nonzero(e > 0)[0][-1])
            margins[i] = np.min(np.abs(cum - u * tot)) / tot
            q_rows[i] = e / tot
        path[i] = cand_ids[i, j]
        prev = j
    return {"path": path, "q_rows": q_rows, "scores": scores, "status": status, "margins": margins}


def viterbi_path(scores: np.ndarray, cand_ids: np.ndarray) -> Dict:
    """Globally best path through the selector lattice, the ablation of the
    sequential walk ([VLLM] PR description: walk the best path from the verified
    anchor, read here as the path of highest total edge score).  scores [P][K][K] =
    s_i(p -> c), position 1's rows all from the anchor; cand_ids [P][K].

    Dynamic programming over positions (Viterbi): best_1(c) = s_1(c);
    best_i(c) = max_p best_{i-1}(p) + s_i(p, c), equal sums -> the predecessor with
    the smaller vocabulary id; the path ends at argmax_c best_P(c) (equal -> smaller
    id) and is read back through the recorded predecessors.  The decision is taken
    on float32 scores with float32 sums in this order (the kernel's precision).
    Returns dict(index int[P] into the candidates, path int32[P] vocabulary ids,
    q_rows one-hot [P][K], total float32)."""
    P, K = cand_ids.shape
    s32 = np.asarray(scores, np.float32)
    best = s32[0, 0].copy()
    back = np.zeros((P, K), np.int64)
    for i in range(1, P):
        nb = np.empty(K, np.float32)
        for c in range(K):
            v = (best + s32[i, :, c]).astype(np.float32)   # float32 sums
            top = v.max()
            tied = [p for p in range(K) if v[p] == top]
            p = min(tied, key=lambda pp: cand_ids[i - 1, pp])
            nb[c] = v[p]
            back[i, c] = p
        best = nb
    top = best.max()
    c = min((cc for cc in range(K) if best[cc] == top), key=lambda cc: cand_ids[P - 1, cc])
    index = np.zeros(P, np.int64)
    for i in range(P - 1, -1, -1):
        index[i] = c
        c = back[i, c]
    q_rows = np.zeros((P, K))
    q_rows[np.arange(P), index] = 1.0
    return {"index": index, "path": cand_ids[np.arange(P), index].astype(np.int32), "q_rows": q_rows,
            "total": np.float32(top)}


# ----------------------------------------------------------------------------- draft tree (DDTree)

def ddtree_build(scores: np.ndarray, cand_ids: np.ndarray, budget: int) -> Dict:
    """Draft tree with selector-scored branches ([LUCE] DDTree commit: each expansion
    scores candidates as the draft log-prob plus the selector compatibility with the
    branch's actual parent, log-softmax-normalised per position, so that cumulative
    best-first comparisons across depths stay on a log-prob scale).

    scores [P][K][K]: the selector lattice (selector_lattice: unary drafter logit +
    compatibility), whose vocabulary log-normaliser is a per-position constant and
    cancels in the per-parent normalisation.  Readings:
      * the root is the verified anchor (depth 0, not counted in the budget); a node
        at depth d < P has the K candidates of block position d + 1 as children;
      * child c of a node whose own candidate index is p (p = 0 for the root, whose
        row repeats) scores log q(c | p) = s[d][p][c] - logsumexp_c' s[d][p][c'];
        a node's score is the sum of log q along its path from the root;
      * best-first: repeatedly add the highest-scoring child, over every node already
        in the tree, that is not in it yet, until `budget` nodes are in; equal scores
        -> the child of the earlier-added parent (the root first), then the smaller
        candidate index (top-k order).
    Returns dict(token int32[n], parent int32[n] (-1 = the root, else the index of an
    earlier node), depth int32[n] (1..P), cand int32[n] (candidate index), score
    float64[n], margins float64[n]: each step's gap between the added node's score and
    the best remaining one (inf when none remains)).  n = min(budget, the K + K^2 + ...
    nodes that exist)."""
    P, K = cand_ids.shape
    logq = np.zeros((P, K, K))
    for d in range(P):
        for p in range(K):
            row = np.asarray(scores[d][p], np.float64)
            m = row.max()
            logq[d][p] = row - (m + math.log(np.exp(row - m).sum()))
    token, parent, depth, cand, score, margins = [], [], [], [], [], []
    # a node is (depth, own candidate index, cumulative score); the root is index -1
    node_depth = {-1: 0}
    node_cand = {-1: 0}
    node_score = {-1: 0.0}
    taken = {-1: set()}
    while len(token) < budget:
        options = []
        for q in [-1] + list(range(len(token))):
            d = node_depth[q]
            if d >= P:
                continue
            for c in range(K):
                if c in taken[q]:
                    continue
                options.append((node_score[q] + logq[d][node_cand[q]][c], q, c))
        if not options:
            break
        # highest score; equal -> earlier parent (root -1 first), then smaller candidate index
        options.sort(key=lambda o: (-o[0], o[1], o[2]))
        best = options[0]
        margins.append(best[0] - options[1][0] if len(options) > 1 else math.inf)
        sc, q, c = best
        d = node_depth[q] + 1
        idx = len(token)
        token.append(int(cand_ids[d - 1][c]))
        parent.append(q)
        depth.append(d)
        cand.append(c)
        score.append(sc)
        taken[q].add(c)
        node_depth[idx], node_cand[idx], node_score[idx], taken[idx] = d, c, sc, set()
    return {"token": np.array(token, np.int32), "parent": np.array(parent, np.int32),
            "depth": np.array(depth, np.int32), "cand": np.array(cand, np.int32),
            "score": np.array(score), "margins": np.array(margins)}


def ddtree_verify(target_rows: np.ndarray, token: np.ndarray, parent: np.ndarray, status_in: int = STATUS_OK,
                  block: int = 8):
    """Greedy verification of a draft tree ([LUCE] DDTree commits: tree verification
    emits the same text as plain decoding; [LSE] first paragraph: greedy requests are
    deterministic).  target_rows [n + 1][V]: row 0 is the target's distribution after
    the anchor (the root), row 1 + k after tree node k.  From the root, move to the
    child whose token is the argmax of the current node's row (ties -> smaller id)
    while one exists; the accepted tokens are the path's, then the argmax of the last
    node's row is emitted.  A used row with NaN or +inf, or a maximum of -inf, makes
    the request nonfinite.  Returns dict(n_accepted, emitted int32[block] (-1 padded),
    n_emitted, status, path (node indices)); a tree is at most block - 1 deep."""
    emitted = np.full(block, -1, np.int32)
    if status_in != STATUS_OK:
        return {"n_accepted": 0, "emitted": emitted, "n_emitted": 0, "status": status_in, "path": []}
    z = np.asarray(target_rows, np.float64)
    n = len(token)
    used = z[: n + 1]
    if np.any(np.isnan(used)) or np.any(np.isposinf(used)) or np.any(~np.isfinite(used.max(axis=1))):
        return {"n_accepted": 0, "emitted": emitted, "n_emitted": 0, "status": STATUS_NONFINITE, "path": []}
    cur, path = -1, []
    while True:
        t = int(np.argmax(z[cur + 1]))
        nxt = [k for k in range(n) if parent[k] == cur and int(token[k]) == t]
        if not nxt:
            break
        cur = nxt[0]
        emitted[len(path)] = t
        path.append(cur)
    emitted[len(path)] = int(np.argmax(z[cur + 1]))
    return {"n_accepted": len(path), "emitted": emitted, "n_emitted": len(path) + 1, "status": STATUS_OK,
            "path": path}


# ----------------------------------------------------------------------------- verify

def verify(target_logits: np.ndarray, path: np.ndarray, cand_ids: np.ndarray, q_rows: np.ndarray,
           temperature: float, seed: int, offset: int, status_in: int = STATUS_OK, uniform_fn=None):
    """Verification of the 7 proposals against the target rows ([LSE] opening
    paragraph: probability-ratio rejection and residual sampling; greedy requests
    deterministic; [LUCE] greedy-width commit: greedy chain verification equals
    plain decode).

    target_logits [8][V]: row j is the target's distribution for block position
    j + 1 (row 7 = the bonus position after all 7 proposals).
    Greedy: t_j = argmax z_j (ties -> smaller id); accept d_{j+1} while it equals
    t_j; emit t_j at the first mismatch, or t_7 if all accepted.
    Sampled: p_j = softmax(z_j / T); accept d if u_a < p_j(d) / q_j(d) (u_a: slot j,
    purpose 1); on rejection draw x from max(0, p_j - q_j) normalised, by inverse
    CDF in vocabulary order (u_r: slot j, purpose 2), from p_j when that mass is
    <= 1e-30; if all are accepted draw the bonus from p_7 (slot 7, purpose 2).
    A row that holds a NaN or +inf, or whose maximum is -inf, makes the request
    nonfinite (then n_accepted = n_emitted = 0).

    Returns dict(n_accepted, emitted int32[8] (-1 padded), n_emitted, status,
    margins, decisions).  `decisions` lists each sampled decision in chain order
    as (kind, row, margin, scale): kind "accept" (margin relative to the ratio
    p/q), "residual" or "bonus" (margin relative to the drawn-from mass, whose
    total in p units is `scale`).  For T > 0 it also returns `p_path` [7] (p_j at
    the proposal of every row), `p_bonus` (p_7 at the bonus token, NaN unless all
    7 were accepted) and `residual_mass` [7] (sum_x max(0, p_j(x) - q_j(x)) of the
    rejected row, NaN elsewhere): the verify probabilities themselves.
    """
    Bk, V = target_logits.shape
    P = Bk - 1
    uni = uniform_fn or (lambda slot, purpose: philox.uniform(seed, offset, slot, purpose))
    emitted = np.full(Bk, -1, np.int32)
    z = np.asarray(target_logits, np.float64)
    if status_in != STATUS_OK:
        return {"n_accepted": 0, "emitted": emitted, "n_emitted": 0, "status": status_in, "margins": [],
                "decisions": []}
    rowmax = z.max(axis=1)
    if np.any(np.isnan(z)) or np.any(np.isposinf(z)) or np.any(~np.isfinite(rowmax)):
        return {"n_accepted": 0, "emitted": emitted, "n_emitted": 0, "status": STATUS_NONFINITE, "margins": [],
                "decisions": []}
    margins = []
    decisions = []
    if temperature == 0.0:
        t = [int(np.argmax(z[j])) for j in range(Bk)]      # argmax returns the first (smallest) index
        n = 0
        while n < P and int(path[n]) == t[n]:
            emitted[n] = path[n]
            n += 1
        emitted[n] = t[n]
        return {"n_accepted": n, "emitted": emitted, "n_emitted": n + 1, "status": STATUS_OK, "margins": margins,
                "decisions": decisions}
    p = np.exp((z - rowmax[:, None]) / temperature)
    p /= p.sum(axis=1, keepdims=True)
    probs = {"p_path": np.array([p[j, int(path[j])] for j in range(P)]), "p_bonus": math.nan,
             "residual_mass": np.full(P, math.nan)}
    for j in range(P):
        d = int(path[j])
        jj = int(np.nonzero(cand_ids[j] == d)[0][0])
        qd = float(q_rows[j, jj])
        u = uni(j, philox.PURPOSE_ACCEPT)
        ratio = p[j, d] / qd if qd > 0 else math.inf
        margins.append(abs(u - ratio) / max(ratio, 1e-300) if math.isfinite(ratio) else math.inf)
        decisions.append(("accept", j, margins[-1], ratio))
        if u < ratio:
            emitted[j] = d
            continue
        q_full = np.zeros(V)
        q_full[cand_ids[j]] = q_rows[j]
        r = np.maximum(0.0, p[j] - q_full)
        probs["residual_mass"][j] = r.sum()
        if r.sum() <= 1e-30:
            r = p[j]
        x, mg = _inverse_cdf(r, uni(j, philox.PURPOSE_RESAMPLE))
        margins.append(mg)
        decisions.append(("residual", j, mg, float(r.sum())))
        emitted[j] = x
        return {"n_accepted": j, "emitted": emitted, "n_emitted": j + 1, "status": STATUS_OK, "margins": margins,
                "decisions": decisions, **probs}
    x, mg = _inverse_cdf(p[P], uni(P, philox.PURPOSE_RESAMPLE))
    margins.append(mg)
    decisions.append(("bonus", P, mg, 1.0))
    emitted[P] = x
    probs["p_bonus"] = p[P, x]
    return {"n_accepted": P, "emitted": emitted, "n_emitted": P + 1, "status": STATUS_OK, "margins": margins,
            "decisions": decisions, **probs}


def _inverse_cdf(w: np.ndarray, u: float):
    """First index x with cumsum(w)[x] > u * sum(w); falls back to the last positive
    entry.  Returns (x, relative distance of u*sum from the nearest cumsum)."""
    cum = np.cumsum(w)
    tot = cum[-1]
    target = u * tot
    x = int(np.searchsorted(cum, target, side="right"))
    if x >= w.size or w[x] <= 0:
        x = int(np.nonzero(w > 0)[0][-1])
    lo = cum[x - 1] if x > 0 else 0.0
    margin = min(abs(target - lo), abs(cum[x] - target)) / tot
    return x, margin


# ----------------------------------------------------------------------------- one step

def advance(ctx_len: int, n_new: int, anchor: int, emitted: Sequence[int], n_emitted: int, offset: int,
            block: int = 8):
    """Request state for the next draft + verify step ([LSE] block paragraph: every
    draft is an anchor plus seven masks; [VLLM] PR description, candidate selector:
    the walk starts at the verified anchor).  Reading: the rows appended this step
    become context; the tokens verify emitted are the next step's new context rows,
    the last of them the next anchor; each step draws from its own Philox counter
    range, the offset advanced by one.  A request with nothing emitted keeps its
    anchor and appends nothing.  Returns (ctx_len, n_new, anchor, offset)."""
    ne = max(0, min(int(n_emitted), block))
    nxt_anchor = int(emitted[ne - 1]) if ne > 0 else int(anchor)
    return int(ctx_len) + max(0, min(int(n_new), block)), ne, nxt_anchor, int(offset) + 1


def block_width(ctx_len: int, n_new: int, block: int, ctx_threshold: int = 8192, narrow_width: int = 8) -> int:
    """Draft-block width of one request for a step ([LUCE] long-context commits: the
    verify's cost scales with the block's rows and the KV length, so past a context
    threshold the block narrows; the rule reads the context length only, never the
    acceptance rate; threshold 0 disables it; the first cut's 32768 default moved to
    8192, with narrowing to 8 inside a block-16 drafter).  Reading: the context is
    the keys the step's block attends to, ctx_len + n_new, and "past" is strictly
    greater.  A narrowed request's step is the step of a block of that width."""
    L = max(0, int(ctx_len)) + max(0, int(n_new))
    return narrow_width if (ctx_threshold > 0 and L > ctx_threshold) else block


def step(g, W: Dict, anchor: int, ctx_len: int, n_new: int, taps, k_cache, v_cache,
         temperature: float, seed: int, offset: int, target_logits_fn) -> Dict:
    """draft_block + top-16 + walk + verify for one request.  target_logits_fn maps the
    drafter logits [7][V] to the target rows [8][V] (the harness's construction)."""
    tr = draft_block(g, W, anchor, ctx_len, n_new, taps, k_cache, v_cache)
    K = g.top_k
    cand = np.zeros((g.block - 1, K), np.int32)
    cl = np.zeros((g.block - 1, K))
    for i in range(g.block - 1):
        cand[i], cl[i] = topk(tr["logits"][i], K)
    sel = walk(g, W["cb_a"], W["cb_b"], anchor, cand, cl, tr["gate"], temperature, seed, offset)
    z = target_logits_fn(tr["logits"])
    ver = verify(z, sel["path"], cand, sel["q_rows"], temperature, seed, offset, sel["status"])
    return {"draft": tr, "cand_ids": cand, "cand_logits": cl, "select": sel, "verify": ver, "target": z}
