"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: numbers the
pages print (tests/golden/lse_dflash2_facts.json), closed forms, textbook
special cases computed by library routines, invariants, and brute force.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import philox
from oracle.dflash2 import matmul_rows
import workloads as wk
from workloads.gen import weight_shapes

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "lse_dflash2_facts.json")))


# ----------------------------------------------------------------------------- geometry

def test_geometry_matches_published_parameter_count():
    """The layer structure the oracle runs sums to the page's exact parameter count,
    BF16 byte count and Q8 tensor count (LSE docs, compatible-drafter and Q8
    paragraphs).  A missing norm, delta projection or bias would break the sums."""
    g = wk.FULL
    shp = weight_shapes(g)
    shared = {"embed", "lm_head"}                     # shared with the target, not in the drafter file
    own = {k: v for k, v in shp.items() if k not in shared}
    n_params = sum(int(np.prod(s)) for s in own.values())
    assert n_params == GOLD["bf16_params"]
    assert len(own) == 81
    header = GOLD["bf16_file_bytes"] - 2 * n_params
    assert 0 < header < 16384                          # safetensors JSON header of 81 tensors
    mats = [k for k, s in own.items() if len(s) == 2 and k.split(".")[-1] in wk.MATRIX_NAMES]
    assert len(mats) == 49
    vecs = [k for k in own if k not in mats]
    n_tensors_q8 = 3 * len(mats) + len(vecs)
    assert n_tensors_q8 == GOLD["q8_tensors"]
    q8_bytes = sum(int(np.prod(own[k])) * 68 // 64 for k in mats) + 2 * sum(int(np.prod(own[k])) for k in vecs)
    assert 0 < GOLD["q8_file_bytes"] - q8_bytes < 32768
    assert (g.hidden, g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, g.ffn) == \
        (GOLD["hidden"], GOLD["layers"], GOLD["q_heads"], GOLD["kv_heads"], GOLD["head_dim"], GOLD["ffn"])
    assert (g.block, g.top_k, g.rank, g.window, g.conv_taps, g.conv_group) == \
        (GOLD["block"], GOLD["top_k"], GOLD["rank"], GOLD["window"], GOLD["conv_taps"], GOLD["conv_group"])


# ----------------------------------------------------------------------------- numbers

def test_round_to_bf16_is_nearest_even():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.normal(0, 1, 4000), rng.normal(0, 1e-3, 1000), rng.normal(0, 300, 1000)])
    r = oracle.round_to_bf16(x)
    for xi, ri in zip(x[:600], r[:600]):
        # brute force: the two bf16 neighbours bracketing xi
        m, e = math.frexp(abs(xi))
        step = 2.0 ** (e - 8)
        lo = math.floor(abs(xi) / step) * step
        hi = lo + step
        d_lo, d_hi = abs(abs(xi) - lo), abs(hi - abs(xi))
        if d_lo < d_hi:
            want = lo
        elif d_hi < d_lo:
            want = hi
        else:
            want = lo if (round(lo / step) % 2 == 0) else hi
        assert abs(ri) == want and (ri == 0 or np.sign(ri) == np.sign(xi))
    # exactly representable in bf16 -> unchanged; matches a float32 -> bf16 bit rounding
    b = wk.bf16_bits_from_f32(x.astype(np.float32))
    y = oracle.bf16_to_f64(b)
    assert np.array_equal(oracle.round_to_bf16(y), y)


def test_q8_dequant_worked_example():
    """w = scale * q + bias per group of 64 (LSE docs, Q8 paragraph: affine Q8, group 64)."""
    codes = np.arange(-128, 128, dtype=np.int8).reshape(2, 128)
    scale = wk.bf16_bits_from_f32(np.array([[2.0 ** -7, 0.5], [1.0, 0.0]], np.float32))
    bias = wk.bf16_bits_from_f32(np.array([[1.0, -2.0], [0.25, 3.0]], np.float32))
    w = oracle.matrix_f64({"kind": "q8", "codes": codes, "scale": scale, "bias": bias})
    q = codes.astype(np.float64)
    assert np.array_equal(w[0, :64], 1.0 + q[0, :64] / 128.0)
    assert np.array_equal(w[0, 64:], -2.0 + 0.5 * q[0, 64:])
    assert np.array_equal(w[1, :64], 0.25 + q[1, :64])
    assert np.array_equal(w[1, 64:], np.full(64, 3.0))


def test_rmsnorm_matches_library():
    rng = np.random.default_rng(2)
    x = rng.normal(0, 3, (8, 512))
    wb = wk.bf16_bits_from_f32(rng.normal(1, 0.02, 512).astype(np.float32))
    w = oracle.bf16_to_f64(wb)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (512,), torch.from_numpy(w), eps=1e-6).numpy()
    assert np.allclose(oracle.rmsnorm(x, wb, 1e-6), ref, rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------------------- RoPE

def test_rope_position_zero_identity_and_norm():
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1, (5, 8, 128))
    assert np.allclose(oracle.rope_neox(x, [0] * 5, 1e7), x, atol=0, rtol=0)
    y = oracle.rope_neox(x, [1, 17, 2055, 33000, 10 ** 6], 1e7)
    # each (j, j+64) pair is rotated: the pair norms are preserved
    n0 = x[..., :64] ** 2 + x[..., 64:] ** 2
    n1 = y[..., :64] ** 2 + y[..., 64:] ** 2
    assert np.allclose(n0, n1, rtol=1e-12)


def test_rope_relative_position_property():
    """<rope(q, m), rope(k, n)> depends only on m - n (the defining property of rotary
    embeddings); a wrong sign, pairing or frequency breaks it."""
    rng = np.random.default_rng(4)
    q = rng.normal(0, 1, (1, 1, 128))
    k = rng.normal(0, 1, (1, 1, 128))
    dots = []
    for m in (5, 1000, 40000):
        qa = oracle.rope_neox(q, [m], 1e7)
        ka = oracle.rope_neox(k, [m - 3], 1e7)
        dots.append(float(np.sum(qa * ka)))
    assert np.allclose(dots, dots[0], rtol=1e-9)
    # and it is not trivially constant across different offsets
    qa = oracle.rope_neox(q, [7], 1e7)
    ka = oracle.rope_neox(k, [0], 1e7)
    assert abs(float(np.sum(qa * ka)) - dots[0]) > 1e-6


def test_rope_frequencies_theta_1e7():
    f = oracle.rope_inv_freq(128, 1e7)
    assert f[0] == 1.0
    assert np.isclose(f[1], 1e7 ** (-2 / 128), rtol=1e-15)
    assert np.isclose(f[-1] / f[-2], 1e7 ** (-2 / 128), rtol=1e-13)
    # NEOX pairing: rotating pair j only moves components j and j+64 (one-hot probe)
    x = np.zeros((1, 1, 128))
    x[0, 0, 5] = 1.0
    y = oracle.rope_neox(x, [1000], 1e7)[0, 0]
    nz = set(np.nonzero(np.abs(y) > 1e-15)[0])
    assert nz <= {5, 69}
    ang = 1000 * f[5]
    assert np.isclose(y[5], math.cos(ang)) and np.isclose(y[69], math.sin(ang))


# ----------------------------------------------------------------------------- conv

def _conv_inputs(B=8, H=64, G=4, seed=5):
    rng = np.random.default_rng(seed)
    return rng.normal(0, 1, (B, H)), rng.normal(0, 1, (2, H)), rng.normal(0, 1, (B, 2, G))


def test_conv_identity_init():
    """Bases (1, 0) with a zero dynamic part is the identity (Speculators PR quoted in the
    vLLM PR thread: identity-initialized, block-local convolutions)."""
    x, _, _ = _conv_inputs()
    base = np.stack([np.ones(64), np.zeros(64)])
    assert np.array_equal(oracle.dyn_conv(x, base, np.zeros((8, 2, 4)), 16), x)


@pytest.mark.parametrize("B", [8, 16])
def test_conv_pure_shift_and_block_boundary(B):
    x, _, _ = _conv_inputs(B=B)
    base = np.stack([np.zeros(64), np.ones(64)])
    y = oracle.dyn_conv(x, base, np.zeros((B, 2, 4)), 16)
    assert np.array_equal(y[0], np.zeros(64))          # the anchor sees nothing before the block
    assert np.array_equal(y[1:], x[:-1])


def test_conv_group_locality_and_linearity():
    x, base, d = _conv_inputs()
    y = oracle.dyn_conv(x, base, d, 16)
    d2 = d.copy()
    d2[3, 1, 2] += 1.0                                 # position 3, tap 1, group 2 (channels 32..47)
    y2 = oracle.dyn_conv(x, base, d2, 16)
    diff = np.abs(y2 - y) > 0
    assert set(np.nonzero(diff.any(axis=1))[0]) == {3}
    assert set(np.nonzero(diff[3])[0]) == set(range(32, 48))
    assert np.allclose(y2[3, 32:48] - y[3, 32:48], x[2, 32:48])
    z = oracle.dyn_conv(2.0 * x - x[::-1], base, d, 16)
    assert np.allclose(z, 2.0 * y - oracle.dyn_conv(x[::-1], base, d, 16))


# ----------------------------------------------------------------------------- attention

def _sdpa(q, k, v, mask=None):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    return torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=mask).numpy()


@pytest.mark.parametrize("B", [8, 16])
def test_attention_dense_case_matches_library(B):
    """With every context key inside the window the block attention is plain
    noncausal GQA softmax attention (torch SDPA in float64), for blocks of 8 and 16."""
    rng = np.random.default_rng(6)
    nq, nkv, hd, L = 8, 2, 128, 300
    q = rng.normal(0, 1, (B, nq, hd))
    kb, vb = rng.normal(0, 1, (B, nkv, hd)), rng.normal(0, 1, (B, nkv, hd))
    kc, vc = rng.normal(0, 1, (L, nkv, hd)), rng.normal(0, 1, (L, nkv, hd))
    out = oracle.block_attention(q, kb, vb, kc, vc, L, 2048).reshape(B, nq, hd)
    K = np.concatenate([kc, kb])
    V = np.concatenate([vc, vb])
    rep = nq // nkv
    Kh = np.repeat(K.transpose(1, 0, 2), rep, axis=0)   # [nq][L+B][hd]
    Vh = np.repeat(V.transpose(1, 0, 2), rep, axis=0)
    ref = _sdpa(q.transpose(1, 0, 2), Kh, Vh).transpose(1, 0, 2)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("B", [8, 16])
def test_attention_window_matches_masked_library_and_ignores_masked_keys(B):
    rng = np.random.default_rng(7)
    nq, nkv, hd, W = 4, 1, 128, 64
    L = 200
    q = rng.normal(0, 1, (B, nq, hd))
    kb, vb = rng.normal(0, 1, (B, nkv, hd)), rng.normal(0, 1, (B, nkv, hd))
    kc, vc = rng.normal(0, 1, (L, nkv, hd)), rng.normal(0, 1, (L, nkv, hd))
    out = oracle.block_attention(q, kb, vb, kc, vc, L, W)
    # boolean mask: query i (position L+i) sees context key k iff L+i-k < W, and all block keys
    mask = np.zeros((B, L + B), bool)
    for i in range(B):
        for k in range(L):
            mask[i, k] = (L + i - k) < W
        mask[i, L:] = True
    K = np.concatenate([kc, kb])[:, 0]
    V = np.concatenate([vc, vb])[:, 0]
    ref = _sdpa(q.transpose(1, 0, 2), np.repeat(K[None], nq, 0), np.repeat(V[None], nq, 0),
                torch.from_numpy(mask)).transpose(1, 0, 2).reshape(B, nq * hd)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[: L - W + 1] = np.nan                          # every key outside all windows
    vc2[: L - W + 1] = np.nan
    assert np.array_equal(oracle.block_attention(q, kb, vb, kc2, vc2, L, W), out)


def test_live_key_counts_match_page():
    """LSE docs, attention test paragraph: live counts 17 and 2055 for 8 queries.
    Reading: keys visible to query 0 = visible context + the 8 block keys; 2055 =
    2047 + 8 once the context fills the 2048 window (a block-uniform window would
    give 2056)."""
    def live(L, i):
        lo, hi = oracle.visible_context_range(L, i, 2048)
        return hi - lo + 8
    assert live(9, 0) == GOLD["attention_live_counts"][0]
    assert live(4096, 0) == GOLD["attention_live_counts"][1]
    assert [live(4096, i) for i in range(8)] == [2055 - i for i in range(8)]


# ----------------------------------------------------------------------------- top-k

def test_topk_matches_stable_sort_and_edge_policy():
    rng = np.random.default_rng(8)
    row = rng.integers(-50, 50, 4097).astype(np.float32)   # many ties
    ids, vals = oracle.topk(row, 16)
    ref = np.argsort(-row.astype(np.float64), kind="stable")[:16]
    assert np.array_equal(ids, ref)
    # edge rows in the manner of the page's 4097-wide edge test (LSE docs, top-k paragraph)
    r = rng.normal(0, 1, 4097).astype(np.float32)
    r[[10, 600, 4000]] = np.nan
    r[[5, 3000]] = np.inf
    r[[7]] = -np.inf
    ids, _ = oracle.topk(r, 16)
    assert list(ids[:3]) == [10, 600, 4000]              # NaNs first, by index
    assert list(ids[3:5]) == [5, 3000]                   # +inf next
    allneg = np.full(4097, -np.inf, np.float32)
    ids, vals = oracle.topk(allneg, 16)
    assert list(ids) == list(range(16)) and np.all(np.isneginf(vals))
    tie = np.zeros(4097, np.float32)
    tie[[512, 513, 1024, 1536, 4096]] = 1.0                # ties across 512-chunk boundaries
    ids, _ = oracle.topk(tie, 16)
    assert list(ids[:5]) == [512, 513, 1024, 1536, 4096] and list(ids[5:]) == list(range(11))


# ----------------------------------------------------------------------------- selector

def _gamma(n):
    u = 2.0 ** -24
    return n * u / (1 - n * u)


def test_selector_scores_library_and_page_rounding_bound():
    """Scores equal an einsum of the rank-256 triple product; a float32 evaluation in
    another order stays inside the page's mixed rounding bound
    gamma_(rank+2) * sum|pred*gate*succ| + 2u/(1-u) * |ref| (LSE docs, selector test)."""
    rng = np.random.default_rng(9)
    P, C, r = 16, 16, 256
    A = rng.normal(0, 0.02, (P, r))
    Bc = rng.normal(0, 0.02, (C, r))
    gate = rng.normal(0, 1.4, r)
    un = rng.normal(0, 1.4, C)
    s = oracle.selector_scores(A, gate, Bc, un)
    ref = np.einsum("pr,r,cr->pc", A, gate, Bc) + un[None, :]
    assert np.allclose(s, ref, rtol=1e-13, atol=1e-15)
    u = 2.0 ** -24
    A32, g32, B32, un32 = (a.astype(np.float32) for a in (A, gate, Bc, un))
    for p in range(P):
        for c in range(C):
            acc = np.float32(0)
            for k in reversed(range(r)):
                acc = np.float32(acc + np.float32(np.float32(A32[p, k] * g32[k]) * B32[c, k]))
            s32 = np.float32(acc + un32[c])
            exact = float(np.sum(A32[p].astype(np.float64) * g32 * B32[c])) + float(un32[c])
            bound = _gamma(r + 2) * float(np.sum(np.abs(A32[p].astype(np.float64) * g32 * B32[c]))) \
                + 2 * u / (1 - u) * abs(exact)
            assert abs(float(s32) - exact) <= bound
    assert P * C * 7 == GOLD["selector_scores_checked"]


def _sel_inputs(seed, V=64, K=4, r=8, P=7, with_q8=False):
    rng = np.random.default_rng(seed)
    A = wk.bf16_bits_from_f32(rng.normal(0, 0.5, (V, r)).astype(np.float32))
    Bm = wk.bf16_bits_from_f32(rng.normal(0, 0.5, (V, r)).astype(np.float32))
    cand = np.stack([rng.choice(V, K, replace=False) for _ in range(P)]).astype(np.int32)
    cl = -np.sort(-rng.normal(0, 1, (P, K)), axis=1)
    gate = rng.normal(0, 1, (P, r))
    return {"kind": "bf16", "w": A}, {"kind": "bf16", "w": Bm}, cand, cl, gate


def test_greedy_walk_is_predecessor_conditioned_argmax():
    """Greedy path = argmax of the edge score from the chosen predecessor, starting at
    the anchor (vLLM PR description); checked by brute force over the candidates."""
    class G:
        block = 8
    for seed in range(5):
        A, Bm, cand, cl, gate = _sel_inputs(seed)
        anchor = 3
        res = oracle.walk(G, A, Bm, anchor, cand, cl, gate, 0.0, 0, 0)
        Af, Bf = oracle.bf16_to_f64(A["w"]), oracle.bf16_to_f64(Bm["w"])
        prev = anchor
        for i in range(7):
            sc = [float(np.sum(Af[prev] * gate[i] * Bf[c])) + cl[i, j] for j, c in enumerate(cand[i])]
            j = int(np.argmax(sc))
            assert res["path"][i] == cand[i, j]
            prev = cand[i, j]
        assert np.allclose(res["q_rows"].sum(axis=1), 1.0)


def test_sampled_walk_low_temperature_equals_greedy_and_distribution():
    class G:
        block = 8
    A, Bm, cand, cl, gate = _sel_inputs(11)
    g0 = oracle.walk(G, A, Bm, 3, cand, cl, gate, 0.0, 0, 0)
    gt = oracle.walk(G, A, Bm, 3, cand, cl, gate, 1e-4, 7, 0)
    assert np.array_equal(g0["path"], gt["path"])
    # first-position draws over many Philox offsets follow softmax(s / T)
    T = 1.0
    n = 4000
    counts = np.zeros(4)
    for off in range(n):
        res = oracle.walk(G, A, Bm, 3, cand[:1], cl[:1], gate[:1], T, 123, off)
        counts[list(cand[0]).index(res["path"][0])] += 1
    q = res["q_rows"][0]
    chi2 = float(np.sum((counts - n * q) ** 2 / (n * q)))
    assert chi2 < 16.3                                  # 3 dof, p = 0.001


# ----------------------------------------------------------------------------- verify

def _breakpoint_integral(fn, points):
    """Integrate a piecewise-constant function of u on [0,1) exactly, given a superset
    of its breakpoints: evaluate at interval midpoints, weight by interval length."""
    pts = sorted(set([0.0, 1.0] + [p for p in points if 0.0 < p < 1.0]))
    out = []
    for a, b in zip(pts[:-1], pts[1:]):
        out.append((b - a, fn(0.5 * (a + b))))
    return out


def test_verify_single_position_is_lossless_exactly():
    """Probability-ratio rejection with residual sampling emits exactly the target
    distribution (LSE docs: the target verifies with probability-ratio rejection and
    residual sampling).  Brute force over a 5-token vocabulary, the draft token drawn
    from q, both uniforms integrated exactly."""
    V, K = 5, 2
    rng = np.random.default_rng(12)
    for trial in range(6):
        z = rng.normal(0, 1.5, (8, V))
        T = [1.0, 0.7, 2.0][trial % 3]
        p0 = np.exp(z[0] / T - (z[0] / T).max())
        p0 /= p0.sum()
        cand = np.zeros((7, K), np.int32)
        cand[0] = rng.choice(V, K, replace=False)
        for i in range(1, 7):
            cand[i] = rng.choice(V, K, replace=False)
        qv = rng.dirichlet(np.ones(K))
        q_rows = np.tile(qv, (7, 1))
        emitted = np.zeros(V)
        for jd in range(K):
            d = cand[0, jd]
            path = np.full(7, d, np.int32)
            path[1:] = cand[1:, 0]
            q_full = np.zeros(V)
            q_full[cand[0]] = qv
            resid = np.maximum(0, p0 - q_full)
            cuts = [p0[d] / qv[jd]] + list(np.cumsum(resid) / max(resid.sum(), 1e-300)) + list(np.cumsum(p0))
            for wa, ua in _breakpoint_integral(lambda u: u, cuts):
                for wr, ur in _breakpoint_integral(lambda u: u, cuts):
                    def uni(slot, purpose, ua=ua, ur=ur):
                        if slot == 0 and purpose == philox.PURPOSE_ACCEPT:
                            return ua
                        if slot == 0 and purpose == philox.PURPOSE_RESAMPLE:
                            return ur
                        return 0.999999                   # later positions: reject (first token only matters)
                    res = oracle.verify(z, path, cand, q_rows, T, 0, 0, uniform_fn=uni)
                    emitted[res["emitted"][0]] += qv[jd] * wa * wr
        assert np.allclose(emitted, p0, atol=1e-12), (emitted, p0)


def test_verify_two_positions_conditional_lossless():
    """Conditioned on the first draft being accepted, the second emitted token follows
    the target's second row exactly (the second draft drawn from its q row, both of
    that position's uniforms integrated exactly)."""
    V, K = 5, 2
    rng = np.random.default_rng(13)
    z = rng.normal(0, 1.0, (8, V))
    T = 1.0
    P = np.exp(z - z.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    cand = np.stack([rng.choice(V, K, replace=False) for _ in range(7)]).astype(np.int32)
    q_rows = rng.dirichlet(np.ones(K), size=7)
    second = np.zeros(V)
    for j0 in range(K):
        for j1 in range(K):
            path = cand[:, 0].copy()
            path[0], path[1] = cand[0, j0], cand[1, j1]
            pq = q_rows[0, j0] * q_rows[1, j1]
            qf = np.zeros(V)
            qf[cand[1]] = q_rows[1]
            resid = np.maximum(0, P[1] - qf)
            cuts = [P[1][path[1]] / q_rows[1, j1]] + list(np.cumsum(resid) / resid.sum())
            for wa, ua in _breakpoint_integral(lambda u: u, cuts):
                for wr, ur in _breakpoint_integral(lambda u: u, cuts):
                    def uni(slot, purpose, ua=ua, ur=ur):
                        if slot == 0:
                            return 0.0 if purpose == philox.PURPOSE_ACCEPT else 0.5   # accept position 1
                        if slot == 1:
                            return ua if purpose == philox.PURPOSE_ACCEPT else ur
                        return 0.999999
                    res = oracle.verify(z, path, cand, q_rows, T, 0, 0, uniform_fn=uni)
                    assert res["n_accepted"] >= 1
                    second[res["emitted"][1]] += pq * wa * wr
    # first draft accepted with u = 0 always: the second token's law given the first is P[1]
    marg = second / second.sum()
    assert np.allclose(marg, P[1], atol=1e-12)


def test_verify_reported_probabilities():
    """The verify probabilities the oracle reports are the ones its decisions use, pinned
    by two identities of speculative sampling, both uniforms integrated exactly:
      * the acceptance probability of a row, with the draft token drawn from q, is
        sum_x min(p(x), q(x)) = 1 - sum_x max(0, p(x) - q(x)): one minus the reported
        residual mass; and P(accept | d) = min(1, p_path / q(d));
      * the bonus token x is drawn from p_7, so E[1 / p_bonus] = the number of tokens
        with p_7 > 0 (all V of them)."""
    V, K = 5, 2
    rng = np.random.default_rng(15)
    for trial in range(4):
        z = rng.normal(0, 1.5, (8, V))
        T = [1.0, 0.7, 2.0, 1.3][trial]
        cand = np.stack([rng.choice(V, K, replace=False) for _ in range(7)]).astype(np.int32)
        qv = rng.dirichlet(np.ones(K))
        q_rows = np.tile(qv, (7, 1))
        acc = 0.0
        resid = []
        for jd in range(K):
            d = cand[0, jd]
            path = cand[:, 0].copy()
            path[0] = d
            acc_d = 0.0
            cuts = list(np.linspace(0, 1, 2001)[1:-1])
            probe = oracle.verify(z, path, cand, q_rows, T, 0, 0, uniform_fn=lambda s, p: 0.0)
            cuts.append(probe["p_path"][0] / qv[jd])
            for wa, ua in _breakpoint_integral(lambda u: u, cuts):
                def uni(slot, purpose, ua=ua):
                    if slot == 0 and purpose == philox.PURPOSE_ACCEPT:
                        return ua
                    return 0.999999 if purpose == philox.PURPOSE_ACCEPT else 0.5
                res = oracle.verify(z, path, cand, q_rows, T, 0, 0, uniform_fn=uni)
                if res["n_accepted"] >= 1:
                    acc_d += wa
                else:
                    resid.append(res["residual_mass"][0])
            assert abs(acc_d - min(1.0, probe["p_path"][0] / qv[jd])) < 1e-12
            acc += qv[jd] * acc_d
        if resid:
            assert np.allclose(resid, resid[0], rtol=0, atol=1e-15)
            assert abs((1.0 - acc) - resid[0]) < 1e-12, (acc, resid[0])
        # bonus: every proposal accepted (u = 0), the bonus uniform integrated exactly
        path = cand[:, 0].copy()
        probe = oracle.verify(z, path, cand, q_rows, T, 0, 0, uniform_fn=lambda s, p: 0.0)
        assert probe["n_accepted"] == 7
        p7 = np.exp((z[7] - z[7].max()) / T)
        cuts = list(np.cumsum(p7 / p7.sum()))
        inv = 0.0
        for wr, ur in _breakpoint_integral(lambda u: u, cuts):
            res = oracle.verify(z, path, cand, q_rows, T, 0, 0,
                                uniform_fn=lambda s, p, ur=ur: ur if p == philox.PURPOSE_RESAMPLE else 0.0)
            inv += wr / res["p_bonus"]
        assert abs(inv - V) < 1e-9, inv


def test_verify_greedy_is_argmax_chain():
    rng = np.random.default_rng(14)
    V = 50
    for trial in range(20):
        z = rng.normal(0, 1, (8, V)).astype(np.float32)
        t = np.argmax(z, axis=1)
        n_match = trial % 8
        path = np.array([t[j] if j < n_match else (t[j] + 1) % V for j in range(7)], np.int32)
        cand = np.stack([np.array([path[j]] + [x for x in range(16) if x != path[j]][:15]) for j in range(7)]).astype(np.int32)
        res = oracle.verify(z, path, cand, np.zeros((7, 16)), 0.0, 0, 0)
        assert res["n_accepted"] == min(n_match, 7)
        assert res["n_emitted"] == res["n_accepted"] + 1
        assert list(res["emitted"][: res["n_emitted"]]) == list(t[: res["n_emitted"]])


def test_verify_nonfinite_rows():
    z = np.zeros((8, 10))
    z[3, 4] = np.nan
    res = oracle.verify(z, np.zeros(7, np.int32), np.zeros((7, 16), np.int32), np.zeros((7, 16)), 1.0, 0, 0)
    assert res["status"] == oracle.STATUS_NONFINITE and res["n_emitted"] == 0
    z = np.zeros((8, 10))
    z[0] = -np.inf
    res = oracle.verify(z, np.zeros(7, np.int32), np.zeros((7, 16), np.int32), np.zeros((7, 16)), 0.0, 0, 0)
    assert res["status"] == oracle.STATUS_NONFINITE


# ----------------------------------------------------------------------------- drafter layer

def _torch_layer_reference(g, W, x, c, kctx, vctx, L, pos_blk):
    """A Qwen3 decoder layer from torch library ops (F.rms_norm, F.linear, SDPA, F.silu),
    used for the special case of identity convolutions (bases (1,0), zero delta)."""
    F = torch.nn.functional
    T = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    w = lambda n: T(oracle.matrix_f64(W[n]))
    v = lambda n: T(oracle.bf16_to_f64(W[n]))
    H, hd, nq, nkv = g.hidden, g.head_dim, g.n_q_heads, g.n_kv_heads
    x = T(x)
    a = F.rms_norm(x, (H,), v("l0.input_norm"), eps=g.rms_eps)
    B = x.shape[0]
    q = F.rms_norm(F.linear(a, w("l0.q")).view(B, nq, hd), (hd,), v("l0.q_norm"), eps=g.rms_eps)
    k = F.rms_norm(F.linear(a, w("l0.k")).view(B, nkv, hd), (hd,), v("l0.k_norm"), eps=g.rms_eps)
    vv = F.linear(a, w("l0.v")).view(B, nkv, hd)
    inv = T(oracle.rope_inv_freq(hd, g.rope_theta))
    ang = T(pos_blk)[:, None] * inv[None]
    rot = lambda t: torch.view_as_real(torch.view_as_complex(
        torch.stack([t[..., :hd // 2], t[..., hd // 2:]], -1).contiguous()) *
        torch.polar(torch.ones_like(ang), ang)[:, None, :])
    def rope(t):
        r = rot(t)
        return torch.cat([r[..., 0], r[..., 1]], -1)
    q, k = rope(q), rope(k)
    K = torch.cat([T(kctx), k])
    V = torch.cat([T(vctx), vv])
    rep = nq // nkv
    o = F.scaled_dot_product_attention(q.transpose(0, 1), K.transpose(0, 1).repeat_interleave(rep, 0),
                                       V.transpose(0, 1).repeat_interleave(rep, 0))
    x = x + F.linear(o.transpose(0, 1).reshape(B, nq * hd), w("l0.o"))
    m = F.rms_norm(x, (H,), v("l0.post_norm"), eps=g.rms_eps)
    x = x + F.linear(F.silu(F.linear(m, w("l0.gate"))) * F.linear(m, w("l0.up")), w("l0.down"))
    return x.numpy()


@pytest.mark.parametrize("block", [8, 16])
def test_draft_layer_reduces_to_qwen3_layer_with_identity_conv(block):
    """With identity convolutions a draft layer is a Qwen3 decoder layer over the
    block rows (anchor + block-1 masks, noncausal) and the context keys, for blocks
    of 8 and of 16 positions ([LUCE] greedy-width commit: block 16)."""
    import dataclasses
    g = dataclasses.replace(wk.TOY, hidden=256, ffn=512, vocab=1024, n_q_heads=4, n_kv_heads=2, block=block)
    W = wk.make_weights(g, "bf16", 21)
    for n in ("l0.attn_base", "l0.mlp_base"):
        W[n] = wk.bf16_bits_from_f32(np.stack([np.ones(g.hidden), np.zeros(g.hidden)] * 2).astype(np.float32))
    for n in ("l0.attn_delta", "l0.mlp_delta"):
        W[n] = {"kind": "bf16", "w": np.zeros_like(W[n]["w"])}
    rng = np.random.default_rng(22)
    ctx_len, n_new = 40, block
    cap = 64
    kc = [wk.bf16_bits_from_f32(rng.normal(0, 1, (cap, 2, 128)).astype(np.float32))]
    vc = [wk.bf16_bits_from_f32(rng.normal(0, 1, (cap, 2, 128)).astype(np.float32))]
    taps = rng.normal(0, 1, (n_new, 5 * g.hidden)).astype(np.float32)
    tr = oracle.draft_block(g, W, 17, ctx_len, n_new, taps, kc, vc)
    L = ctx_len + n_new
    x0 = oracle.bf16_to_f64(W["embed"][[17] + [g.mask_id] * (block - 1)])
    ref = _torch_layer_reference(g, W, x0, tr["c"], oracle.bf16_to_f64(kc[0][:L]), oracle.bf16_to_f64(vc[0][:L]),
                                 L, np.arange(L, L + block))
    assert np.allclose(tr["x0"], ref, rtol=1e-10, atol=1e-10)
    # the appended context rows are the taps projection through W_k / W_v of that layer
    c = tr["c"]
    kref = oracle.rope_neox(oracle.rmsnorm((c @ oracle.matrix_f64(W["l0.k"]).T).reshape(block, 2, 128),
                                           W["l0.k_norm"], g.rms_eps), np.arange(ctx_len, L), g.rope_theta)
    assert np.allclose(oracle.bf16_to_f64(kc[0][ctx_len:L]), kref, rtol=2 ** -8, atol=1e-30)


def test_draft_block_window_isolation():
    """Cache rows that no block query can see do not affect the draft (window), and the
    taps only enter through the appended context rows."""
    import dataclasses
    g = dataclasses.replace(wk.TOY, window=32, vocab=512)
    W = wk.make_weights(g, "bf16", 31)
    rng = np.random.default_rng(32)
    cap, ctx_len = 128, 90
    kc = [wk.bf16_bits_from_f32(rng.normal(0, 1, (cap, 1, 128)).astype(np.float32))]
    vc = [wk.bf16_bits_from_f32(rng.normal(0, 1, (cap, 1, 128)).astype(np.float32))]
    taps = rng.normal(0, 1, (8, 5 * g.hidden)).astype(np.float32)
    a = oracle.draft_block(g, W, 5, ctx_len, 8, taps, [kc[0].copy()], [vc[0].copy()])
    L = ctx_len + 8
    k2, v2 = kc[0].copy(), vc[0].copy()
    k2[: L - 32 + 1] = 0x7FC0                            # NaN in every row outside the window
    v2[: L - 32 + 1] = 0x7FC0
    b = oracle.draft_block(g, W, 5, ctx_len, 8, taps, [k2], [v2])
    assert np.array_equal(a["logits"], b["logits"])
    k3, v3 = kc[0].copy(), vc[0].copy()
    k3[L - 32 + 1] ^= 0x0101                             # the oldest visible row does matter
    c3 = oracle.draft_block(g, W, 5, ctx_len, 8, taps, [k3], [v3.copy()])
    assert not np.array_equal(a["logits"], c3["logits"])


def test_philox_structure():
    """Known structural facts of the definition: the key schedule and that ten rounds
    of a bijection on the counter give distinct outputs for distinct counters."""
    outs = {philox.philox4x32_10((i, 0, 0, 0), (1, 2)) for i in range(2000)}
    assert len(outs) == 2000
    u = [philox.uniform(42, 0, s, p) for s in range(8) for p in range(3)]
    assert all(0.0 <= x < 1.0 for x in u) and len(set(u)) == 24


def test_advance_worked_examples():
    """The serving-loop state update on hand-worked cases: the appended rows become
    context, the last emitted token the next anchor, the emitted tokens the next new
    rows, the Philox offset advances by one; nothing emitted keeps the anchor."""
    assert oracle.advance(100, 8, 5, [11, 12, 13, -1, -1, -1, -1, -1], 3, 7) == (108, 3, 13, 8)
    assert oracle.advance(108, 3, 13, [-1] * 8, 0, 8) == (111, 0, 13, 9)          # verify emitted nothing
    assert oracle.advance(0, 0, 2, [4, 5, 6, 7, 8, 9, 10, 11], 8, 1 << 32) == (0, 8, 11, (1 << 32) + 1)
    # a whole loop: context grows by the previous step's emitted count
    ctx, nn, anc, off = 50, 8, 1, 0
    for ne in (2, 8, 1, 0, 5):
        ctx_before, nn_before = ctx, nn
        ctx, nn, anc, off = oracle.advance(ctx, nn, anc, list(range(100, 108)), ne, off)
        assert ctx == ctx_before + nn_before and nn == ne
    assert (ctx, nn, anc, off) == (50 + 8 + 2 + 8 + 1 + 0, 5, 104, 5)


def test_viterbi_path_brute_force_and_examples():
    """The Viterbi selector on small lattices: its path is the one of highest total
    score over all K^P paths (brute force, tie-free random scores), greedy and Viterbi
    differ on a hand-made lattice, and equal totals go to smaller candidate ids."""
    import itertools
    rng = np.random.default_rng(77)
    for trial in range(20):
        P, K = 4, 5
        sc = rng.normal(0, 1, (P, K, K))
        sc[0] = np.repeat(sc[0, :1], K, axis=0)          # position 1: every row from the anchor
        ids = np.stack([rng.permutation(100)[:K] for _ in range(P)]).astype(np.int32)
        res = oracle.viterbi_path(sc, ids)
        s32 = sc.astype(np.float32)
        best, arg = None, None
        for path in itertools.product(range(K), repeat=P):
            tot = s32[0, 0, path[0]] + sum(s32[i, path[i - 1], path[i]] for i in range(1, P))
            if best is None or tot > best:
                best, arg = tot, path
        assert tuple(res["index"]) == arg
        assert abs(float(res["total"]) - float(best)) <= 1e-5 * max(1.0, abs(float(best)))
    # greedy takes 1.0 then 0 (total 1.0); the best path takes 0.9 then 5 (total 5.9)
    sc = np.zeros((2, 2, 2))
    sc[0] = [[1.0, 0.9], [1.0, 0.9]]
    sc[1] = [[0.0, 0.0], [5.0, 0.0]]
    ids = np.array([[10, 20], [30, 40]], np.int32)
    assert list(oracle.viterbi_path(sc, ids)["path"]) == [20, 30]
    # all-equal scores: the smallest ids at every position
    ids = np.array([[7, 3, 9], [5, 2, 8], [6, 1, 4]], np.int32)
    assert list(oracle.viterbi_path(np.zeros((3, 3, 3)), ids)["path"]) == [3, 2, 1]


# ----------------------------------------------------------------------------- draft tree (DDTree)

def _all_paths(scores, K, P):
    """Every root path of the tree (tuples of candidate indices) with its probability,
    enumerated by brute force: the product of the per-parent softmax of the lattice
    rows along the path (position 1 uses the anchor row 0)."""
    out = {}
    def rec(path, prob):
        d = len(path)
        if d == P:
            return
        prev = path[-1] if path else 0
        row = np.asarray(scores[d][prev], np.float64)
        pr = np.exp(row - row.max())
        pr /= pr.sum()
        for c in range(K):
            np_ = path + (c,)
            out[np_] = prob * pr[c]
            rec(np_, prob * pr[c])
    rec((), 1.0)
    return out


def test_ddtree_is_the_budget_most_probable_nodes():
    """Best-first growth on log-softmax-normalised scores yields exactly the `budget`
    most probable nodes of the whole tree (a child is never more probable than its
    parent), each after its parent (LUCE DDTree commit: cumulative best-first
    comparisons on a log-prob scale).  Brute force over every path, K = 3, depth 4."""
    rng = np.random.default_rng(31)
    K, P = 3, 4
    cand = np.arange(100, 100 + P * K, dtype=np.int32).reshape(P, K)
    for trial in range(20):
        scores = rng.normal(0, 1.5, (P, K, K))
        scores[0] = scores[0][0][None, :]               # position 1: the anchor row repeats
        paths = _all_paths(scores, K, P)
        ranked = sorted(paths.items(), key=lambda kv: -kv[1])
        for budget in (1, 4, 12, len(paths)):
            tr = oracle.ddtree_build(scores, cand, budget)
            assert len(tr["token"]) == min(budget, len(paths))
            got = {}
            for k in range(len(tr["token"])):
                pre = () if tr["parent"][k] < 0 else got[int(tr["parent"][k])]
                assert tr["parent"][k] < k                  # parents come first
                got[k] = pre + (int(tr["cand"][k]),)
                assert tr["depth"][k] == len(got[k])
                assert tr["token"][k] == cand[tr["depth"][k] - 1][tr["cand"][k]]
                assert abs(tr["score"][k] - math.log(paths[got[k]])) < 1e-12
            want = {p for p, _ in ranked[:len(tr["token"])]}
            assert set(got.values()) == want, (trial, budget)


def test_ddtree_children_of_a_node_normalise():
    """The normalised scores of a node's K children are log-probabilities: their
    exponentials, relative to the parent, sum to one."""
    rng = np.random.default_rng(32)
    K, P = 4, 3
    cand = np.arange(K * P, dtype=np.int32).reshape(P, K)
    scores = rng.normal(0, 2.0, (P, K, K))
    scores[0] = scores[0][0][None, :]
    full = K + K * K + K ** 3
    tr = oracle.ddtree_build(scores, cand, full)
    assert len(tr["token"]) == full
    for q in [-1] + list(range(full)):
        kids = [k for k in range(full) if tr["parent"][k] == q]
        if not kids:
            continue
        base = 0.0 if q < 0 else tr["score"][q]
        assert len(kids) == K
        assert abs(sum(math.exp(tr["score"][k] - base) for k in kids) - 1.0) < 1e-12


def test_ddtree_verify_on_a_chain_is_the_greedy_verify():
    """A tree that is a single chain verifies exactly as the chain (the greedy verify,
    pinned above as the argmax chain)."""
    rng = np.random.default_rng(33)
    V = 40
    for trial in range(20):
        z = rng.normal(0, 1, (8, V))
        t = np.argmax(z, axis=1)
        n_match = trial % 8
        path = np.array([t[j] if j < n_match else (t[j] + 1) % V for j in range(7)], np.int32)
        res = oracle.ddtree_verify(z, path, np.arange(-1, 6, dtype=np.int32))
        ref = oracle.verify(z, path, np.zeros((7, 16), np.int32), np.zeros((7, 16)), 0.0, 0, 0)
        assert res["n_accepted"] == ref["n_accepted"] and res["n_emitted"] == ref["n_emitted"]
        assert np.array_equal(res["emitted"], ref["emitted"])


def test_ddtree_verify_accepts_the_deepest_fully_matching_node():
    """Brute force on random trees: a node is accepted iff every node on its root path
    carries the argmax token of its parent's row; the verify ends at the deepest such
    node (unique: siblings carry distinct tokens) and emits that node's row argmax."""
    rng = np.random.default_rng(34)
    V = 6
    for trial in range(200):
        n = int(rng.integers(1, 14))
        parent = np.array([int(rng.integers(-1, k)) for k in range(n)], np.int32)
        token = np.zeros(n, np.int32)
        for k in range(n):  # siblings distinct
            used = {int(token[j]) for j in range(k) if parent[j] == parent[k]}
            token[k] = int(rng.choice([x for x in range(V) if x not in used])) if len(used) < V else 0
        depth = np.zeros(n, int)
        for k in range(n):
            depth[k] = 1 if parent[k] < 0 else depth[parent[k]] + 1
        if depth.max() > 7 or any(len({int(token[j]) for j in range(n) if parent[j] == q}) !=
                                  sum(1 for j in range(n) if parent[j] == q) for q in range(-1, n)):
            continue
        z = rng.integers(0, 3, (n + 1, V)).astype(np.float64)   # integer rows: ties to the smaller id
        am = [int(np.argmax(z[k])) for k in range(n + 1)]
        def matched(k):
            while k >= 0:
                if int(token[k]) != am[parent[k] + 1]:
                    return False
                k = parent[k]
            return True
        ok = [k for k in range(n) if matched(k)]
        deepest = max(ok, key=lambda k: depth[k]) if ok else -1
        res = oracle.ddtree_verify(z, token, parent)
        assert res["n_accepted"] == (depth[deepest] if deepest >= 0 else 0)
        assert res["emitted"][res["n_accepted"]] == am[deepest + 1]
        assert res["n_emitted"] == res["n_accepted"] + 1


# ----------------------------------------------------------------------------- wider blocks, narrowing

def _plain_next(seq, V):
    """A deterministic stand-in for the target's greedy next token: a fixed hash of the
    last three tokens (any function of the prefix would do)."""
    a, b, c = (list(seq[-3:]) + [0, 0, 0])[:3]
    return (a * 1_000_003 + b * 7_919 + c * 104_729 + len(seq) * 31) % V


@pytest.mark.parametrize("block", [8, 10, 12, 16, 20, 24])
def test_greedy_chain_equals_plain_decode_at_any_width(block):
    """[LUCE] greedy-width commit: greedy chain verification emits exactly what plain
    decoding emits at any draft width (byte-identical completions at widths 8 to 24).
    Drafts that are right with probability 0.7 per position (else a random token) go
    through the oracle's greedy verify and serving-loop update, with target rows whose
    argmax is the stand-in target's next token after the proposals; the emitted text
    must equal plain decoding's, and every step must emit between 1 and block tokens."""
    V = 97
    rng = np.random.default_rng(block)
    prompt = [5, 9, 13]
    plain = list(prompt)
    for _ in range(200):
        plain.append(_plain_next(plain, V))
    seq = list(prompt)
    ctx, nn, anchor, off = len(prompt) - 1, 1, prompt[-1], 0
    steps = 0
    while len(seq) < len(plain):
        path = []
        for j in range(block - 1):
            right = _plain_next(seq + path, V)
            path.append(right if rng.random() < 0.7 else int(rng.integers(V)))
        z = rng.normal(0, 1, (block, V))
        for j in range(block):
            z[j, _plain_next(seq + path[:j], V)] = 10.0
        res = oracle.verify(z, np.array(path), np.zeros((block - 1, 16), np.int32), np.zeros((block - 1, 16)),
                            0.0, 0, off)
        ne = res["n_emitted"]
        assert 1 <= ne <= block and res["n_accepted"] == ne - 1
        em = [int(t) for t in res["emitted"][:ne]]
        assert list(res["emitted"][ne:]) == [-1] * (block - ne)
        seq += em
        ctx, nn, anchor, off = oracle.advance(ctx, nn, anchor, res["emitted"], ne, off, block)
        assert anchor == seq[-1] and nn == ne
        steps += 1
    n = min(len(seq), len(plain))
    assert seq[:n] == plain[:n]
    assert steps < len(plain) - len(prompt)      # wider than one token per step on average


def test_block_width_rule_page_points():
    """[LUCE] long-context commits: past the threshold (default 8192 after the first
    cut's 32768) a block-16 drafter narrows to 8; below it nothing changes; the rule
    reads the context length only; 0 disables it.  The page's measured prompts:
    6,208 keeps the wide block, 13,148 / 26,728 / 39,861 / 81,365 narrow."""
    bw = oracle.block_width
    assert bw(6_208, 16, 16) == 16
    for ctx in (13_148, 26_728, 39_861, 81_365):
        assert bw(ctx, 16, 16) == 8
    assert bw(39_861, 16, 16, ctx_threshold=32_768) == 8 and bw(26_728, 16, 16, ctx_threshold=32_768) == 16
    assert bw(81_365, 16, 16, ctx_threshold=0) == 16
    # the boundary (reading: strictly past the threshold; the context is ctx_len + n_new)
    assert bw(8_192 - 16, 16, 16) == 16 and bw(8_192 - 15, 16, 16) == 8
    assert bw(8_000, 0, 8) == 8                  # a block-8 drafter has nothing to narrow


def test_advance_block16():
    """The serving-loop update with blocks of 16: up to 16 emitted tokens become the next
    step's new rows."""
    em = list(range(200, 216))
    assert oracle.advance(1000, 16, 3, em, 16, 0, 16) == (1016, 16, 215, 1)
    assert oracle.advance(1016, 16, 215, em[:11] + [-1] * 5, 11, 1, 16) == (1032, 11, 210, 2)
    assert oracle.advance(1032, 11, 210, [-1] * 16, 0, 2, 16) == (1043, 0, 210, 3)


def test_ddtree_verify_block16_depth():
    """A chain tree as deep as a block of 16 allows (15 nodes) accepted end to end emits
    16 tokens."""
    V = 50
    tok = np.arange(1, 16, dtype=np.int32)
    par = np.arange(-1, 14, dtype=np.int32)
    z = np.zeros((16, V))
    for j in range(15):
        z[j, tok[j]] = 1.0
    z[15, 42] = 1.0
    res = oracle.ddtree_verify(z, tok, par, block=16)
    assert res["n_accepted"] == 15 and res["n_emitted"] == 16
    assert list(res["emitted"]) == list(range(1, 16)) + [42]
