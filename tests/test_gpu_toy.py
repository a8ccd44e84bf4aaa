"""GPU parity of the CUDA path against the oracle on the toy workload (1 layer,
width 512, vocab 8192) and on small multi-request variants, through the C ABI."""
import dataclasses

import numpy as np
import pytest
import torch

import block_drafter_pos_gb300 as bd
import oracle
import workloads as wk
from oracle import philox

from gpu_common import (BF16_NAN, GpuStep, certified_topk, compare_verify, compare_walk, i16, lattice_error_bounds,
                        new_caches, oracle_draft, rel_l2, topk_of, verify_decided)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    bd.build()
    assert torch.cuda.is_available()


def _draft_case(wl, fmt_override=None):
    if fmt_override:
        wl = dataclasses.replace(wl, weight_format=fmt_override)
    W = wk.make_weights(wl.geom, wl.weight_format, wl.seed)
    inp = wk.make_request_inputs(wl)
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    kct, vct = i16(kc), i16(vc)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    step.draft(t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"]), t(inp["taps"]), kct, vct)
    torch.cuda.synchronize()
    return wl, W, inp, kc, vc, step, kct, vct


@pytest.mark.parametrize("fmt", ["bf16", "q8"])
def test_draft_block_toy_matches_oracle(fmt):
    wl, W, inp, kc, vc, step, kct, vct = _draft_case(wk.workload(1), fmt)
    logits = step.logits.cpu().numpy()
    gate = step.gate.cpu().numpy()
    ids = step.cand_ids.cpu().numpy()
    cl = step.cand_logits.cpu().numpy()
    kc_gpu = kct.cpu().numpy().view(np.uint16)
    vc_gpu = vct.cpu().numpy().view(np.uint16)
    near = 0
    for r in range(wl.n_req):
        tr = oracle_draft(wl, W, inp, kc, vc, r)
        assert np.all(np.isfinite(logits[r]))
        assert rel_l2(logits[r], tr["logits"]) < 2e-2
        assert rel_l2(gate[r], tr["gate"]) < 2e-2
        # appended context rows (k after k_norm + RoPE, v), BF16 in the cache
        ctx, nn = int(inp["ctx_len"][r]), int(inp["n_new"][r])
        for l in range(wl.geom.n_layers):
            kg = oracle.bf16_to_f64(kc_gpu[l, r, ctx:ctx + nn])
            ko = oracle.bf16_to_f64(tr["k_cache"][l][ctx:ctx + nn])
            assert rel_l2(kg, ko) < 2e-2
            vg = oracle.bf16_to_f64(vc_gpu[l, r, ctx:ctx + nn])
            vo = oracle.bf16_to_f64(tr["v_cache"][l][ctx:ctx + nn])
            assert rel_l2(vg, vo) < 2e-2
            # rows outside the append range are untouched
            assert np.array_equal(kc_gpu[l, r, :ctx], kc[l, r, :ctx])
            assert np.array_equal(kc_gpu[l, r, ctx + nn:], kc[l, r, ctx + nn:])
        for i in range(7):
            # the kernel's top-16 is exactly the policy's top-16 of its own logits
            assert np.array_equal(ids[r, i], topk_of(logits[r, i]))
            assert np.array_equal(cl[r, i], logits[r, i][ids[r, i]])
            err = float(np.max(np.abs(logits[r, i] - tr["logits"][i])))
            near += certified_topk(ids[r, i], tr["logits"][i], err)
    assert near < 7 * 16 // 2          # most ranks are decided exactly


def test_draft_block_deterministic():
    wl = wk.workload(1)
    outs = []
    for _ in range(2):
        _, _, _, _, _, step, kct, _ = _draft_case(wl)
        outs.append((step.logits.cpu().numpy().copy(), step.gate.cpu().numpy().copy(), kct.cpu().numpy().copy()))
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b)


def test_draft_block_multi_request_ragged():
    """4 requests with different cache lengths (one beyond the window) and n_new 0..8."""
    g = dataclasses.replace(wk.TOY, window=256)
    wl = wk.Workload("toy_r4", g, "bf16", 4, [40, 300, 700, 20], [0.0, 0.7, 1.0, 0.0], [0.5] * 4, seed=11)
    W = wk.make_weights(g, "bf16", wl.seed)
    inp = wk.make_request_inputs(wl)
    inp["n_new"] = np.array([8, 3, 0, 5], np.int32)
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    kct, vct = i16(kc), i16(vc)
    step.draft(t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"]), t(inp["taps"]), kct, vct)
    torch.cuda.synchronize()
    logits = step.logits.cpu().numpy()
    for r in range(4):
        tr = oracle_draft(wl, W, inp, kc, vc, r)
        assert rel_l2(logits[r], tr["logits"]) < 2e-2, r


def test_draft_block_gqa_two_layers_full_window():
    """2 layers, 8 query / 2 KV heads (GQA group mapping), the 2048-key window at its
    full size (one request past it), 2 requests."""
    g = dataclasses.replace(wk.TOY, hidden=1024, n_layers=2, n_q_heads=8, n_kv_heads=2, ffn=2048, vocab=16384)
    wl = wk.Workload("mid_r2", g, "bf16", 2, [300, 2600], [0.0, 0.0], [0.5] * 2, seed=12)
    W = wk.make_weights(g, "bf16", wl.seed)
    inp = wk.make_request_inputs(wl)
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    step.draft(t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"]), t(inp["taps"]), i16(kc), i16(vc))
    torch.cuda.synchronize()
    logits = step.logits.cpu().numpy()
    gate = step.gate.cpu().numpy()
    for r in range(2):
        tr = oracle_draft(wl, W, inp, kc, vc, r)
        assert rel_l2(logits[r], tr["logits"]) < 1e-3, r
        assert rel_l2(gate[r], tr["gate"]) < 1e-3, r


def _select_case(V, R, seed, integer, temps):
    si = wk.make_selector_inputs(V, R, seed, integer=integer)
    g = dataclasses.replace(wk.TOY, vocab=V)
    W = wk.make_weights(g, "bf16", 5)
    if integer:
        rng = np.random.default_rng(seed)
        for n in ("cb_a", "cb_b"):
            W[n] = {"kind": "bf16", "w": wk.bf16_bits_from_f32(rng.integers(-2, 3, (V, 256)).astype(np.float32))}
    wl = wk.Workload("sel", g, "bf16", R, [64] * R, list(temps), [1.0] * R, seed=seed)
    return si, W, wl


@pytest.mark.parametrize("integer", [True, False])
def test_select_matches_oracle(integer):
    """The selector kernel against the oracle's walk fed the same candidates, logits and
    gate, over 50 seeds x 4 requests (greedy, greedy, T 0.7, T 1.0): every lattice score
    within the LSE page's mixed rounding bound (exact for integer inputs), the path
    bit-exact wherever the decision lies outside that rounding (counted otherwise:
    at most 2% of the requests), q rows at rel-L2 <= 1e-4."""
    R, V = 4, 8192
    temps = [float(np.float32(x)) for x in (0.0, 0.0, 0.7, 1.0)]  # the kernel's FP32 temperatures
    si, W, wl = _select_case(V, R, 3, integer, temps)
    step = GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    u = 2.0 ** -24
    gam = 258 * u / (1 - 258 * u)
    A = oracle.bf16_to_f64(W["cb_a"]["w"])
    B = oracle.bf16_to_f64(W["cb_b"]["w"])
    undecided = compared = 0
    q_pairs = []
    for trial in range(50):
        si = wk.make_selector_inputs(V, R, 1000 + trial, integer=integer)
        seeds = np.array([42 + trial, 43, 44 + 7 * trial, 45], np.uint64)
        offs = np.array([trial, 1 << 32, (2 << 32) + trial, 3 << 32], np.uint64)
        step.select(t(si["anchors"]), t(np.array(temps, np.float32)), t(seeds.view(np.int64)),
                    t(offs.view(np.int64)), t(si["cand_ids"]), t(si["cand_logits"]), t(si["gate"]))
        torch.cuda.synchronize()
        path = step.path.cpu().numpy()
        q = step.q_rows.cpu().numpy()
        scores = step.scores.cpu().numpy()
        st = step.status.cpu().numpy()
        for r in range(R):
            res = oracle.walk(wl.geom, W["cb_a"], W["cb_b"], int(si["anchors"][r]), si["cand_ids"][r],
                              si["cand_logits"][r].astype(np.float64), si["gate"][r].astype(np.float64), temps[r],
                              int(seeds[r]), int(offs[r]))
            assert st[r] == 0
            bounds = lattice_error_bounds(W, int(si["anchors"][r]), si["cand_ids"][r],
                                          si["gate"][r].astype(np.float64), res["scores"], False)
            if trial < 5:  # every lattice score within the page's mixed rounding bound
                for i in range(7):
                    preds = [si["anchors"][r]] * 16 if i == 0 else si["cand_ids"][r, i - 1]
                    for p in range(16):
                        absprod = np.abs(A[preds[p]][None, :] * si["gate"][r, i][None, :]
                                         * B[si["cand_ids"][r, i]]).sum(1)
                        bound = gam * absprod + 2 * u / (1 - u) * np.abs(res["scores"][i, p])
                        assert np.all(np.abs(scores[r, i, p] - res["scores"][i, p]) <= bound)
            if integer:
                assert np.array_equal(scores[r], res["scores"].astype(np.float32))
            n_cmp, und, qs = compare_walk(res, path[r], q[r], bounds, temps[r], si["cand_ids"][r], exact=integer)
            undecided += und
            compared += not und
            q_pairs += qs
    print(f"select: {compared} requests compared in full, {undecided} stopped at an undecided step")
    assert undecided <= 4 and compared >= 196
    qg, qo = np.array([a for a, _ in q_pairs]), np.array([b for _, b in q_pairs])
    assert rel_l2(qg, qo) <= 1e-4


def test_select_rejects_nonfinite():
    R, V = 2, 8192
    si, W, wl = _select_case(V, R, 4, False, [0.0, 1.0])
    si["cand_logits"][1, 3, 5] = np.nan
    step = GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    seeds = np.zeros(2, np.int64)
    step.select(t(si["anchors"]), t(np.array([0.0, 1.0], np.float32)), t(seeds), t(seeds), t(si["cand_ids"]),
                t(si["cand_logits"]), t(si["gate"]))
    torch.cuda.synchronize()
    st = step.status.cpu().numpy()
    assert st[0] == 0 and st[1] == bd.binding.E_NONFINITE
    assert np.all(step.path.cpu().numpy()[1] == -1)


@pytest.mark.parametrize("integer", [True, False])
def test_verify_matches_oracle(integer):
    """The verify kernel against the oracle fed the same target rows, path, candidates and
    q rows, over 50 seeds x 4 requests with varied acceptance depths: n_accepted, emitted
    and n_emitted bit-exact wherever every sampled decision lies outside the kernel's
    FP32 rounding (counted otherwise: at most 2% of the requests), the verify
    probabilities (p at each proposal, the residual mass, the bonus p) at rel-L2 <= 1e-4."""
    R, V = 4, 8192
    temps = [float(np.float32(x)) for x in ((0.0, 0.0, 0.7, 1.0) if not integer else (0.0,) * 4)]
    g = dataclasses.replace(wk.TOY, vocab=V)
    W = wk.make_weights(g, "bf16", 5)
    wl = wk.Workload("ver", g, "bf16", R, [64] * R, temps, [1.0] * R, seed=9)
    step = GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    undecided = compared = 0
    pairs = []
    for trial in range(50):
        depth = [trial % 8, (trial + 3) % 8, (trial * 5) % 8, (trial * 3 + 1) % 8]
        vi = wk.make_verify_inputs(V, R, 100 + trial, temps, integer=integer, accept_depth=depth)
        seeds = np.array([7 + trial, 8, 9 + 3 * trial, 10], np.uint64)
        offs = np.array([5, 6 + trial, 7, (8 << 32) + trial], np.uint64)
        step.status.zero_()
        step.verify(t(vi["target"]), t(vi["temps"]), t(seeds.view(np.int64)), t(offs.view(np.int64)),
                    t(vi["path"]), t(vi["cand_ids"]), t(vi["q_rows"]))
        torch.cuda.synchronize()
        na = step.n_acc.cpu().numpy()
        em = step.emitted.cpu().numpy()
        ne = step.n_emit.cpu().numpy()
        probs = step.probs.cpu().numpy()
        for r in range(R):
            res = oracle.verify(vi["target"][r].astype(np.float64), vi["path"][r], vi["cand_ids"][r],
                                vi["q_rows"][r].astype(np.float64), temps[r], int(seeds[r]), int(offs[r]))
            if temps[r] == 0.0 or verify_decided(res):
                pairs += compare_verify(res, na[r], em[r], ne[r], probs[r], temps[r])
                compared += 1
            else:
                undecided += 1
    print(f"verify: {compared} requests compared, {undecided} with an undecided sampled decision")
    assert undecided <= 4 and compared >= 196
    if pairs:
        pg, po = np.array([a for a, _ in pairs], np.float64), np.array([b for _, b in pairs])
        assert rel_l2(pg, po) <= 1e-4, rel_l2(pg, po)


def test_verify_nonfinite_and_skip():
    R, V = 3, 8192
    vi = wk.make_verify_inputs(V, R, 10, [1.0, 0.0, 1.0])
    vi["target"][0, 4, 100] = np.nan
    g = dataclasses.replace(wk.TOY, vocab=V)
    wl = wk.Workload("ver", g, "bf16", R, [64] * R, [1.0, 0.0, 1.0], [1.0] * R, seed=9)
    step = GpuStep(wl, wk.make_weights(g, "bf16", 5))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    step.status.copy_(torch.tensor([0, 0, 2], dtype=torch.int32))
    z = np.zeros(R, np.int64)
    step.verify(t(vi["target"]), t(vi["temps"]), t(z), t(z), t(vi["path"]), t(vi["cand_ids"]), t(vi["q_rows"]))
    torch.cuda.synchronize()
    st = step.status.cpu().numpy()
    ne = step.n_emit.cpu().numpy()
    assert st[0] == bd.binding.E_NONFINITE and ne[0] == 0
    assert st[1] == 0 and ne[1] >= 1
    assert st[2] == 2 and ne[2] == 0


def test_pipeline_error_reported_by_select_and_skipped_by_verify():
    """The device error path, driven from the host (no kernel waits out its limit): the
    handle's pipeline error word is set after a draft, as a bounded weight-pipeline wait
    that gave up would set it.  The selector then reports DFLASH2_E_CUDA for every
    request (path -1, q rows 0) and verify emits nothing for them; the next draft
    clears the word and the step is healthy again."""
    R = 3
    g = dataclasses.replace(wk.TOY, window=256)
    wl = wk.Workload("toy_err", g, "bf16", R, [64, 100, 200], [0.0, 0.7, 1.0], [0.5] * R, seed=23)
    W = wk.make_weights(g, "bf16", wl.seed)
    inp = wk.make_request_inputs(wl)
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    temps = t(np.array(wl.temps, np.float32))
    z = t(np.zeros(R, np.int64))
    target = torch.zeros((R, 8, g.vocab), dtype=torch.float32, device="cuda")
    for inject in (True, False):
        step.draft(t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"]), t(inp["taps"]), i16(kc), i16(vc))
        if inject:
            bd.dflash2_debug_set_pipeline_error(step.drafter.handle)
        step.status.fill_(-7)
        step.select(t(inp["anchors"]), temps, z, z)
        target[:, :7] = step.logits
        target[:, 7] = step.logits[:, 6]
        step.verify(target, temps, z, z)
        torch.cuda.synchronize()
        st = step.status.cpu().numpy()
        ne = step.n_emit.cpu().numpy()
        if inject:
            assert np.all(st == bd.binding.E_CUDA), st
            assert np.all(step.path.cpu().numpy() == -1)
            assert np.all(step.q_rows.cpu().numpy() == 0)
            assert np.all(ne == 0) and np.all(step.n_acc.cpu().numpy() == 0)
            assert np.all(step.emitted.cpu().numpy() == -1)
        else:
            assert np.all(st == 0), st
            assert np.all(ne >= 1)


def test_head_topk_exact_integer_logits_with_ties_nan_inf():
    """Integer weights and hidden states make every logit exact in FP32, so the top-16
    (ties, NaN, +/-inf policy) must equal the oracle's bit for bit."""
    V = 8192
    g = dataclasses.replace(wk.TOY, vocab=V)
    W = wk.make_weights(g, "bf16", 6)
    rng = np.random.default_rng(6)
    lm = rng.integers(-3, 4, (V, g.hidden)).astype(np.float32)
    lm_bits = wk.bf16_bits_from_f32(lm)
    lm_bits[[17, 4000, 4097]] = 0x7FC0                      # NaN rows -> NaN logits
    lm_bits[[513, 2000], 0] = 0x7F80                        # +inf logits (x[:, 0] = 1)
    lm_bits[700, 0] = 0xFF80                                # -inf logit
    W["lm_head"] = lm_bits
    wl = wk.Workload("head", g, "bf16", 1, [64], [0.0], [1.0], seed=6)
    step = GpuStep(wl, W)
    x = rng.integers(-1, 2, (8, g.hidden)).astype(np.float32)
    x[:, 0] = 1.0
    xb = wk.bf16_bits_from_f32(x)
    ids = torch.zeros((1, 7, 16), dtype=torch.int32, device="cuda")
    vals = torch.zeros((1, 7, 16), dtype=torch.float32, device="cuda")
    logits = torch.zeros((1, 7, V), dtype=torch.float32, device="cuda")
    bd.dflash2_head_topk(step.drafter.handle, 8, i16(xb), ids, vals, logits)
    torch.cuda.synchronize()
    Wf = oracle.bf16_to_f64(lm_bits)
    for i in range(1, 8):
        with np.errstate(invalid="ignore"):
            ref = (Wf * x[i][None, :].astype(np.float64)).sum(1)
        rid, rv = oracle.topk(ref, 16)
        got = ids.cpu().numpy()[0, i - 1]
        assert np.array_equal(got, rid), (i, got, rid)
        lg = logits.cpu().numpy()[0, i - 1]
        fin = np.isfinite(ref)
        assert np.array_equal(lg[fin], ref[fin].astype(np.float32))


@pytest.mark.parametrize("integer", [True, False])
def test_select_viterbi_mode_matches_oracle(integer):
    """Selector mode 1: greedy requests take the globally best path.  The oracle's
    dynamic program on the GPU's own lattice (float32 sums in the kernel's order)
    gives the same path exactly; its total is never below the sequential walk's;
    requests with T > 0 still walk and sample."""
    R, V = 4, 8192
    temps = [0.0, 0.0, 0.7, 0.0]
    si, W, wl = _select_case(V, R, 21, integer, temps)
    step = GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    seeds = np.array([42, 43, 44, 45], np.uint64)
    offs = np.array([0, 1 << 32, 2 << 32, 3 << 32], np.uint64)
    args = (t(si["anchors"]), t(np.array(temps, np.float32)), t(seeds.view(np.int64)), t(offs.view(np.int64)),
            t(si["cand_ids"]), t(si["cand_logits"]), t(si["gate"]))
    step.select(*args)
    torch.cuda.synchronize()
    walk_path = step.path.cpu().numpy().copy()
    bd.dflash2_set_select_mode(step.drafter.handle, 1)
    step.select(*args)
    torch.cuda.synchronize()
    bd.dflash2_set_select_mode(step.drafter.handle, 0)
    path, q = step.path.cpu().numpy(), step.q_rows.cpu().numpy()
    scores = step.scores.cpu().numpy()
    st = step.status.cpu().numpy()
    for r in range(R):
        assert st[r] == 0
        if temps[r] == 0.0:
            ref = oracle.viterbi_path(scores[r], si["cand_ids"][r])
            assert np.array_equal(path[r], ref["path"]), r
            assert np.array_equal(q[r], ref["q_rows"].astype(np.float32))
            idx_w = [int(np.nonzero(si["cand_ids"][r, i] == walk_path[r, i])[0][0]) for i in range(7)]
            s32 = scores[r].astype(np.float32)
            tot_w = s32[0, 0, idx_w[0]] + sum(s32[i, idx_w[i - 1], idx_w[i]] for i in range(1, 7))
            assert ref["total"] >= tot_w - 1e-4 * max(1.0, abs(float(tot_w)))
        else:
            assert np.array_equal(path[r], walk_path[r])  # sampled requests are unaffected by the mode


@pytest.mark.parametrize("fmt,R", [("bf16", 3), ("q8", 5)])
def test_draft_block_empty_context(fmt, R):
    """Degenerate contexts: nothing in the cache and no new rows (the block attends to
    its own 8 keys only), or only this call's new rows; every other cache row holds the
    NaN sentinel.  GEMV path (3 bf16 requests) and tensor-core path (5 Q8 requests)."""
    g = dataclasses.replace(wk.TOY, window=256)
    wl = wk.Workload("toy_empty_ctx", g, fmt, R, [8] * R, [0.0] * R, [0.5] * R, seed=17)
    W = wk.make_weights(g, fmt, wl.seed)
    inp = wk.make_request_inputs(wl)
    inp["n_new"] = np.array([0, 5, 8, 0, 1][:R], np.int32)  # ctx_len is 0 for every request
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    kct, vct = i16(kc), i16(vc)
    step.draft(t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"]), t(inp["taps"]), kct, vct)
    torch.cuda.synchronize()
    logits = step.logits.cpu().numpy()
    kc_gpu = kct.cpu().numpy().view(np.uint16)
    assert np.isfinite(logits).all()
    for r in range(R):
        tr = oracle_draft(wl, W, inp, kc, vc, r)
        assert rel_l2(logits[r], tr["logits"]) < 2e-2, r
        nn = int(inp["n_new"][r])
        for l in range(g.n_layers):
            if nn:
                assert rel_l2(oracle.bf16_to_f64(kc_gpu[l, r, :nn]), oracle.bf16_to_f64(tr["k_cache"][l][:nn])) < 2e-2
            assert np.array_equal(kc_gpu[l, r, nn:], kc[l, r, nn:])  # nothing written past the new rows


def test_draft_block_fills_the_cache_to_capacity():
    """The new rows end exactly at the cache's capacity (request 0: 256 keys after the
    append in a 256-row cache, beyond the 256-key window) next to a shorter request."""
    g = dataclasses.replace(wk.TOY, window=256)
    wl = wk.Workload("toy_full_cache", g, "bf16", 2, [256, 100], [0.0, 0.0], [0.5] * 2, seed=19, steps=0)
    assert wl.kv_capacity == 256
    W = wk.make_weights(g, "bf16", wl.seed)
    inp = wk.make_request_inputs(wl)
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    kct, vct = i16(kc), i16(vc)
    step.draft(t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"]), t(inp["taps"]), kct, vct)
    torch.cuda.synchronize()
    logits = step.logits.cpu().numpy()
    kc_gpu, vc_gpu = kct.cpu().numpy().view(np.uint16), vct.cpu().numpy().view(np.uint16)
    for r in range(2):
        tr = oracle_draft(wl, W, inp, kc, vc, r)
        assert rel_l2(logits[r], tr["logits"]) < 2e-2, r
        ctx, nn = int(inp["ctx_len"][r]), int(inp["n_new"][r])
        for l in range(g.n_layers):
            assert rel_l2(oracle.bf16_to_f64(vc_gpu[l, r, ctx:ctx + nn]),
                          oracle.bf16_to_f64(tr["v_cache"][l][ctx:ctx + nn])) < 2e-2, r
            assert np.array_equal(kc_gpu[l, r, :ctx], kc[l, r, :ctx])
            assert np.array_equal(kc_gpu[l, r, ctx + nn:], kc[l, r, ctx + nn:])
