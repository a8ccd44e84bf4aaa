"""GPU parity of blocks of 16 positions and of the long-context narrowing against the
oracle, through the C ABI ("qwen35: DSpark speculative decoding (Qwen3.8-27B drafters)
- #625": the greedy-width commit's block 16, the long-context commits' narrowing of
the block past a context threshold).

A request narrowed to width w inside a block-16 handle is compared with the oracle's
block of w positions of the same drafter (its first w rows; the rest is padding)."""
import dataclasses

import numpy as np
import pytest
import torch

import block_drafter_pos_gb300 as bd
import oracle
import workloads as wk

from gpu_common import (GpuStep, certified_topk, compare_verify, compare_walk, i16, lattice_error_bounds, new_caches,
                        rel_l2, topk_of, verify_decided)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    bd.build()
    assert torch.cuda.is_available()


def t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _oracle_draft(wl, W, inp, kc, vc, r, width):
    """The oracle's draft of request r as a block of `width` positions (caches copied)."""
    g = dataclasses.replace(wl.geom, block=width)
    kl = [kc[l, r].copy() for l in range(g.n_layers)]
    vl = [vc[l, r].copy() for l in range(g.n_layers)]
    nn = int(inp["n_new"][r])
    tr = oracle.draft_block(g, W, int(inp["anchors"][r]), int(inp["ctx_len"][r]), nn, inp["taps"][r][:nn], kl, vl)
    tr["k_cache"], tr["v_cache"] = kl, vl
    return tr


def _case(fmt, R, ctx, n_new, width, window=2048, seed=31):
    g = dataclasses.replace(wk.TOY, block=16, window=window)
    wl = wk.Workload("toy_b16", g, fmt, R, ctx, [0.0] * R, [0.5] * R, seed=seed)
    W = wk.make_weights(g, fmt, wl.seed)
    inp = wk.make_request_inputs(wl)
    inp["n_new"] = np.array(n_new, np.int32)
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    if width is not None:
        step.width = t(np.array(width, np.int32))
    kct, vct = i16(kc), i16(vc)
    step.draft(t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"]), t(inp["taps"]), kct, vct)
    torch.cuda.synchronize()
    return wl, W, inp, kc, vc, step, kct, vct


@pytest.mark.parametrize("fmt,R", [("bf16", 2), ("bf16", 3), ("q8", 1), ("q8", 2)])
def test_draft_block16_matches_oracle(fmt, R):
    """Blocks of 16 (two 8-row tiles per request: the convolutions cross the tile
    boundary inside a block), ragged n_new and cache lengths, one request past the
    window; the GEMV path (bf16 up to 32 rows, Q8 below 32) and the tensor-core GEMM
    (bf16 48 rows, Q8 32 rows): logits and gate at rel-L2 < 2e-2 (the toy tolerance
    of blocks of 8), the appended cache rows, and the kernel's top-16 exactly the
    policy's top-16 of its own logits, rank by rank against the oracle outside
    near-ties."""
    wl, W, inp, kc, vc, step, kct, vct = _case(fmt, R, [300, 700, 90][:R], [16, 5, 11][:R], None, window=512)
    logits, gate = step.logits.cpu().numpy(), step.gate.cpu().numpy()
    ids, cl = step.cand_ids.cpu().numpy(), step.cand_logits.cpu().numpy()
    kc_gpu, vc_gpu = kct.cpu().numpy().view(np.uint16), vct.cpu().numpy().view(np.uint16)
    near = 0
    for r in range(R):
        tr = _oracle_draft(wl, W, inp, kc, vc, r, 16)
        assert logits[r].shape == tr["logits"].shape == (15, wl.geom.vocab)
        assert rel_l2(logits[r], tr["logits"]) < 2e-2, r
        assert rel_l2(gate[r], tr["gate"]) < 2e-2, r
        ctx, nn = int(inp["ctx_len"][r]), int(inp["n_new"][r])
        for l in range(wl.geom.n_layers):
            assert rel_l2(oracle.bf16_to_f64(kc_gpu[l, r, ctx:ctx + nn]),
                          oracle.bf16_to_f64(tr["k_cache"][l][ctx:ctx + nn])) < 2e-2
            assert np.array_equal(kc_gpu[l, r, ctx + nn:], kc[l, r, ctx + nn:])
        for i in range(15):
            assert np.array_equal(ids[r, i], topk_of(logits[r, i]))
            assert np.array_equal(cl[r, i], logits[r, i][ids[r, i]])
            err = float(np.max(np.abs(logits[r, i] - tr["logits"][i])))
            near += certified_topk(ids[r, i], tr["logits"][i], err)
    if R * 16 < (40 if fmt == "bf16" else 32):
        # the GEMV path: most ranks decided exactly (the tensor-core GEMM reads one
        # 16-bit activation plane, ~2^-9 relative: its near-ties are many more)
        assert near < R * 15 * 16 // 2


def test_draft_block16_gqa_two_layers_tight():
    """2 layers, 8 query / 2 KV heads, blocks of 16, 2 requests (one past the 2048-key
    window): the tighter tolerance of the mid-size blocks-of-8 case."""
    g = dataclasses.replace(wk.TOY, hidden=1024, n_layers=2, n_q_heads=8, n_kv_heads=2, ffn=2048, vocab=16384,
                            block=16)
    wl = wk.Workload("mid_b16", g, "bf16", 2, [300, 2600], [0.0, 0.0], [0.5] * 2, seed=12)
    W = wk.make_weights(g, "bf16", wl.seed)
    inp = wk.make_request_inputs(wl)
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    step.draft(t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"]), t(inp["taps"]), i16(kc), i16(vc))
    torch.cuda.synchronize()
    logits, gate = step.logits.cpu().numpy(), step.gate.cpu().numpy()
    for r in range(2):
        tr = _oracle_draft(wl, W, inp, kc, vc, r, 16)
        assert rel_l2(logits[r], tr["logits"]) < 1e-3, r
        assert rel_l2(gate[r], tr["gate"]) < 1e-3, r


@pytest.mark.parametrize("widths,tol", [([16, 5], 1e-3), ([16, 8, 2], 2e-2)])
def test_narrowed_request_is_a_block_of_its_width(widths, tol):
    """Requests of different widths in one block-16 call: each request's first w rows
    equal the oracle's block of w positions (its later rows are unspecified).  Two
    requests run on the GEMV path (the tight tolerance of the mid-size case), three
    (48 rows) on the tensor-core GEMM (its one-plane tolerance)."""
    g = dataclasses.replace(wk.TOY, hidden=1024, n_layers=2, n_q_heads=8, n_kv_heads=2, ffn=2048, vocab=16384,
                            block=16)
    R = len(widths)
    wl = wk.Workload("mid_narrow", g, "bf16", R, [300, 500, 900][:R], [0.0] * R, [0.5] * R, seed=13)
    W = wk.make_weights(g, "bf16", wl.seed)
    inp = wk.make_request_inputs(wl)
    inp["n_new"] = np.array([16, 4, 2][:R], np.int32)
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    step.width = t(np.array(widths, np.int32))
    kct = i16(kc)
    step.draft(t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"]), t(inp["taps"]), kct, i16(vc))
    torch.cuda.synchronize()
    logits, gate = step.logits.cpu().numpy(), step.gate.cpu().numpy()
    kc_gpu = kct.cpu().numpy().view(np.uint16)
    for r, w in enumerate(widths):
        tr = _oracle_draft(wl, W, inp, kc, vc, r, w)
        assert rel_l2(logits[r, :w - 1], tr["logits"]) < tol, r
        assert rel_l2(gate[r, :w - 1], tr["gate"]) < tol, r
        ctx, nn = int(inp["ctx_len"][r]), int(inp["n_new"][r])
        assert rel_l2(oracle.bf16_to_f64(kc_gpu[0, r, ctx:ctx + nn]),
                      oracle.bf16_to_f64(tr["k_cache"][0][ctx:ctx + nn])) < max(tol, 1e-2)


def test_block16_tensor_core_and_gemv_paths_agree():
    """One block-16 handle for 3 requests (48 rows: tensor-core GEMM): a 2-request call
    (32 rows, GEMV path) and the 3-request call agree on the first two requests up to
    the paths' rounding, and the GEMV call matches the oracle tightly, so the GEMM
    path's larger deviation from the oracle is its one-plane rounding, not the block."""
    g = dataclasses.replace(wk.TOY, hidden=1024, n_layers=2, n_q_heads=8, n_kv_heads=2, ffn=2048, vocab=16384,
                            block=16)
    wl = wk.Workload("mid_paths", g, "bf16", 3, [300, 500, 900], [0.0] * 3, [0.5] * 3, seed=14)
    W = wk.make_weights(g, "bf16", wl.seed)
    inp = wk.make_request_inputs(wl)
    kc, vc = new_caches(wl, inp)
    s3 = GpuStep(wl, W)
    s3.draft(t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"]), t(inp["taps"]), i16(kc), i16(vc))
    ids = torch.zeros((2, 15, 16), dtype=torch.int32, device="cuda")
    vals = torch.zeros((2, 15, 16), dtype=torch.float32, device="cuda")
    gate = torch.zeros((2, 15, g.rank), dtype=torch.float32, device="cuda")
    logits = torch.zeros((2, 15, g.vocab), dtype=torch.float32, device="cuda")
    bd.dflash2_draft_block(s3.drafter.handle, 2, t(inp["anchors"][:2]), t(inp["ctx_len"][:2]), t(inp["n_new"][:2]),
                           t(inp["taps"][:2]), i16(kc), i16(vc), ids, vals, gate, logits)
    torch.cuda.synchronize()
    l2, l3 = logits.cpu().numpy(), s3.logits.cpu().numpy()[:2]
    assert rel_l2(l3, l2) < 2e-2
    for r in range(2):
        tr = _oracle_draft(wl, W, inp, kc, vc, r, 16)
        assert rel_l2(l2[r], tr["logits"]) < 1e-3, r
        # the GEMM path's deviation is of the one-plane size at every block position,
        # the positions past the first tile (8..15) included
        e3 = [rel_l2(l3[r, i], tr["logits"][i]) for i in range(15)]
        assert max(e3) < 2e-2 and max(e3[7:]) < 3 * max(e3[:7]), e3


def test_block_width_matches_oracle():
    """dflash2_block_width against the oracle's rule on lengths around the threshold,
    the page's default (8192, narrowing to 8), another threshold and 0 (disabled)."""
    g = dataclasses.replace(wk.TOY, block=16)
    wl = wk.Workload("bw", g, "bf16", 8, [64] * 8, [0.0] * 8, [1.0] * 8, seed=3)
    step = GpuStep(wl, wk.make_weights(g, "bf16", 3))
    h = step.drafter.handle
    rng = np.random.default_rng(4)
    for thr, narrow in ((8192, 8), (32768, 8), (0, 8), (4000, 2), (100, 16)):
        for trial in range(3):
            ctx = rng.integers(thr - 20 if thr else 0, thr + 20 if thr else 100_000, size=8).astype(np.int32)
            ctx = np.maximum(ctx, 0)
            nn = rng.integers(0, 17, size=8).astype(np.int32)
            out = torch.full((8,), -1, dtype=torch.int32, device="cuda")
            bd.dflash2_block_width(h, 8, t(ctx), t(nn), thr, narrow, out)
            torch.cuda.synchronize()
            want = [oracle.block_width(int(c), int(n), 16, thr, narrow) for c, n in zip(ctx, nn)]
            assert out.cpu().numpy().tolist() == want
    out = torch.zeros((8,), dtype=torch.int32, device="cuda")
    z = t(np.zeros(8, np.int32))
    for bad in ((8192, 1), (8192, 17), (-1, 8)):
        with pytest.raises(bd.Dflash2Error):
            bd.dflash2_block_width(h, 8, z, z, bad[0], bad[1], out)


def test_select_block16_and_narrowed_matches_oracle():
    """The selector at blocks of 16 against the oracle's walk fed the same candidates,
    logits and gate (15 positions, or the first w - 1 for a narrowed request): path and
    q rows wherever every decision lies outside the FP32 rounding (counted otherwise);
    positions past the width hold path -1 and q 0."""
    R, V = 4, 8192
    temps = [float(np.float32(x)) for x in (0.0, 0.0, 0.7, 1.0)]
    g = dataclasses.replace(wk.TOY, vocab=V, block=16)
    W = wk.make_weights(g, "bf16", 5)
    wl = wk.Workload("sel16", g, "bf16", R, [64] * R, temps, [1.0] * R, seed=3)
    step = GpuStep(wl, W)
    widths = np.array([16, 8, 16, 5], np.int32)
    step.width = t(widths)
    undecided = compared = 0
    q_pairs = []
    for trial in range(30):
        si = wk.make_selector_inputs(V, R, 2000 + trial, P=15)
        seeds = np.array([42 + trial, 43, 44 + 7 * trial, 45], np.uint64)
        offs = np.array([trial, 1 << 32, (2 << 32) + trial, 3 << 32], np.uint64)
        step.select(t(si["anchors"]), t(np.array(temps, np.float32)), t(seeds.view(np.int64)),
                    t(offs.view(np.int64)), t(si["cand_ids"]), t(si["cand_logits"]), t(si["gate"]))
        torch.cuda.synchronize()
        path, q, st = step.path.cpu().numpy(), step.q_rows.cpu().numpy(), step.status.cpu().numpy()
        for r in range(R):
            w = int(widths[r])
            P = w - 1
            res = oracle.walk(g, W["cb_a"], W["cb_b"], int(si["anchors"][r]), si["cand_ids"][r, :P],
                              si["cand_logits"][r, :P].astype(np.float64), si["gate"][r, :P].astype(np.float64),
                              temps[r], int(seeds[r]), int(offs[r]))
            assert st[r] == 0
            assert np.all(path[r, P:] == -1) and np.all(q[r, P:] == 0)
            bounds = lattice_error_bounds(W, int(si["anchors"][r]), si["cand_ids"][r, :P],
                                          si["gate"][r, :P].astype(np.float64), res["scores"], False)
            _, und, qs = compare_walk(res, path[r], q[r], bounds, temps[r], si["cand_ids"][r, :P])
            undecided += und
            compared += not und
            q_pairs += qs
    print(f"select (block 16): {compared} requests compared in full, {undecided} stopped at an undecided step")
    assert undecided <= 4 and compared >= 116
    qg, qo = np.array([a for a, _ in q_pairs]), np.array([b for _, b in q_pairs])
    assert rel_l2(qg, qo) <= 1e-4


def test_verify_block16_and_narrowed_matches_oracle():
    """The verify at blocks of 16 against the oracle on the same target rows, path,
    candidates and q rows (16 rows, or the first w for a narrowed request; NaN in the
    rows past the width must not be read), acceptance depths 0..15: outputs bit-exact
    wherever every sampled decision is decided (counted otherwise), the verify
    probabilities at rel-L2 <= 1e-4."""
    R, V = 4, 8192
    temps = [float(np.float32(x)) for x in (0.0, 0.7, 1.0, 0.0)]
    g = dataclasses.replace(wk.TOY, vocab=V, block=16)
    W = wk.make_weights(g, "bf16", 5)
    wl = wk.Workload("ver16", g, "bf16", R, [64] * R, temps, [1.0] * R, seed=9)
    step = GpuStep(wl, W)
    widths = np.array([16, 16, 8, 12], np.int32)
    step.width = t(widths)
    undecided = compared = 0
    pairs = []
    for trial in range(40):
        depth = [trial % 16, (trial * 7 + 3) % 16, (trial * 5) % 8, (trial * 3 + 1) % 12]
        vi = wk.make_verify_inputs(V, R, 300 + trial, temps, accept_depth=depth, block=16)
        for r in range(R):
            vi["target"][r, widths[r]:] = np.nan       # rows past the width are not read
        seeds = np.array([7 + trial, 8, 9 + 3 * trial, 10], np.uint64)
        offs = np.array([5, 6 + trial, 7, (8 << 32) + trial], np.uint64)
        step.status.zero_()
        step.verify(t(vi["target"]), t(vi["temps"]), t(seeds.view(np.int64)), t(offs.view(np.int64)),
                    t(vi["path"]), t(vi["cand_ids"]), t(vi["q_rows"]))
        torch.cuda.synchronize()
        na, em, ne = step.n_acc.cpu().numpy(), step.emitted.cpu().numpy(), step.n_emit.cpu().numpy()
        probs, st = step.probs.cpu().numpy(), step.status.cpu().numpy()
        for r in range(R):
            w = int(widths[r])
            assert st[r] == 0
            res = oracle.verify(vi["target"][r, :w].astype(np.float64), vi["path"][r, :w - 1],
                                vi["cand_ids"][r, :w - 1], vi["q_rows"][r, :w - 1].astype(np.float64), temps[r],
                                int(seeds[r]), int(offs[r]))
            if temps[r] == 0.0 or verify_decided(res):
                pairs += compare_verify(res, na[r], em[r], ne[r], probs[r], temps[r])
                compared += 1
            else:
                undecided += 1
    print(f"verify (block 16): {compared} requests compared, {undecided} with an undecided sampled decision")
    assert undecided <= 4 and compared >= 156
    pg, po = np.array([a for a, _ in pairs], np.float64), np.array([b for _, b in pairs])
    assert rel_l2(pg, po) <= 1e-4


def test_device_loop_block16():
    """Blocks of 16 through draft, select, verify and the device-side state update for
    several steps, greedy, with target rows that accept a chosen number k of the
    proposals (0..15; 15 = every proposal and the bonus row): verify emits path[:k] and
    the target's token at row k, and the state update matches the oracle's (context
    grows by the appended rows, the last emitted token is the next anchor, the emitted
    count the next n_new)."""
    V = 8192
    g = dataclasses.replace(wk.TOY, vocab=V, block=16)
    R = 2
    wl = wk.Workload("loop16", g, "bf16", R, [200, 300], [0.0] * R, [1.0] * R, seed=15, steps=10)
    W = wk.make_weights(g, "bf16", wl.seed)
    inp = wk.make_request_inputs(wl)
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    kct, vct = i16(kc), i16(vc)
    anchors, ctx, nn = t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"])
    taps = t(inp["taps"])
    offs = t(np.zeros(R, np.int64))
    temps = t(np.zeros(R, np.float32))
    state = [(int(inp["ctx_len"][r]), int(inp["n_new"][r]), int(inp["anchors"][r]), 0) for r in range(R)]
    rng = np.random.default_rng(5)
    for it in range(10):
        step.draft(anchors, ctx, nn, taps, kct, vct, with_logits=False)
        step.select(anchors, temps, offs, offs)
        path = step.path.cpu().numpy()
        target = rng.normal(0, 1, (R, 16, V)).astype(np.float32)
        ks = [int(rng.integers(0, 16)) if it else 15 for _ in range(R)]
        want = []
        for r in range(R):
            k = ks[r]
            for j in range(k):
                target[r, j, path[r, j]] = 20.0
            tok = int(rng.integers(V))
            if k < 15 and tok == path[r, k]:
                tok = (tok + 1) % V
            target[r, k, tok] = 20.0
            want.append(path[r, :k].tolist() + [tok])
        step.verify(t(target), temps, offs, offs)
        em, ne = step.emitted.cpu().numpy(), step.n_emit.cpu().numpy()
        for r in range(R):
            assert ne[r] == ks[r] + 1 and em[r, :ne[r]].tolist() == want[r], (it, r)
            assert np.all(em[r, ne[r]:] == -1)
        bd.dflash2_advance(step.drafter.handle, R, step.emitted, step.n_emit, anchors, ctx, nn, offs)
        torch.cuda.synchronize()
        for r in range(R):
            state[r] = oracle.advance(*state[r][:3], em[r], int(ne[r]), state[r][3], 16)
        assert ctx.cpu().numpy().tolist() == [s[0] for s in state]
        assert nn.cpu().numpy().tolist() == [s[1] for s in state]
        assert anchors.cpu().numpy().tolist() == [s[2] for s in state]
