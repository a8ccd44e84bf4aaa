"""GPU parity of the tensor-core path against the oracle: a call with many
requests runs every projection and the LM head on the tcgen05 GEMM (128-row weight
blocks, activations one 16-bit plane) and the top-16 on the chunked kernel.  Toy
width (512, vocab 8192) with 5 and 16 requests, ragged contexts and appends, both
weight formats, every request against the FP64 oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import block_drafter_pos_gb300 as bd
import oracle
import workloads as wk

from gpu_common import GpuStep, certified_topk, i16, new_caches, oracle_draft, rel_l2, topk_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    bd.build()
    assert torch.cuda.is_available()


def _wide_workload(fmt, R, window=256):
    g = dataclasses.replace(wk.TOY, window=window)
    rng = np.random.default_rng(100 + R)
    ctx = [int(x) for x in rng.integers(8, 600, size=R)]
    temps = [[0.0, 0.7, 1.0][r % 3] for r in range(R)]
    return wk.Workload(f"toy_wide_{fmt}_r{R}", g, fmt, R, ctx, temps, [0.5] * R, seed=20 + R)


def _run(wl, W, inp, step=None):
    kc, vc = new_caches(wl, inp)
    step = step or GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    kct, vct = i16(kc), i16(vc)
    step.draft(t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"]), t(inp["taps"]), kct, vct)
    torch.cuda.synchronize()
    return kc, vc, step, kct, vct


@pytest.mark.parametrize("fmt,R", [("bf16", 16), ("q8", 16), ("q8", 5), ("bf16", 7)])
def test_wide_path_matches_oracle(fmt, R):
    wl = _wide_workload(fmt, R)
    W = wk.make_weights(wl.geom, fmt, wl.seed)
    inp = wk.make_request_inputs(wl)
    inp["n_new"] = (np.arange(R) % 9).astype(np.int32)  # 0..8 new context rows, ragged
    kc, vc, step, kct, vct = _run(wl, W, inp)
    logits = step.logits.cpu().numpy()
    gate = step.gate.cpu().numpy()
    ids = step.cand_ids.cpu().numpy()
    cl = step.cand_logits.cpu().numpy()
    kc_gpu = kct.cpu().numpy().view(np.uint16)
    vc_gpu = vct.cpu().numpy().view(np.uint16)
    for r in range(R):
        tr = oracle_draft(wl, W, inp, kc, vc, r)
        assert np.all(np.isfinite(logits[r]))
        assert rel_l2(logits[r], tr["logits"]) < 2e-2, r
        assert rel_l2(gate[r], tr["gate"]) < 2e-2, r
        ctx, nn = int(inp["ctx_len"][r]), int(inp["n_new"][r])
        for l in range(wl.geom.n_layers):
            if nn:
                assert rel_l2(oracle.bf16_to_f64(kc_gpu[l, r, ctx:ctx + nn]),
                              oracle.bf16_to_f64(tr["k_cache"][l][ctx:ctx + nn])) < 2e-2, r
                assert rel_l2(oracle.bf16_to_f64(vc_gpu[l, r, ctx:ctx + nn]),
                              oracle.bf16_to_f64(tr["v_cache"][l][ctx:ctx + nn])) < 2e-2, r
            assert np.array_equal(kc_gpu[l, r, :ctx], kc[l, r, :ctx])
            assert np.array_equal(kc_gpu[l, r, ctx + nn:], kc[l, r, ctx + nn:])
            assert np.array_equal(vc_gpu[l, r, ctx + nn:], vc[l, r, ctx + nn:])
        for i in range(7):
            assert np.array_equal(ids[r, i], topk_of(logits[r, i]))
            assert np.array_equal(cl[r, i], logits[r, i][ids[r, i]])
            err = float(np.max(np.abs(logits[r, i] - tr["logits"][i])))
            certified_topk(ids[r, i], tr["logits"][i], err)


def test_wide_and_gemv_paths_agree_on_one_handle():
    """One handle created for 16 requests: a 3-request call (GEMV path) and a
    16-request call (tensor-core path) whose first three requests are the same give
    the same drafts up to the paths' rounding.  Both calls use caches laid out for
    the handle's 16 requests."""
    wl = _wide_workload("q8", 16)
    W = wk.make_weights(wl.geom, "q8", wl.seed)
    inp = wk.make_request_inputs(wl)
    _, _, s16, _, _ = _run(wl, W, inp)
    kc, vc = new_caches(wl, inp)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    g = wl.geom
    ids = torch.zeros((3, 7, 16), dtype=torch.int32, device="cuda")
    vals = torch.zeros((3, 7, 16), dtype=torch.float32, device="cuda")
    gate = torch.zeros((3, 7, g.rank), dtype=torch.float32, device="cuda")
    logits = torch.zeros((3, 7, g.vocab), dtype=torch.float32, device="cuda")
    bd.dflash2_draft_block(s16.drafter.handle, 3, t(inp["anchors"][:3]), t(inp["ctx_len"][:3]), t(inp["n_new"][:3]),
                           t(inp["taps"][:3]), i16(kc), i16(vc), ids, vals, gate, logits)
    torch.cuda.synchronize()
    assert rel_l2(s16.logits.cpu().numpy()[:3], logits.cpu().numpy()) < 2e-2
    assert rel_l2(s16.gate.cpu().numpy()[:3], gate.cpu().numpy()) < 2e-2


def test_head_topk_many_rows_exact_integer_logits():
    """dflash2_head_topk with 128 rows (tensor-core GEMM + chunked top-16): small
    integer weights and hidden values make every logit an exact integer in fp32, so
    ids and values must equal the policy's top-16 of the exact product, ties to the
    smaller id."""
    g = dataclasses.replace(wk.TOY)
    W = wk.make_weights(g, "bf16", 3)
    rng = np.random.default_rng(9)
    lm = rng.integers(-2, 3, (g.vocab, g.hidden)).astype(np.float32)
    W["lm_head"] = wk.bf16_bits_from_f32(lm)
    wl = wk.Workload("toy_r16", g, "bf16", 16, [64] * 16, [0.0] * 16, [1.0] * 16, seed=3)
    d = bd.Drafter(g, "bf16", W, 16, wl.kv_capacity)
    hid = rng.integers(-2, 3, (128, g.hidden)).astype(np.float32)
    hid_t = torch.from_numpy(wk.bf16_bits_from_f32(hid).view(np.int16)).cuda()
    ids = torch.zeros((16, 7, 16), dtype=torch.int32, device="cuda")
    vals = torch.zeros((16, 7, 16), dtype=torch.float32, device="cuda")
    logits = torch.zeros((16, 7, g.vocab), dtype=torch.float32, device="cuda")
    bd.dflash2_head_topk(d.handle, 128, hid_t, ids, vals, logits)
    torch.cuda.synchronize()
    exact = hid.astype(np.float64) @ lm.astype(np.float64).T
    got = logits.cpu().numpy()
    ids_h, vals_h = ids.cpu().numpy(), vals.cpu().numpy()
    for n in range(128):
        if n % 8 == 0:
            continue
        r, i = n // 8, n % 8 - 1
        assert np.array_equal(got[r, i], exact[n])
        want = topk_of(exact[n])
        assert np.array_equal(ids_h[r, i], want)
        assert np.array_equal(vals_h[r, i], exact[n][want])


def test_wide_path_many_stages_per_cta():
    """A mid-size geometry (width 2048, FFN 4096, vocabulary 32768, 2 layers) with 16
    requests and Q8 weights: every CTA of the tensor-core GEMM runs many stages and
    crosses weight blocks (the fc projection ~8 stages per CTA, the LM head ~27), so
    the rings wrap, accumulators are reused and partial planes are added, which the
    toy width (one stage per CTA) never does.  Four requests against the oracle."""
    g = dataclasses.replace(wk.TOY, hidden=2048, n_layers=2, n_q_heads=16, n_kv_heads=4, ffn=4096, vocab=32768,
                            window=256)
    rng = np.random.default_rng(77)
    R = 16
    ctx = [int(x) for x in rng.integers(8, 400, size=R)]
    wl = wk.Workload("mid_wide_q8_r16", g, "q8", R, ctx, [0.0] * R, [0.5] * R, seed=31)
    W = wk.make_weights(g, "q8", wl.seed)
    inp = wk.make_request_inputs(wl)
    kc, vc, step, kct, vct = _run(wl, W, inp)
    logits = step.logits.cpu().numpy()
    gate = step.gate.cpu().numpy()
    ids = step.cand_ids.cpu().numpy()
    for r in (0, 5, 10, 15):
        tr = oracle_draft(wl, W, inp, kc, vc, r)
        assert rel_l2(logits[r], tr["logits"]) < 2e-2, r
        assert rel_l2(gate[r], tr["gate"]) < 2e-2, r
        for i in range(7):
            assert np.array_equal(ids[r, i], topk_of(logits[r, i]))
            err = float(np.max(np.abs(logits[r, i] - tr["logits"][i])))
            certified_topk(ids[r, i], tr["logits"][i], err)
