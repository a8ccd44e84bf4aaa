"""GPU parity of a multi-step serving loop through the C ABI: draft, select, verify
and the device-side state update (dflash2_advance), four consecutive steps, with the
oracle following the same loop.  Each step: the drafts and the appended cache rows
against the oracle's (which keeps its own caches), select and verify against the
oracle fed the GPU's candidates (wherever the oracle's decision margins are clear
of rounding), and the advanced state equal to the oracle's update of the GPU's
emitted tokens.  Both paths: 3 bf16 requests (GEMV) and 5 Q8 requests (tensor
cores)."""
import dataclasses

import numpy as np
import pytest
import torch

import block_drafter_pos_gb300 as bd
import oracle
import workloads as wk

from gpu_common import GpuStep, i16, new_caches, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    bd.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("fmt,R", [("bf16", 3), ("q8", 5)])
def test_serving_loop(fmt, R):
    g = dataclasses.replace(wk.TOY, window=256)
    rng = np.random.default_rng(200 + R)
    ctx = [int(x) for x in rng.integers(20, 300, size=R)]
    temps = [[0.0, 0.7, 1.0][r % 3] for r in range(R)]
    steps = 4
    offs0 = [(r << 32) + 3 for r in range(R)]
    wl = wk.Workload(f"toy_loop_{fmt}_r{R}", g, fmt, R, ctx, temps, [0.5] * R, seed=40 + R, philox_seed=42,
                     philox_offsets=offs0, steps=steps)
    W = wk.make_weights(g, fmt, wl.seed)
    inp = wk.make_request_inputs(wl)
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    anchors, ctx_len, n_new = t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"])
    temps_t = t(np.array(temps, np.float32))
    seeds = t(np.full(R, 42, np.uint64).view(np.int64))
    offs = t(np.array(offs0, np.uint64).view(np.int64))
    kct, vct = i16(kc), i16(vc)
    # the oracle's own state and caches
    state = [(int(inp["ctx_len"][r]), int(inp["n_new"][r]), int(inp["anchors"][r]), offs0[r]) for r in range(R)]
    kl = [[kc[l, r].copy() for l in range(g.n_layers)] for r in range(R)]
    vl = [[vc[l, r].copy() for l in range(g.n_layers)] for r in range(R)]
    compared = 0
    for s in range(steps):
        taps = np.random.default_rng(1000 + s).normal(0, 1, (R, 8, g.n_taps * g.hidden)).astype(np.float32)
        step.draft(anchors, ctx_len, n_new, t(taps), kct, vct)
        torch.cuda.synchronize()
        logits = step.logits.cpu().numpy()
        ids, cl, gate = step.cand_ids.cpu().numpy(), step.cand_logits.cpu().numpy(), step.gate.cpu().numpy()
        kc_gpu = kct.cpu().numpy().view(np.uint16)
        for r in range(R):
            c0, nn, anc, _ = state[r]
            tr = oracle.draft_block(g, W, anc, c0, nn, taps[r][:nn], kl[r], vl[r])
            assert rel_l2(logits[r], tr["logits"]) < 2e-2, (s, r)
            for l in range(g.n_layers):
                if nn:
                    assert rel_l2(oracle.bf16_to_f64(kc_gpu[l, r, c0:c0 + nn]),
                                  oracle.bf16_to_f64(kl[r][l][c0:c0 + nn])) < 2e-2, (s, r)
        target = np.zeros((R, 8, g.vocab), np.float32)
        for r in range(R):
            nz = wk.make_target_noise(wl, s, r)
            target[r, :7] = logits[r] + nz[:7]
            target[r, 7] = logits[r, 6] + nz[7]
        step.select(anchors, temps_t, seeds, offs)
        step.verify(t(target), temps_t, seeds, offs)
        torch.cuda.synchronize()
        path, q = step.path.cpu().numpy(), step.q_rows.cpu().numpy()
        st, na = step.status.cpu().numpy(), step.n_acc.cpu().numpy()
        em, ne = step.emitted.cpu().numpy(), step.n_emit.cpu().numpy()
        for r in range(R):
            assert st[r] == 0
            off = state[r][3]
            sel = oracle.walk(g, W["cb_a"], W["cb_b"], state[r][2], ids[r], cl[r].astype(np.float64),
                              gate[r].astype(np.float64), temps[r], 42, off)
            clear = all(m > (1e-4 if temps[r] == 0.0 else 1e-5) for m in sel["margins"])
            if clear:
                assert np.array_equal(path[r], sel["path"]), (s, r)
                ver = oracle.verify(target[r], path[r], ids[r], q[r].astype(np.float64), temps[r], 42, off)
                if temps[r] == 0.0 or all(m > 1e-5 for m in ver["margins"]):
                    assert na[r] == ver["n_accepted"] and ne[r] == ver["n_emitted"], (s, r)
                    assert np.array_equal(em[r], ver["emitted"]), (s, r)
                    compared += 1
            assert ne[r] == na[r] + 1 and np.array_equal(em[r, :na[r]], path[r, :na[r]])
        bd.dflash2_advance(step.drafter.handle, R, step.emitted, step.n_emit, anchors, ctx_len, n_new, offs)
        torch.cuda.synchronize()
        for r in range(R):
            c0, nn, anc, off = state[r]
            state[r] = oracle.advance(c0, nn, anc, em[r], int(ne[r]), off)
        got = list(zip(ctx_len.cpu().numpy().tolist(), n_new.cpu().numpy().tolist(), anchors.cpu().numpy().tolist(),
                       offs.cpu().numpy().view(np.uint64).tolist()))
        assert [tuple(int(v) for v in x) for x in got] == state, s
    assert compared >= steps * R // 2  # most steps' decisions are clear of rounding
