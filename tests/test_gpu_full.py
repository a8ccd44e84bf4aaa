"""GPU parity at the full DFlash2 geometry (5 layers, width 5120, vocab 248320) on
the benchmark workloads (and configuration 2's request with blocks of 16): the
drafter outputs of every request (a spread of four of the 16 requests of
configuration 5, which runs on the tensor-core path) against
the FP64 oracle; the selector walk and the verification of EVERY request against
the oracle fed the GPU's own candidates, candidate logits, gate, path, q rows and
target rows (discrete outputs bit-exact wherever the decision lies outside the
kernels' FP32 rounding, such near-boundary decisions counted: at most one per
configuration; verify probabilities and q rows at rel-L2 <= 1e-4); and properties
that hold at any size."""
import numpy as np
import pytest
import torch

import block_drafter_pos_gb300 as bd
import oracle
import workloads as wk

from gpu_common import (GpuStep, certified_topk, compare_verify, compare_walk, i16, lattice_error_bounds, new_caches,
                        oracle_draft, rel_l2, topk_of, verify_decided)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    bd.build()
    assert torch.cuda.is_available()


# requests checked against the oracle (all of them, or a spread for 16 requests)
ORACLE_REQS = {5: (0, 5, 10, 15)}


@pytest.mark.parametrize("cfg", [2, 3, 4, 5, 9])
def test_full_geometry_step(cfg):
    wl = wk.workload(cfg)
    g = wl.geom
    W = wk.make_weights(g, wl.weight_format, wl.seed)
    inp = wk.make_request_inputs(wl)
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    kct, vct = i16(kc), i16(vc)
    R = wl.n_req
    B, P = g.block, g.block - 1  # configuration 9: blocks of 16
    step.draft(t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"]), t(inp["taps"]), kct, vct)
    torch.cuda.synchronize()
    logits = step.logits.cpu().numpy()
    ids = step.cand_ids.cpu().numpy()
    gate = step.gate.cpu().numpy()
    kc_gpu = kct.cpu().numpy().view(np.uint16)
    near = 0
    for r in ORACLE_REQS.get(cfg, range(R)):
        tr = oracle_draft(wl, W, inp, kc, vc, r)
        assert rel_l2(logits[r], tr["logits"]) < 2e-2, r
        assert rel_l2(gate[r], tr["gate"]) < 2e-2, r
        ctx = int(inp["ctx_len"][r])
        for l in range(g.n_layers):
            assert rel_l2(oracle.bf16_to_f64(kc_gpu[l, r, ctx:ctx + B]),
                          oracle.bf16_to_f64(tr["k_cache"][l][ctx:ctx + B])) < 2e-2
        for i in range(P):
            assert np.array_equal(ids[r, i], topk_of(logits[r, i]))
            err = float(np.max(np.abs(logits[r, i] - tr["logits"][i])))
            near += certified_topk(ids[r, i], tr["logits"][i], err)
    # select + verify on the drafted candidates, target = drafter logits + noise
    target = np.zeros((R, B, g.vocab), np.float32)
    for r in range(R):
        nz = wk.make_target_noise(wl, 0, r)
        target[r, :P] = logits[r] + nz[:P]
        target[r, P] = logits[r, P - 1] + nz[P]
    temps = t(np.array(wl.temps, np.float32))
    seeds = t(np.full(R, wl.philox_seed, np.uint64).view(np.int64))
    offs = t(np.array(wl.philox_offsets or [0] * R, np.uint64).view(np.int64))
    step.select(t(inp["anchors"]), temps, seeds, offs)
    step.verify(t(target), temps, seeds, offs)
    torch.cuda.synchronize()
    path = step.path.cpu().numpy()
    q = step.q_rows.cpu().numpy()
    st = step.status.cpu().numpy()
    na, em, ne = step.n_acc.cpu().numpy(), step.emitted.cpu().numpy(), step.n_emit.cpu().numpy()
    probs = step.probs.cpu().numpy()
    cl = step.cand_logits.cpu().numpy()
    # the oracle's walk and verify on the GPU's own inputs, every request
    offs_h = wl.philox_offsets or [0] * R
    undecided_walk = undecided_verify = 0
    q_pairs, p_pairs = [], []
    for r in range(R):
        T = float(np.float32(wl.temps[r]))  # the kernel's FP32 temperature
        res = oracle.walk(g, W["cb_a"], W["cb_b"], int(inp["anchors"][r]), ids[r], cl[r].astype(np.float64),
                          gate[r].astype(np.float64), T, wl.philox_seed, int(offs_h[r]))
        assert res["status"] == 0
        bounds = lattice_error_bounds(W, int(inp["anchors"][r]), ids[r], gate[r].astype(np.float64), res["scores"],
                                      wl.weight_format == "q8")
        n_cmp, und, qs = compare_walk(res, path[r], q[r], bounds, T, ids[r])
        undecided_walk += und
        q_pairs += qs
        ver = oracle.verify(target[r].astype(np.float64), path[r], ids[r], q[r].astype(np.float64), T,
                            wl.philox_seed, int(offs_h[r]))
        if verify_decided(ver):
            p_pairs += compare_verify(ver, na[r], em[r], ne[r], probs[r], T)
        else:
            undecided_verify += 1
    print(f"cfg {cfg}: walk undecided {undecided_walk}/{R}, verify undecided {undecided_verify}/{R}")
    assert undecided_walk <= 1 and undecided_verify <= 1
    if q_pairs:
        qg, qo = np.array([a for a, _ in q_pairs]), np.array([b for _, b in q_pairs])
        assert rel_l2(qg, qo) <= 1e-4, rel_l2(qg, qo)
    if p_pairs:
        pg, po = np.array([a for a, _ in p_pairs], np.float64), np.array([b for _, b in p_pairs])
        assert rel_l2(pg, po) <= 1e-4, rel_l2(pg, po)
    for r in range(R):
        assert st[r] == 0
        for i in range(P):
            assert path[r, i] in ids[r, i]
            assert abs(q[r, i].sum() - 1.0) < 1e-5
        assert ne[r] == na[r] + 1 and 0 <= na[r] <= P
        assert np.array_equal(em[r, :na[r]], path[r, :na[r]])
        assert 0 <= em[r, na[r]] < g.vocab and np.all(em[r, ne[r]:] == -1)
        if wl.temps[r] == 0.0:
            am = np.argmax(target[r], axis=1)
            assert np.array_equal(em[r, :ne[r]], am[:ne[r]])
            if na[r] < P:
                assert path[r, na[r]] != am[na[r]]
