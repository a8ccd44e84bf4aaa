"""GPU parity at the full DFlash2 geometry (5 layers, width 5120, vocab 248320) on
the benchmark workloads: the drafter outputs of every request (a spread of four
of the 16 requests of configuration 5, which runs on the tensor-core path) against
the FP64 oracle, and the select/verify outputs against properties that hold at any
size."""
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


# requests checked against the oracle (all of them, or a spread for 16 requests)
ORACLE_REQS = {5: (0, 5, 10, 15)}


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
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
            assert rel_l2(oracle.bf16_to_f64(kc_gpu[l, r, ctx:ctx + 8]),
                          oracle.bf16_to_f64(tr["k_cache"][l][ctx:ctx + 8])) < 2e-2
        for i in range(7):
            assert np.array_equal(ids[r, i], topk_of(logits[r, i]))
            err = float(np.max(np.abs(logits[r, i] - tr["logits"][i])))
            near += certified_topk(ids[r, i], tr["logits"][i], err)
    # select + verify on the drafted candidates, target = drafter logits + noise
    target = np.zeros((R, 8, g.vocab), np.float32)
    for r in range(R):
        nz = wk.make_target_noise(wl, 0, r)
        target[r, :7] = logits[r] + nz[:7]
        target[r, 7] = logits[r, 6] + nz[7]
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
    for r in range(R):
        assert st[r] == 0
        for i in range(7):
            assert path[r, i] in ids[r, i]
            assert abs(q[r, i].sum() - 1.0) < 1e-5
        assert ne[r] == na[r] + 1 and 0 <= na[r] <= 7
        assert np.array_equal(em[r, :na[r]], path[r, :na[r]])
        assert 0 <= em[r, na[r]] < g.vocab and np.all(em[r, ne[r]:] == -1)
        if wl.temps[r] == 0.0:
            am = np.argmax(target[r], axis=1)
            assert np.array_equal(em[r, :ne[r]], am[:ne[r]])
            if na[r] < 7:
                assert path[r, na[r]] != am[na[r]]
