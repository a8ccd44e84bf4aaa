"""GPU parity of the draft tree (DDTree: selector-scored, log-softmax-normalised
branches grown best-first under a node budget; greedy tree verification) against
the oracle, through the C ABI.

The tree build is compared with the oracle's best-first growth fed the GPU's own
selector lattice: node for node while each step's choice is farther from the next
best option than the FP32 rounding of the per-row log-softmax and the cumulative
sums can move it (counted otherwise).  The tree verify is compared bit-exactly:
it only takes argmaxes of the target rows."""
import dataclasses

import numpy as np
import pytest
import torch

import block_drafter_pos_gb300 as bd
import oracle
import workloads as wk

from gpu_common import GpuStep, i16, new_caches, rel_l2

pytestmark = pytest.mark.gpu

# Bound on the FP32 error of a node's cumulative score: each level's log q carries a
# few roundings of values up to ~|lattice| (exp, the 16-term sum, log, the
# subtraction); seven levels of ~1e-6 each, times ten for safety.
TREE_ABS = 1e-4


@pytest.fixture(scope="module", autouse=True)
def built():
    bd.build()
    assert torch.cuda.is_available()


class TreeBufs:
    def __init__(self, R, budget, V):
        dev = "cuda"
        self.token = torch.full((R, budget), -7, dtype=torch.int32, device=dev)
        self.parent = torch.full((R, budget), -7, dtype=torch.int32, device=dev)
        self.depth = torch.full((R, budget), -7, dtype=torch.int32, device=dev)
        self.score = torch.zeros((R, budget), dtype=torch.float32, device=dev)
        self.n = torch.zeros((R,), dtype=torch.int32, device=dev)
        self.lat = torch.zeros((R, 7, 16, 16), dtype=torch.float32, device=dev)
        self.status = torch.zeros((R,), dtype=torch.int32, device=dev)
        self.n_acc = torch.zeros((R,), dtype=torch.int32, device=dev)
        self.emitted = torch.zeros((R, 8), dtype=torch.int32, device=dev)
        self.n_emit = torch.zeros((R,), dtype=torch.int32, device=dev)


def compare_tree(res, tok, par, dep, sc, n_gpu):
    """Node-by-node equality while decided; returns (nodes compared, undecided)."""
    n = len(res["token"])
    assert n_gpu == n
    for k in range(n):
        if k > 0 and res["margins"][k - 1] <= TREE_ABS:
            return k, True  # an earlier choice was a near-tie: later nodes may differ
        if res["margins"][k] <= TREE_ABS:
            return k, True
        assert tok[k] == res["token"][k] and par[k] == res["parent"][k] and dep[k] == res["depth"][k], k
        assert abs(sc[k] - res["score"][k]) <= TREE_ABS
    return n, False


def _tree_case(V, R, seed):
    si = wk.make_selector_inputs(V, R, seed)
    g = dataclasses.replace(wk.TOY, vocab=V)
    W = wk.make_weights(g, "bf16", 5)
    wl = wk.Workload("tree", g, "bf16", R, [64] * R, [0.0] * R, [1.0] * R, seed=seed)
    return si, W, wl


def test_tree_build_matches_oracle():
    R, V = 4, 8192
    si, W, wl = _tree_case(V, R, 40)
    step = GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    undecided = compared = 0
    for budget in (1, 8, 12, 32):
        tb = TreeBufs(R, budget, V)
        for trial in range(10):
            si = wk.make_selector_inputs(V, R, 500 + 17 * budget + trial)
            bd.dflash2_tree_build(step.drafter.handle, R, budget, t(si["anchors"]), t(si["cand_ids"]),
                                  t(si["cand_logits"]), t(si["gate"]), tb.token, tb.parent, tb.depth, tb.score, tb.n,
                                  tb.lat, tb.status)
            torch.cuda.synchronize()
            assert np.all(tb.status.cpu().numpy() == 0)
            lat = tb.lat.cpu().numpy()
            tok, par, dep = tb.token.cpu().numpy(), tb.parent.cpu().numpy(), tb.depth.cpu().numpy()
            sc, n = tb.score.cpu().numpy(), tb.n.cpu().numpy()
            for r in range(R):
                res = oracle.ddtree_build(lat[r].astype(np.float64), si["cand_ids"][r], budget)
                k, und = compare_tree(res, tok[r], par[r], dep[r], sc[r], int(n[r]))
                undecided += und
                compared += not und
                # structure holds for every node: parents first, depth = parent's + 1, the
                # token is a candidate of its position
                for j in range(int(n[r])):
                    assert -1 <= par[r, j] < j
                    assert dep[r, j] == (1 if par[r, j] < 0 else dep[r, par[r, j]] + 1)
                    assert tok[r, j] in si["cand_ids"][r, dep[r, j] - 1]
    print(f"tree build: {compared} trees compared in full, {undecided} stopped at a near-tie")
    assert undecided <= 3 and compared >= 157


def _target_rows(rng, tree_tok, tree_par, n, budget, V, boost_path):
    """Target rows [budget + 1][V]: N(0, 1.5) with the argmax of each row on the path
    steered onto the chosen child, so acceptance runs down that path."""
    z = rng.normal(0, 1.5, (budget + 1, V)).astype(np.float32)
    cur = -1
    for k in boost_path:
        z[cur + 1, tree_tok[k]] = z[cur + 1].max() + 4.0
        cur = k
    return z


def test_tree_verify_matches_oracle():
    R, V, budget = 4, 8192, 12
    si, W, wl = _tree_case(V, R, 41)
    step = GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    tb = TreeBufs(R, budget, V)
    rng = np.random.default_rng(41)
    depths_seen = set()
    for trial in range(20):
        si = wk.make_selector_inputs(V, R, 700 + trial)
        bd.dflash2_tree_build(step.drafter.handle, R, budget, t(si["anchors"]), t(si["cand_ids"]),
                              t(si["cand_logits"]), t(si["gate"]), tb.token, tb.parent, tb.depth, tb.score, tb.n,
                              None, tb.status)
        torch.cuda.synchronize()
        tok, par, n = tb.token.cpu().numpy(), tb.parent.cpu().numpy(), tb.n.cpu().numpy()
        target = np.zeros((R, budget + 1, V), np.float32)
        for r in range(R):
            # steer acceptance down the path to a random node
            end = int(rng.integers(-1, n[r]))
            path = []
            while end >= 0:
                path.append(end)
                end = int(par[r, end])
            target[r] = _target_rows(rng, tok[r], par[r], n[r], budget, V, path[::-1])
        if trial == 3:
            target[2, 0, 17] = np.nan  # a nonfinite root row
        tb.status.zero_()
        if trial == 5:
            tb.status[1] = 2  # a request skipped by an earlier stage
        bd.dflash2_tree_verify(step.drafter.handle, R, budget, t(target), tb.token, tb.parent, tb.n, tb.n_acc,
                               tb.emitted, tb.n_emit, tb.status)
        torch.cuda.synchronize()
        na, em, ne, st = (x.cpu().numpy() for x in (tb.n_acc, tb.emitted, tb.n_emit, tb.status))
        for r in range(R):
            st_in = 2 if (trial == 5 and r == 1) else 0
            res = oracle.ddtree_verify(target[r].astype(np.float64), tok[r, :n[r]], par[r, :n[r]], st_in)
            assert st[r] == res["status"], (trial, r)
            assert na[r] == res["n_accepted"] and ne[r] == res["n_emitted"], (trial, r)
            assert np.array_equal(em[r], res["emitted"]), (trial, r)
            depths_seen.add(int(na[r]))
    assert len(depths_seen) >= 4  # acceptance ran to several depths


def test_tree_on_full_geometry_draft():
    """Configuration 2's drafted block (V = 248,320): tree of budget 12 against the oracle
    on the GPU's lattice, then greedy verification on target rows built from the
    drafter's logits plus noise (row of a node at depth d: block position d + 1's
    logits, position 7's for the deepest), bit-exact against the oracle."""
    wl = wk.workload(2)
    g = wl.geom
    W = wk.make_weights(g, wl.weight_format, wl.seed)
    inp = wk.make_request_inputs(wl)
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    step.draft(t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"]), t(inp["taps"]), i16(kc), i16(vc))
    budget = 12
    tb = TreeBufs(1, budget, g.vocab)
    bd.dflash2_tree_build(step.drafter.handle, 1, budget, t(inp["anchors"]), step.cand_ids, step.cand_logits,
                          step.gate, tb.token, tb.parent, tb.depth, tb.score, tb.n, tb.lat, tb.status)
    torch.cuda.synchronize()
    assert tb.status.item() == 0
    res = oracle.ddtree_build(tb.lat.cpu().numpy()[0].astype(np.float64), step.cand_ids.cpu().numpy()[0], budget)
    k, und = compare_tree(res, tb.token.cpu().numpy()[0], tb.parent.cpu().numpy()[0], tb.depth.cpu().numpy()[0],
                          tb.score.cpu().numpy()[0], int(tb.n.item()))
    assert not und
    logits = step.logits.cpu().numpy()[0]
    dep = tb.depth.cpu().numpy()[0]
    rng = np.random.default_rng(2)
    rows = np.zeros((budget + 1, g.vocab), np.float32)
    rows[0] = logits[0] + rng.normal(0, 1.0, g.vocab).astype(np.float32)
    for j in range(int(tb.n.item())):
        rows[1 + j] = logits[min(int(dep[j]), 6)] + rng.normal(0, 1.0, g.vocab).astype(np.float32)
    bd.dflash2_tree_verify(step.drafter.handle, 1, budget, t(rows[None]), tb.token, tb.parent, tb.n, tb.n_acc,
                           tb.emitted, tb.n_emit, tb.status)
    torch.cuda.synchronize()
    n = int(tb.n.item())
    ref = oracle.ddtree_verify(rows.astype(np.float64), tb.token.cpu().numpy()[0, :n],
                               tb.parent.cpu().numpy()[0, :n])
    assert tb.status.item() == 0
    assert tb.n_acc.item() == ref["n_accepted"] and tb.n_emit.item() == ref["n_emitted"]
    assert np.array_equal(tb.emitted.cpu().numpy()[0], ref["emitted"])
