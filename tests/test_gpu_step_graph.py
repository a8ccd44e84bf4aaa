"""GPU test of dflash2_step (include/dflash2.h): one draft + select + verify step
replayed from the handle's CUDA graph of its argument set.  Over several steps of a
serving loop (the state advanced on the device between steps, new taps and target
rows copied into the same buffers), its outputs equal those of the three separate
calls bit for bit, on both paths (3 bf16 requests: GEMV; 5 Q8 requests: tensor
cores), and a replay counts the same kernels as a step of separate calls.  More
argument sets than the handle keeps replace the least recently used graph and still
give the same results, and a change of the selector mode is not replayed from a
graph captured under the other mode."""
import numpy as np
import pytest
import torch

import block_drafter_pos_gb300 as bd

from gpu_common import GpuStep, i16, new_caches
from test_gpu_loop import STEPS, _loop_setup

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    bd.build()
    assert torch.cuda.is_available()


def t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class Side:
    """One copy of the loop state and of the step's outputs (device buffers whose
    addresses stay fixed across steps)."""

    def __init__(self, g, inp, kc, vc, temps, offs0, R):
        self.anchors, self.ctx_len, self.n_new = t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"])
        self.offs = t(np.array(offs0, np.uint64).view(np.int64))
        self.temps = t(np.array(temps, np.float32))
        self.seeds = t(np.full(R, 42, np.uint64).view(np.int64))
        self.kc, self.vc = i16(kc), i16(vc)
        self.taps = torch.zeros((R, 8, g.n_taps * g.hidden), dtype=torch.float32, device="cuda")
        self.target = torch.zeros((R, 8, g.vocab), dtype=torch.float32, device="cuda")
        P = g.block - 1
        z = lambda shape, dt: torch.zeros(shape, dtype=dt, device="cuda")
        self.cand_ids, self.cand_logits = z((R, P, 16), torch.int32), z((R, P, 16), torch.float32)
        self.gate = z((R, P, g.rank), torch.float32)
        self.path, self.q_rows = z((R, P), torch.int32), z((R, P, 16), torch.float32)
        self.status, self.n_acc, self.n_emit = z((R,), torch.int32), z((R,), torch.int32), z((R,), torch.int32)
        self.emitted = z((R, g.block), torch.int32)

    def outputs(self):
        return {k: getattr(self, k).cpu().numpy() for k in (
            "cand_ids", "cand_logits", "gate", "path", "q_rows", "status", "n_acc", "emitted", "n_emit", "anchors",
            "ctx_len", "n_new", "offs", "kc", "vc")}


def _separate(h, R, S):
    bd.dflash2_draft_block(h, R, S.anchors, S.ctx_len, S.n_new, S.taps, S.kc, S.vc, S.cand_ids, S.cand_logits, S.gate,
                           None)
    bd.dflash2_select(h, R, S.anchors, S.cand_ids, S.cand_logits, S.gate, S.temps, S.seeds, S.offs, S.path, S.q_rows,
                      None, S.status)
    bd.dflash2_verify(h, R, S.target, S.path, S.cand_ids, S.q_rows, S.temps, S.seeds, S.offs, S.n_acc, S.emitted,
                      S.n_emit, None, S.status)


def _step(h, R, S, status=None):
    bd.dflash2_step(h, R, S.anchors, S.ctx_len, S.n_new, S.taps, S.kc, S.vc, S.cand_ids, S.cand_logits, S.gate,
                    S.temps, S.seeds, S.offs, S.path, S.q_rows, S.status if status is None else status, S.target,
                    S.n_acc, S.emitted, S.n_emit)


def _advance(h, R, S):
    bd.dflash2_advance(h, R, S.emitted, S.n_emit, S.anchors, S.ctx_len, S.n_new, S.offs)


@pytest.mark.parametrize("fmt,R", [("bf16", 3), ("q8", 5)])
def test_step_graph_equals_the_three_calls(fmt, R):
    g, wl, W, inp, temps, offs0, taps, noise = _loop_setup(fmt, R)
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    h = step.drafter.handle
    A = Side(g, inp, kc, vc, temps, offs0, R)  # separate calls
    Bs = Side(g, inp, kc, vc, temps, offs0, R)  # dflash2_step
    rng = np.random.default_rng(7 + R)
    for s in range(STEPS):
        tg = (rng.standard_normal((R, 8, g.vocab)) * 3.0).astype(np.float32)
        for S in (A, Bs):
            S.taps.copy_(t(taps[s]))
            S.target.copy_(t(tg))
        n0 = bd.dflash2_launch_count(h)
        _separate(h, R, A)
        n_sep = bd.dflash2_launch_count(h) - n0
        _advance(h, R, A)
        torch.cuda.synchronize()
        n0 = bd.dflash2_launch_count(h)
        _step(h, R, Bs)  # step 0: the calls as they are, then the capture; later steps: the graph
        n_step = bd.dflash2_launch_count(h) - n0
        _advance(h, R, Bs)
        torch.cuda.synchronize()
        assert n_step == n_sep, (s, n_step, n_sep)
        a, b = A.outputs(), Bs.outputs()
        for k in a:
            assert np.array_equal(a[k], b[k]), (s, k)
        assert np.all(a["status"] == 0) and np.all(a["n_emit"] >= 1), s


def test_step_graph_more_argument_sets_than_kept():
    """DFLASH2_STEP_GRAPHS + 1 argument sets (each its own status buffer), used in
    turn twice: every call after the first of a set is a replay or, once the set was
    replaced, a new capture; all give the separate calls' results."""
    fmt, R = "bf16", 3
    g, wl, W, inp, temps, offs0, taps, noise = _loop_setup(fmt, R)
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    h = step.drafter.handle
    A = Side(g, inp, kc, vc, temps, offs0, R)
    Bs = Side(g, inp, kc, vc, temps, offs0, R)
    n_sets = 5
    statuses = [torch.zeros((R,), dtype=torch.int32, device="cuda") for _ in range(n_sets)]
    rng = np.random.default_rng(11)
    for it in range(2 * n_sets):
        tg = (rng.standard_normal((R, 8, g.vocab)) * 3.0).astype(np.float32)
        for S in (A, Bs):
            S.taps.copy_(t(taps[it % STEPS]))
            S.target.copy_(t(tg))
        _separate(h, R, A)
        _step(h, R, Bs, status=statuses[it % n_sets])
        torch.cuda.synchronize()
        a, b = A.outputs(), Bs.outputs()
        b["status"] = statuses[it % n_sets].cpu().numpy()
        for k in a:
            assert np.array_equal(a[k], b[k]), (it, k)
    bd.dflash2_step_graphs_clear(h)


def test_step_graph_follows_the_selector_mode():
    """A set captured under the sequential walk, then the Viterbi mode (mode 1, for the
    greedy requests): the step must use the mode in force, like the separate calls."""
    fmt, R = "bf16", 3
    g, wl, W, inp, temps, offs0, taps, noise = _loop_setup(fmt, R)
    # selector tables 16x larger (a power of two: exact in bf16), so that the pairwise
    # scores outweigh the candidates' logits and the best path is often not the walk's
    W = dict(W)
    for name in ("cb_a", "cb_b"):
        f = (W[name]["w"].astype(np.uint32) << 16).view(np.float32) * np.float32(16.0)
        W[name] = {"kind": "bf16", "w": (f.view(np.uint32) >> 16).astype(np.uint16)}
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    h = step.drafter.handle
    greedy = [0.0] * R  # mode 1 changes the greedy requests' paths only
    A = Side(g, inp, kc, vc, greedy, offs0, R)
    Bs = Side(g, inp, kc, vc, greedy, offs0, R)
    rng = np.random.default_rng(5)
    differs = 0  # requests whose mode-1 path differs from the walk's (else the test proves nothing)
    for it, mode in enumerate((0, 0, 1, 1, 1, 1, 0)):
        bd.dflash2_set_select_mode(h, mode)
        tg = (rng.standard_normal((R, 8, g.vocab)) * 3.0).astype(np.float32)
        for S in (A, Bs):
            S.taps.copy_(t(taps[it % STEPS]))
            S.target.copy_(t(tg))
        _separate(h, R, A)
        _step(h, R, Bs)
        torch.cuda.synchronize()
        a, b = A.outputs(), Bs.outputs()
        for k in a:
            assert np.array_equal(a[k], b[k]), (it, mode, k)
        if mode == 1:
            bd.dflash2_set_select_mode(h, 0)
            walk_path = torch.empty_like(A.path)
            bd.dflash2_select(h, R, A.anchors, A.cand_ids, A.cand_logits, A.gate, A.temps, A.seeds, A.offs, walk_path,
                              torch.empty_like(A.q_rows), None, torch.empty_like(A.status))
            torch.cuda.synchronize()
            wp = walk_path.cpu().numpy()
            differs += sum(int(not np.array_equal(wp[r], a["path"][r])) for r in range(R))
    bd.dflash2_set_select_mode(h, 0)
    assert differs >= 1
    bd.dflash2_step_graphs_clear(h)
