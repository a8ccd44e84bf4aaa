"""GPU parity of a multi-step serving loop through the C ABI: draft, select, verify
and the device-side state update (dflash2_advance), four consecutive steps, with the
oracle following the same loop.  Each step: the drafts and the appended cache rows
against the oracle's (which keeps its own caches), select and verify against the
oracle fed the GPU's candidates (wherever the oracle's decision margins are clear
of rounding), and the advanced state equal to the oracle's update of the GPU's
emitted tokens.  Both paths: 3 bf16 requests (GEMV) and 5 Q8 requests (tensor
cores).  The loop runs once step by step from the host and once as one CUDA graph
of all four steps with no host synchronisation between them (how the bench times
the 16-request loop): there each step's first kernel reads the ids and lengths that
the previous step's update has just written."""
import dataclasses

import numpy as np
import pytest
import torch

import block_drafter_pos_gb300 as bd
import oracle
import workloads as wk

from gpu_common import GpuStep, i16, new_caches, rel_l2

pytestmark = pytest.mark.gpu

STEPS = 4


@pytest.fixture(scope="module", autouse=True)
def built():
    bd.build()
    assert torch.cuda.is_available()


def _loop_setup(fmt, R):
    g = dataclasses.replace(wk.TOY, window=256)
    rng = np.random.default_rng(200 + R)
    ctx = [int(x) for x in rng.integers(20, 300, size=R)]
    temps = [[0.0, 0.7, 1.0][r % 3] for r in range(R)]
    offs0 = [(r << 32) + 3 for r in range(R)]
    wl = wk.Workload(f"toy_loop_{fmt}_r{R}", g, fmt, R, ctx, temps, [0.5] * R, seed=40 + R, philox_seed=42,
                     philox_offsets=offs0, steps=STEPS)
    W = wk.make_weights(g, fmt, wl.seed)
    inp = wk.make_request_inputs(wl)
    taps = [np.random.default_rng(1000 + s).normal(0, 1, (R, 8, g.n_taps * g.hidden)).astype(np.float32)
            for s in range(STEPS)]
    noise = [np.stack([wk.make_target_noise(wl, s, r) for r in range(R)]) for s in range(STEPS)]
    return g, wl, W, inp, temps, offs0, taps, noise


class OracleLoop:
    """The oracle's side of the loop: its own request state and caches, checked step
    by step against what the GPU produced in that step."""

    def __init__(self, g, W, inp, kc, vc, temps, offs0):
        R = len(temps)
        self.g, self.W, self.temps = g, W, temps
        self.state = [(int(inp["ctx_len"][r]), int(inp["n_new"][r]), int(inp["anchors"][r]), offs0[r]) for r in range(R)]
        self.kl = [[kc[l, r].copy() for l in range(g.n_layers)] for r in range(R)]
        self.vl = [[vc[l, r].copy() for l in range(g.n_layers)] for r in range(R)]
        self.appended = [[] for _ in range(R)]  # (first row, rows) appended per step
        self.compared = 0

    def check_step(self, s, taps, logits, ids, cl, gate, target, path, q, st, na, em, ne, new_state):
        g, W = self.g, self.W
        for r in range(len(self.temps)):
            c0, nn, anc, off = self.state[r]
            tr = oracle.draft_block(g, W, anc, c0, nn, taps[r][:nn], self.kl[r], self.vl[r])
            assert rel_l2(logits[r], tr["logits"]) < 2e-2, (s, r)
            self.appended[r].append((c0, nn))
            assert st[r] == 0, (s, r)
            sel = oracle.walk(g, W["cb_a"], W["cb_b"], anc, ids[r], cl[r].astype(np.float64),
                              gate[r].astype(np.float64), self.temps[r], 42, off)
            if all(m > (1e-4 if self.temps[r] == 0.0 else 1e-5) for m in sel["margins"]):
                assert np.array_equal(path[r], sel["path"]), (s, r)
                ver = oracle.verify(target[r], path[r], ids[r], q[r].astype(np.float64), self.temps[r], 42, off)
                if self.temps[r] == 0.0 or all(m > 1e-5 for m in ver["margins"]):
                    assert na[r] == ver["n_accepted"] and ne[r] == ver["n_emitted"], (s, r)
                    assert np.array_equal(em[r], ver["emitted"]), (s, r)
                    self.compared += 1
            assert ne[r] == na[r] + 1 and np.array_equal(em[r, :na[r]], path[r, :na[r]])
            self.state[r] = oracle.advance(c0, nn, anc, em[r], int(ne[r]), off)
        assert [tuple(int(v) for v in x) for x in new_state] == self.state, s

    def check_cache(self, kc_gpu):
        """Every row the loop appended, against the oracle's."""
        for r, rows in enumerate(self.appended):
            for c0, nn in rows:
                for l in range(self.g.n_layers):
                    if nn:
                        assert rel_l2(oracle.bf16_to_f64(kc_gpu[l, r, c0:c0 + nn]),
                                      oracle.bf16_to_f64(self.kl[r][l][c0:c0 + nn])) < 2e-2, (r, c0)


def _state_tuple(ctx_len, n_new, anchors, offs):
    return list(zip(ctx_len.tolist(), n_new.tolist(), anchors.tolist(), offs.view(np.uint64).tolist()))


@pytest.mark.parametrize("fmt,R", [("bf16", 3), ("q8", 5)])
def test_serving_loop(fmt, R):
    g, wl, W, inp, temps, offs0, taps, noise = _loop_setup(fmt, R)
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    anchors, ctx_len, n_new = t(inp["anchors"]), t(inp["ctx_len"]), t(inp["n_new"])
    temps_t = t(np.array(temps, np.float32))
    seeds = t(np.full(R, 42, np.uint64).view(np.int64))
    offs = t(np.array(offs0, np.uint64).view(np.int64))
    kct, vct = i16(kc), i16(vc)
    ol = OracleLoop(g, W, inp, kc, vc, temps, offs0)
    for s in range(STEPS):
        step.draft(anchors, ctx_len, n_new, t(taps[s]), kct, vct)
        torch.cuda.synchronize()
        logits = step.logits.cpu().numpy()
        target = np.zeros((R, 8, g.vocab), np.float32)
        target[:, :7] = logits + noise[s][:, :7]
        target[:, 7] = logits[:, 6] + noise[s][:, 7]
        step.select(anchors, temps_t, seeds, offs)
        step.verify(t(target), temps_t, seeds, offs)
        torch.cuda.synchronize()
        outs = [x.cpu().numpy() for x in (step.cand_ids, step.cand_logits, step.gate)]
        res = [x.cpu().numpy() for x in (step.path, step.q_rows, step.status, step.n_acc, step.emitted, step.n_emit)]
        bd.dflash2_advance(step.drafter.handle, R, step.emitted, step.n_emit, anchors, ctx_len, n_new, offs)
        torch.cuda.synchronize()
        new_state = _state_tuple(ctx_len.cpu().numpy(), n_new.cpu().numpy(), anchors.cpu().numpy(), offs.cpu().numpy())
        ol.check_step(s, taps[s], logits, *outs, target, *res, new_state)
    ol.check_cache(kct.cpu().numpy().view(np.uint16))
    assert ol.compared >= STEPS * R // 2  # most steps' decisions are clear of rounding


@pytest.mark.parametrize("fmt,R", [("bf16", 3), ("q8", 5)])
def test_serving_loop_in_one_graph(fmt, R):
    g, wl, W, inp, temps, offs0, taps, noise = _loop_setup(fmt, R)
    kc, vc = new_caches(wl, inp)
    step = GpuStep(wl, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    state0 = {"anchors": t(inp["anchors"]), "ctx_len": t(inp["ctx_len"]), "n_new": t(inp["n_new"]),
              "offs": t(np.array(offs0, np.uint64).view(np.int64))}
    S = {k: v.clone() for k, v in state0.items()}
    temps_t = t(np.array(temps, np.float32))
    seeds = t(np.full(R, 42, np.uint64).view(np.int64))
    kct, vct = i16(kc), i16(vc)
    taps_all, noise_all = t(np.stack(taps)), t(np.stack(noise))
    taps_buf = torch.empty_like(taps_all[0])
    target = torch.empty((R, 8, g.vocab), dtype=torch.float32, device="cuda")
    rec = {k: torch.empty((STEPS,) + tuple(x.shape), dtype=x.dtype, device="cuda") for k, x in (
        ("logits", step.logits), ("cand_ids", step.cand_ids), ("cand_logits", step.cand_logits), ("gate", step.gate),
        ("target", target), ("path", step.path), ("q_rows", step.q_rows), ("status", step.status),
        ("n_acc", step.n_acc), ("emitted", step.emitted), ("n_emit", step.n_emit),
        ("anchors", S["anchors"]), ("ctx_len", S["ctx_len"]), ("n_new", S["n_new"]), ("offs", S["offs"]))}

    def one_step(s):
        taps_buf.copy_(taps_all[s])
        step.draft(S["anchors"], S["ctx_len"], S["n_new"], taps_buf, kct, vct)
        target[:, :7] = step.logits + noise_all[s][:, :7]
        target[:, 7] = step.logits[:, 6] + noise_all[s][:, 7]
        step.select(S["anchors"], temps_t, seeds, S["offs"])
        step.verify(target, temps_t, seeds, S["offs"])
        bd.dflash2_advance(step.drafter.handle, R, step.emitted, step.n_emit, S["anchors"], S["ctx_len"], S["n_new"],
                           S["offs"])
        for k in ("logits", "cand_ids", "cand_logits", "gate", "path", "q_rows", "status", "n_acc", "emitted",
                  "n_emit"):
            rec[k][s].copy_(getattr(step, k))
        rec["target"][s].copy_(target)
        for k in ("anchors", "ctx_len", "n_new", "offs"):
            rec[k][s].copy_(S[k])

    # one eager step first (kernel attributes are set on first use), then the
    # initial state again: the graph's first step rewrites the same cache rows
    one_step(0)
    torch.cuda.synchronize()
    for k, v in state0.items():
        S[k].copy_(v)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for s in range(STEPS):
                one_step(s)
    torch.cuda.current_stream().wait_stream(cap)
    for k, v in state0.items():
        S[k].copy_(v)
    graph.replay()
    torch.cuda.synchronize()
    out = {k: v.cpu().numpy() for k, v in rec.items()}
    ol = OracleLoop(g, W, inp, kc, vc, temps, offs0)
    for s in range(STEPS):
        new_state = _state_tuple(out["ctx_len"][s], out["n_new"][s], out["anchors"][s], out["offs"][s])
        ol.check_step(s, taps[s], out["logits"][s], out["cand_ids"][s], out["cand_logits"][s], out["gate"][s],
                      out["target"][s], out["path"][s], out["q_rows"][s], out["status"][s], out["n_acc"][s],
                      out["emitted"][s], out["n_emit"][s], new_state)
    ol.check_cache(kct.cpu().numpy().view(np.uint16))
    assert ol.compared >= STEPS * R // 2
