"""Shared helpers of the GPU parity tests: set up a drafter from a workload, run the
CUDA path through the C ABI, run the oracle on the same seeded inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import block_drafter_pos_gb300 as bd
import oracle
import workloads as wk

BF16_NAN = 0x7FC0


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def i16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def new_caches(wl, inp, fill=BF16_NAN):
    """Host K/V caches [L][R][cap][nkv][hd] (BF16 bits): visible rows from the workload,
    every other row the fill pattern (NaN: any read of a masked row would show)."""
    g = wl.geom
    cap = wl.kv_capacity
    shp = (g.n_layers, wl.n_req, cap, g.n_kv_heads, g.head_dim)
    kc = np.full(shp, fill, np.uint16)
    vc = np.full(shp, fill, np.uint16)
    for l in range(g.n_layers):
        for r in range(wl.n_req):
            K, V = inp["kv"][l][r]
            lo = int(inp["kv_lo"][r])
            kc[l, r, lo:lo + len(K)] = K
            vc[l, r, lo:lo + len(V)] = V
    return kc, vc


class GpuStep:
    """Device buffers of one workload's step and the three ABI calls."""

    def __init__(self, wl, W, drafter=None):
        self.wl = wl
        g = wl.geom
        self.g = g
        self.drafter = drafter or bd.Drafter(g, wl.weight_format, W, wl.n_req, wl.kv_capacity)
        R = wl.n_req
        dev = "cuda"
        self.cand_ids = torch.zeros((R, 7, 16), dtype=torch.int32, device=dev)
        self.cand_logits = torch.zeros((R, 7, 16), dtype=torch.float32, device=dev)
        self.gate = torch.zeros((R, 7, g.rank), dtype=torch.float32, device=dev)
        self.logits = torch.zeros((R, 7, g.vocab), dtype=torch.float32, device=dev)
        self.path = torch.zeros((R, 7), dtype=torch.int32, device=dev)
        self.q_rows = torch.zeros((R, 7, 16), dtype=torch.float32, device=dev)
        self.scores = torch.zeros((R, 7, 16, 16), dtype=torch.float32, device=dev)
        self.status = torch.zeros((R,), dtype=torch.int32, device=dev)
        self.n_acc = torch.zeros((R,), dtype=torch.int32, device=dev)
        self.emitted = torch.zeros((R, 8), dtype=torch.int32, device=dev)
        self.n_emit = torch.zeros((R,), dtype=torch.int32, device=dev)

    def draft(self, anchors, ctx_len, n_new, taps, kc, vc, with_logits=True):
        h = self.drafter.handle
        R = self.wl.n_req
        bd.dflash2_draft_block(h, R, anchors, ctx_len, n_new, taps, kc, vc, self.cand_ids, self.cand_logits,
                               self.gate, self.logits if with_logits else None)

    def select(self, anchors, temps, seeds, offsets, cand_ids=None, cand_logits=None, gate=None):
        h = self.drafter.handle
        bd.dflash2_select(h, self.wl.n_req, anchors, self.cand_ids if cand_ids is None else cand_ids,
                          self.cand_logits if cand_logits is None else cand_logits,
                          self.gate if gate is None else gate, temps, seeds, offsets, self.path, self.q_rows,
                          self.scores, self.status)

    def verify(self, target, temps, seeds, offsets, path=None, cand_ids=None, q_rows=None):
        h = self.drafter.handle
        bd.dflash2_verify(h, self.wl.n_req, target, self.path if path is None else path,
                          self.cand_ids if cand_ids is None else cand_ids, self.q_rows if q_rows is None else q_rows,
                          temps, seeds, offsets, self.n_acc, self.emitted, self.n_emit, self.status)


def oracle_draft(wl, W, inp, kc_host, vc_host, r):
    """Oracle draft block of request r on copies of the host caches."""
    g = wl.geom
    kl = [kc_host[l, r].copy() for l in range(g.n_layers)]
    vl = [vc_host[l, r].copy() for l in range(g.n_layers)]
    nn = int(inp["n_new"][r])
    tr = oracle.draft_block(g, W, int(inp["anchors"][r]), int(inp["ctx_len"][r]), nn, inp["taps"][r][:nn], kl, vl)
    tr["k_cache"] = kl
    tr["v_cache"] = vl
    return tr


def topk_of(row: np.ndarray, k: int = 16) -> np.ndarray:
    """Reference ordering of the top-k policy applied by the test itself (NaN first by
    index, value descending, ties to the smaller index), for self-consistency checks."""
    idx = np.arange(row.size)
    nan = np.isnan(row)
    order = np.lexsort((idx, np.where(nan, 0.0, -row.astype(np.float64)), ~nan))
    return order[:k].astype(np.int32)


def certified_topk(gpu_ids: np.ndarray, ref_logits: np.ndarray, err: float, k: int = 16):
    """Checks a GPU top-k list against FP64 reference logits whose GPU counterparts may
    differ by up to `err`.  Reference ranks are grouped into clusters of values closer
    than 2*err; ranks in a singleton cluster must hold exactly the reference id, a
    cluster inside the top-k must hold the same ids in some order, and the cluster
    that straddles rank k may hold any of its members.  Returns the number of ranks
    that were decided inside a near-tie cluster."""
    extra = topk_of(ref_logits, min(ref_logits.size, 4 * k))
    vals = ref_logits[extra]
    assert len(set(gpu_ids.tolist())) == k
    near = 0
    j = 0
    while j < k:
        e = j
        while e + 1 < vals.size and vals[e] - vals[e + 1] <= 2 * err:
            e += 1
        members = set(extra[j:e + 1].tolist())
        hi = min(e, k - 1)
        if e == j:
            assert gpu_ids[j] == extra[j], (j, gpu_ids, extra[:k])
        else:
            got = set(gpu_ids[j:hi + 1].tolist())
            assert got <= members, (j, e, got, members)
            if e < k:
                assert got == members
            near += hi - j + 1
        j = e + 1
    return near
