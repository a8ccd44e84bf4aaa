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
        B, P = g.block, g.block - 1
        dev = "cuda"
        self.cand_ids = torch.zeros((R, P, 16), dtype=torch.int32, device=dev)
        self.cand_logits = torch.zeros((R, P, 16), dtype=torch.float32, device=dev)
        self.gate = torch.zeros((R, P, g.rank), dtype=torch.float32, device=dev)
        self.logits = torch.zeros((R, P, g.vocab), dtype=torch.float32, device=dev)
        self.path = torch.zeros((R, P), dtype=torch.int32, device=dev)
        self.q_rows = torch.zeros((R, P, 16), dtype=torch.float32, device=dev)
        self.scores = torch.zeros((R, P, 16, 16), dtype=torch.float32, device=dev)
        self.status = torch.zeros((R,), dtype=torch.int32, device=dev)
        self.n_acc = torch.zeros((R,), dtype=torch.int32, device=dev)
        self.emitted = torch.zeros((R, B), dtype=torch.int32, device=dev)
        self.n_emit = torch.zeros((R,), dtype=torch.int32, device=dev)
        self.probs = torch.zeros((R, B, 2), dtype=torch.float32, device=dev)
        self.width = None  # [R] int32 device tensor of block widths, or None (full blocks)

    def draft(self, anchors, ctx_len, n_new, taps, kc, vc, with_logits=True):
        h = self.drafter.handle
        R = self.wl.n_req
        bd.dflash2_draft_block(h, R, anchors, ctx_len, n_new, taps, kc, vc, self.cand_ids, self.cand_logits,
                               self.gate, self.logits if with_logits else None, width=self.width)

    def select(self, anchors, temps, seeds, offsets, cand_ids=None, cand_logits=None, gate=None):
        h = self.drafter.handle
        bd.dflash2_select(h, self.wl.n_req, anchors, self.cand_ids if cand_ids is None else cand_ids,
                          self.cand_logits if cand_logits is None else cand_logits,
                          self.gate if gate is None else gate, temps, seeds, offsets, self.path, self.q_rows,
                          self.scores, self.status, width=self.width)

    def verify(self, target, temps, seeds, offsets, path=None, cand_ids=None, q_rows=None):
        h = self.drafter.handle
        bd.dflash2_verify(h, self.wl.n_req, target, self.path if path is None else path,
                          self.cand_ids if cand_ids is None else cand_ids, self.q_rows if q_rows is None else q_rows,
                          temps, seeds, offsets, self.n_acc, self.emitted, self.n_emit, self.probs, self.status,
                          width=self.width)


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


# ----------------------------------------------------------------------------- sampled-decision parity
# The oracle decides in FP64; the kernels in FP32.  A decision of the oracle is
# "decided" when it sits farther from its boundary than the kernels' rounding can
# move it; only those must match bit for bit.  Undecided ones are counted.

U24 = 2.0 ** -24


def lattice_error_bounds(W, anchor, cand_ids, gate, scores, q8: bool):
    """Rounding bound of each FP32 lattice score s_i(p -> c) of the selector kernel:
    |fl(s) - s| <= gamma_n * sum_r |a_r g_r b_r| + 2u/(1-u) |s|, the mixed bound of the
    LSE page's selector test paragraph (n = 256 products + 2 roundings per term; Q8
    codebooks add the two dequantisations per term).  scores: the oracle's FP64
    lattice [P][16][16] (row p of position 1 repeats the anchor row).  -> [P][16][16]"""
    n = 262 if q8 else 258
    gam = n * U24 / (1 - n * U24)
    P = len(cand_ids)
    out = np.zeros((P, 16, 16))
    B_all = [np.abs(oracle.codebook_rows(W["cb_b"], cand_ids[i])) for i in range(P)]
    for i in range(P):
        preds = [anchor] * 16 if i == 0 else cand_ids[i - 1]
        A = np.abs(oracle.codebook_rows(W["cb_a"], preds))                 # [16][r]
        absprod = (A * np.abs(gate[i])[None, :]) @ B_all[i].T              # [p][c]
        out[i] = gam * absprod + 2 * U24 / (1 - U24) * np.abs(scores[i])
    return out


def compare_walk(res, gpu_path, gpu_q, bounds, T, cand_ids, exact=False):
    """Follows the oracle's walk (fed the GPU's candidates, logits and gate) and checks
    the GPU's path position by position while each decision is decided:
      greedy: the top-2 gap exceeds 3x the row's largest score bound (the FP64 order
      and the kernel's FP32 order agree), or exact (integer inputs: exact scores);
      sampled: |u * sum - nearest cumsum| / sum exceeds 4 E / T + 64 u (a score error E
      moves each q by at most a factor exp(2E/T); FP32 exp, 16-term sums and the
      product u * sum add well under 64 ulp).
    Returns (positions compared, undecided: bool, list of (gpu q row, oracle q row))."""
    prev = 0
    qs = []
    P = len(res["path"])
    for i in range(P):
        E = 0.0 if exact else float(np.max(bounds[i, prev]))  # integer inputs: every score is exact
        if T == 0.0:
            decided = exact or res["margins"][i] > 3 * E
        else:
            decided = res["margins"][i] > 4 * E / T + 64 * U24
        if not decided:
            return i, True, qs
        assert gpu_path[i] == res["path"][i], (i, gpu_path, res["path"])
        qs.append((gpu_q[i], res["q_rows"][i]))
        prev = int(np.nonzero(cand_ids[i] == res["path"][i])[0][0])
    return P, False, qs


# Decision thresholds of the verify comparison.  The kernel's p at one entry carries
# a few FP32 roundings (exp, the scaled argument, one division): relative ~2e-7 for the
# tokens a ratio test meets, so an accept test is decided beyond 4e-6 of the ratio.
# Its inverse-CDF draws accumulate in FP64 over compensated chunk sums, leaving the
# independent per-entry FP32 roundings (~1e-9 of probability mass at V = 248,320);
# a draw is decided beyond 2e-8 of mass.  A draw lands that close to a boundary with
# probability about 2 * 2e-8 * V: 1% of draws at the full vocabulary.
ACCEPT_REL = 4e-6
DRAW_ABS = 2e-8


def verify_decided(res) -> bool:
    """Every sampled decision of the oracle's chain lies beyond the thresholds above."""
    for kind, _row, margin, scale in res["decisions"]:
        if kind == "accept":
            if margin <= ACCEPT_REL:
                return False
        elif margin * scale <= DRAW_ABS:
            return False
    return True


def compare_verify(res, na, em, ne, probs, T):
    """Bit-exact outputs; the verify probabilities (T > 0) as pairs for a rel-L2 check:
    p at every proposal, and the residual mass / bonus p where both sides took that
    branch (the same branch whenever the outputs agree).  The oracle's verify may run
    on fewer rows w than the GPU's block (a narrowed request): the GPU's entries past
    them are padding (emitted -1, probabilities NaN)."""
    assert na == res["n_accepted"] and ne == res["n_emitted"], (na, ne, res["n_accepted"], res["n_emitted"])
    w = len(res["emitted"])
    assert np.array_equal(em[:w], res["emitted"]), (em, res["emitted"])
    assert np.all(em[w:] == -1)
    P = w - 1
    pairs = []
    if T > 0:
        pairs += list(zip(probs[:P, 0], res["p_path"]))
        if res["n_accepted"] < P:
            j = res["n_accepted"]
            pairs.append((probs[j, 1], res["residual_mass"][j]))
            assert np.all(np.isnan(np.delete(probs[:P, 1], j)))
        else:
            pairs.append((probs[P, 0], res["p_bonus"]))
        assert np.all(np.isnan(probs[w:]))
    else:
        assert np.all(np.isnan(probs))
    return pairs
