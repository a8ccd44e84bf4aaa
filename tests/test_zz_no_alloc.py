"""The LM head + top-16 entry point that allocates no device memory.

It exists for callers that cannot call cudaMalloc.  Some run inside a runtime
whose allocator owns all of HBM, or as a plug-in of another framework's memory
pool.  Others must not risk an allocation, and the synchronisation or
out-of-memory failure it can bring, in the middle of a step.  Its scratch is one
fixed device array inside the library, shared by every call.  So the GPU test
makes two calls in a row, on different inputs and row counts, and checks each
against the handle-based dflash2_head_topk on the same input: anything the
second call read from the first would show.

This file is named to be collected last: the GPU test also passes run alone in a
fresh process (the first call on the device does the array's address lookup).
"""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

import block_drafter_pos_gb300 as bd
import workloads as wk


def _call_status(**kw):
    args = dict(lm_head=ctypes.c_void_p(16), vocab=8192, hidden_dim=512, n_rows=8, hidden=ctypes.c_void_p(16),
                cand_ids=ctypes.c_void_p(16), cand_logits=ctypes.c_void_p(16))
    args.update(kw)
    L = bd.lib()
    return L.dflash2_head_topk_noalloc(args["lm_head"], args["vocab"], args["hidden_dim"], args["n_rows"],
                                       args["hidden"], args["cand_ids"], args["cand_logits"], None, None)


def test_noalloc_rejects_bad_sizes_before_any_device_work():
    """Host-side checks return before the first CUDA call, so this runs without a GPU."""
    assert _call_status(n_rows=8 * 5) == bd.binding.E_UNSUPPORTED        # beyond the 32-row scratch
    assert _call_status(vocab=8200) == bd.binding.E_UNSUPPORTED          # not a multiple of 16
    assert _call_status(hidden_dim=520) == bd.binding.E_UNSUPPORTED      # not a multiple of 128
    assert _call_status(n_rows=0) == bd.binding.E_INVAL
    assert _call_status(n_rows=12) == bd.binding.E_INVAL
    assert _call_status(vocab=8) == bd.binding.E_INVAL
    assert _call_status(lm_head=None) == bd.binding.E_INVAL
    assert _call_status(hidden=ctypes.c_void_p(8)) == bd.binding.E_INVAL  # not 16-byte aligned


def _i16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


@pytest.mark.gpu
def test_noalloc_matches_handle_head_topk_on_two_calls_in_a_row():
    V = 8192
    g = dataclasses.replace(wk.TOY, vocab=V)
    W = wk.make_weights(g, "bf16", 11)
    drafter = bd.Drafter(g, "bf16", W, 2, 256)
    lm = _i16(W["lm_head"])                       # the caller's own copy of the LM head
    rng = np.random.default_rng(11)
    try:
        for call, n_rows in enumerate((16, 8)):
            R = n_rows // 8
            x = wk.bf16_bits_from_f32(rng.standard_normal((n_rows, g.hidden)).astype(np.float32))
            xd = _i16(x)
            outs = []
            for noalloc in (False, True):
                ids = torch.full((R, 7, 16), -1, dtype=torch.int32, device="cuda")
                vals = torch.full((R, 7, 16), float("nan"), dtype=torch.float32, device="cuda")
                logits = torch.full((R, 7, V), float("nan"), dtype=torch.float32, device="cuda")
                if noalloc:
                    bd.dflash2_head_topk_noalloc(lm, V, g.hidden, n_rows, xd, ids, vals, logits)
                else:
                    bd.dflash2_head_topk(drafter.handle, n_rows, xd, ids, vals, logits)
                torch.cuda.synchronize()
                outs.append((ids.cpu().numpy(), vals.cpu().numpy(), logits.cpu().numpy()))
            (ri, rv, rl), (gi, gv, gl) = outs
            # same kernels, same per-row arithmetic: the ids must be identical and the
            # values within the LM-head tolerance of the other GPU tests (here exact)
            assert np.array_equal(gi, ri), call
            assert np.isfinite(gl).all() and np.isfinite(gv).all()
            assert np.linalg.norm(gl - rl) <= 1e-6 * np.linalg.norm(rl), call
            assert np.linalg.norm(gv - rv) <= 1e-6 * np.linalg.norm(rv), call
    finally:
        drafter.close()


def _f64_topk(ref):
    """Top-16 of float64 logits built here (value descending, equal values -> smaller id)."""
    order = np.lexsort((np.arange(ref.size), -ref))
    return order[:16]


@pytest.mark.gpu
@pytest.mark.parametrize("n_rows,vocab,hidden", [(32, 8192, 512), (24, 8208, 384), (8, 8208, 384)])
def test_noalloc_shapes_against_float64_matmul(n_rows, vocab, hidden):
    """Shapes the handle path never runs through this call: 32 rows (the array's row
    bound, four 8-row tiles), 24 rows (three tiles in the four-tile kernel), a
    vocabulary that ends inside a 64-row block (8208), and an odd number of 128-wide
    K stages (384).  Integer weights and hidden states make every logit exact, so the
    ids and logits equal a float64 matmul's top-16 computed here, bit for bit."""
    rng = np.random.default_rng(n_rows + vocab + hidden)
    lm = rng.integers(-3, 4, (vocab, hidden)).astype(np.float32)
    x = rng.integers(-1, 2, (n_rows, hidden)).astype(np.float32)
    R = n_rows // 8
    ids = torch.full((R, 7, 16), -1, dtype=torch.int32, device="cuda")
    vals = torch.full((R, 7, 16), float("nan"), dtype=torch.float32, device="cuda")
    logits = torch.full((R, 7, vocab), float("nan"), dtype=torch.float32, device="cuda")
    for _ in range(2):  # two calls in a row on the shared array
        bd.dflash2_head_topk_noalloc(_i16(wk.bf16_bits_from_f32(lm)), vocab, hidden, n_rows,
                                     _i16(wk.bf16_bits_from_f32(x)), ids, vals, logits)
        torch.cuda.synchronize()
    gi, gv, gl = ids.cpu().numpy(), vals.cpu().numpy(), logits.cpu().numpy()
    ref = x.astype(np.float64) @ lm.astype(np.float64).T          # [n_rows][vocab]
    for n in range(n_rows):
        if n % 8 == 0:
            continue                                             # the anchor position is not projected
        rq, pos = n // 8, n % 8
        want = _f64_topk(ref[n])
        assert np.array_equal(gi[rq, pos - 1], want), (n, gi[rq, pos - 1], want)
        assert np.array_equal(gv[rq, pos - 1], ref[n][want].astype(np.float32))
        assert np.array_equal(gl[rq, pos - 1], ref[n].astype(np.float32))


@pytest.mark.gpu
def test_noalloc_device_error_writes_the_sentinel():
    """A failed pipeline wait cannot be reported by the return value (the call does not
    synchronise), so the call writes cand_ids = -1 and cand_logits = NaN.  Driven from
    the host by the test hook that starts the call's error word set; the next call with
    the hook off is correct again."""
    V, H = 8192, 512
    rng = np.random.default_rng(5)
    lm = _i16(wk.bf16_bits_from_f32(rng.integers(-3, 4, (V, H)).astype(np.float32)))
    x = _i16(wk.bf16_bits_from_f32(rng.integers(-1, 2, (16, H)).astype(np.float32)))
    ids = torch.zeros((2, 7, 16), dtype=torch.int32, device="cuda")
    vals = torch.zeros((2, 7, 16), dtype=torch.float32, device="cuda")
    try:
        bd.dflash2_debug_noalloc_inject_error(True)
        bd.dflash2_head_topk_noalloc(lm, V, H, 16, x, ids, vals, None)
        torch.cuda.synchronize()
        assert np.all(ids.cpu().numpy() == -1)
        assert np.all(np.isnan(vals.cpu().numpy()))
    finally:
        bd.dflash2_debug_noalloc_inject_error(False)
    bd.dflash2_head_topk_noalloc(lm, V, H, 16, x, ids, vals, None)
    torch.cuda.synchronize()
    assert np.all(ids.cpu().numpy() >= 0) and np.all(np.isfinite(vals.cpu().numpy()))
