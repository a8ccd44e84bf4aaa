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
