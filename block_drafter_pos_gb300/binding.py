"""Thin ctypes binding of the C ABI in include/dflash2.h (same names, argument
marshalling only).  Tensors are torch CUDA tensors; their data pointers and the
current CUDA stream are passed straight through.  Every computation happens in
the CUDA library; there is no CPU path.  If the library has not been built, or
no GPU is present when a call needs one, the binding raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

from .builder import LIB

MAX_LAYERS = 8
OK, E_INVAL, E_NONFINITE, E_CUDA, E_UNSUPPORTED = 0, 1, 2, 3, 4
WEIGHTS_BF16, WEIGHTS_Q8G64 = 0, 1


class Dflash2Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({_status_string(status)})")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "hidden", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "n_taps", "block",
        "top_k", "rank", "window", "conv_taps", "conv_group", "mask_token_id", "weight_format")] + [
        ("rope_theta", ctypes.c_double), ("rms_eps", ctypes.c_float)]


class Matrix(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("bias", ctypes.c_void_p)]


_LAYER_MATS = ("q", "k", "v", "o", "gate", "up", "down", "attn_delta", "mlp_delta")


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("input_norm", "post_norm", "q_norm", "k_norm", "attn_base",
                                                 "mlp_base")] + [(n, Matrix) for n in _LAYER_MATS]


class StepArgs(ctypes.Structure):
    """dflash2_step_args: the device buffers of one draft + select + verify step."""
    _fields_ = [("n_req", ctypes.c_int32)] + [(n, ctypes.c_void_p) for n in (
        "anchor_ids", "ctx_len", "n_new", "taps", "k_cache", "v_cache", "cand_ids", "cand_logits", "gate",
        "temperature", "seed", "philox_offset", "path", "q_rows", "status", "target_logits", "n_accepted",
        "emitted", "n_emitted", "width")]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("embed", "lm_head", "hidden_norm", "final_norm")] + [
        (n, Matrix) for n in ("fc", "sel_proj", "cb_a", "cb_b")] + [("layers", LayerWeights * MAX_LAYERS)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libdflash2.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"libdflash2.so is not built ({LIB}); run block_drafter_pos_gb300.build()")
        L = ctypes.CDLL(LIB)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.dflash2_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), i32, i32, ctypes.POINTER(vp)]
        L.dflash2_destroy.argtypes = [vp]
        L.dflash2_draft_block.argtypes = [vp, i32] + [vp] * 12
        L.dflash2_select.argtypes = [vp, i32] + [vp] * 13
        L.dflash2_verify.argtypes = [vp, i32] + [vp] * 14
        L.dflash2_advance.argtypes = [vp, i32] + [vp] * 7
        L.dflash2_block_width.argtypes = [vp, i32, vp, vp, i32, i32, vp, vp]
        L.dflash2_set_select_mode.argtypes = [vp, i32]
        L.dflash2_head_topk.argtypes = [vp, i32] + [vp] * 5
        L.dflash2_head_topk.restype = i32
        L.dflash2_head_topk_noalloc.argtypes = [vp, i32, i32, i32] + [vp] * 5
        L.dflash2_head_topk_noalloc.restype = i32
        L.dflash2_launch_count.argtypes = [vp]
        L.dflash2_launch_count.restype = i64
        L.dflash2_set_lmhead_events.argtypes = [vp, vp, vp]
        L.dflash2_lmhead_bytes.argtypes = [vp, i32]
        L.dflash2_lmhead_bytes.restype = i64
        L.dflash2_tree_build.argtypes = [vp, i32, i32] + [vp] * 12
        L.dflash2_tree_build.restype = i32
        L.dflash2_tree_verify.argtypes = [vp, i32, i32] + [vp] * 9
        L.dflash2_tree_verify.restype = i32
        L.dflash2_set_projection_events.argtypes = [vp, vp, i32]
        L.dflash2_set_projection_events.restype = i32
        L.dflash2_projection_launches.argtypes = [vp]
        L.dflash2_projection_launches.restype = i32
        L.dflash2_projection_bytes.argtypes = [vp]
        L.dflash2_projection_bytes.restype = i64
        L.dflash2_debug_set_pipeline_error.argtypes = [vp, vp]
        L.dflash2_debug_set_pipeline_error.restype = i32
        L.dflash2_debug_noalloc_inject_error.argtypes = [i32]
        L.dflash2_debug_noalloc_inject_error.restype = i32
        L.dflash2_step.argtypes = [vp, ctypes.POINTER(StepArgs), vp]
        L.dflash2_step.restype = i32
        L.dflash2_step_graphs_clear.argtypes = [vp]
        L.dflash2_step_graphs_clear.restype = i32
        L.dflash2_status_string.argtypes = [i32]
        L.dflash2_status_string.restype = ctypes.c_char_p
        for f in ("dflash2_create", "dflash2_destroy", "dflash2_draft_block", "dflash2_select", "dflash2_verify",
                  "dflash2_advance", "dflash2_set_select_mode",
                  "dflash2_set_lmhead_events"):
            getattr(L, f).restype = i32
        _lib = L
    return _lib


def _status_string(s: int) -> str:
    try:
        return lib().dflash2_status_string(s).decode()
    except Exception:  # noqa: BLE001 - message only
        return "?"


def _check(s: int, what: str):
    if s != OK:
        raise Dflash2Error(s, what)


def _p(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


# ----------------------------------------------------------------------------- C entry points

def dflash2_create(cfg: Config, weights: Weights, max_requests: int, kv_capacity: int) -> int:
    h = ctypes.c_void_p()
    _check(lib().dflash2_create(ctypes.byref(cfg), ctypes.byref(weights), max_requests, kv_capacity, ctypes.byref(h)),
           "dflash2_create")
    return h.value


def dflash2_destroy(h: int):
    _check(lib().dflash2_destroy(h), "dflash2_destroy")


def dflash2_draft_block(h, n_req, anchor_ids, ctx_len, n_new, taps, k_cache, v_cache, cand_ids, cand_logits, gate,
                        logits_out=None, width=None, stream=None):
    _check(lib().dflash2_draft_block(h, n_req, _p(anchor_ids), _p(ctx_len), _p(n_new), _p(taps), _p(k_cache),
                                     _p(v_cache), _p(cand_ids), _p(cand_logits), _p(gate), _p(logits_out),
                                     _p(width), _stream(stream)), "dflash2_draft_block")


def dflash2_select(h, n_req, anchor_ids, cand_ids, cand_logits, gate, temperature, seed, philox_offset, path, q_rows,
                   scores_out, status, width=None, stream=None):
    _check(lib().dflash2_select(h, n_req, _p(anchor_ids), _p(cand_ids), _p(cand_logits), _p(gate), _p(temperature),
                                _p(seed), _p(philox_offset), _p(path), _p(q_rows), _p(scores_out), _p(status),
                                _p(width), _stream(stream)), "dflash2_select")


def dflash2_verify(h, n_req, target_logits, path, cand_ids, q_rows, temperature, seed, philox_offset, n_accepted,
                   emitted, n_emitted, probs_out, status, width=None, stream=None):
    _check(lib().dflash2_verify(h, n_req, _p(target_logits), _p(path), _p(cand_ids), _p(q_rows), _p(temperature),
                                _p(seed), _p(philox_offset), _p(n_accepted), _p(emitted), _p(n_emitted),
                                _p(probs_out), _p(status), _p(width), _stream(stream)), "dflash2_verify")


def dflash2_tree_build(h, n_req, budget, anchor_ids, cand_ids, cand_logits, gate, node_token, node_parent, node_depth,
                       node_score, n_nodes, scores_out, status, stream=None):
    _check(lib().dflash2_tree_build(h, n_req, budget, _p(anchor_ids), _p(cand_ids), _p(cand_logits), _p(gate),
                                    _p(node_token), _p(node_parent), _p(node_depth), _p(node_score), _p(n_nodes),
                                    _p(scores_out), _p(status), _stream(stream)), "dflash2_tree_build")


def dflash2_tree_verify(h, n_req, budget, target_logits, node_token, node_parent, n_nodes, n_accepted, emitted,
                        n_emitted, status, stream=None):
    _check(lib().dflash2_tree_verify(h, n_req, budget, _p(target_logits), _p(node_token), _p(node_parent),
                                     _p(n_nodes), _p(n_accepted), _p(emitted), _p(n_emitted), _p(status),
                                     _stream(stream)), "dflash2_tree_verify")


def dflash2_step(h, n_req, anchor_ids, ctx_len, n_new, taps, k_cache, v_cache, cand_ids, cand_logits, gate,
                 temperature, seed, philox_offset, path, q_rows, status, target_logits, n_accepted, emitted,
                 n_emitted, width=None, stream=None):
    """One draft + select + verify step, replayed from the handle's CUDA graph of this
    argument set after its first call (dflash2.h, dflash2_step)."""
    a = StepArgs(n_req, _p(anchor_ids), _p(ctx_len), _p(n_new), _p(taps), _p(k_cache), _p(v_cache), _p(cand_ids),
                 _p(cand_logits), _p(gate), _p(temperature), _p(seed), _p(philox_offset), _p(path), _p(q_rows),
                 _p(status), _p(target_logits), _p(n_accepted), _p(emitted), _p(n_emitted), _p(width))
    _check(lib().dflash2_step(h, ctypes.byref(a), _stream(stream)), "dflash2_step")


def dflash2_step_graphs_clear(h):
    _check(lib().dflash2_step_graphs_clear(h), "dflash2_step_graphs_clear")


def dflash2_set_select_mode(h, mode: int):
    _check(lib().dflash2_set_select_mode(h, mode), "dflash2_set_select_mode")


def dflash2_advance(h, n_req, emitted, n_emitted, anchor_ids, ctx_len, n_new, philox_offset, stream=None):
    _check(lib().dflash2_advance(h, n_req, _p(emitted), _p(n_emitted), _p(anchor_ids), _p(ctx_len), _p(n_new),
                                 _p(philox_offset), _stream(stream)), "dflash2_advance")


def dflash2_block_width(h, n_req, ctx_len, n_new, ctx_threshold: int, narrow_width: int, width, stream=None):
    _check(lib().dflash2_block_width(h, n_req, _p(ctx_len), _p(n_new), ctx_threshold, narrow_width, _p(width),
                                     _stream(stream)), "dflash2_block_width")


def dflash2_head_topk(h, n_rows, hidden, cand_ids, cand_logits, logits_out=None, stream=None):
    _check(lib().dflash2_head_topk(h, n_rows, _p(hidden), _p(cand_ids), _p(cand_logits), _p(logits_out),
                                   _stream(stream)), "dflash2_head_topk")


def dflash2_head_topk_noalloc(lm_head, vocab, hidden_dim, n_rows, hidden, cand_ids, cand_logits, logits_out=None,
                              stream=None):
    """LM head + top-16 that allocates nothing: for callers that cannot call
    cudaMalloc (its scratch is a fixed device array inside the library)."""
    _check(lib().dflash2_head_topk_noalloc(_p(lm_head), vocab, hidden_dim, n_rows, _p(hidden), _p(cand_ids),
                                           _p(cand_logits), _p(logits_out), _stream(stream)),
           "dflash2_head_topk_noalloc")


def dflash2_debug_set_pipeline_error(h, stream=None):
    _check(lib().dflash2_debug_set_pipeline_error(h, _stream(stream)), "dflash2_debug_set_pipeline_error")


def dflash2_debug_noalloc_inject_error(on: bool):
    _check(lib().dflash2_debug_noalloc_inject_error(1 if on else 0), "dflash2_debug_noalloc_inject_error")


def dflash2_launch_count(h) -> int:
    return int(lib().dflash2_launch_count(h))


def dflash2_set_lmhead_events(h, start, stop):
    _check(lib().dflash2_set_lmhead_events(h, start.cuda_event if start is not None else None,
                                           stop.cuda_event if stop is not None else None),
           "dflash2_set_lmhead_events")


def dflash2_set_projection_events(h, events):
    """events: a flat list of torch.cuda.Event (start, stop, start, stop, ...), already
    created on the device (recorded once), or None.  The ctypes array is kept on the
    binding while set."""
    global _proj_events_keep
    if events is None:
        _proj_events_keep = None
        _check(lib().dflash2_set_projection_events(h, None, 0), "dflash2_set_projection_events")
        return
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _proj_events_keep = arr
    _check(lib().dflash2_set_projection_events(h, ctypes.cast(arr, ctypes.c_void_p), len(events) // 2),
           "dflash2_set_projection_events")


_proj_events_keep = None


def dflash2_projection_launches(h) -> int:
    return int(lib().dflash2_projection_launches(h))


def dflash2_projection_bytes(h) -> int:
    return int(lib().dflash2_projection_bytes(h))


def dflash2_lmhead_bytes(h, n_req) -> int:
    return int(lib().dflash2_lmhead_bytes(h, n_req))


# ----------------------------------------------------------------------------- convenience

def make_config(geom, weight_format: str) -> Config:
    c = Config()
    for n in ("hidden", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "n_taps", "block",
              "top_k", "rank", "window", "conv_taps", "conv_group"):
        setattr(c, n, getattr(geom, n))
    c.mask_token_id = geom.mask_id
    c.weight_format = WEIGHTS_BF16 if weight_format == "bf16" else WEIGHTS_Q8G64
    c.rope_theta = geom.rope_theta
    c.rms_eps = geom.rms_eps
    return c


def upload_weights(W: Dict[str, object], device="cuda"):
    """Copies a weight dict (numpy, layout of workloads.gen) to the device.  Returns
    (dict of torch tensors keeping them alive, ctypes Weights)."""
    import numpy as np
    import torch

    keep = {}

    def dev(name, arr):
        a = np.ascontiguousarray(arr)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        t = torch.from_numpy(a).to(device)
        keep[name] = t
        return t.data_ptr()

    def mat(name, m):
        x = Matrix()
        if m["kind"] == "bf16":
            x.w = dev(name, m["w"])
        else:
            x.w = dev(name + ".codes", m["codes"])
            x.scale = dev(name + ".scale", m["scale"])
            x.bias = dev(name + ".bias", m["bias"])
        return x

    w = Weights()
    for n in ("embed", "lm_head", "hidden_norm", "final_norm"):
        setattr(w, n, dev(n, W[n]))
    for n in ("fc", "sel_proj", "cb_a", "cb_b"):
        setattr(w, n, mat(n, W[n]))
    l = 0
    while f"l{l}.q" in W:
        L = w.layers[l]
        p = f"l{l}."
        for n in ("input_norm", "post_norm", "q_norm", "k_norm", "attn_base", "mlp_base"):
            setattr(L, n, dev(p + n, W[p + n]))
        for n in _LAYER_MATS:
            setattr(L, n, mat(p + n, W[p + n]))
        l += 1
    return keep, w


class Drafter:
    """Owns a handle and the device weights of one synthetic drafter."""

    def __init__(self, geom, weight_format: str, W: Dict[str, object], max_requests: int, kv_capacity: int):
        self.geom = geom
        self.cfg = make_config(geom, weight_format)
        self._keep, self._w = upload_weights(W)
        self.max_requests = max_requests
        self.kv_capacity = kv_capacity
        self.handle = dflash2_create(self.cfg, self._w, max_requests, kv_capacity)

    def close(self):
        if self.handle:
            dflash2_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001
            pass
