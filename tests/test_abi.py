"""The C-ABI library builds for sm_103a, loads, and exports every entry point the
header declares (no GPU needed: nothing is called that touches the device)."""
import ctypes
import os
import re

import pytest

import block_drafter_pos_gb300 as bd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "dflash2.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash2_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_step_calls():
    syms = declared_symbols()
    for s in ("dflash2_create", "dflash2_destroy", "dflash2_draft_block", "dflash2_select", "dflash2_verify"):
        assert s in syms


def test_library_exports_every_declared_symbol():
    lib_path = bd.build()
    lib = ctypes.CDLL(lib_path)
    for s in declared_symbols():
        assert hasattr(lib, s), s


def test_host_validation_without_device_work():
    """Bad arguments are rejected on the host before any launch."""
    lib = bd.lib()
    lib.dflash2_draft_block.argtypes = [ctypes.c_void_p, ctypes.c_int32] + [ctypes.c_void_p] * 11
    assert lib.dflash2_draft_block(None, 1, *([None] * 11)) == bd.binding.E_INVAL
    assert lib.dflash2_status_string(2) == b"nonfinite logit or selector score"
    h = ctypes.c_void_p()
    cfg = bd.binding.Config()
    w = bd.binding.Weights()
    # head_dim 64 has no kernels -> unsupported (checked before any device call)
    cfg.hidden, cfg.n_layers, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim = 512, 1, 4, 1, 64
    cfg.ffn, cfg.vocab, cfg.n_taps, cfg.block, cfg.top_k, cfg.rank = 1536, 8192, 5, 8, 16, 256
    cfg.window, cfg.conv_taps, cfg.conv_group, cfg.mask_token_id = 2048, 2, 16, 8191
    cfg.rope_theta, cfg.rms_eps = 1e7, 1e-6
    assert lib.dflash2_create(ctypes.byref(cfg), ctypes.byref(w), 1, 1024, ctypes.byref(h)) == bd.binding.E_UNSUPPORTED
    cfg.head_dim = 128
    assert lib.dflash2_create(ctypes.byref(cfg), ctypes.byref(w), 1, 1024, ctypes.byref(h)) == bd.binding.E_INVAL
