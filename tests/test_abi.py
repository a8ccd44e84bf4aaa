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
    lib.dflash2_draft_block.argtypes = [ctypes.c_void_p, ctypes.c_int32] + [ctypes.c_void_p] * 12
    assert lib.dflash2_draft_block(None, 1, *([None] * 12)) == bd.binding.E_INVAL
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


def _toy_config(**kw):
    cfg = bd.binding.Config()
    cfg.hidden, cfg.n_layers, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim = 512, 1, 4, 1, 128
    cfg.ffn, cfg.vocab, cfg.n_taps, cfg.block, cfg.top_k, cfg.rank = 1536, 8192, 5, 8, 16, 256
    cfg.window, cfg.conv_taps, cfg.conv_group, cfg.mask_token_id = 2048, 2, 16, 8191
    cfg.rope_theta, cfg.rms_eps, cfg.weight_format = 1e7, 1e-6, 0
    for k, v in kw.items():
        setattr(cfg, k, v)
    return cfg


@pytest.mark.parametrize("kw,max_req,want", [
    # geometry the kernels are not instantiated for (the header's dflash2_create limits)
    (dict(hidden=384), 1, "E_UNSUPPORTED"),                    # hidden % 256
    (dict(ffn=1600), 1, "E_UNSUPPORTED"),                      # bf16: ffn % 128
    (dict(ffn=1664, weight_format=1), 1, "E_UNSUPPORTED"),     # Q8: ffn % 256
    (dict(n_q_heads=8), 1, "E_UNSUPPORTED"),                   # 4 query heads per KV head
    (dict(vocab=8200, mask_token_id=8199), 1, "E_UNSUPPORTED"),  # vocab % 16
    (dict(), 17, "E_UNSUPPORTED"),                             # more than DFLASH2_MAX_REQUESTS
    (dict(block=12), 1, "E_UNSUPPORTED"),                      # blocks of 8 or 16 only
    (dict(block=16), 9, "E_UNSUPPORTED"),                      # more than 128 block rows
    (dict(block=16, vocab=8208, mask_token_id=8207), 3, "E_UNSUPPORTED"),  # bf16 tensor-core path: 48 rows
    (dict(block=16, vocab=8208, mask_token_id=8207), 2, "E_INVAL"),       # 32 rows: GEMV path
    (dict(block=16, vocab=8208, mask_token_id=8207, weight_format=1), 2, "E_UNSUPPORTED"),  # Q8 from 32 rows
    (dict(block=16, vocab=8208, mask_token_id=8207, weight_format=1), 1, "E_INVAL"),
    (dict(vocab=8208, mask_token_id=8207), 5, "E_UNSUPPORTED"),  # tensor-core path: vocab % 128
    (dict(hidden=768, ffn=1536, n_q_heads=4), 5, "E_UNSUPPORTED"),  # tensor-core path: hidden/4 % 128
    (dict(vocab=8208, mask_token_id=8207, weight_format=1), 4, "E_UNSUPPORTED"),  # Q8 from 4 requests
    # within the limits, the next check is the (missing) weights: invalid argument
    (dict(vocab=8208, mask_token_id=8207), 4, "E_INVAL"),      # bf16 GEMV path up to 4 requests
    (dict(vocab=8208, mask_token_id=8207, weight_format=1), 3, "E_INVAL"),
    (dict(mask_token_id=8192), 1, "E_INVAL"),                  # mask id outside the vocabulary
    (dict(weight_format=2), 1, "E_INVAL"),
    (dict(window=1), 1, "E_INVAL"),
])
def test_create_geometry_limits_on_the_host(kw, max_req, want):
    """dflash2_create rejects unsupported geometry and bad arguments before any device call."""
    lib = bd.lib()
    h = ctypes.c_void_p()
    rc = lib.dflash2_create(ctypes.byref(_toy_config(**kw)), ctypes.byref(bd.binding.Weights()), max_req, 1024,
                            ctypes.byref(h))
    assert rc == getattr(bd.binding, want)
    assert not h.value


def test_entry_points_reject_a_null_handle_or_bad_sizes():
    lib = bd.lib()
    E = bd.binding.E_INVAL
    assert lib.dflash2_select(None, 1, *([None] * 13)) == E
    assert lib.dflash2_verify(None, 1, *([None] * 14)) == E
    lib.dflash2_block_width.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    assert lib.dflash2_block_width(None, 1, None, None, 8192, 8, None, None) == E
    lib.dflash2_tree_build.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32] + [ctypes.c_void_p] * 12
    lib.dflash2_tree_verify.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32] + [ctypes.c_void_p] * 9
    assert lib.dflash2_tree_build(None, 1, 12, *([None] * 12)) == E
    assert lib.dflash2_tree_verify(None, 1, 12, *([None] * 9)) == E
    assert lib.dflash2_advance(None, 1, *([None] * 7)) == E
    assert lib.dflash2_set_select_mode(None, 0) == E
    assert lib.dflash2_head_topk(None, 8, *([None] * 5)) == E
    assert lib.dflash2_destroy(None) == E
    assert lib.dflash2_step(None, None, None) == E
    assert lib.dflash2_step_graphs_clear(None) == E
    # the entry that allocates nothing: its size checks come before any device call
    buf = (ctypes.c_char * 64)()
    p = ctypes.cast(ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16, ctypes.c_void_p)
    assert lib.dflash2_head_topk_noalloc(None, 8192, 512, 8, p, p, p, None, None) == E
    assert lib.dflash2_head_topk_noalloc(p, 8192, 512, 12, p, p, p, None, None) == E     # rows % 8
    assert lib.dflash2_head_topk_noalloc(p, 8, 512, 8, p, p, p, None, None) == E         # vocab < 16
    assert lib.dflash2_head_topk_noalloc(p, 8200, 512, 8, p, p, p, None, None) == bd.binding.E_UNSUPPORTED
    assert lib.dflash2_head_topk_noalloc(p, 8192, 576, 8, p, p, p, None, None) == bd.binding.E_UNSUPPORTED


def test_stream_k_plane_map_against_brute_force(tmp_path):
    """The closed-form plane map (internal.h) that the partial-plane consumers use,
    against the stream-K partition enumerated stage by stage (host code, g++)."""
    import shutil
    import subprocess
    gxx = shutil.which("g++")
    cuda_inc = "/usr/local/cuda/include"
    if gxx is None or not os.path.exists(os.path.join(cuda_inc, "cuda.h")):
        pytest.skip("g++ or the CUDA headers are missing")
    exe = str(tmp_path / "plane_map_check")
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "block_drafter_pos_gb300", "csrc"),
                    "-I", cuda_inc, os.path.join(ROOT, "tests", "plane_map_check.cpp"), "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout
    assert out.stdout.startswith("ok ") and int(out.stdout.split()[1]) > 10000


def test_attention_part_length_rule(tmp_path):
    """The attention's context chunks per part (internal.h): the lengths measured best
    at 1, 4 and 16 requests on the drafter's geometry, and the rule's limits for every
    shape in range (host code, g++)."""
    import shutil
    import subprocess
    gxx = shutil.which("g++")
    cuda_inc = "/usr/local/cuda/include"
    if gxx is None or not os.path.exists(os.path.join(cuda_inc, "cuda.h")):
        pytest.skip("g++ or the CUDA headers are missing")
    exe = str(tmp_path / "attn_parts_check")
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "block_drafter_pos_gb300", "csrc"),
                    "-I", cuda_inc, os.path.join(ROOT, "tests", "attn_parts_check.cpp"), "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout
    assert out.stdout.startswith("ok ") and int(out.stdout.split()[1]) > 100000


def test_binding_structures_match_the_header(tmp_path):
    """The ctypes structures of the binding have the C header's sizes and field
    offsets (a small C program built with the host compiler prints them)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "abi_layout")
    subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "abi_layout.c"),
                    "-o", exe], check=True)
    got = dict(line.split() for line in subprocess.run([exe], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    b = bd.binding
    want = {
        "dflash2_config": ctypes.sizeof(b.Config),
        "dflash2_config.hidden": b.Config.hidden.offset,
        "dflash2_config.mask_token_id": b.Config.mask_token_id.offset,
        "dflash2_config.weight_format": b.Config.weight_format.offset,
        "dflash2_config.rope_theta": b.Config.rope_theta.offset,
        "dflash2_config.rms_eps": b.Config.rms_eps.offset,
        "dflash2_matrix": ctypes.sizeof(b.Matrix),
        "dflash2_layer_weights": ctypes.sizeof(b.LayerWeights),
        "dflash2_layer_weights.mlp_base": b.LayerWeights.mlp_base.offset,
        "dflash2_layer_weights.q": b.LayerWeights.q.offset,
        "dflash2_layer_weights.mlp_delta": b.LayerWeights.mlp_delta.offset,
        "dflash2_weights": ctypes.sizeof(b.Weights),
        "dflash2_weights.final_norm": b.Weights.final_norm.offset,
        "dflash2_weights.fc": b.Weights.fc.offset,
        "dflash2_weights.cb_b": b.Weights.cb_b.offset,
        "dflash2_weights.layers": b.Weights.layers.offset,
        "dflash2_step_args": ctypes.sizeof(b.StepArgs),
        "dflash2_step_args.anchor_ids": b.StepArgs.anchor_ids.offset,
        "dflash2_step_args.status": b.StepArgs.status.offset,
        "dflash2_step_args.width": b.StepArgs.width.offset,
    }
    assert {k: int(v) for k, v in got.items()} == want
