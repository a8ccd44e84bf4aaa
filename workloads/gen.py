"""Seeded generators: weights, request inputs, target noise.

Every tensor is drawn from its own PCG64 stream, keyed by (seed, tensor name,
chunk index), so any chunk can be regenerated alone and generation runs on all
host cores.  BF16 tensors are returned as uint16 bit patterns; a Q8/group64
matrix as (int8 codes, uint16 bf16 scale, uint16 bf16 bias).

Weight layout (row-major [out][in] for every matrix):

  global : embed [V][H] bf16, lm_head [V][H] bf16, fc [H][n_taps*H],
           hidden_norm [H], final_norm [H], sel_proj [rank][H],
           cb_a [V][rank], cb_b [V][rank]
  layer l: input_norm [H], post_norm [H], q [nq*hd][H], k [nkv*hd][H],
           v [nkv*hd][H], o [H][nq*hd], q_norm [hd], k_norm [hd],
           gate [F][H], up [F][H], down [H][F],
           attn_delta [2*taps*G][H], attn_base [2*taps][H],
           mlp_delta  [2*taps*G][H], mlp_base  [2*taps][H]

A delta row index is (io*taps + t)*G + g with io 0 = conv before the sublayer,
1 = conv after it; a base row is io*taps + t.
"""
from __future__ import annotations

import os
import zlib
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, List

import numpy as np

from .configs import Geometry, Workload

WEIGHT_NAMES_GLOBAL = ["embed", "lm_head", "fc", "hidden_norm", "final_norm", "sel_proj", "cb_a", "cb_b"]
WEIGHT_NAMES_LAYER = ["input_norm", "post_norm", "q", "k", "v", "o", "q_norm", "k_norm", "gate", "up",
                      "down", "attn_delta", "attn_base", "mlp_delta", "mlp_base"]
# matrices that the Q8/group64 format quantizes (49 at 5 layers); embed and lm_head stay BF16
MATRIX_NAMES = ["fc", "sel_proj", "cb_a", "cb_b", "q", "k", "v", "o", "gate", "up", "down",
                "attn_delta", "mlp_delta"]

_CHUNK = 1 << 22
_THREADS = max(1, min(32, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else 8))


def _pool():
    return ThreadPoolExecutor(_THREADS)


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    xf, of = x.reshape(-1), out.reshape(-1)

    def job(s):
        u = xf[s:s + _CHUNK].view(np.uint32)
        r = ((u >> 16) & 1) + np.uint32(0x7FFF)
        of[s:s + _CHUNK] = ((u + r) >> 16).astype(np.uint16)

    if xf.size <= _CHUNK:
        job(0)
    else:
        with _pool() as ex:
            list(ex.map(job, range(0, xf.size, _CHUNK)))
    return out


def f32_from_bf16_bits(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _key(name: str) -> int:
    return zlib.crc32(name.encode())


def normal_f32(shape, std: float, mean: float, seed: int, name: str) -> np.ndarray:
    """N(mean, std^2) float32, chunked by _CHUNK elements, each chunk its own stream."""
    n = int(np.prod(shape))
    out = np.empty(n, np.float32)

    def job(ci):
        s = ci * _CHUNK
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _key(name), ci])))
        v = out[s:s + _CHUNK]
        g.standard_normal(out=v, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        if mean != 0.0:
            v += np.float32(mean)

    nch = (n + _CHUNK - 1) // _CHUNK
    if nch == 1:
        job(0)
    else:
        with _pool() as ex:
            list(ex.map(job, range(nch)))
    return out.reshape(shape)


def quantize_q8g64(w_bits: np.ndarray):
    """Affine Q8 with groups of 64 along the input dimension.

    scale = bf16((max-min)/255), bias = bf16(min + 128*scale); codes are chosen
    against the stored (rounded) scale and bias: q = clamp(rne((w-bias)/scale),
    -128, 127), q = 0 where scale = 0.  (LSE DFlash2 docs, Q8 conversion
    paragraph: affine Q8/g64, BF16 scale and bias, codes against stored values.)
    """
    M, K = w_bits.shape
    assert K % 64 == 0
    codes = np.empty((M, K), np.int8)
    scale = np.empty((M, K // 64), np.uint16)
    bias = np.empty((M, K // 64), np.uint16)
    rows = max(1, _CHUNK // K)

    def job(r0):
        w = f32_from_bf16_bits(w_bits[r0:r0 + rows]).reshape(-1, K // 64, 64)
        mn = w.min(axis=2)
        mx = w.max(axis=2)
        s_bits = bf16_bits_from_f32((mx - mn) / np.float32(255.0))
        s = f32_from_bf16_bits(s_bits)
        b_bits = bf16_bits_from_f32(mn + np.float32(128.0) * s)
        b = f32_from_bf16_bits(b_bits)
        safe = np.where(s == 0, np.float32(1.0), s)
        q = np.rint((w - b[..., None]) / safe[..., None])
        q = np.where(s[..., None] == 0, 0.0, q)
        codes[r0:r0 + rows] = np.clip(q, -128, 127).astype(np.int8).reshape(-1, K)
        scale[r0:r0 + rows] = s_bits
        bias[r0:r0 + rows] = b_bits

    with _pool() as ex:
        list(ex.map(job, range(0, M, rows)))
    return codes, scale, bias


def _bf16_tensor(shape, std, mean, seed, name):
    return bf16_bits_from_f32(normal_f32(shape, std, mean, seed, name))


def _matrix(shape, seed, name, fmt, std=0.02):
    bits = _bf16_tensor(shape, std, 0.0, seed, name)
    if fmt == "bf16":
        return {"kind": "bf16", "w": bits}
    codes, scale, bias = quantize_q8g64(bits)
    return {"kind": "q8", "codes": codes, "scale": scale, "bias": bias}


def weight_shapes(g: Geometry) -> Dict[str, tuple]:
    H, V, r = g.hidden, g.vocab, g.rank
    shp = {
        "embed": (V, H), "lm_head": (V, H), "fc": (H, g.n_taps * H), "hidden_norm": (H,),
        "final_norm": (H,), "sel_proj": (r, H), "cb_a": (V, r), "cb_b": (V, r),
    }
    for l in range(g.n_layers):
        p = f"l{l}."
        shp.update({
            p + "input_norm": (H,), p + "post_norm": (H,), p + "q": (g.q_dim, H),
            p + "k": (g.kv_dim, H), p + "v": (g.kv_dim, H), p + "o": (H, g.q_dim),
            p + "q_norm": (g.head_dim,), p + "k_norm": (g.head_dim,), p + "gate": (g.ffn, H),
            p + "up": (g.ffn, H), p + "down": (H, g.ffn), p + "attn_delta": (g.delta_dim, H),
            p + "attn_base": (2 * g.conv_taps, H), p + "mlp_delta": (g.delta_dim, H),
            p + "mlp_base": (2 * g.conv_taps, H),
        })
    return shp


def _base_init(g: Geometry, seed: int, name: str) -> np.ndarray:
    """Conv bases: tap 0 = 1 + N(0, 0.02), other taps N(0, 0.02) (near-identity)."""
    t = g.conv_taps
    x = normal_f32((2 * t, g.hidden), 0.02, 0.0, seed, name)
    for io in range(2):
        x[io * t + 0] += np.float32(1.0)
    return bf16_bits_from_f32(x)


def make_weights(g: Geometry, fmt: str, seed: int) -> Dict[str, object]:
    """All weights of one synthetic drafter.  Matrices ~N(0, 0.02) in BF16 (then Q8/g64
    when fmt == 'q8'); norm weights 1 + N(0, 0.02); conv bases near identity."""
    assert fmt in ("bf16", "q8")
    shp = weight_shapes(g)
    W: Dict[str, object] = {}
    for name, s in shp.items():
        base = name.split(".")[-1]
        if base in ("embed", "lm_head"):
            W[name] = _bf16_tensor(s, 0.02, 0.0, seed, name)
        elif base.endswith("norm"):
            W[name] = _bf16_tensor(s, 0.02, 1.0, seed, name)
        elif base.endswith("_base"):
            W[name] = _base_init(g, seed, name)
        else:
            W[name] = _matrix(s, seed, name, fmt)
    return W


def tap_rows(g: Geometry, seed: int, req: int, positions) -> np.ndarray:
    """Target feature taps (n_taps * H floats, ~N(0,1)) for absolute context positions
    of one request.  Keyed by (seed, request, position), so any step can rebuild them."""
    out = np.empty((len(positions), g.n_taps * g.hidden), np.float32)
    for i, p in enumerate(positions):
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0x7A95, req, int(p)])))
        rng.standard_normal(out=out[i], dtype=np.float32)
    return out


def kv_rows(g: Geometry, seed: int, layer: int, req: int, lo: int, hi: int):
    """Context K and V rows [hi-lo][nkv][hd] as BF16 bits, ~N(0,1), for positions lo..hi-1.
    Rows are drawn in blocks of 256 positions, each its own stream."""
    nk = g.kv_dim
    K = np.empty((hi - lo, nk), np.float32)
    V = np.empty((hi - lo, nk), np.float32)
    for b0 in range((lo // 256) * 256, hi, 256):
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0x4B56, layer, req, b0])))
        blk = rng.standard_normal((2, 256, nk), dtype=np.float32)
        s, e = max(lo, b0), min(hi, b0 + 256)
        K[s - lo:e - lo] = blk[0, s - b0:e - b0]
        V[s - lo:e - lo] = blk[1, s - b0:e - b0]
    shp = (hi - lo, g.n_kv_heads, g.head_dim)
    return bf16_bits_from_f32(K).reshape(shp), bf16_bits_from_f32(V).reshape(shp)


def make_request_inputs(wl: Workload) -> Dict[str, object]:
    """First-step inputs: anchors, cache lengths, n_new = block, taps of the new rows,
    and the visible part of the pre-filled context cache.

    ctx_len (keys before this step's append) = ctx - block.  Only positions that
    any of the workload's steps can see (the last window + block before the
    append) are drawn; the harness fills older cache rows with a sentinel.
    """
    g = wl.geom
    R = wl.n_req
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([wl.seed, 0xA11C])))
    anchors = rng.integers(0, g.mask_id, size=R).astype(np.int32)
    n_new = np.full(R, g.block, np.int32)
    ctx_len = np.array([c - g.block for c in wl.ctx], np.int32)
    taps = np.zeros((R, g.block, g.n_taps * g.hidden), np.float32)
    for r in range(R):
        taps[r] = tap_rows(g, wl.seed, r, range(ctx_len[r], ctx_len[r] + g.block))
    kv_lo = np.maximum(0, ctx_len - (g.window + g.block)).astype(np.int32)
    kv: List[List[tuple]] = []
    for l in range(g.n_layers):
        kv.append([kv_rows(g, wl.seed, l, r, int(kv_lo[r]), int(ctx_len[r])) for r in range(R)])
    return {"anchors": anchors, "ctx_len": ctx_len, "n_new": n_new, "taps": taps,
            "kv_lo": kv_lo, "kv": kv}


def make_target_noise(wl: Workload, step: int, req: int) -> np.ndarray:
    """N(0, sigma_req^2) noise [block][V] added to drafter logits to form target logits."""
    g = wl.geom
    return normal_f32((g.block, g.vocab), wl.sigma[req], 0.0, wl.seed, f"noise/{step}/{req}")


def make_selector_inputs(V: int, R: int, seed: int, integer: bool = False, K: int = 16, P: int = 7, rank: int = 256):
    """Synthetic selector inputs shaped like a draft block's output: distinct candidate
    ids per position, candidate logits in descending order, a gate vector per position.
    integer=True draws small integers (exact in every precision, with many ties)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0x5E1])))
    anchors = rng.integers(0, V, size=R).astype(np.int32)
    cand = np.stack([np.stack([rng.choice(V, K, replace=False) for _ in range(P)]) for _ in range(R)]).astype(np.int32)
    if integer:
        cl = -np.sort(-rng.integers(-3, 4, size=(R, P, K)), axis=2).astype(np.float32)
        gate = rng.integers(-2, 3, size=(R, P, rank)).astype(np.float32)
    else:
        cl = -np.sort(-rng.normal(0, 1.4, size=(R, P, K)), axis=2).astype(np.float32)
        gate = rng.normal(0, 1.4, size=(R, P, rank)).astype(np.float32)
    return {"anchors": anchors, "cand_ids": cand, "cand_logits": cl, "gate": gate}


def make_verify_inputs(V: int, R: int, seed: int, temps, integer: bool = False, accept_depth=None, K: int = 16,
                       block: int = 8):
    """Synthetic verify inputs: target rows [R][block][V], a path through distinct
    candidate ids [R][block-1][16] with q rows [R][block-1][16].  Target rows are
    N(0, 1.5) (integers in [-4, 4] when integer=True) with the path token raised by
    `boost` on the first accept_depth[r] rows, so acceptance depths vary."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0x7E2])))
    P = block - 1
    if integer:
        z = rng.integers(-4, 5, size=(R, block, V)).astype(np.float32)
    else:
        z = rng.normal(0, 1.5, size=(R, block, V)).astype(np.float32)
    cand = np.stack([np.stack([rng.choice(V, K, replace=False) for _ in range(P)]) for _ in range(R)]).astype(np.int32)
    q = rng.dirichlet(np.ones(K) * 0.5, size=(R, P)).astype(np.float32)
    pick = rng.integers(0, K, size=(R, P))
    path = np.take_along_axis(cand, pick[..., None], axis=2)[..., 0].astype(np.int32)
    depth = accept_depth if accept_depth is not None else rng.integers(0, block, size=R)
    for r in range(R):
        for j in range(min(int(depth[r]), P)):
            z[r, j, path[r, j]] += 6.0 if not integer else 8.0
    return {"target": z, "path": path, "cand_ids": cand, "q_rows": q,
            "temps": np.asarray(temps, np.float32)}
