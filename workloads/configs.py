"""Geometry and workload definitions (seeded, synthetic).

The full geometry is the DFlash2 drafter of the LSE DFlash2 docs page
("DFLASH2.md", the paragraph on the compatible drafter): 5 layers, width 5120,
32 query heads, 8 KV heads, head dim 128, FFN 17408, RoPE theta 1e7, a block of
8 positions, top-16 candidates and rank-256 selector codebooks, a 2048-key
sliding window, 2-tap dynamic convolution over groups of 16 channels.  The
vocabulary (248320) is the width of the selector codebooks and shared head
(vLLM PR #52816, "What the conv and the selector cost").

The toy geometry keeps every structural choice at a size a CPU finishes in
seconds.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Geometry:
    name: str
    hidden: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    n_taps: int = 5
    block: int = 8
    top_k: int = 16
    rank: int = 256
    window: int = 2048
    conv_taps: int = 2
    conv_group: int = 16
    rope_theta: float = 1e7
    rms_eps: float = 1e-6
    mask_token_id: int = -1          # -1: last vocabulary id

    @property
    def mask_id(self) -> int:
        return self.vocab - 1 if self.mask_token_id < 0 else self.mask_token_id

    @property
    def groups(self) -> int:
        return self.hidden // self.conv_group

    @property
    def delta_dim(self) -> int:
        # [in/out][tap][group]
        return 2 * self.conv_taps * self.groups

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim


TOY = Geometry("toy", hidden=512, n_layers=1, n_q_heads=4, n_kv_heads=1, head_dim=128,
               ffn=1536, vocab=8192)
FULL = Geometry("full", hidden=5120, n_layers=5, n_q_heads=32, n_kv_heads=8, head_dim=128,
                ffn=17408, vocab=248320)


@dataclasses.dataclass
class Workload:
    """One benchmark/parity workload.

    ctx: keys in the context cache after the first step's append (n_new = 8 on
    the first step), per request.
    temps: sampling temperature per request (0 = greedy).
    sigma: std of the Gaussian noise added to the drafter logits to make the
    synthetic target logits, per request.
    """
    name: str
    geom: Geometry
    weight_format: str               # "bf16" or "q8"
    n_req: int
    ctx: List[int]
    temps: List[float]
    sigma: List[float]
    seed: int = 0
    philox_seed: int = 0
    philox_offsets: Optional[List[int]] = None
    steps: int = 1
    description: str = ""

    @property
    def kv_capacity(self) -> int:
        need = max(self.ctx) + self.geom.block * self.steps
        return ((need + 255) // 256) * 256


def _cfg5() -> Workload:
    rng = np.random.default_rng(5)
    ctx = [int(x) for x in rng.integers(512, 32768 + 1, size=16)]
    sig = [float(x) for x in rng.uniform(0.5, 3.0, size=16)]
    temps = [[0.0, 0.7, 1.0][r % 3] for r in range(16)]
    return Workload("cfg5_q8_r16_ragged", FULL, "q8", 16, ctx, temps, sig, seed=5, philox_seed=42,
                    philox_offsets=[r << 32 for r in range(16)], steps=100,
                    description="full geometry, Q8/g64, 16 requests (128 draft rows), ctx U[512,32768], "
                                "T round-robin {0,0.7,1.0}, 100 steps with accepted-prefix append")


def _cfg4() -> Workload:
    rng = np.random.default_rng(4)
    sig = [float(x) for x in rng.uniform(0.5, 2.0, size=4)]
    return Workload("cfg4_q8_r4_ctx8192", FULL, "q8", 4, [8192] * 4, [0.7] * 4, sig, seed=4,
                    philox_seed=42, philox_offsets=[r << 32 for r in range(4)],
                    description="full geometry, Q8/g64, 4 requests, ctx 8192 (window masks old keys), T=0.7")


WORKLOADS = {
    1: Workload("cfg1_toy", TOY, "bf16", 1, [512], [0.0], [0.5], seed=0,
                description="toy: 1 layer, width 512, 4q/1kv, FFN 1536, vocab 8192, ctx 512, greedy"),
    2: Workload("cfg2_bf16_r1_ctx1024", FULL, "bf16", 1, [1024], [0.0], [1.0], seed=2,
                description="full geometry, BF16 weights, 1 request, ctx 1024, greedy"),
    3: Workload("cfg3_q8_r1_ctx2048", FULL, "q8", 1, [2048], [1.0], [1.5], seed=3, philox_seed=42,
                philox_offsets=[0],
                description="full geometry, Q8/g64 drafter, 1 request, ctx 2048, T=1.0, Philox seed 42"),
    4: _cfg4(),
    5: _cfg5(),
}


# Profiling-only workload (not one of the benchmark configurations): one layer of the
# full width with a small vocabulary, so a profiler capture holds about 1 GB.
WORKLOADS[6] = Workload("profile_one_full_layer", Geometry("full_width_1layer", hidden=5120, n_layers=1, n_q_heads=32,
                                                            n_kv_heads=8, head_dim=128, ffn=17408, vocab=16384),
                        "bf16", 1, [1024], [0.0], [1.0], seed=6,
                        description="profiling: one full-width layer, vocab 16384, 1 request, ctx 1024")


# Profiling-only workload for the tensor-core path: the same layer with 16 Q8 requests
# whose 2048-key windows are full, as in configuration 5 (about 1 GB on the device).
WORKLOADS[7] = Workload("profile_q8_r16_one_full_layer",
                        Geometry("full_width_1layer", hidden=5120, n_layers=1, n_q_heads=32, n_kv_heads=8,
                                 head_dim=128, ffn=17408, vocab=16384),
                        "q8", 16, [2048] * 16, [0.0, 0.7, 1.0, 0.0] * 4, [1.0] * 16, seed=7, philox_seed=42,
                        philox_offsets=[r << 32 for r in range(16)],
                        description="profiling: one full-width layer, vocab 16384, Q8, 16 requests, ctx 2048")


# Profiling-only workload for the one-request int8 GEMV: the same layer with one Q8
# request (about 0.6 GB on the device).
WORKLOADS[8] = Workload("profile_q8_r1_one_full_layer",
                        Geometry("full_width_1layer", hidden=5120, n_layers=1, n_q_heads=32, n_kv_heads=8,
                                 head_dim=128, ffn=17408, vocab=16384),
                        "q8", 1, [2048], [1.0], [1.5], seed=8, philox_seed=42, philox_offsets=[0],
                        description="profiling: one full-width layer, vocab 16384, Q8, 1 request, ctx 2048, T=1.0")


# The one-request BF16 workload with blocks of 16 positions (anchor + 15 masks): the
# wider draft block of the DSpark pull request's greedy-width commit, on the drafter
# geometry otherwise unchanged.
WORKLOADS[9] = Workload("cfg2_bf16_r1_ctx1024_block16", dataclasses.replace(FULL, block=16), "bf16", 1, [1024],
                        [0.0], [1.0], seed=2,
                        description="full geometry with blocks of 16, BF16 weights, 1 request, ctx 1024, greedy")


def workload(i: int) -> Workload:
    return WORKLOADS[i]
