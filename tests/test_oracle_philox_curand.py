"""Pin of the oracle's Philox4x32-10 against the cuRAND host generator (a library
implementation of the same published generator), run on the CPU."""
import os
import shutil
import subprocess
import tempfile

import pytest

from oracle import philox

HERE = os.path.dirname(os.path.abspath(__file__))


def _cuda_root():
    for d in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "curand.h")):
            return d
    return None


@pytest.fixture(scope="module")
def curand_blocks():
    root = _cuda_root()
    if root is None or shutil.which("gcc") is None:
        pytest.skip("cuRAND headers or gcc not available")
    tmp = tempfile.mkdtemp()
    exe = os.path.join(tmp, "blocks")
    subprocess.check_call(["gcc", "-O1", os.path.join(HERE, "curand_philox_blocks.c"), "-I", root + "/include",
                           "-L", root + "/lib64", "-lcurand", "-o", exe])
    env = dict(os.environ, LD_LIBRARY_PATH=root + "/lib64:" + os.environ.get("LD_LIBRARY_PATH", ""))

    def run(seed, first, n):
        out = subprocess.check_output([exe, str(seed), str(first), str(n)], env=env).decode().split()
        vals = [int(v) for v in out]
        return [tuple(vals[4 * i:4 * i + 4]) for i in range(n)]
    yield run
    shutil.rmtree(tmp, ignore_errors=True)


@pytest.mark.parametrize("seed", [0, 42, 0x123456789ABCDEF, 0xFFFFFFFFFFFFFFFF])
def test_philox_matches_curand_host(curand_blocks, seed):
    key = (seed & 0xFFFFFFFF, seed >> 32)
    # the host generator lays block b out as counter (hi lo32, hi hi32, b mod 2^16, 0)
    # with hi = b >> 16 (found by probing the library; it exercises counter words 0..2)
    for first in (0, 1000, 65530, 0xFFFFFF00, (1 << 48) + 3 * 65536 - 20):
        blocks = curand_blocks(seed, first, 40)
        for i, got in enumerate(blocks):
            b = first + i
            hi = b >> 16
            assert philox.philox4x32_10((hi & 0xFFFFFFFF, hi >> 32, b & 0xFFFF, 0), key) == got
