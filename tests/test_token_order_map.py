"""The raster token order's address map (token_row / block_patch in the CUDA
library's internal.h, host-callable) against the oracle's tile order: the
row token_row gives for tile position p must be the raster token the oracle's
permutation places at p, for every p of several image sizes. Built as a tiny
host program with nvcc (no GPU needed)."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "hierarchical_sparse_attention_mean_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstdlib>
#include "internal.h"
int main(int argc, char** argv) {
    const int side = atoi(argv[1]);
    const int n = side * side;
    for (long long slice = 0; slice < 2; slice++)
        for (int t = 0; t < n; t++)
            printf("%lld\n", llsa::token_row(slice, n, 1, side, t));
    return 0;
}
"""


@pytest.fixture(scope="module")
def mapper(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    d = tmp_path_factory.mktemp("tokmap")
    src, exe = d / "map.cu", d / "map"
    src.write_text(PROGRAM)
    subprocess.run([nvcc, "-std=c++17", "-I", os.path.join(ROOT, "include"), "-I", CSRC, str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    return str(exe)


@pytest.mark.parametrize("side", [4, 16, 64, 256])
def test_token_row_is_the_tile_order(mapper, side):
    out = subprocess.run([mapper, str(side)], check=True, capture_output=True, text=True).stdout.split()
    rows = np.array(out, dtype=np.int64).reshape(2, side * side)
    src = oracle.tile_order(side, side, 16)
    n = side * side
    assert np.array_equal(rows[0], src)          # slice 0: the raster token at tile position p
    assert np.array_equal(rows[1], n + src)      # slice 1: offset by one image
