"""The sparse index transpose through the C ABI against the oracle's counting
transpose, bit-exact, on selections shaped to reach every branch of the CUDA
path: spatially local rows (the pixel workloads), uniform rows, unsorted rows,
rows that all pick the same blocks (long column runs), fewer rows than the
CTAs that share a slice, and, for the multi-kernel form, a slice too large
for the one-kernel form's shared memory and more slices than clusters that
are resident at once."""
import numpy as np
import pytest
import torch

import oracle
import hierarchical_sparse_attention_mean_gb300 as llsa
from hierarchical_sparse_attention_mean_gb300 import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    oracle.build()


def _selection(slices, T, K, pattern, seed):
    """[slices, T, K] int32, K distinct entries per row in [0, T)."""
    rng = np.random.default_rng(seed)
    out = np.empty((slices, T, K), np.int64)
    for s in range(slices):
        if pattern == "local":
            side = int(round(np.sqrt(T)))
            assert side * side == T
            r = 3
            offs = np.array([(dy, dx) for dy in range(-r, r + 1) for dx in range(-r, r + 1)])
            score = rng.random((T, len(offs))) - 0.02 * (offs ** 2).sum(1)
            top = np.argsort(-score, axis=1)[:, :K]
            y, x = np.arange(T) // side, np.arange(T) % side
            out[s] = ((y[:, None] + offs[top, 0]) % side) * side + (x[:, None] + offs[top, 1]) % side
        elif pattern == "uniform":
            w = T // K
            out[s] = np.arange(K)[None, :] * w + rng.integers(0, w, (T, K))
        elif pattern == "hot":
            out[s] = np.arange(K)[None, :] + np.zeros((T, 1), np.int64)
        elif pattern == "half-hot":
            w = T // K
            out[s] = np.arange(K)[None, :] * w + rng.integers(0, w, (T, K))
            out[s, ::2] = np.arange(K)[None, :]
        else:
            raise ValueError(pattern)
        out[s] = rng.permuted(out[s], axis=1)  # rows need not be sorted
    return out.astype(np.int32)


CASES = {
    # id: (batch, heads, n, block, topk, pattern)
    "tiny-T5": (1, 3, 20, 4, 2, "uniform"),
    "n65536-K8-local": (1, 3, 65536, 16, 8, "local"),
    "n262144-K16-local": (1, 2, 262144, 16, 16, "local"),
    "n262144-K16-uniform": (1, 2, 262144, 16, 16, "uniform"),
    "n32768-K16-hot": (1, 2, 32768, 16, 16, "hot"),
    "n32768-K16-half-hot": (2, 1, 32768, 16, 16, "half-hot"),
    "n4096-B4-K3-uniform": (1, 2, 4096, 4, 3, "uniform"),
    # T = 32768 with K = 16: beyond the one-kernel form's shared memory
    "n524288-K16-multikernel": (1, 1, 524288, 16, 16, "uniform"),
    # 64 slices: more clusters than are resident at once (multi-kernel form)
    "n16384-64slices-local": (4, 16, 16384, 16, 8, "local"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_transpose_matches_oracle(name):
    b, h, n, B, K, pattern = CASES[name]
    p = llsa.Params(b, h, n, 64, block=B, topk=K)
    s = llsa.get_sizes(p)
    T, K1 = s.n_blocks, s.topk_level[1]
    assert K1 == K
    sel = _selection(s.slices, T, K1, pattern, seed=500 + list(CASES).index(name))
    col_ptr = torch.full((s.slices, T + 1), -7, dtype=torch.int32, device="cuda")
    row_idx = torch.full((s.slices, T * K1), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(16, llsa.workspace_bytes(p, llsa.OP_TRANSPOSE)), dtype=torch.uint8, device="cuda")
    llsa.llsa_index_transpose(p, torch.from_numpy(sel).cuda(), col_ptr, row_idx, ws)
    torch.cuda.synchronize()
    assert llsa.llsa_get_status() == 0
    cp, ri = col_ptr.cpu().numpy(), row_idx.cpu().numpy()
    for sl in range(s.slices):
        ref_cp, ref_ri = oracle.transpose(sel[sl], T)
        np.testing.assert_array_equal(cp[sl], ref_cp)
        np.testing.assert_array_equal(ri[sl], ref_ri)


@pytest.mark.parametrize("shape", [(1, 2, 16384, 16, 8), (1, 1, 524288, 16, 16)], ids=["cluster", "multikernel"])
def test_transpose_skips_and_reports_out_of_range_entries(shape):
    """An entry outside [0, T) is skipped by both forms and reported through
    the status word; the valid entries form the CSC (brute force over the
    input), col_ptr[T] counts them and nothing past that count is written."""
    b, h, n, B, K = shape
    p = llsa.Params(b, h, n, 64, block=B, topk=K)
    s = llsa.get_sizes(p)
    T = s.n_blocks
    sel = _selection(s.slices, T, K, "uniform", seed=900 + T)
    sel[0, 3, 2] = T + 5
    sel[-1, 10, 0] = -1
    col_ptr = torch.full((s.slices, T + 1), -7, dtype=torch.int32, device="cuda")
    row_idx = torch.full((s.slices, T * K), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(16, llsa.workspace_bytes(p, llsa.OP_TRANSPOSE)), dtype=torch.uint8, device="cuda")
    llsa.llsa_index_transpose(p, torch.from_numpy(sel).cuda(), col_ptr, row_idx, ws)
    torch.cuda.synchronize()
    assert llsa.llsa_get_status() == -10
    assert llsa.llsa_get_status() == 0
    cp, ri = col_ptr.cpu().numpy(), row_idx.cpu().numpy()
    for sl in range(s.slices):
        rows = np.repeat(np.arange(T), K)
        cols = sel[sl].reshape(-1)
        keep = (cols >= 0) & (cols < T)
        order = np.lexsort((rows[keep], cols[keep]))  # by column, then row
        ref_ri = rows[keep][order]
        ref_cp = np.concatenate([[0], np.cumsum(np.bincount(cols[keep], minlength=T))])
        np.testing.assert_array_equal(cp[sl], ref_cp)
        np.testing.assert_array_equal(ri[sl, :len(ref_ri)], ref_ri)
        assert (ri[sl, len(ref_ri):] == -7).all()
