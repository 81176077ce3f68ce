"""The no-allocation index transpose, through the C ABI.

llsa_index_transpose_noalloc serves callers that cannot allocate device
memory or hand the library a workspace (an allocator-free runtime, code living
inside another owner's memory pool or budget). Its scratch sits in a fixed
device array inside the library, shared by every call; only the multi-kernel
form of the transpose (count, scan, scatter, order) touches it. These checks
run shapes that take that form -- a slice too large for the one-kernel form's
shared memory, and more slices than thread-block clusters resident at once --
confirm from the library's launch records that the counting kernels ran, and
compare two calls in a row on different selections with the workspace-taking
llsa_index_transpose (bit-exact, the transpose's own tolerance), so counts
left in the array by the first call would show in the second. Sizes beyond
the array are refused. This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import hierarchical_sparse_attention_mean_gb300 as llsa
from hierarchical_sparse_attention_mean_gb300 import build

pytestmark = pytest.mark.gpu

MAX_COUNTERS = 1 << 20   # LLSA_NOALLOC_TRANSPOSE_MAX_COUNTERS of include/llsa.h


def _noalloc_fn():
    build.build()
    lib = llsa._load()
    f = lib.llsa_index_transpose_noalloc
    f.argtypes = [ctypes.POINTER(llsa._Params), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def _selection(slices, T, K, seed, hot):
    """[slices, T, K] int32, K distinct blocks per row (unsorted). With hot,
    every other row picks blocks 0..K-1, so the two calls of a test leave very
    different column counts behind."""
    rng = np.random.default_rng(seed)
    w = T // K
    sel = np.arange(K)[None, None, :] * w + rng.integers(0, w, (slices, T, K))
    if hot:
        sel[:, ::2] = np.arange(K)
    sel = rng.permuted(sel, axis=2)
    return torch.from_numpy(sel.astype(np.int32)).cuda()


@pytest.mark.parametrize("shape", [(1, 1, 524288, 16, 16), (4, 16, 16384, 16, 8)],
                         ids=["T32768-too-large-for-cluster", "64-slices-beyond-resident-clusters"])
def test_noalloc_matches_workspace_transpose_twice(shape):
    fn = _noalloc_fn()
    b, h, n, B, K = shape
    p = llsa.Params(b, h, n, 64, block=B, topk=K)
    s = llsa.get_sizes(p)
    assert s.slices * s.n_blocks <= MAX_COUNTERS
    stream = torch.cuda.current_stream().cuda_stream
    for call, (seed, hot) in enumerate(((11, True), (12, False))):
        sel = _selection(s.slices, s.n_blocks, s.topk_level[1], seed, hot)
        ref_ptr = torch.empty((s.slices, s.n_blocks + 1), dtype=torch.int32, device="cuda")
        ref_idx = torch.empty((s.slices, s.n_blocks * s.topk_level[1]), dtype=torch.int32, device="cuda")
        ws = torch.empty(llsa.workspace_bytes(p, llsa.OP_TRANSPOSE), dtype=torch.uint8, device="cuda")
        llsa.llsa_index_transpose(p, sel, ref_ptr, ref_idx, ws)
        col_ptr = torch.full_like(ref_ptr, -1)
        row_idx = torch.full_like(ref_idx, -1)
        torch.cuda.synchronize()
        llsa.profile_reset()
        llsa.profile_enable(True)
        try:
            rc = fn(ctypes.byref(p.c()), sel.data_ptr(), col_ptr.data_ptr(), row_idx.data_ptr(), stream)
            torch.cuda.synchronize()
            launched = {name for name, _ in llsa.profile_read()}
        finally:
            llsa.profile_enable(False)
            llsa.profile_reset()
        assert rc == 0, llsa.strerror(rc)
        # the form that uses the fixed array ran
        assert {"transpose_count", "transpose_scatter"} <= launched, launched
        assert torch.equal(col_ptr, ref_ptr), f"call {call}: col_ptr differs"
        assert torch.equal(row_idx, ref_idx), f"call {call}: row_idx differs"
        # and the result is the transpose: every (row, column) entry appears once
        cp, ri, sl = col_ptr.cpu().numpy(), row_idx.cpu().numpy(), sel.cpu().numpy()
        for bb in range(0, s.slices, max(1, s.slices // 4)):
            cols = np.repeat(np.arange(s.n_blocks), np.diff(cp[bb]))
            pairs = set(zip(ri[bb].tolist(), cols.tolist()))
            assert len(pairs) == sl[bb].size
            assert all((i, int(j)) in pairs for i in range(0, s.n_blocks, 97) for j in sl[bb, i])
    assert llsa.llsa_get_status() == 0


def test_noalloc_refuses_sizes_beyond_its_scratch():
    fn = _noalloc_fn()
    # 65 slices x 16384 key blocks > 2^20 counters: refused before any work
    p = llsa.Params(1, 65, 262144, 64, topk=8)
    assert llsa.get_sizes(p).slices * llsa.get_sizes(p).n_blocks > MAX_COUNTERS
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    rc = fn(ctypes.byref(p.c()), dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    assert rc == -8   # LLSA_ERR_UNSUPPORTED
