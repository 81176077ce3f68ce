"""The no-allocation index transpose, through the C ABI.

llsa_index_transpose_noalloc serves callers that cannot allocate device
memory or hand the library a workspace (an allocator-free runtime, code living
inside another owner's memory pool or budget). Its scratch sits in a fixed
device array inside the library, shared by every call. These checks call it
twice in a row on different selections and compare each result with the
workspace-taking llsa_index_transpose (bit-exact, the transpose's own
tolerance), so leftovers of the first call would show in the second; and they
check that sizes beyond the fixed array are refused. This file is named to be
collected last.
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


def _random_selection(p, seed):
    s = llsa.get_sizes(p)
    g = torch.Generator().manual_seed(seed)
    rows = [torch.randperm(s.n_blocks, generator=g)[:s.topk_level[1]].sort().values
            for _ in range(s.slices * s.n_blocks)]
    return torch.stack(rows).view(s.slices, s.n_blocks, s.topk_level[1]).to(torch.int32).cuda()


def test_noalloc_matches_workspace_transpose_twice():
    fn = _noalloc_fn()
    p = llsa.Params(2, 3, 16384, 64, topk=8)
    s = llsa.get_sizes(p)
    stream = torch.cuda.current_stream().cuda_stream
    for seed in (1, 2):
        sel = _random_selection(p, seed)
        ref_ptr = torch.empty((s.slices, s.n_blocks + 1), dtype=torch.int32, device="cuda")
        ref_idx = torch.empty((s.slices, s.n_blocks * s.topk_level[1]), dtype=torch.int32, device="cuda")
        ws = torch.empty(llsa.workspace_bytes(p, llsa.OP_TRANSPOSE), dtype=torch.uint8, device="cuda")
        llsa.llsa_index_transpose(p, sel, ref_ptr, ref_idx, ws)
        col_ptr = torch.full_like(ref_ptr, -1)
        row_idx = torch.full_like(ref_idx, -1)
        rc = fn(ctypes.byref(p.c()), sel.data_ptr(), col_ptr.data_ptr(), row_idx.data_ptr(), stream)
        assert rc == 0, llsa.strerror(rc)
        torch.cuda.synchronize()
        assert torch.equal(col_ptr, ref_ptr)
        assert torch.equal(row_idx, ref_idx)
        # and the result is the transpose: every (row, column) entry appears once
        cp, ri, sl = col_ptr.cpu().numpy(), row_idx.cpu().numpy(), sel.cpu().numpy()
        for b in range(s.slices):
            cols = np.repeat(np.arange(s.n_blocks), np.diff(cp[b]))
            pairs = set(zip(ri[b].tolist(), cols.tolist()))
            assert len(pairs) == sl[b].size
            assert all((i, int(j)) in pairs for i in range(0, s.n_blocks, 97) for j in sl[b, i])
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
