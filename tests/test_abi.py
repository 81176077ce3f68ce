"""The C-ABI library: it loads, exports every function include/llsa.h
declares, and validates parameters on the host (no GPU needed: these calls
fail or return before any device work)."""
import ctypes
import os
import re

import pytest

import hierarchical_sparse_attention_mean_gb300 as llsa
from hierarchical_sparse_attention_mean_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return llsa._load()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_ ]*?[\s\*]+(llsa_[a-z0-9_]+)\s*\(", text,
                                re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ("llsa_pool", "llsa_select", "llsa_fwd", "llsa_index_transpose", "llsa_bwd",
              "llsa_workspace_bytes", "llsa_get_status", "llsa_strerror"):
        assert f in names


def test_library_exports_every_declared_symbol(lib):
    cdll = ctypes.CDLL(llsa.lib_path())
    missing = [n for n in declared_functions() if not hasattr(cdll, n)]
    assert not missing, missing


def test_sizes_of_the_workloads(lib):
    cases = [  # (n, d, K, L, K1*B + L, T)
        (1024, 64, 4, 1, 65, 64),
        (4096, 64, 8, 2, 130, 256),
        (16384, 64, 8, 2, 130, 1024),
        (65536, 64, 8, 3, 131, 4096),
        (262144, 128, 16, 3, 259, 16384),
    ]
    for n, d, K, L, kpq, T in cases:
        s = llsa.get_sizes(llsa.Params(1, 2, n, d, topk=K))
        assert s.levels == L and s.keys_per_query == kpq and s.n_blocks == T
        assert s.n_level == tuple(n // 16 ** l for l in range(L + 1))
        assert abs(s.scale - d ** -0.5) < 1e-7


def test_topk_clamps_to_candidates(lib):
    s = llsa.get_sizes(llsa.Params(1, 1, 4096, 64, topk=300))
    assert s.topk_level[2] == 16 and s.topk_level[1] == 256   # full selection
    s = llsa.get_sizes(llsa.Params(1, 1, 8, 8, block=2, topk=1))   # Figure 1
    assert s.levels == 2 and s.n_level == (8, 4, 2) and s.keys_per_query == 2 + 2


@pytest.mark.parametrize("kw,code", [
    (dict(n=255), -2),             # N < B^2
    (dict(n=4096 + 16), -2),       # not divisible by B^L
    (dict(d=60), -2),              # d not a multiple of 8
    (dict(levels=3), -2),          # above floor(log_B N - 1)
    (dict(enrich_levels=5), -2),
    (dict(topk=0), -1),
    (dict(block=1), -2),
])
def test_invalid_parameters_rejected_on_host(lib, kw, code):
    base = dict(batch=1, heads=1, n=4096, d=64)
    base.update(kw)
    with pytest.raises(llsa.LLSAError) as e:
        llsa.get_sizes(llsa.Params(**base))
    assert e.value.code == code


def test_enrichment_rules(lib):
    for rule in ("top1", "ancestor"):
        s = llsa.get_sizes(llsa.Params(1, 1, 4096, 64, enrich_rule=rule))
        assert (s.keys_per_query, s.coarse_cols, s.enrich_cols) == (8 * 16 + 2, 2, 2)
    # ALLK: K_l columns per level (N = 4096, B = 16: n_2 = 16 tokens, K_2 = 8)
    s = llsa.get_sizes(llsa.Params(1, 1, 4096, 64, enrich_rule="allk"))
    assert (s.keys_per_query, s.coarse_cols, s.enrich_cols) == (8 * 16 + 16, 16, 16)
    s = llsa.get_sizes(llsa.Params(1, 1, 4096, 64, enrich_rule="allk", enrich_levels=1))
    assert (s.keys_per_query, s.coarse_cols, s.enrich_cols) == (8 * 16 + 8, 16, 8)
    # the coarsest level clamps K to its tokens: K = 32 keeps 16 at level 2
    s = llsa.get_sizes(llsa.Params(1, 1, 4096, 64, topk=32, enrich_rule="allk"))
    assert (s.coarse_cols, s.enrich_cols) == (48, 48)
    # more than 64 coarse keys per query is beyond the kernels
    with pytest.raises(llsa.LLSAError):
        llsa.get_sizes(llsa.Params(1, 1, 65536, 64, topk=32, enrich_rule="allk"))
    p = llsa.Params(1, 1, 4096, 64).c()
    p.enrich_rule = 3  # no such rule
    s = llsa._Sizes()
    assert lib.llsa_get_sizes(ctypes.byref(p), ctypes.byref(s)) == -1
    with pytest.raises(ValueError):
        llsa.Params(1, 1, 4096, 64, enrich_rule="all").c()


def test_bad_dtype_and_empty_input(lib):
    p = llsa.Params(1, 1, 4096, 64).c()
    p.dtype = 7
    assert lib.llsa_pool(ctypes.byref(p), None, None, None, None, None, 0, None) == -3
    empty = llsa.Params(0, 8, 4096, 64).c()  # batch 0: valid, nothing to do
    for f, nargs in (("llsa_pool", 7), ("llsa_select", 7), ("llsa_fwd", 11), ("llsa_index_transpose", 6)):
        assert getattr(lib, f)(ctypes.byref(empty), *([0] * nargs)) == 0
    assert lib.llsa_bwd(ctypes.byref(empty), *([0] * 17)) == 0


def test_null_and_misaligned_pointers_rejected_before_device_work(lib):
    p = llsa.Params(1, 1, 4096, 64).c()
    assert lib.llsa_pool(ctypes.byref(p), None, None, None, None, None, 0, None) == -1
    assert lib.llsa_index_transpose(ctypes.byref(p), 16, 32, 48, None, 0, None) == -6  # no workspace
    assert lib.llsa_pool(ctypes.byref(p), 16, 32, 40, 64, None, 0, None) == -4        # misaligned


def test_workspace_sizes(lib):
    p = llsa.Params(1, 12, 65536, 64)
    assert llsa.workspace_bytes(p, llsa.OP_TRANSPOSE) == 12 * 4096 * 4
    assert llsa.workspace_bytes(p, llsa.OP_BWD) > 12 * 65536 * 4
    # the grouping of query blocks: order and group list per slice, group
    # counts per window of 1024 query blocks, and a 512-byte record per group
    assert llsa.workspace_bytes(p, llsa.OP_FWD) == 2 * 12 * 4096 * 4 + 256 + 12 * 4096 * 512
    # shapes the grouped forward does not take need no forward workspace
    assert llsa.workspace_bytes(llsa.Params(1, 2, 4096, 128, topk=16), llsa.OP_FWD) == 0
    assert llsa.workspace_bytes(llsa.Params(1, 2, 1024, 64, dtype="fp32"), llsa.OP_FWD) == 0
    assert llsa.strerror(-9) == "device wait timed out"


def test_test_hook_flags(lib):
    assert lib.llsa_test_set_wait_limit(0, 8) == -1  # no such switch
    both = llsa.LLSA_TEST_FORCE_GROUPED | llsa.LLSA_TEST_FORCE_PER_BLOCK
    assert lib.llsa_test_set_wait_limit(0, both) == -1
    for f in (llsa.LLSA_TEST_FORCE_GROUPED, llsa.LLSA_TEST_FORCE_PER_BLOCK, llsa.LLSA_TEST_NO_COPIES, 0):
        assert lib.llsa_test_set_wait_limit(0, f) == 0
    assert lib.llsa_test_set_wait_limit(0, 0) == 0


def test_token_order_validation(lib):
    # raster order: B = 16 and a square image of side 4^m
    for n in (256, 4096, 65536, 1 << 20):
        s = llsa.get_sizes(llsa.Params(1, 2, n, 64, token_order="raster"))
        assert s.n_blocks == n // 16
    for kw, code in ((dict(n=1024), -2),                     # side 32 is not a power of 4
                     (dict(n=512 * 512), -2),                # nor is 512
                     (dict(n=4096, block=4, levels=2), -2),  # B != 16
                     (dict(n=2 * 4096), -2)):                # not a square
        with pytest.raises(llsa.LLSAError) as e:
            llsa.get_sizes(llsa.Params(1, 1, d=64, token_order="raster", **kw))
        assert e.value.code == code
    # raster order takes the per-query-block forward: no grouping workspace
    assert llsa.workspace_bytes(llsa.Params(1, 12, 65536, 64, token_order="raster"), llsa.OP_FWD) == 0
    p = llsa.Params(1, 1, 4096, 64).c()
    p.token_order = 2  # no such order
    assert lib.llsa_get_sizes(ctypes.byref(p), ctypes.byref(llsa._Sizes())) == -1
    with pytest.raises(ValueError):
        llsa.Params(1, 1, 4096, 64, token_order="zorder").c()
