"""Log-linear Sparse Attention (LLSA) for GB300 (sm_103a): Python binding.

A thin ctypes layer over the C ABI of ``include/llsa.h`` (libllsa.so, built
in-tree by ``build.build()``). The functions keep the C names -- ``llsa_pool``,
``llsa_select``, ``llsa_fwd``, ``llsa_index_transpose``, ``llsa_bwd`` -- and do
argument marshalling only: every step of the computation runs in the
library's CUDA kernels on the caller's current torch stream. PyTorch supplies
device memory and streams. There is no CPU fallback: if the library is not
built or the device is not a GB300, calls raise.

Method: "Trainable Log-linear Sparse Attention for Efficient Diffusion
Transformers" (arXiv 2512.16615), as described on its Pith review page
("Core claim", "What carries the argument").
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libllsa.so")
_lib = None

LLSA_DTYPE_BF16, LLSA_DTYPE_F32 = 0, 1
LLSA_ENRICH_TOP1 = 0
LLSA_ENRICH_ANCESTOR = 1
LLSA_ENRICH_ALLK = 2
_RULES = {"top1": LLSA_ENRICH_TOP1, "ancestor": LLSA_ENRICH_ANCESTOR, "allk": LLSA_ENRICH_ALLK}
LLSA_ORDER_TILE, LLSA_ORDER_RASTER = 0, 1
_ORDERS = {"tile": LLSA_ORDER_TILE, "raster": LLSA_ORDER_RASTER}
OP_POOL, OP_SELECT, OP_FWD, OP_TRANSPOSE, OP_BWD = range(5)
MAX_LEVELS = 8


class LLSAError(RuntimeError):
    """A negative LLSA_* status from the library."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (code {code})")


class _Params(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("heads", ctypes.c_int), ("n", ctypes.c_int), ("d", ctypes.c_int),
                ("block", ctypes.c_int), ("levels", ctypes.c_int), ("topk", ctypes.c_int),
                ("enrich_levels", ctypes.c_int), ("dtype", ctypes.c_int), ("scale", ctypes.c_float),
                ("enrich_rule", ctypes.c_int), ("token_order", ctypes.c_int)]


class _Sizes(ctypes.Structure):
    _fields_ = [("levels", ctypes.c_int), ("enrich_levels", ctypes.c_int),
                ("n_level", ctypes.c_int * (MAX_LEVELS + 1)), ("topk_level", ctypes.c_int * (MAX_LEVELS + 1)),
                ("row_offset", ctypes.c_int * (MAX_LEVELS + 1)), ("pyr_rows", ctypes.c_int),
                ("n_blocks", ctypes.c_int), ("keys_per_query", ctypes.c_int), ("slices", ctypes.c_longlong),
                ("level_idx_offset", ctypes.c_longlong * (MAX_LEVELS + 1)),
                ("level_idx_per_slice", ctypes.c_longlong), ("scale", ctypes.c_float),
                ("coarse_cols", ctypes.c_int), ("enrich_cols", ctypes.c_int)]


def lib_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"LLSA CUDA library not built ({_LIB_PATH}); run "
                           "hierarchical_sparse_attention_mean_gb300.build.build()")
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.POINTER(_Params)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    lib.llsa_get_sizes.argtypes = [P, ctypes.POINTER(_Sizes)]
    lib.llsa_workspace_bytes.argtypes = [P, ctypes.c_int]
    lib.llsa_workspace_bytes.restype = sz
    lib.llsa_pool.argtypes = [P, vp, vp, vp, vp, vp, sz, vp]
    lib.llsa_select.argtypes = [P, vp, vp, vp, vp, vp, sz, vp]
    lib.llsa_fwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.llsa_index_transpose.argtypes = [P, vp, vp, vp, vp, sz, vp]
    lib.llsa_reorder.argtypes = [P, ctypes.c_int, ctypes.c_int, vp, vp, ctypes.c_int, vp]
    lib.llsa_select_exhaustive.argtypes = [P, vp, vp, vp]
    lib.llsa_bwd.argtypes = [P] + [vp] * 14 + [vp, sz, vp]
    lib.llsa_get_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    lib.llsa_strerror.argtypes = [ctypes.c_int]
    lib.llsa_strerror.restype = ctypes.c_char_p
    lib.llsa_launch_count.restype = ctypes.c_ulonglong
    lib.llsa_test_set_wait_limit.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.llsa_profile_enable.argtypes = [ctypes.c_int]
    lib.llsa_profile_only.argtypes = [ctypes.c_char_p]
    lib.llsa_profile_read.argtypes = [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float), ctypes.c_int]
    _lib = lib
    return lib


def strerror(code: int) -> str:
    return _load().llsa_strerror(code).decode()


def _check(rc: int, where: str):
    if rc != 0:
        raise LLSAError(rc, where)


@dataclass(frozen=True)
class Params:
    """Problem description; mirrors llsa_params of include/llsa.h."""
    batch: int
    heads: int
    n: int
    d: int
    block: int = 16
    topk: int = 8
    levels: int = 0            # 0: floor(log_B n - 1)
    enrich_levels: int = -1    # -1: all levels; 0: no enrichment
    dtype: str = "bf16"        # "bf16" or "fp32"
    scale: float = 0.0         # 0: 1/sqrt(d)
    enrich_rule: str = "top1"  # "top1", "ancestor" or "allk"
    token_order: str = "tile"  # "tile" or "raster" (raster order of a square image)

    def c(self) -> _Params:
        dt = {"bf16": LLSA_DTYPE_BF16, "fp32": LLSA_DTYPE_F32}.get(self.dtype)
        if dt is None:
            raise ValueError(f"dtype must be 'bf16' or 'fp32', not {self.dtype!r}")
        rule = _RULES.get(self.enrich_rule)
        if rule is None:
            raise ValueError(f"enrich_rule must be 'top1', 'ancestor' or 'allk', not {self.enrich_rule!r}")
        order = _ORDERS.get(self.token_order)
        if order is None:
            raise ValueError(f"token_order must be 'tile' or 'raster', not {self.token_order!r}")
        return _Params(self.batch, self.heads, self.n, self.d, self.block, self.levels, self.topk,
                       self.enrich_levels, dt, self.scale, rule, order)

    @staticmethod
    def like(q, **kw) -> "Params":
        import torch
        b, h, n, d = q.shape
        dtype = {torch.bfloat16: "bf16", torch.float32: "fp32"}.get(q.dtype)
        if dtype is None:
            raise ValueError("q must be bfloat16 or float32")
        return Params(b, h, n, d, dtype=dtype, **kw)


@dataclass(frozen=True)
class Sizes:
    levels: int
    enrich_levels: int
    n_level: tuple
    topk_level: tuple
    row_offset: tuple
    pyr_rows: int
    n_blocks: int
    keys_per_query: int
    slices: int
    level_idx_offset: tuple
    level_idx_per_slice: int
    scale: float
    coarse_cols: int   # entries per coarse_idx row (levels 1..L)
    enrich_cols: int   # coarse keys per query (columns of levels 1..L_e)


def get_sizes(p: Params) -> Sizes:
    s = _Sizes()
    _check(_load().llsa_get_sizes(ctypes.byref(p.c()), ctypes.byref(s)), "llsa_get_sizes")
    L = s.levels
    return Sizes(L, s.enrich_levels, tuple(s.n_level[:L + 1]), tuple(s.topk_level[:L + 1]),
                 tuple(s.row_offset[:L + 1]), s.pyr_rows, s.n_blocks, s.keys_per_query, s.slices,
                 tuple(s.level_idx_offset[:L + 1]), s.level_idx_per_slice, s.scale, s.coarse_cols, s.enrich_cols)


def workspace_bytes(p: Params, op: int) -> int:
    return int(_load().llsa_workspace_bytes(ctypes.byref(p.c()), op))


def _ptr(t, name, dtype=None):
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ws(ws):
    if ws is None:
        return None, 0
    return _ptr(ws, "ws"), ws.numel() * ws.element_size()


def _tok_dtype(p: Params):
    import torch
    return torch.bfloat16 if p.dtype == "bf16" else torch.float32


# ------------------------------------------------------------------ C calls

def llsa_pool(p: Params, q, k, v, pyr, ws=None, stream=None):
    import torch
    td = _tok_dtype(p)
    w, wb = _ws(ws)
    _check(_load().llsa_pool(ctypes.byref(p.c()), _ptr(q, "q", td), _ptr(k, "k", td), _ptr(v, "v", td),
                             _ptr(pyr, "pyr", torch.float32), w, wb, _stream(stream)), "llsa_pool")


def llsa_select(p: Params, pyr, sel_idx, coarse_idx, level_idx=None, ws=None, stream=None):
    import torch
    w, wb = _ws(ws)
    _check(_load().llsa_select(ctypes.byref(p.c()), _ptr(pyr, "pyr", torch.float32),
                               _ptr(sel_idx, "sel_idx", torch.int32), _ptr(coarse_idx, "coarse_idx", torch.int32),
                               _ptr(level_idx, "level_idx", torch.int32), w, wb, _stream(stream)), "llsa_select")


def llsa_fwd(p: Params, q, k, v, pyr, sel_idx, coarse_idx, o, lse, ws=None, stream=None):
    import torch
    td = _tok_dtype(p)
    w, wb = _ws(ws)
    _check(_load().llsa_fwd(ctypes.byref(p.c()), _ptr(q, "q", td), _ptr(k, "k", td), _ptr(v, "v", td),
                            _ptr(pyr, "pyr", torch.float32), _ptr(sel_idx, "sel_idx", torch.int32),
                            _ptr(coarse_idx, "coarse_idx", torch.int32), _ptr(o, "o", td),
                            _ptr(lse, "lse", torch.float32), w, wb, _stream(stream)), "llsa_fwd")


def llsa_index_transpose(p: Params, sel_idx, col_ptr, row_idx, ws, stream=None):
    import torch
    w, wb = _ws(ws)
    _check(_load().llsa_index_transpose(ctypes.byref(p.c()), _ptr(sel_idx, "sel_idx", torch.int32),
                                        _ptr(col_ptr, "col_ptr", torch.int32), _ptr(row_idx, "row_idx", torch.int32),
                                        w, wb, _stream(stream)), "llsa_index_transpose")


def llsa_select_exhaustive(p: Params, pyr, sel_idx, stream=None):
    """Exhaustive level-1 Top-K: sel_idx int32 [batch*heads, T, min(K, T)]."""
    import torch
    _check(_load().llsa_select_exhaustive(ctypes.byref(p.c()), _ptr(pyr, "pyr", torch.float32),
                                          _ptr(sel_idx, "sel_idx", torch.int32), _stream(stream)),
           "llsa_select_exhaustive")


def routing_recall(hier_sel, exhaustive_sel) -> float:
    """Share of the exhaustive level-1 Top-K entries that the hierarchical
    selection also holds, over all rows (both int32 [.., T, K] tensors)."""
    import torch
    h = hier_sel.reshape(-1, hier_sel.shape[-1]).long()
    e = exhaustive_sel.reshape(-1, exhaustive_sel.shape[-1]).long()
    hit = (e[:, :, None] == h[:, None, :]).any(-1)
    return float(hit.double().mean())


def llsa_reorder(p: Params, height: int, width: int, x, out, inverse: bool = False, stream=None):
    """Hierarchical tile order of the N = height * width tokens of x
    [batch, heads, N, d] into out (inverse=True maps back to raster order)."""
    td = _tok_dtype(p)
    _check(_load().llsa_reorder(ctypes.byref(p.c()), int(height), int(width), _ptr(x, "x", td), _ptr(out, "out", td),
                                1 if inverse else 0, _stream(stream)), "llsa_reorder")


def llsa_bwd(p: Params, q, k, v, o, lse, dout, pyr, sel_idx, coarse_idx, col_ptr, row_idx, dq, dk, dv, ws,
             stream=None):
    import torch
    td = _tok_dtype(p)
    w, wb = _ws(ws)
    i32, f32 = torch.int32, torch.float32
    _check(_load().llsa_bwd(ctypes.byref(p.c()), _ptr(q, "q", td), _ptr(k, "k", td), _ptr(v, "v", td),
                            _ptr(o, "o", td), _ptr(lse, "lse", f32), _ptr(dout, "dout", td), _ptr(pyr, "pyr", f32),
                            _ptr(sel_idx, "sel_idx", i32), _ptr(coarse_idx, "coarse_idx", i32),
                            _ptr(col_ptr, "col_ptr", i32), _ptr(row_idx, "row_idx", i32), _ptr(dq, "dq", td),
                            _ptr(dk, "dk", td), _ptr(dv, "dv", td), w, wb, _stream(stream)), "llsa_bwd")


def llsa_get_status(stream=None) -> int:
    st = ctypes.c_int(0)
    _check(_load().llsa_get_status(_stream(stream), ctypes.byref(st)), "llsa_get_status")
    return st.value


LLSA_TEST_NO_COPIES = 1
LLSA_TEST_FORCE_GROUPED = 2
LLSA_TEST_FORCE_PER_BLOCK = 4


def test_set_wait_limit(polls: int = 0, flags: int = 0):
    """Test hook (llsa_test_set_wait_limit): polls before a bounded device wait
    gives up (0: the kernels' own limit) and test switches
    (LLSA_TEST_NO_COPIES: the copy warps issue nothing; LLSA_TEST_FORCE_GROUPED
    / LLSA_TEST_FORCE_PER_BLOCK: which tensor-core forward llsa_fwd takes)."""
    _check(_load().llsa_test_set_wait_limit(int(polls), int(flags)), "llsa_test_set_wait_limit")


def llsa_launch_count() -> int:
    return int(_load().llsa_launch_count())


def profile_enable(on: bool = True):
    _load().llsa_profile_enable(1 if on else 0)


def profile_reset():
    _load().llsa_profile_reset()


def profile_only(prefix: str | None = None):
    """Time only kernels whose name starts with `prefix` (None: all)."""
    _load().llsa_profile_only(prefix.encode() if prefix else None)


def profile_read(cap: int = 4096):
    names = (ctypes.c_char_p * cap)()
    ms = (ctypes.c_float * cap)()
    n = _load().llsa_profile_read(names, ms, cap)
    return [(names[i].decode(), float(ms[i])) for i in range(n)]


# ------------------------------------------------------- buffer management

class Buffers:
    """Device buffers of one problem (allocated by torch, owned here)."""

    def __init__(self, p: Params, device="cuda"):
        import torch
        s = get_sizes(p)
        self.p, self.s = p, s
        bh = s.slices
        dev = torch.device(device)
        td = _tok_dtype(p)
        self.pyr = torch.empty((3, bh, s.pyr_rows, p.d), dtype=torch.float32, device=dev)
        self.sel_idx = torch.empty((bh, s.n_blocks, s.topk_level[1]), dtype=torch.int32, device=dev)
        self.coarse_idx = torch.empty((bh, s.n_blocks, s.coarse_cols), dtype=torch.int32, device=dev)
        self.level_idx = torch.empty((bh, max(1, s.level_idx_per_slice)), dtype=torch.int32, device=dev)
        self.o = torch.empty((p.batch, p.heads, p.n, p.d), dtype=td, device=dev)
        self.lse = torch.empty((p.batch, p.heads, p.n), dtype=torch.float32, device=dev)
        self.col_ptr = torch.empty((bh, s.n_blocks + 1), dtype=torch.int32, device=dev)
        self.row_idx = torch.empty((bh, s.n_blocks * s.topk_level[1]), dtype=torch.int32, device=dev)
        self.ws_f = torch.empty(max(16, workspace_bytes(p, OP_FWD)), dtype=torch.uint8, device=dev)
        self.ws_t = torch.empty(max(16, workspace_bytes(p, OP_TRANSPOSE)), dtype=torch.uint8, device=dev)
        self.ws_b = torch.empty(max(16, workspace_bytes(p, OP_BWD)), dtype=torch.uint8, device=dev)
        # the sparse-index transpose that forward() issues on a side stream
        self._side = None          # that stream (made on first use)
        self._sel_ready = None     # event: the selection it reads is written
        self._transposed = None    # event: col_ptr / row_idx are written
        self._pending = False      # a transpose was issued that backward() has not waited for

    def side_stream(self):
        import torch
        if self._side is None:
            self._side = torch.cuda.Stream(device=self.sel_idx.device)
            self._sel_ready = torch.cuda.Event()
            self._transposed = torch.cuda.Event()
        return self._side

    def level(self, l: int):
        """I^(l) as [bh, n_l, K_l] (l >= 2) view of level_idx; I^(1) = sel_idx."""
        if l == 1:
            return self.sel_idx
        s = self.s
        off = s.level_idx_offset[l]
        return self.level_idx[:, off:off + s.n_level[l] * s.topk_level[l]].view(-1, s.n_level[l], s.topk_level[l])


def _as_stream(stream, device):
    import torch
    if stream is None:
        return torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return stream
    return torch.cuda.ExternalStream(int(stream), device=device)


def forward(p: Params, q, k, v, bufs: Buffers | None = None, stream=None) -> Buffers:
    """pool -> select -> fwd. Returns the buffers (o, lse, indices, pyramids).

    The sparse-index transpose that backward() needs depends on the selection
    alone: it is issued here on a side stream, after select, so that it runs
    beside the forward's grouping pass; backward() waits for it."""
    b = bufs or Buffers(p, q.device)
    st = _as_stream(stream, q.device)
    if b._pending:
        st.wait_event(b._transposed)  # the previous transpose still reads sel_idx
    llsa_pool(p, q, k, v, b.pyr, stream=st)
    llsa_select(p, b.pyr, b.sel_idx, b.coarse_idx, b.level_idx, stream=st)
    side = b.side_stream()
    b._sel_ready.record(st)
    side.wait_event(b._sel_ready)
    llsa_index_transpose(p, b.sel_idx, b.col_ptr, b.row_idx, b.ws_t, stream=side)
    b._transposed.record(side)
    b._pending = True
    for t in (b.sel_idx, b.col_ptr, b.row_idx, b.ws_t):
        t.record_stream(side)  # in use there until the transpose is done
    llsa_fwd(p, q, k, v, b.pyr, b.sel_idx, b.coarse_idx, b.o, b.lse, b.ws_f, stream=st)
    return b


def backward(p: Params, q, k, v, dout, b: Buffers, dq=None, dk=None, dv=None, stream=None):
    """bwd after forward() (and its index transpose). Returns (dq, dk, dv)."""
    import torch
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    st = _as_stream(stream, q.device)
    if b._pending:
        st.wait_event(b._transposed)
        b._pending = False
    else:
        llsa_index_transpose(p, b.sel_idx, b.col_ptr, b.row_idx, b.ws_t, stream=st)
    stream = st
    llsa_bwd(p, q, k, v, b.o, b.lse, dout, b.pyr, b.sel_idx, b.coarse_idx, b.col_ptr, b.row_idx, dq, dk, dv,
             b.ws_b, stream=stream)
    return dq, dk, dv


def _autograd_function():
    import torch

    class LLSAFunction(torch.autograd.Function):
        """Differentiable LLSA over [batch, heads, N, d] tensors."""

        @staticmethod
        def forward(ctx, q, k, v, block, topk, levels, enrich_levels, scale, token_order):
            q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
            p = Params.like(q, block=block, topk=topk, levels=levels, enrich_levels=enrich_levels, scale=scale,
                            token_order=token_order)
            b = forward(p, q, k, v)
            ctx.p, ctx.b = p, b
            ctx.save_for_backward(q, k, v)
            return b.o

        @staticmethod
        def backward(ctx, do):
            q, k, v = ctx.saved_tensors
            dq, dk, dv = backward(ctx.p, q, k, v, do.contiguous(), ctx.b)
            return dq, dk, dv, None, None, None, None, None, None

    return LLSAFunction


_FN = None


def llsa_attention(q, k, v, block: int = 16, topk: int = 8, levels: int = 0, enrich_levels: int = -1,
                   scale: float = 0.0, token_order: str = "tile"):
    """Autograd entry point: o = LLSA(q, k, v). token_order "raster": q, k, v
    (and o, the gradients) are in the raster order of a square image, reordered
    inside the kernels."""
    global _FN
    if _FN is None:
        _FN = _autograd_function()
    return _FN.apply(q, k, v, block, topk, levels, enrich_levels, scale, token_order)


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)
