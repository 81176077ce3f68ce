"""CPU oracle for Log-linear Sparse Attention (LLSA) -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never links, imports or
calls it, and it shares no code with the CUDA library.

The arithmetic lives in ``llsa_oracle.c`` (plain loops, fp64 throughout); this
module compiles it with gcc and wraps each entry point with ctypes. ctypes
releases the GIL during a foreign call, so independent (batch, head) slices can
run on a thread pool; ``run()`` does that.

What it follows: the Pith review page of "Trainable Log-linear Sparse Attention
for Efficient Diffusion Transformers" (arXiv 2512.16615), sections "Core claim"
and "What carries the argument", the referee report's comments on Algorithm 1,
Eq. (6) and KV Reweighting, and Figure 1. Each C function names the passage it
follows.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "llsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libllsa_oracle.so")
_lib = None

_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_ll = ctypes.c_longlong


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (strict IEEE double: no fast-math, no FMA
    contraction, so x86 and Arm produce the same bits)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    lib.orc_num_levels.argtypes = [_ll, ctypes.c_int]
    lib.orc_num_levels.restype = ctypes.c_int
    lib.orc_level_topk.argtypes = [_ll, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p]
    lib.orc_pool.argtypes = [_f32p, _ll, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f64p]
    lib.orc_select_level.argtypes = [_f64p, _f64p, _ll, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                     _i32p, _i32p, ctypes.POINTER(_ll)]
    lib.orc_pair_scores.argtypes = [_f64p, _f64p, ctypes.c_int, _i64p, _i64p, _ll, _f64p]
    lib.orc_select_all.argtypes = [_f64p, _f64p, _ll, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, _i32p, _i32p, _i32p, ctypes.POINTER(_ll)]
    lib.orc_coarse_cols.argtypes = [_ll, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    lib.orc_coarse_cols.restype = ctypes.c_int
    lib.orc_fwd.argtypes = [_f32p, _f32p, _f32p, _f64p, _f64p, _ll, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                            ctypes.c_int, ctypes.c_int, _i32p, _i32p, ctypes.c_int, _i32p, ctypes.c_double,
                            ctypes.c_void_p, _ll, _f64p, _f64p]
    lib.orc_transpose.argtypes = [_i32p, _ll, ctypes.c_int, _ll, _i32p, _i32p]
    lib.orc_bwd.argtypes = [_f32p, _f32p, _f32p, _f64p, _f64p, _f64p, _f64p, _f32p, _ll, ctypes.c_int,
                            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, _i32p,
                            ctypes.c_int, _i32p, ctypes.c_double, _f64p, _f64p, _f64p]
    lib.orc_bwd_dq_rows.argtypes = [_f32p, _f32p, _f32p, _f64p, _f64p, _f64p, _f64p, _f32p, _ll, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, _i32p,
                                    ctypes.c_int, _i32p, ctypes.c_double, _i64p, _ll, _f64p]
    lib.orc_bwd_dkv_blocks.argtypes = [_f32p, _f32p, _f32p, _f64p, _f64p, _f64p, _f64p, _f32p, _ll, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, _i32p,
                                       ctypes.c_int, _i32p, ctypes.c_double, _i64p, _ll, _f64p, _f64p]
    _lib = lib
    return lib


def _check(rc, what):
    if rc < 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")
    return rc


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


# --------------------------------------------------------------------------
# Level bookkeeping
# --------------------------------------------------------------------------

def num_levels(n: int, B: int) -> int:
    """L = floor(log_B n - 1) ("What carries the argument")."""
    return _load().orc_num_levels(n, B)


def level_sizes(n: int, B: int, L: int) -> list[int]:
    """[n_0, n_1, ..., n_L] with n_l = n / B^l."""
    out = [n]
    for _ in range(L):
        if out[-1] % B:
            raise ValueError("n is not divisible by B^L")
        out.append(out[-1] // B)
    return out


def level_topk(n: int, B: int, L: int, K: int) -> list[int]:
    """[_, K_1, ..., K_L]: Top-K clamped to each level's candidate count."""
    out = np.zeros(L + 1, np.int32)
    _check(_load().orc_level_topk(n, B, L, K, out), "level_topk")
    return [int(x) for x in out]


# --------------------------------------------------------------------------
# Stages, one (batch, head) slice per call
# --------------------------------------------------------------------------

def pool(x, B: int, L: int) -> np.ndarray:
    """Mean pyramid of x [n, d]: levels 1..L stacked, float64 [sum n_l, d]."""
    x = _f32(x)
    n, d = x.shape
    rows = sum(level_sizes(n, B, L)[1:])
    out = np.empty((rows, d), np.float64)
    _check(_load().orc_pool(x, n, d, B, L, out), "pool")
    return out


def level_rows(n: int, B: int, L: int) -> list[tuple[int, int]]:
    """(row offset, rows) of each level 1..L inside a pyramid (index 0 unused)."""
    sizes = level_sizes(n, B, L)
    out, off = [(0, n)], 0
    for l in range(1, L + 1):
        out.append((off, sizes[l]))
        off += sizes[l]
    return out


def select_level(qpyr_l, kpyr_l, B: int, parent_sel, K: int):
    """Selection of one level. parent_sel is None at the coarsest level.
    Returns (sel [n_l, K_l] ascending, top1 [n_l], scored-pair count)."""
    qpyr_l, kpyr_l = _f64(qpyr_l), _f64(kpyr_l)
    n_l, d = qpyr_l.shape
    if parent_sel is None:
        C, Kp, pptr = n_l, 0, None
    else:
        parent_sel = _i32(parent_sel)
        Kp = parent_sel.shape[1]
        C, pptr = Kp * B, parent_sel.ctypes.data
    Kl = min(K, C)
    sel = np.empty((n_l, Kl), np.int32)
    top1 = np.empty(n_l, np.int32)
    work = _ll(0)
    _check(_load().orc_select_level(qpyr_l, kpyr_l, n_l, d, B, pptr, Kp, K, sel, top1, ctypes.byref(work)),
           "select_level")
    return sel, top1, int(work.value)


def pair_scores(qpyr_l, kpyr_l, rows, cols) -> np.ndarray:
    """Selection score (raw pooled dot product) of arbitrary pairs."""
    qpyr_l, kpyr_l = _f64(qpyr_l), _f64(kpyr_l)
    rows = np.ascontiguousarray(rows, np.int64).ravel()
    cols = np.ascontiguousarray(cols, np.int64).ravel()
    out = np.empty(rows.size, np.float64)
    _check(_load().orc_pair_scores(qpyr_l, kpyr_l, qpyr_l.shape[1], rows, cols, rows.size, out), "pair_scores")
    return out


RULES = {"top1": 0, "ancestor": 1, "allk": 2}


def coarse_levels(n: int, B: int, L: int, K: int, rule: str = "top1") -> np.ndarray:
    """Level (1..L) of each column of a query block's enrichment row: one
    column per level for "top1" and "ancestor", K_l columns for level l under
    "allk"."""
    lib = _load()
    ncol = _check(lib.orc_coarse_cols(n, B, L, K, RULES[rule], None), "coarse_cols")
    clev = np.empty(ncol, np.int32)
    lib.orc_coarse_cols(n, B, L, K, RULES[rule], clev.ctypes.data)
    return clev


def _clev(coarse, L, clev):
    """The column levels of a coarse table: given, or one column per level."""
    if clev is not None:
        return _i32(clev)
    if coarse.shape[1] != L:
        raise ValueError("coarse has more columns than levels: pass clev")
    return np.arange(1, L + 1, dtype=np.int32)


def select_all(qpyr, kpyr, n: int, B: int, L: int, K: int, rule: str = "top1") -> dict:
    """All levels coarsest-first plus the enrichment index (rule "top1": the
    rank-1 selection of the query block's level-l ancestor; "ancestor": that
    ancestor itself; "allk": all K_l selections of level l for that ancestor).
    Returns {'levels': [None, I1, ..., IL], 'top1': [None, t1, ...],
             'coarse': int32 [n_1, C], 'clev': int32 [C] (column levels),
             'work': scored pairs}."""
    qpyr, kpyr = _f64(qpyr), _f64(kpyr)
    d = qpyr.shape[1]
    sizes = level_sizes(n, B, L)
    kl = level_topk(n, B, L, K)
    idx_all = np.empty(sum(sizes[l] * kl[l] for l in range(1, L + 1)), np.int32)
    top1_all = np.empty(sum(sizes[1:]), np.int32)
    clev = coarse_levels(n, B, L, K, rule)
    coarse = np.empty((sizes[1], clev.size), np.int32)
    work = _ll(0)
    _check(_load().orc_select_all(qpyr, kpyr, n, d, B, L, K, RULES[rule], idx_all, top1_all, coarse,
                                  ctypes.byref(work)),
           "select_all")
    levels, top1 = [None], [None]
    io, to = 0, 0
    for l in range(1, L + 1):
        levels.append(idx_all[io:io + sizes[l] * kl[l]].reshape(sizes[l], kl[l]))
        top1.append(top1_all[to:to + sizes[l]])
        io += sizes[l] * kl[l]
        to += sizes[l]
    return {"levels": levels, "top1": top1, "coarse": coarse, "clev": clev, "work": int(work.value)}


def fwd(q, k, v, kpyr, vpyr, B, L, Le, sel, coarse, scale, qlist=None, clev=None):
    """Forward of one slice; returns (o float64 [rows, d], lse float64 [rows])
    for all tokens, or for the tokens in qlist (in list order). clev: the
    levels of coarse's columns (default: one column per level)."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    kpyr, vpyr = _f64(kpyr), _f64(vpyr)
    sel, coarse = _i32(sel), _i32(coarse)
    n, d = q.shape
    if qlist is None:
        nq, qptr, keep = n, None, None
    else:
        keep = np.ascontiguousarray(qlist, np.int64)
        nq, qptr = keep.size, keep.ctypes.data
    o = np.empty((nq, d), np.float64)
    lse = np.empty(nq, np.float64)
    cl = _clev(coarse, L, clev)
    _check(_load().orc_fwd(q, k, v, kpyr, vpyr, n, d, B, L, Le, sel.shape[1], sel, coarse, cl.size, cl,
                           float(scale), qptr, nq, o, lse), "fwd")
    return o, lse


def transpose(sel, ncols: int):
    """CSR (rows x K) -> CSC: (col_ptr [ncols+1], row_idx [rows*K])."""
    sel = _i32(sel)
    T, K = sel.shape
    col_ptr = np.empty(ncols + 1, np.int32)
    row_idx = np.empty(T * K, np.int32)
    _check(_load().orc_transpose(sel, T, K, ncols, col_ptr, row_idx), "transpose")
    return col_ptr, row_idx


def bwd(q, k, v, kpyr, vpyr, o, lse, dout, B, L, Le, sel, coarse, scale, clev=None):
    """Backward of one slice; returns (dq, dk, dv) float64 [n, d]."""
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    n, d = q.shape
    dq, dk, dv = (np.empty((n, d), np.float64) for _ in range(3))
    sel, coarse = _i32(sel), _i32(coarse)
    cl = _clev(coarse, L, clev)
    _check(_load().orc_bwd(q, k, v, _f64(kpyr), _f64(vpyr), _f64(o), _f64(lse), dout, n, d, B, L, Le,
                           sel.shape[1], sel, coarse, cl.size, cl, float(scale), dq, dk, dv), "bwd")
    return dq, dk, dv


def bwd_dq_rows(q, k, v, kpyr, vpyr, o_rows, lse_rows, dout, B, L, Le, sel, coarse, scale, qlist, clev=None):
    """dq of the listed tokens only (o_rows, lse_rows in list order)."""
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    n, d = q.shape
    ql = np.ascontiguousarray(qlist, np.int64)
    out = np.empty((ql.size, d), np.float64)
    sel, coarse = _i32(sel), _i32(coarse)
    cl = _clev(coarse, L, clev)
    _check(_load().orc_bwd_dq_rows(q, k, v, _f64(kpyr), _f64(vpyr), _f64(o_rows), _f64(lse_rows), dout, n, d,
                                   B, L, Le, sel.shape[1], sel, coarse, cl.size, cl, float(scale), ql, ql.size,
                                   out),
           "bwd_dq_rows")
    return out


def bwd_dkv_blocks(q, k, v, kpyr, vpyr, o, lse, dout, B, L, Le, sel, coarse, scale, kblocks, clev=None):
    """dk, dv of the fine tokens of the listed key blocks: [len*B, d] each."""
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    n, d = q.shape
    kb = np.ascontiguousarray(kblocks, np.int64)
    dk = np.empty((kb.size * B, d), np.float64)
    dv = np.empty((kb.size * B, d), np.float64)
    sel, coarse = _i32(sel), _i32(coarse)
    cl = _clev(coarse, L, clev)
    _check(_load().orc_bwd_dkv_blocks(q, k, v, _f64(kpyr), _f64(vpyr), _f64(o), _f64(lse), dout, n, d, B, L,
                                      Le, sel.shape[1], sel, coarse, cl.size, cl, float(scale), kb, kb.size, dk,
                                      dv),
           "bwd_dkv_blocks")
    return dk, dv


# --------------------------------------------------------------------------
# Whole path over [bh, n, d] arrays
# --------------------------------------------------------------------------

def run(q, k, v, dout=None, *, B=16, K=8, L=None, Le=None, scale=None, threads=1, backward=True, rule="top1"):
    """The whole hot path for every (batch, head) slice of q, k, v [bh, n, d]
    (any leading shape is flattened to bh). Returns a dict of per-slice lists
    plus stacked outputs 'o', 'lse', and, with dout, 'dq', 'dk', 'dv'."""
    q, k, v = (np.asarray(a, np.float32) for a in (q, k, v))
    n, d = q.shape[-2:]
    q3, k3, v3 = (a.reshape(-1, n, d) for a in (q, k, v))
    do3 = None if dout is None else np.asarray(dout, np.float32).reshape(-1, n, d)
    bh = q3.shape[0]
    if L is None:
        L = num_levels(n, B)
    if L < 1:
        raise ValueError("need at least one pooled level (n >= B^2)")
    if Le is None:
        Le = L
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    T = n // B

    def one(s):
        qp, kp, vp = pool(q3[s], B, L), pool(k3[s], B, L), pool(v3[s], B, L)
        sel = select_all(qp, kp, n, B, L, K, rule)
        I1, coarse, clev = sel["levels"][1], sel["coarse"], sel["clev"]
        o, lse = fwd(q3[s], k3[s], v3[s], kp, vp, B, L, Le, I1, coarse, scale, clev=clev)
        col_ptr, row_idx = transpose(I1, T)
        res = {"qpyr": qp, "kpyr": kp, "vpyr": vp, "sel": sel, "o": o, "lse": lse,
               "col_ptr": col_ptr, "row_idx": row_idx}
        if do3 is not None and backward:
            res["dq"], res["dk"], res["dv"] = bwd(q3[s], k3[s], v3[s], kp, vp, o, lse, do3[s], B, L, Le,
                                                  I1, coarse, scale, clev=clev)
        return res

    if threads > 1 and bh > 1:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            per = list(ex.map(one, range(bh)))
    else:
        per = [one(s) for s in range(bh)]
    out = {"slices": per, "L": L, "Le": Le, "scale": scale, "B": B, "K": K,
           "o": np.stack([r["o"] for r in per]), "lse": np.stack([r["lse"] for r in per])}
    if do3 is not None and backward:
        for key in ("dq", "dk", "dv"):
            out[key] = np.stack([r[key] for r in per])
    return out


def tile_order(height: int, width: int, B: int) -> np.ndarray:
    """Hierarchical tile order of an s^m x s^m raster image, B = s^2 (reading of
    the page's index reordering, referee comments on Sec. 5.1 / Figure 2):
    pixel (r, c) with base-s digits r_k, c_k goes to position
    sum_k (r_k * s + c_k) * B^k, so every run of B^l consecutive positions is
    an s^l x s^l square. Returns src with src[p] = the raster token at
    position p (the forward permutation reads in[src[p]] into out[p])."""
    s = int(round(math.sqrt(B)))
    if s * s != B or s < 2 or height != width:
        raise ValueError("need B = s^2 and a square image")
    m, side = 0, height
    while side > 1:
        if side % s:
            raise ValueError("side must be a power of sqrt(B)")
        side //= s
        m += 1
    r, c = np.divmod(np.arange(height * width, dtype=np.int64), width)
    pos = np.zeros(height * width, np.int64)
    for k in range(m):
        rk, ck = (r // s ** k) % s, (c // s ** k) % s
        pos += (rk * s + ck) * B ** k
    src = np.empty_like(pos)
    src[pos] = np.arange(height * width)
    return src


def select_exhaustive(qpyr, kpyr, n: int, B: int, L: int, K: int) -> np.ndarray:
    """Single-level full scoring of the level-1 tokens (the reference of
    routing recall): every level-1 query token keeps its min(K, T) best of all
    T level-1 key tokens by the selection's score; ties to the lower index;
    rows ascending. This is the coarsest level's rule applied to level 1."""
    off, nl = level_rows(n, B, L)[1]
    sel, _, _ = select_level(np.asarray(qpyr)[off:off + nl], np.asarray(kpyr)[off:off + nl], B, None, K)
    return sel


def routing_recall(hier_sel, exhaustive_sel) -> float:
    """Share of the exhaustive level-1 Top-K entries that the hierarchical
    level-1 selection also holds (rows aligned, [T, K] each)."""
    h, e = np.asarray(hier_sel), np.asarray(exhaustive_sel)
    hits = sum(len(set(e[i].tolist()) & set(h[i].tolist())) for i in range(e.shape[0]))
    return hits / e.size
