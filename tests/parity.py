"""Helpers of the GPU parity tests: run the CUDA path through the C ABI, run
the oracle on the same seeded inputs, compare with the acceptance rules.

Acceptance (the method's stated tolerances):
  * index sets (every level of the selection, the enrichment index) identical,
    except where the oracle's score of a differing index lies within 1e-3
    relative of the oracle's K-th score (a near-tie swap); the sparse index
    transpose bit-exact;
  * o, dq, dk, dv: max-abs 2e-2 for bf16; for fp32 max-abs <= 1e-4 * max|ref|
    and, element by element, |got - ref| <= 1e-4 * |ref| + FP32_FLOOR * max|ref|
    (the floor covers elements that cancel to near zero: fp32 accumulation
    leaves them an absolute error of a few ulps of the terms summed, which are
    bounded by the tensor's scale);
  * lse: abs 1e-3.
No value computed by the CUDA path is ever fed to the oracle: stage tests feed
the CUDA path the oracle's indices; the end-to-end test compares outputs only
where the two selections agree and checks that the rest are legal near-tie
swaps (judged with the oracle's own scores of the indices the GPU chose).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import hierarchical_sparse_attention_mean_gb300 as llsa
from hierarchical_sparse_attention_mean_gb300 import synth

TIE_REL = 1e-3
BF16_ABS = 2e-2
FP32_REL = 1e-4
FP32_FLOOR = 1e-6   # absolute floor of the element-wise fp32 check, times max|ref| (~8 ulps)
LSE_ABS = 1e-3


def params_of(w: synth.Workload, **kw) -> llsa.Params:
    base = dict(block=w.block, topk=w.topk, dtype=w.dtype)
    base.update(kw)
    return llsa.Params(w.batch, w.heads, w.n, w.d, **base)


def to_dev(x: np.ndarray, dtype: str, shape=None):
    t = torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16 if dtype == "bf16" else torch.float32)
    if shape is not None:
        t = t.reshape(shape)
    return t.cuda().contiguous()


def dev_inputs(w: synth.Workload, x: dict) -> dict:
    shape = (w.batch, w.heads, w.n, w.d)
    return {k: to_dev(v, w.dtype, shape) for k, v in x.items()}


def f64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def out_tol_ok(got, ref, dtype):
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    if dtype == "bf16":
        return err <= BF16_ABS, err
    scale = max(float(np.abs(ref).max()), 1e-30)
    # worst element against its own bound (<= 1 passes)
    elem = float((np.abs(got - ref) / (FP32_REL * np.abs(ref) + FP32_FLOOR * scale)).max()) if got.size else 0.0
    return err <= FP32_REL * scale and elem <= 1.0, max(err / scale, elem * FP32_REL)


def assert_close(name, got, ref, dtype):
    ok, err = out_tol_ok(got, ref, dtype)
    assert ok, f"{name}: error {err:.3e} beyond tolerance ({dtype})"
    return err


def assert_lse(got, ref):
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    assert err <= LSE_ABS, f"lse: error {err:.3e}"
    return err


# --------------------------------------------------------------- selection

def legal_row(gpu_row, cand, scores, K):
    """Is gpu_row a legal Top-K of candidates `cand` whose oracle scores are
    `scores`: distinct, and every chosen index scores at least the K-th best
    score less a near-tie margin of TIE_REL relative."""
    order = np.lexsort((cand, -scores))
    kth = scores[order[min(K, len(cand)) - 1]]
    pos = {int(c): i for i, c in enumerate(cand)}
    tol = TIE_REL * max(abs(kth), 1e-30)
    if len(set(int(g) for g in gpu_row)) != len(gpu_row):
        return False
    for g in gpu_row:
        if int(g) not in pos or scores[pos[int(g)]] < kth - tol:
            return False
    return True


def check_selection(qpyr, kpyr, n, B, L, K, gpu_levels, gpu_coarse, ref):
    """Compares the GPU selection of one slice with the oracle's, level by
    level, coarsest first. Rows are equal, or legal near-tie swaps judged with
    oracle scores of the GPU row's own candidate set. Returns (set of query
    blocks whose key set differs from the oracle's, T)."""
    sizes = oracle.level_sizes(n, B, L)
    rows = oracle.level_rows(n, B, L)
    kl = oracle.level_topk(n, B, L, K)
    differ = {}
    for l in range(L, 0, -1):
        off, nl = rows[l]
        Q, Kp = qpyr[off:off + nl], kpyr[off:off + nl]
        g, r = np.asarray(gpu_levels[l]), ref["levels"][l]
        assert g.shape == r.shape, (l, g.shape, r.shape)
        bad = np.nonzero((g != r).any(axis=1))[0]
        for i in bad:
            if l == L:
                cand = np.arange(nl)
            else:
                parents = np.asarray(gpu_levels[l + 1])[i // B]
                cand = (parents[:, None] * B + np.arange(B)[None, :]).ravel()
            sc = oracle.pair_scores(Q, Kp, np.full(cand.size, i), cand)
            assert legal_row(g[i], cand, sc, kl[l]), f"level {l} row {i}: {g[i]} vs oracle {r[i]}"
        differ[l] = set(int(i) for i in bad)
    # enrichment: coarse[i][l-1] is the rank-1 of the GPU's level-l row of i's
    # ancestor; it must match the oracle's or be a near-tie of the best
    T = sizes[1]
    gc = np.asarray(gpu_coarse)
    cbad = np.nonzero((gc != ref["coarse"]).any(axis=1))[0]
    for i in cbad:
        for l in range(1, L + 1):
            if gc[i, l - 1] == ref["coarse"][i, l - 1]:
                continue
            off, nl = rows[l]
            a = i // B ** (l - 1)
            row = np.asarray(gpu_levels[l])[a]
            sc = oracle.pair_scores(qpyr[off:off + nl], kpyr[off:off + nl], np.full(row.size, a), row)
            best = sc.max()
            got = oracle.pair_scores(qpyr[off:off + nl], kpyr[off:off + nl], [a], [gc[i, l - 1]])[0]
            assert gc[i, l - 1] in row and got >= best - TIE_REL * max(abs(best), 1e-30), (i, l)
    qb = set(int(i) for i in cbad) | differ.get(1, set())
    return qb, T


# ------------------------------------------------------------ GPU runs

def gpu_stage_outputs(w, x, p=None, backward=True, oracle_sel=None):
    """Runs the CUDA path. With oracle_sel (per-slice oracle results), the
    attention stages get the ORACLE's indices instead of the GPU selection."""
    p = p or params_of(w)
    d = dev_inputs(w, x)
    b = llsa.Buffers(p)
    llsa.llsa_pool(p, d["q"], d["k"], d["v"], b.pyr)
    llsa.llsa_select(p, b.pyr, b.sel_idx, b.coarse_idx, b.level_idx)
    out = {"pyr": b.pyr.cpu().numpy(), "gpu_sel": b.sel_idx.cpu().numpy(), "gpu_coarse": b.coarse_idx.cpu().numpy(),
           "gpu_levels": [None] + [b.level(l).cpu().numpy() for l in range(1, b.s.levels + 1)]}
    if oracle_sel is not None:
        b.sel_idx.copy_(torch.from_numpy(np.stack([r["sel"]["levels"][1] for r in oracle_sel])))
        b.coarse_idx.copy_(torch.from_numpy(np.stack([r["sel"]["coarse"] for r in oracle_sel])))
    llsa.llsa_fwd(p, d["q"], d["k"], d["v"], b.pyr, b.sel_idx, b.coarse_idx, b.o, b.lse, b.ws_f)
    out["o"] = f64(b.o).reshape(-1, w.n, w.d)
    out["lse"] = f64(b.lse).reshape(-1, w.n)
    llsa.llsa_index_transpose(p, b.sel_idx, b.col_ptr, b.row_idx, b.ws_t)
    out["col_ptr"] = b.col_ptr.cpu().numpy()
    out["row_idx"] = b.row_idx.cpu().numpy()
    if backward:
        dq, dk, dv = llsa.backward(p, d["q"], d["k"], d["v"], d["dout"], b)
        out["dq"], out["dk"], out["dv"] = (f64(t).reshape(-1, w.n, w.d) for t in (dq, dk, dv))
    torch.cuda.synchronize()
    assert llsa.llsa_get_status() == 0
    return out, b
