"""Exhaustive level-1 selection on the GPU (the reference of routing recall)
against the oracle's single-level full scoring: rows equal or legal near-tie
swaps; the recall the GPU reports equals the recall the oracle computes from
the same two index sets."""
import numpy as np
import pytest
import torch

import oracle
import hierarchical_sparse_attention_mean_gb300 as llsa
from hierarchical_sparse_attention_mean_gb300 import build, synth

from parity import dev_inputs, legal_row, params_of

pytestmark = pytest.mark.gpu

W = synth.Workload


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    oracle.build()


@pytest.mark.parametrize("w", [
    W("ex-4096", 2, 3, 4096, 64, amplitude=0.5, seed=111),
    W("ex-k16-d128", 1, 2, 4096, 128, topk=16, amplitude=0.5, seed=112),
    W("ex-fp32-b4", 1, 2, 1024, 32, block=4, topk=3, dtype="fp32", seed=113),
    W("ex-grf", 1, 2, 16384, 64, kind="grf", grid=(128, 128), seed=114),
], ids=lambda w: w.name)
def test_exhaustive_selection_and_recall(w):
    x = synth.make_inputs(w, with_dout=False)
    p = params_of(w)
    s = llsa.get_sizes(p)
    d = dev_inputs(w, x)
    b = llsa.Buffers(p)
    llsa.llsa_pool(p, d["q"], d["k"], d["v"], b.pyr)
    llsa.llsa_select(p, b.pyr, b.sel_idx, b.coarse_idx, b.level_idx)
    T = s.n_blocks
    kx = min(w.topk, T)
    ex = torch.empty(w.bh, T, kx, dtype=torch.int32, device="cuda")
    llsa.llsa_select_exhaustive(p, b.pyr, ex)
    torch.cuda.synchronize()
    assert llsa.llsa_get_status() == 0
    gex, gsel = ex.cpu().numpy(), b.sel_idx.cpu().numpy()
    L = s.levels
    off, nl = oracle.level_rows(w.n, w.block, L)[1]
    swaps = 0
    for sl in range(w.bh):
        qp = oracle.pool(x["q"][sl], w.block, L)
        kp = oracle.pool(x["k"][sl], w.block, L)
        ref = oracle.select_exhaustive(qp, kp, w.n, w.block, L, w.topk)
        bad = np.nonzero((gex[sl] != ref).any(axis=1))[0]
        swaps += bad.size
        cand = np.arange(T)
        for i in bad:
            sc = oracle.pair_scores(qp[off:off + nl], kp[off:off + nl], np.full(T, i), cand)
            assert legal_row(gex[sl][i], cand, sc, kx), (sl, i)
    assert swaps <= max(1, 0.01 * w.bh * T)
    r_gpu = llsa.routing_recall(b.sel_idx, ex)
    r_orc = np.mean([oracle.routing_recall(gsel[sl], gex[sl]) for sl in range(w.bh)])
    assert abs(r_gpu - r_orc) < 1e-9
    assert 0.0 < r_gpu <= 1.0
