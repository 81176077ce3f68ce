"""Host-side logic of bench.py that needs no GPU: the work model's counts,
which workloads the tile-order side metric accepts, and that every entry of
the hyperparameter sweep either derives sizes or is refused with an LLSA
error (never a crash)."""
import math

import pytest

import bench
import hierarchical_sparse_attention_mean_gb300 as llsa
from hierarchical_sparse_attention_mean_gb300 import build, synth


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def test_work_model_counts_pairs_and_flops():
    w = synth.WORKLOADS[synth.HEADLINE]
    p = llsa.Params(w.batch, w.heads, w.n, w.d, block=w.block, topk=w.topk)
    s = llsa.get_sizes(p)
    m = bench.work_model(w, s)
    # 8 selected blocks of 16 tokens plus one pooled token per level
    assert s.keys_per_query == 8 * 16 + 3
    assert m["pairs"] == w.bh * w.n * s.keys_per_query
    assert m["step_flops"] == 14 * w.d * m["pairs"] == m["fwd_flops"] + m["bwd_flops"]
    # scored candidates: n_L^2 at the coarsest level, K_{l+1} B per token below
    n = [w.n // w.block ** l for l in range(4)]
    assert m["select_flops"] == 2 * w.d * w.bh * (n[3] ** 2 + n[2] * 8 * 16 + n[1] * 8 * 16)


def test_work_model_partials_follow_enrichment_columns():
    w = synth.WORKLOADS[synth.HEADLINE]
    one = llsa.get_sizes(llsa.Params(w.batch, w.heads, w.n, w.d))
    allk = llsa.get_sizes(llsa.Params(w.batch, w.heads, w.n, w.d, enrich_rule="allk"))
    b1 = bench.work_model(w, one)["kernels"]["bwd_dq"][0]
    b2 = bench.work_model(w, allk)["kernels"]["bwd_dq"][0]
    # the pooled-level partials grow with the enrichment columns (3 -> 24)
    assert b2 - b1 == 2 * w.bh * one.n_blocks * (allk.enrich_cols - one.enrich_cols) * w.d * 4


def test_reorder_side_metric_needs_a_power_of_the_tile_side():
    # 256 = 4^4 (headline); 128 is not a power of 4: reported unavailable, no launch
    w128 = synth.WORKLOADS["llsa-n16384-d64-b2h12-K8-bf16"]
    assert "unavailable" in bench.reorder_rate(w128, None, {"hbm_gbs": 1.0})
    w_iid = synth.WORKLOADS["llsa-fwd-n4096-d64-b2h8-K8-bf16"]     # 64 = 4^3: accepted shape
    side = int(round(math.sqrt(w_iid.n)))
    assert side == 64 and 4 ** 3 == side


@pytest.mark.parametrize("entry", bench.SWEEP, ids=lambda e: e[0])
def test_sweep_entries_derive_or_are_refused(entry):
    label, B, K, L, Le, *rule = entry
    w = synth.WORKLOADS[synth.HEADLINE]
    p = llsa.Params(w.batch, w.heads, w.n, w.d, block=B, topk=K, levels=L, enrich_levels=Le,
                    enrich_rule=rule[0] if rule else "top1")
    try:
        s = llsa.get_sizes(p)
    except llsa.LLSAError as e:
        assert e.code < 0
        return
    assert s.keys_per_query == s.topk_level[1] * B + s.enrich_cols
    assert s.levels == (L or s.levels)


def test_spread_is_nearest_rank_percentiles():
    assert bench.spread([]) is None
    assert bench.spread([2.5]) == {"p10": 2.5, "median": 2.5, "p90": 2.5}
    v = [float(x) for x in range(101)]  # 0 .. 100: the percentiles are the values themselves
    assert bench.spread(list(reversed(v))) == {"p10": 10.0, "median": 50.0, "p90": 90.0}
