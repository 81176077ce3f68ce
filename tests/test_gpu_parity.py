"""Parity of the CUDA path (through the C ABI) with the CPU oracle, stage by
stage and end to end, on seeded synthetic inputs that span several tiles and
ragged tails, plus the method's degenerate cases."""
import numpy as np
import pytest
import torch

import oracle
import hierarchical_sparse_attention_mean_gb300 as llsa
from hierarchical_sparse_attention_mean_gb300 import build, synth

from parity import assert_close, assert_lse, check_selection, dev_inputs, gpu_stage_outputs, params_of

pytestmark = pytest.mark.gpu

W = synth.Workload
CASES = {
    # the 32x32 fp32 forward workload, full size
    "n1024-fp32": synth.WORKLOADS["llsa-fwd-n1024-d64-b1h1-K4-fp32"],
    # the 64x64 bf16 forward workload, full size (16 slices)
    "n4096-bf16": synth.WORKLOADS["llsa-fwd-n4096-d64-b2h8-K8-bf16"],
    # 768 query blocks: not a multiple of the SM count
    "ragged-h3": W("ragged", 1, 3, 4096, 64, amplitude=0.5, seed=77),
    "d128-K16": W("d128", 1, 2, 4096, 128, topk=16, amplitude=0.5, seed=78),
    # the two tensor-core instances with fewer shared-memory stages (d = 64
    # with K = 16; d = 128 with K = 8), on a ragged block count and on a
    # spatially structured field
    "d64-K16": W("d64k16", 1, 3, 4096, 64, topk=16, amplitude=0.5, seed=82),
    "d128-K8-grf": W("d128k8", 1, 3, 4096, 128, topk=8, kind="grf", length_scale=4.0, grid=(64, 64), seed=83),
    # K_1 = 4: the grouped forward always runs (no per-block tensor-core
    # forward for 64 keys) and the backward's dQ uses an M = 64 key tile;
    # d = 128 takes the CUDA-core forward and the tensor-core backward
    "d64-K4": W("d64k4", 1, 3, 4096, 64, topk=4, amplitude=0.5, seed=84),
    "d128-K4-grf": W("d128k4", 1, 2, 4096, 128, topk=4, kind="grf", length_scale=4.0, grid=(64, 64), seed=85),
    # K_1 = 32 (512 fine keys per query block): four key tiles with one ring
    # stage in the per-block forward and in dQ
    "d64-K32-grf": W("d64k32", 1, 2, 4096, 64, topk=32, kind="grf", length_scale=4.0, grid=(64, 64), seed=86),
    # 512 level-1 candidates per row (16 per lane): the selection's threshold
    # form of the Top-K
    "n16384-K32": W("n16k32", 1, 2, 16384, 64, topk=32, amplitude=0.5, seed=87),
    "B4-L4-fp32": W("b4", 1, 2, 1024, 32, block=4, topk=3, dtype="fp32", seed=79),
    "B2-fig1": W("fig1", 1, 1, 8, 8, block=2, topk=1, dtype="fp32", seed=80),
    "B8-d16-bf16": W("b8", 2, 1, 512, 16, block=8, topk=5, amplitude=0.5, seed=81),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    oracle.build()


def run_oracle(w, x, **kw):
    return oracle.run(x["q"], x["k"], x["v"], x.get("dout"), B=w.block, K=w.topk, threads=16, **kw)


@pytest.fixture(scope="module")
def case_data():
    cache = {}

    def get(name):
        if name not in cache:
            w = CASES[name]
            x = synth.make_inputs(w)
            cache[name] = (w, x, run_oracle(w, x))
        return cache[name]
    return get


@pytest.mark.parametrize("name", list(CASES))
def test_pool(case_data, name):
    w, x, ref = case_data(name)
    out, _ = gpu_stage_outputs(w, x, backward=False)
    for s, r in enumerate(ref["slices"]):
        for t, key in enumerate(("qpyr", "kpyr", "vpyr")):
            err = np.abs(out["pyr"][t, s] - r[key]).max()
            assert err <= 1e-5 * max(1.0, np.abs(r[key]).max()), (s, key, err)


@pytest.mark.parametrize("name", list(CASES))
def test_select(case_data, name):
    w, x, ref = case_data(name)
    out, _ = gpu_stage_outputs(w, x, backward=False)
    L = ref["L"]
    total = 0
    for s, r in enumerate(ref["slices"]):
        levels = [None] + [out["gpu_levels"][l][s] for l in range(1, L + 1)]
        differ, T = check_selection(r["qpyr"], r["kpyr"], w.n, w.block, L, w.topk, levels,
                                    out["gpu_coarse"][s], r["sel"])
        total += len(differ)
    assert total <= max(1, 0.01 * w.bh * (w.n // w.block)), total


# the cases that can take the grouped tensor-core forward (bf16, d = 64,
# B = 16, K_1 in {8, 16}): their forward is checked on both tensor-core paths
# as well as on the one llsa_fwd picks
GROUPABLE = [n for n, w in CASES.items() if w.dtype == "bf16" and w.d == 64 and w.block == 16 and w.topk in (8, 16)]
PATHS = {"auto": 0, "grouped": llsa.LLSA_TEST_FORCE_GROUPED, "per_block": llsa.LLSA_TEST_FORCE_PER_BLOCK}


def forced(path):
    """Context manager: llsa_fwd takes `path` until exit."""
    import contextlib

    @contextlib.contextmanager
    def ctx():
        llsa.test_set_wait_limit(0, PATHS[path])
        try:
            yield
        finally:
            llsa.test_set_wait_limit(0, 0)
    return ctx()


@pytest.mark.parametrize("name,path", [(n, "auto") for n in CASES] +
                         [(n, p) for n in GROUPABLE for p in ("grouped", "per_block")])
def test_fwd_with_oracle_indices(case_data, name, path):
    w, x, ref = case_data(name)
    with forced(path):
        out, _ = gpu_stage_outputs(w, x, backward=False, oracle_sel=ref["slices"])
    assert_close("o", out["o"], ref["o"], w.dtype)
    assert_lse(out["lse"], ref["lse"])


@pytest.mark.parametrize("name", list(CASES))
def test_transpose_bit_exact(case_data, name):
    w, x, ref = case_data(name)
    out, _ = gpu_stage_outputs(w, x, backward=False, oracle_sel=ref["slices"])
    for s, r in enumerate(ref["slices"]):
        np.testing.assert_array_equal(out["col_ptr"][s], r["col_ptr"])
        np.testing.assert_array_equal(out["row_idx"][s], r["row_idx"])


@pytest.mark.parametrize("name", [n for n in CASES if CASES[n].backward])
def test_bwd_with_oracle_indices(case_data, name):
    w, x, ref = case_data(name)
    out, _ = gpu_stage_outputs(w, x, backward=True, oracle_sel=ref["slices"])
    for key in ("dq", "dk", "dv"):
        assert_close(key, out[key], ref[key], w.dtype)


def compare_end_to_end(w, ref, out):
    """Outputs compared wherever the GPU and oracle selections agree; where
    they differ the swaps were shown legal by check_selection."""
    L, B = ref["L"], w.block
    excluded = 0
    for s, r in enumerate(ref["slices"]):
        levels = [None] + [out["gpu_levels"][l][s] for l in range(1, L + 1)]
        differ, T = check_selection(r["qpyr"], r["kpyr"], w.n, B, L, w.topk, levels, out["gpu_coarse"][s],
                                    r["sel"])
        tok = np.ones(w.n, bool)
        kblk = np.ones(T, bool)
        for i in differ:
            tok[i * B:(i + 1) * B] = False
            for row in (out["gpu_sel"][s][i], r["sel"]["levels"][1][i]):
                kblk[row] = False
            for crow in (out["gpu_coarse"][s][i], r["sel"]["coarse"][i]):
                for l in range(1, L + 1):
                    span = B ** (l - 1)
                    kblk[crow[l - 1] * span:(crow[l - 1] + 1) * span] = False
        excluded += len(differ)
        ktok = np.repeat(kblk, B)
        assert_close("o", out["o"][s][tok], r["o"][tok], w.dtype)
        assert_lse(out["lse"][s][tok], r["lse"][tok])
        if "dq" in out:
            assert_close("dq", out["dq"][s][tok], r["dq"][tok], w.dtype)
            assert_close("dk", out["dk"][s][ktok], r["dk"][ktok], w.dtype)
            assert_close("dv", out["dv"][s][ktok], r["dv"][ktok], w.dtype)
    return excluded


@pytest.mark.parametrize("name", list(CASES))
def test_end_to_end(case_data, name):
    w, x, ref = case_data(name)
    out, _ = gpu_stage_outputs(w, x, backward=w.backward)
    excluded = compare_end_to_end(w, ref, out)
    assert excluded <= max(1, 0.01 * w.bh * (w.n // w.block))


# ------------------------------------------------------------ edge cases

@pytest.mark.parametrize("n,K,g", [(4096, 8, 0.5), (16384, 32, 0.02)])
def test_constant_inputs_tie_break_bit_exact(n, K, g):
    """Every score ties: the lower index wins at every level, on both sides
    (at 16,384 tokens with K = 32 through the threshold form of the Top-K).
    Every query block then selects the same key blocks, so dv of those keys
    sums all N queries; the output gradient g keeps it near 1 there (with 0.5
    it reaches about 31, where one bf16 step is 0.125, above the bf16 bound)."""
    w = W("const", 1, 2, n, 64, topk=K, seed=1)
    x = {k: np.full((2, n, 64), 0.5, np.float32) for k in ("q", "k", "v")}
    x["dout"] = np.full((2, n, 64), g, np.float32)
    ref = run_oracle(w, x)
    out, _ = gpu_stage_outputs(w, x)
    for s, r in enumerate(ref["slices"]):
        np.testing.assert_array_equal(out["gpu_sel"][s], r["sel"]["levels"][1])
        np.testing.assert_array_equal(out["gpu_coarse"][s], r["sel"]["coarse"])
        np.testing.assert_array_equal(out["gpu_levels"][2][s], r["sel"]["levels"][2])
    assert_close("o", out["o"], ref["o"], "bf16")
    for key in ("dq", "dk", "dv"):
        assert_close(key, out[key], ref[key], "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_full_selection_is_dense_plus_enrichment(dtype):
    """K*B >= N: every block selected; equals dense attention over all tokens
    plus the enrichment tokens."""
    w = W("full", 1, 2, 1024, 32, topk=64, dtype=dtype, amplitude=0.5, seed=5)
    x = synth.make_inputs(w)
    ref = run_oracle(w, x)
    out, _ = gpu_stage_outputs(w, x)
    assert (out["gpu_sel"] == np.arange(64)[None, None, :]).all()
    assert_close("o", out["o"], ref["o"], dtype)
    assert_lse(out["lse"], ref["lse"])
    for key in ("dq", "dk", "dv"):
        assert_close(key, out[key], ref[key], dtype)


def test_no_enrichment_is_sparse_softmax():
    w = W("noenr", 1, 2, 4096, 64, amplitude=0.5, seed=6)
    x = synth.make_inputs(w)
    ref = run_oracle(w, x, Le=0)
    out, _ = gpu_stage_outputs(w, x, p=params_of(w, enrich_levels=0), oracle_sel=ref["slices"])
    assert_close("o", out["o"], ref["o"], "bf16")
    assert_lse(out["lse"], ref["lse"])
    for key in ("dq", "dk", "dv"):
        assert_close(key, out[key], ref[key], "bf16")


def test_partial_enrichment_and_fewer_levels():
    w = W("le1", 1, 2, 16384, 64, amplitude=0.5, seed=7)
    x = synth.make_inputs(w)
    ref = run_oracle(w, x, L=1, Le=1)
    out, _ = gpu_stage_outputs(w, x, p=params_of(w, levels=1, enrich_levels=1), oracle_sel=ref["slices"])
    assert_close("o", out["o"], ref["o"], "bf16")
    for key in ("dq", "dk", "dv"):
        assert_close(key, out[key], ref[key], "bf16")


def test_empty_batch_is_a_no_op():
    p = llsa.Params(0, 4, 4096, 64)
    z = torch.empty((0, 4, 4096, 64), dtype=torch.bfloat16, device="cuda")
    b = llsa.Buffers(p)
    llsa.forward(p, z, z, z, b)
    llsa.backward(p, z, z, z, z, b)
    torch.cuda.synchronize()


def test_out_of_range_index_sets_status():
    """An index outside [0, T) is caught by the kernel's bounds check: the
    access is clamped and the device status word reports it."""
    w = W("bad", 1, 1, 4096, 64, amplitude=0.5, seed=8)
    x = dev_inputs(w, synth.make_inputs(w, with_dout=False))
    p = params_of(w)
    b = llsa.forward(p, x["q"], x["k"], x["v"])
    torch.cuda.synchronize()
    assert llsa.llsa_get_status() == 0
    b.sel_idx[0, 3, 2] = 10_000
    llsa.llsa_fwd(p, x["q"], x["k"], x["v"], b.pyr, b.sel_idx, b.coarse_idx, b.o, b.lse, b.ws_f)
    assert llsa.llsa_get_status() == -10
    assert llsa.llsa_get_status() == 0   # reading clears it


def test_autograd_function_matches_direct_calls():
    w = W("ag", 1, 2, 4096, 64, amplitude=0.5, seed=9)
    x = dev_inputs(w, synth.make_inputs(w))
    q, k, v = (x[a].clone().requires_grad_(True) for a in ("q", "k", "v"))
    o = llsa.llsa_attention(q, k, v, block=16, topk=8)
    o.backward(x["dout"])
    p = params_of(w)
    b = llsa.forward(p, x["q"], x["k"], x["v"])
    dq, dk, dv = llsa.backward(p, x["q"], x["k"], x["v"], x["dout"], b)
    torch.cuda.synchronize()
    assert torch.equal(o.detach(), b.o)
    assert torch.equal(q.grad, dq) and torch.equal(k.grad, dk) and torch.equal(v.grad, dv)


def test_deterministic_across_runs():
    w = W("det", 1, 3, 4096, 64, amplitude=0.5, seed=10)
    x = dev_inputs(w, synth.make_inputs(w))
    p = params_of(w)
    outs = []
    for _ in range(2):
        b = llsa.forward(p, x["q"], x["k"], x["v"])
        g = llsa.backward(p, x["q"], x["k"], x["v"], x["dout"], b)
        outs.append([b.o.clone(), b.lse.clone(), b.col_ptr.clone(), b.row_idx.clone()] + [t.clone() for t in g])
    torch.cuda.synchronize()
    for a, c in zip(*outs):
        assert torch.equal(a, c)


@pytest.mark.parametrize("path", ["grouped", "per_block"])
def test_fine_logits_far_above_pooled_logits(path):
    """Keys whose block means cancel (so every pooled key is zero and every
    pooled logit is its ln B^l bias) against queries that are, on alternate
    query blocks, large multiples of the keys' direction: there the fine
    logits exceed the pooled ones by about 70 nats, beyond the range the
    forward's pooled-logit shift covers, so those blocks take the exact-maximum
    path while the others keep the shifted one."""
    n, d, B = 4096, 64, 16
    w = W("wide", 1, 2, n, d, amplitude=0.5, seed=8)
    x = synth.make_inputs(w)
    rng = np.random.default_rng(8)
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    sign = np.where(np.arange(n) % 2 == 0, 1.0, -1.0)        # block means of K are exactly zero
    big = np.sqrt(80.0 * np.sqrt(d))                           # scale * |q| * |k| = 80 on large blocks
    cq = np.where((np.arange(n) // B) % 2 == 0, big, 0.3)      # alternate query blocks large / small
    k = (big * sign)[:, None] * u[None, :]
    q = cq[:, None] * u[None, :]
    for s in range(2):
        x["k"][s] = synth.bf16_round(k.astype(np.float32))
        x["q"][s] = synth.bf16_round(q.astype(np.float32))
    # |q|, |k| ~ 25 make dk, dq ~ 25x larger than usual; dO / 32 (exact in bf16)
    # keeps the gradients on the scale the absolute bf16 tolerance assumes
    x["dout"] = x["dout"] / 32.0
    ref = run_oracle(w, x)
    with forced(path):
        out, _ = gpu_stage_outputs(w, x, oracle_sel=ref["slices"])
    assert_close("o", out["o"], ref["o"], "bf16")
    assert_lse(out["lse"], ref["lse"])
    for key in ("dq", "dk", "dv"):
        assert_close(key, out[key], ref[key], "bf16")


@pytest.mark.parametrize("name", ["n4096-bf16", "B4-L4-fp32", "d128-K16"])
def test_ancestor_rule_end_to_end(name):
    """ANCESTOR enrichment: selection identical to TOP1's, the enrichment index
    is each block's own ancestor, outputs and gradients match the oracle."""
    w = CASES[name]
    x = synth.make_inputs(w)
    ref = run_oracle(w, x, rule="ancestor")
    out, _ = gpu_stage_outputs(w, x, p=params_of(w, enrich_rule="ancestor"), backward=w.backward)
    T, L = w.n // w.block, ref["L"]
    for s in range(w.bh):
        for l in range(1, L + 1):
            np.testing.assert_array_equal(out["gpu_coarse"][s][:, l - 1], np.arange(T) // w.block ** (l - 1))
    excluded = compare_end_to_end(w, ref, out)
    assert excluded <= max(1, 0.01 * w.bh * (w.n // w.block))


@pytest.mark.parametrize("name,Le", [("ragged-h3", None), ("ragged-h3", 1), ("B4-L4-fp32", None),
                                     ("d128-K16", None), ("n4096-bf16", None)])
def test_allk_rule(name, Le):
    """ALLK enrichment (every token a level keeps for the block's ancestor):
    the selection equals TOP1's; the enrichment table holds, for each level,
    the GPU's own ascending row of the ancestor; on the oracle's indices the
    outputs and gradients match the oracle."""
    w = CASES[name]
    x = synth.make_inputs(w)
    kw = {} if Le is None else {"enrich_levels": Le}
    p = params_of(w, enrich_rule="allk", **kw)
    out, _ = gpu_stage_outputs(w, x, p=p, backward=False)
    top1, _ = gpu_stage_outputs(w, x, p=params_of(w, **kw), backward=False)
    L = len(out["gpu_levels"]) - 1
    clev = oracle.coarse_levels(w.n, w.block, L, w.topk, "allk")
    T = w.n // w.block
    for l in range(1, L + 1):
        np.testing.assert_array_equal(out["gpu_levels"][l], top1["gpu_levels"][l])
        cols = np.nonzero(clev == l)[0]
        anc = np.arange(T) // w.block ** (l - 1)
        for s in range(w.bh):
            np.testing.assert_array_equal(out["gpu_coarse"][s][:, cols], out["gpu_levels"][l][s][anc])
    ref = run_oracle(w, x, rule="allk", **({} if Le is None else {"Le": Le}))
    got, _ = gpu_stage_outputs(w, x, p=p, backward=w.backward, oracle_sel=ref["slices"])
    assert_close("o", got["o"], ref["o"], w.dtype)
    assert_lse(got["lse"], ref["lse"])
    if w.backward:
        for key in ("dq", "dk", "dv"):
            assert_close(key, got[key], ref[key], w.dtype)
