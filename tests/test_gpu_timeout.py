"""Failure detection of the tensor-core kernels, without faulting a GPU.

Every wait of these kernels is bounded; when one runs out the kernel records
LLSA_ERR_TIMEOUT in the device status word, the CTA drains (no copy or MMA in
flight), frees its tensor memory and exits, and the context stays usable. The
test hook llsa_test_set_wait_limit lowers the wait limit and switches the copy
warps off (LLSA_TEST_NO_COPIES), so the consumers' first waits run out. Each
case checks that the status reads TIMEOUT and then clears, and that the next
normal call is correct again (against the oracle, or for the 2^20-token case
against the same call made before the timeout)."""
import numpy as np
import pytest
import torch

import oracle
import hierarchical_sparse_attention_mean_gb300 as llsa
from hierarchical_sparse_attention_mean_gb300 import build, synth

from parity import assert_close, assert_lse, dev_inputs, params_of

pytestmark = pytest.mark.gpu

TIMEOUT = -9
LIMIT = 256  # polls: a fraction of a millisecond instead of about a second


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    oracle.build()
    yield
    llsa.test_set_wait_limit(0, 0)


def _timed_out(fn):
    llsa.test_set_wait_limit(LIMIT, llsa.LLSA_TEST_NO_COPIES)
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        llsa.test_set_wait_limit(0, 0)
    assert llsa.llsa_get_status() == TIMEOUT
    assert llsa.llsa_get_status() == 0   # read and cleared


# d = 64: the grouped forward, the dQ and dK/dV kernels (d = 64 instances);
# d = 128: the few-stage forward and the d = 128 backward instances
@pytest.mark.parametrize("d", [64, 128])
def test_forward_and_backward_time_out_then_recover(d):
    w = synth.Workload("to", 1, 2, 4096, d, topk=8, amplitude=0.5, seed=95)
    x = synth.make_inputs(w)
    ref = oracle.run(x["q"], x["k"], x["v"], x["dout"], B=w.block, K=w.topk, threads=8)
    p = params_of(w)
    dv_ = dev_inputs(w, x)
    b = llsa.Buffers(p)
    _timed_out(lambda: llsa.forward(p, dv_["q"], dv_["k"], dv_["v"], b))
    # the next normal forward is correct; the oracle's selection is used so
    # that outputs compare element by element
    llsa.forward(p, dv_["q"], dv_["k"], dv_["v"], b)
    b.sel_idx.copy_(torch.from_numpy(np.stack([r["sel"]["levels"][1] for r in ref["slices"]])))
    b.coarse_idx.copy_(torch.from_numpy(np.stack([r["sel"]["coarse"] for r in ref["slices"]])))
    llsa.llsa_fwd(p, dv_["q"], dv_["k"], dv_["v"], b.pyr, b.sel_idx, b.coarse_idx, b.o, b.lse, b.ws_f)
    torch.cuda.synchronize()
    assert llsa.llsa_get_status() == 0
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64).reshape(-1, w.n, w.d)
    assert_close("o", f64(b.o), ref["o"], w.dtype)
    assert_lse(b.lse.cpu().numpy().reshape(-1, w.n), ref["lse"])
    # the backward kernels time out, then recover
    _timed_out(lambda: llsa.backward(p, dv_["q"], dv_["k"], dv_["v"], dv_["dout"], b))
    dq, dk, dv = llsa.backward(p, dv_["q"], dv_["k"], dv_["v"], dv_["dout"], b)
    torch.cuda.synchronize()
    assert llsa.llsa_get_status() == 0
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close(name, f64(got), ref[name], w.dtype)


def test_pipelined_forward_times_out_then_recovers():
    """2^20 tokens (L = 4 enrichment levels) take the pipelined forward; its
    recovered output equals the one computed before the timeout, bit for bit
    (the kernels are deterministic)."""
    w = synth.Workload("to4", 1, 1, 1 << 20, 64, topk=8, amplitude=0.5, seed=96, backward=False)
    x = synth.make_inputs(w, with_dout=False)
    p = params_of(w)
    assert llsa.get_sizes(p).enrich_levels == 4
    dv_ = dev_inputs(w, x)
    b = llsa.Buffers(p)
    llsa.forward(p, dv_["q"], dv_["k"], dv_["v"], b)
    torch.cuda.synchronize()
    assert llsa.llsa_get_status() == 0
    o0, lse0 = b.o.clone(), b.lse.clone()
    llsa.profile_reset()
    llsa.profile_enable(True)
    try:
        _timed_out(lambda: llsa.forward(p, dv_["q"], dv_["k"], dv_["v"], b))
        launched = {n for n, _ in llsa.profile_read()}
    finally:
        llsa.profile_enable(False)
        llsa.profile_reset()
    assert "fwd_tc" in launched, launched
    llsa.forward(p, dv_["q"], dv_["k"], dv_["v"], b)
    torch.cuda.synchronize()
    assert llsa.llsa_get_status() == 0
    assert torch.equal(b.o, o0) and torch.equal(b.lse, lse0)


def test_test_hook_rejects_unknown_switches():
    with pytest.raises(llsa.LLSAError):
        llsa.test_set_wait_limit(0, 8)
    with pytest.raises(llsa.LLSAError):  # both forward paths forced at once
        llsa.test_set_wait_limit(0, llsa.LLSA_TEST_FORCE_GROUPED | llsa.LLSA_TEST_FORCE_PER_BLOCK)
