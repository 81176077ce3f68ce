"""Kernel timing of the library (llsa_profile_*): with every kernel timed, one
forward + backward step records each of its launches; with the timing
restricted to one kernel name, only that kernel's launches are recorded, each
with a positive duration, and the launch count still counts every kernel."""
import pytest
import torch

import hierarchical_sparse_attention_mean_gb300 as llsa
from hierarchical_sparse_attention_mean_gb300 import build, synth

from parity import dev_inputs, params_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    yield
    llsa.profile_enable(False)
    llsa.profile_only(None)
    llsa.profile_reset()


def _step_records(prefix):
    w = synth.WORKLOADS["llsa-fwd-n4096-d64-b2h8-K8-bf16"]
    x = synth.make_inputs(w)
    p = params_of(w)
    d = dev_inputs(w, x)
    b = llsa.Buffers(p)
    dq, dk, dv = (torch.empty_like(d["q"]) for _ in range(3))
    llsa.forward(p, d["q"], d["k"], d["v"], b)  # warm-up, untimed
    torch.cuda.synchronize()
    llsa.profile_reset()
    llsa.profile_only(prefix)
    llsa.profile_enable(True)
    n0 = llsa.llsa_launch_count()
    llsa.forward(p, d["q"], d["k"], d["v"], b)
    llsa.backward(p, d["q"], d["k"], d["v"], d["dout"], b, dq, dk, dv)
    torch.cuda.synchronize()
    launched = llsa.llsa_launch_count() - n0
    llsa.profile_enable(False)
    llsa.profile_only(None)
    rec = llsa.profile_read()
    llsa.profile_reset()
    assert llsa.llsa_get_status() == 0
    return rec, launched


def test_every_kernel_timed():
    rec, launched = _step_records(None)
    names = [n for n, _ in rec]
    assert len(rec) == launched
    assert any(n.startswith("select_level") for n in names) and any(n.startswith("bwd_dkv") for n in names)
    assert all(ms > 0 for _, ms in rec)


def test_timing_restricted_to_one_kernel():
    full, launched = _step_records(None)
    rec, launched2 = _step_records("bwd_dkv")
    assert launched2 == launched  # every kernel still ran and was counted
    expect = [n for n, _ in full if n.startswith("bwd_dkv")]
    assert [n for n, _ in rec] == expect and len(expect) >= 1
    assert all(ms > 0 for _, ms in rec)
