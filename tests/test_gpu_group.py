"""The grouping of query blocks that the tensor-core forward gathers together
(csrc/group.cu), read back from the forward's workspace and checked
bit-exact against a numpy restatement of its rule: the anchor of query block
i is the selected key block with the smallest bit-reversed index; within each
window of 1024 consecutive query blocks, blocks sorted by (anchor, i) and runs
of equal anchors cut into groups of at most 8. The groups must partition the
query blocks, whatever the selection. The grouping changes no result, so the
forward parity tests cover its use."""
import numpy as np
import pytest
import torch

import hierarchical_sparse_attention_mean_gb300 as llsa
from hierarchical_sparse_attention_mean_gb300 import build, synth

from parity import dev_inputs, params_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def bitrev(j, bits):
    j = np.asarray(j, np.int64)
    r = np.zeros_like(j)
    for b in range(bits):
        r |= ((j >> b) & 1) << (bits - 1 - b)
    return r


WIN = 1024


def expected_groups(sel, T):
    """Per window: (order of its query blocks, [(start in the slice's order, count)])."""
    bits = int(np.ceil(np.log2(T))) if T > 1 else 0
    h = bitrev(sel, bits)
    anchor = sel[np.arange(T), np.argmin(h, axis=1)]
    out = []
    for w0 in range(0, T, WIN):
        idx = np.arange(w0, min(T, w0 + WIN))
        order = idx[np.lexsort((idx, anchor[idx]))]
        groups = []
        p = 0
        while p < len(order):
            q = p
            while q < len(order) and anchor[order[q]] == anchor[order[p]]:
                q += 1
            for s0 in range(p, q, 8):
                groups.append((w0 + s0, min(8, q - s0)))
            p = q
        out.append((order, groups))
    return out


def read_groups(b, slices, T):
    windows = (T + WIN - 1) // WIN
    ws = b.ws_f.view(torch.int32).cpu().numpy()
    a = ((4 * slices * T + 255) // 256) * 256 // 4
    c = ((4 * slices * windows + 255) // 256) * 256 // 4
    order = ws[:slices * T].reshape(slices, T)
    gdesc = ws[a:a + slices * T].reshape(slices, T)
    ngroups = ws[2 * a:2 * a + slices * windows].reshape(slices, windows)
    recs = ws[2 * a + c:2 * a + c + slices * T * 128].reshape(slices, T, 128)  # 512-byte records
    return order, gdesc, ngroups, recs


def check_record(rec, members, sel_rows, coarse_rows, Le, sl):
    """A group record: mask words [8][4], union (uint16 [128]), query blocks
    (uint16 [8]), enrichment tokens (uint16 [8][4]), count, union size, slice."""
    mask = rec[:32].view(np.uint32).reshape(8, 4)
    u16 = rec[32:].view(np.uint16)
    uni, qb, ce = u16[:128], u16[128:136], u16[136:168].reshape(8, 4)
    count, nslots, slice_ = rec[116], rec[117], rec[118]
    union = np.unique(sel_rows[members])
    assert count == len(members) and slice_ == sl and nslots == len(union)
    np.testing.assert_array_equal(uni[:nslots], union)
    np.testing.assert_array_equal(qb[:count], members)
    for q, m in enumerate(members):
        bits = [(int(mask[q, u >> 5]) >> (u & 31)) & 1 for u in range(nslots)]
        assert [union[u] for u in range(nslots) if bits[u]] == sorted(sel_rows[m].tolist())
        np.testing.assert_array_equal(ce[q, :Le], coarse_rows[m, :Le])


@pytest.mark.parametrize("name", ["llsa-fwd-n4096-d64-b2h8-K8-bf16", "grf-64x64-K16", "grf-128x128-K4", "n65536-grf-2heads"])
def test_grouping_rule_and_partition(name):
    if name == "grf-64x64-K16":
        w = synth.Workload("g", 1, 3, 4096, 64, topk=16, kind="grf", length_scale=4.0, grid=(64, 64), seed=91)
    elif name == "grf-128x128-K4":
        w = synth.Workload("g4", 1, 2, 16384, 64, topk=4, kind="grf", length_scale=4.0, grid=(128, 128), seed=93)
    elif name == "n65536-grf-2heads":
        w = synth.Workload("g2", 1, 2, 65536, 64, kind="grf", length_scale=8.0, grid=(256, 256), seed=92)
    else:
        w = synth.WORKLOADS[name]
    x = synth.make_inputs(w, with_dout=False)
    p = params_of(w)
    d = dev_inputs(w, x)
    b = llsa.forward(p, d["q"], d["k"], d["v"])
    torch.cuda.synchronize()
    assert llsa.llsa_get_status() == 0
    s = llsa.get_sizes(p)
    T = s.n_blocks
    order, gdesc, ngroups, recs = read_groups(b, s.slices, T)
    sel = b.sel_idx.cpu().numpy()
    coarse = b.coarse_idx.cpu().numpy()
    sizes = []
    for sl in range(s.slices):
        covered = []
        for wi, (ref_order, ref_groups) in enumerate(expected_groups(sel[sl], T)):
            w0 = wi * WIN
            np.testing.assert_array_equal(order[sl, w0:w0 + len(ref_order)], ref_order)
            assert ngroups[sl, wi] == len(ref_groups)
            got = [(int(g) & 0xFFFF, int(g) >> 16) for g in gdesc[sl, w0:w0 + ngroups[sl, wi]]]
            assert got == ref_groups
            covered += [order[sl][a0:a0 + c] for a0, c in got]
            sizes += [c for _, c in got]
            for k, (a0, c) in enumerate(got):
                if k % 7 == 0:   # a sample of the records
                    check_record(recs[sl, w0 + k], order[sl][a0:a0 + c], sel[sl], coarse[sl], s.enrich_levels, sl)
        assert sorted(np.concatenate(covered).tolist()) == list(range(T))   # a partition
    if w.kind == "grf":
        # spatially structured selections group well (several blocks per group)
        assert np.mean(sizes) > 3.0, np.mean(sizes)
