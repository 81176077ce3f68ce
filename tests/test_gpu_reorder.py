"""Index reordering on the GPU (hierarchical tile order of an image's tokens)
against the oracle's definition: bit-exact, both directions, plus the shape
checks of the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import parity
import hierarchical_sparse_attention_mean_gb300 as llsa
from hierarchical_sparse_attention_mean_gb300 import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


@pytest.mark.parametrize("b,h,side,B,d,dtype", [
    (2, 3, 64, 16, 64, "bf16"),
    (1, 12, 256, 16, 64, "bf16"),     # the 256x256 pixel-token shape
    (1, 2, 32, 4, 32, "fp32"),
    (1, 1, 27, 9, 16, "bf16"),        # s = 3
    (1, 2, 64, 16, 128, "fp32"),
])
def test_reorder_bit_exact_both_ways(b, h, side, B, d, dtype):
    n = side * side
    p = llsa.Params(b, h, n, d, block=B, dtype=dtype)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator().manual_seed(side * 7 + d)
    x = torch.randn(b, h, n, d, generator=g).to(td)
    src = torch.from_numpy(oracle.tile_order(side, side, B))
    xd = x.cuda()
    y = torch.empty_like(xd)
    llsa.llsa_reorder(p, side, side, xd, y)
    back = torch.empty_like(xd)
    llsa.llsa_reorder(p, side, side, y, back, inverse=True)
    torch.cuda.synchronize()
    assert torch.equal(y.cpu(), x[:, :, src])
    assert torch.equal(back.cpu(), x)


def test_reorder_rejects_bad_shapes():
    x = torch.zeros(1, 1, 4096, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    for p, hw, code in ((llsa.Params(1, 1, 4096, 64, block=8, levels=1), (64, 64), -2),   # B not a square
                        (llsa.Params(1, 1, 4096, 64), (32, 128), -2),                   # not square
                        (llsa.Params(1, 1, 4096, 64), (64, 64), None)):
        if code is None:
            llsa.llsa_reorder(p, *hw, x, y)
        else:
            with pytest.raises(llsa.LLSAError) as e:
                llsa.llsa_reorder(p, *hw, x, y)
            assert e.value.code == code
    with pytest.raises(llsa.LLSAError):
        llsa.llsa_reorder(llsa.Params(1, 1, 4096, 64), 64, 64, x, x)     # in place
    torch.cuda.synchronize()


# ------------------------------------------------ reordering inside the path

def _raster_inputs(b, h, side, d, seed):
    g = torch.Generator().manual_seed(seed)
    n = side * side
    return {k: (0.5 * torch.randn(b, h, n, d, generator=g)).to(torch.bfloat16) for k in ("q", "k", "v", "dout")}


def _step(p, x, flags=0):
    dev = {k: t.cuda() for k, t in x.items()}
    llsa.test_set_wait_limit(0, flags)
    try:
        bufs = llsa.forward(p, dev["q"], dev["k"], dev["v"])
        dq, dk, dv = llsa.backward(p, dev["q"], dev["k"], dev["v"], dev["dout"], bufs)
        torch.cuda.synchronize()
    finally:
        llsa.test_set_wait_limit(0, 0)
    assert llsa.llsa_get_status() == 0
    return bufs, dq, dk, dv


@pytest.mark.parametrize("b,h,side,d,K", [
    (2, 3, 64, 64, 8),
    (1, 2, 64, 64, 16),
    (1, 2, 64, 128, 8),
    (1, 2, 64, 128, 16),
    (1, 2, 64, 64, 32),                                 # four key tiles per query block
    (1, 2, 256, 64, 8),                                 # 256 x 256 pixel tokens, three levels
])
def test_raster_order_step_equals_step_on_reordered_tokens(b, h, side, d, K):
    """LLSA_ORDER_RASTER reads the raster tokens as 4 x 4 patches and writes
    o, dq, dk, dv back in raster order: the step must be bit-identical to the
    tile-order step on tokens permuted by the oracle's tile order, run on the
    same (per-query-block) kernels: the same values reach the same arithmetic
    in the same order."""
    x = _raster_inputs(b, h, side, d, seed=side + d + K)
    src = torch.from_numpy(oracle.tile_order(side, side, 16))
    xt = {k: t[:, :, src].contiguous() for k, t in x.items()}
    n = side * side
    pr = llsa.Params(b, h, n, d, topk=K, token_order="raster")
    pt = llsa.Params(b, h, n, d, topk=K)
    assert llsa.workspace_bytes(pr, llsa.OP_FWD) == 0  # no grouping pass in raster order
    br, dqr, dkr, dvr = _step(pr, x)
    bt, dqt, dkt, dvt = _step(pt, xt, llsa.LLSA_TEST_FORCE_PER_BLOCK)
    for name in ("pyr", "sel_idx", "coarse_idx", "lse", "col_ptr", "row_idx"):
        assert torch.equal(getattr(br, name), getattr(bt, name)), name
    for name, got, ref in (("o", br.o, bt.o), ("dq", dqr, dqt), ("dk", dkr, dkt), ("dv", dvr, dvt)):
        assert torch.equal(got[:, :, src.cuda()], ref), name


def test_raster_order_step_against_oracle():
    """The raster-order step against the oracle run on the tokens in the
    oracle's tile order, with the GPU's selection (so near-ties cannot move
    it): pyramids, o and lse (lse stays in tile order), dq, dk, dv."""
    b, h, side, d, K = 1, 2, 64, 64, 8
    n, B = side * side, 16
    x = _raster_inputs(b, h, side, d, seed=77)
    src = oracle.tile_order(side, side, B)
    p = llsa.Params(b, h, n, d, topk=K, token_order="raster")
    bufs, dq, dk, dv = _step(p, x)
    s = llsa.get_sizes(p)
    L, scale = s.levels, s.scale
    xt = {k: t.float().numpy().reshape(b * h, n, d)[:, src] for k, t in x.items()}
    pyr = bufs.pyr.cpu().numpy()
    sel = bufs.sel_idx.cpu().numpy()
    coarse = bufs.coarse_idx.cpu().numpy()
    o_r = parity.f64(bufs.o).reshape(b * h, n, d)
    lse_r = bufs.lse.cpu().numpy().astype(np.float64).reshape(b * h, n)
    grads = [parity.f64(t).reshape(b * h, n, d) for t in (dq, dk, dv)]
    for sl in range(b * h):
        qp, kp, vp = (oracle.pool(xt[k][sl], B, L) for k in ("q", "k", "v"))
        for t, ref in enumerate((qp, kp, vp)):
            assert np.abs(pyr[t, sl] - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())
        o, lse = oracle.fwd(xt["q"][sl], xt["k"][sl], xt["v"][sl], kp, vp, B, L, L, sel[sl], coarse[sl], scale)
        parity.assert_close("o", o_r[sl][src], o, "bf16")
        parity.assert_lse(lse_r[sl], lse)
        ref = oracle.bwd(xt["q"][sl], xt["k"][sl], xt["v"][sl], kp, vp, o, lse, xt["dout"][sl], B, L, L,
                         sel[sl], coarse[sl], scale)
        for name, got, r in zip(("dq", "dk", "dv"), grads, ref):
            parity.assert_close(name, got[sl][src], r, "bf16")


def test_raster_order_outside_the_tensor_core_path_is_refused():
    n, d = 4096, 64
    q = torch.zeros(1, 1, n, d, dtype=torch.float32, device="cuda")
    p = llsa.Params(1, 1, n, d, dtype="fp32", token_order="raster")
    bufs = llsa.Buffers(p)
    llsa.llsa_pool(p, q, q, q, bufs.pyr)  # the pool takes any dtype
    with pytest.raises(llsa.LLSAError) as e:
        llsa.llsa_fwd(p, q, q, q, bufs.pyr, bufs.sel_idx, bufs.coarse_idx, bufs.o, bufs.lse, bufs.ws_f)
    assert e.value.code == -8
    qa = q.to(torch.bfloat16)
    # ALLK (several coarse keys per level) and K_1 = 4 (no per-block
    # tensor-core forward) stay in tile order
    for kw in (dict(enrich_rule="allk"), dict(topk=4)):
        pa = llsa.Params(1, 1, n, d, token_order="raster", **kw)
        ba = llsa.Buffers(pa)
        with pytest.raises(llsa.LLSAError) as e:
            llsa.llsa_fwd(pa, qa, qa, qa, ba.pyr, ba.sel_idx, ba.coarse_idx, ba.o, ba.lse, ba.ws_f)
        assert e.value.code == -8
    torch.cuda.synchronize()
    assert llsa.llsa_get_status() == 0


def test_raster_order_pool_fp32_equals_pool_on_reordered_tokens():
    """The fp32 pool reads raster tokens as 4 x 4 patches in the same order
    as the tile-order pool reads the permuted tokens: the pyramids are equal."""
    side, d = 64, 32
    n = side * side
    g = torch.Generator().manual_seed(5)
    x = {k: torch.randn(1, 2, n, d, generator=g) for k in ("q", "k", "v")}
    src = torch.from_numpy(oracle.tile_order(side, side, 16))
    pr = llsa.Params(1, 2, n, d, dtype="fp32", token_order="raster")
    pt = llsa.Params(1, 2, n, d, dtype="fp32")
    s = llsa.get_sizes(pt)
    out = []
    for p, xs in ((pr, x), (pt, {k: t[:, :, src].contiguous() for k, t in x.items()})):
        dev = {k: t.cuda() for k, t in xs.items()}
        pyr = torch.empty(3, 2, s.pyr_rows, d, device="cuda")
        llsa.llsa_pool(p, dev["q"], dev["k"], dev["v"], pyr)
        out.append(pyr)
    torch.cuda.synchronize()
    assert torch.equal(out[0], out[1])


def test_raster_order_autograd():
    """llsa_attention with token_order="raster": output and input gradients
    equal the tile-order call on permuted tokens (per-block forward forced on
    both, so the arithmetic is the same)."""
    x = _raster_inputs(1, 2, 64, 64, seed=91)
    src = torch.from_numpy(oracle.tile_order(64, 64, 16)).cuda()
    res = []
    llsa.test_set_wait_limit(0, llsa.LLSA_TEST_FORCE_PER_BLOCK)
    try:
        for order in ("raster", "tile"):
            t = {k: v.cuda() for k, v in x.items()}
            if order == "tile":
                t = {k: v[:, :, src].contiguous() for k, v in t.items()}
            q, k, v = (t[n].requires_grad_(True) for n in ("q", "k", "v"))
            o = llsa.llsa_attention(q, k, v, token_order=order)
            o.backward(t["dout"])
            res.append((o.detach(), q.grad, k.grad, v.grad))
        torch.cuda.synchronize()
    finally:
        llsa.test_set_wait_limit(0, 0)
    assert llsa.llsa_get_status() == 0
    for got, ref in zip(res[0], res[1]):
        assert torch.equal(got[:, :, src], ref)
