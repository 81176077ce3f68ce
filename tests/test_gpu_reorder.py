"""Index reordering on the GPU (hierarchical tile order of an image's tokens)
against the oracle's definition: bit-exact, both directions, plus the shape
checks of the C ABI."""
import numpy as np
import pytest
import torch

import oracle
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
