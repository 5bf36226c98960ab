"""Host checks of the diagonal-operand problem description (no GPU): the dense
equivalent the parity tests hand to the oracle is the GEMM with the diagonal
written out, so the oracle's result on it must equal the closed form
d[i] * x(i,j) (left) or x(i,j) * d[j] (right) -- section 5.2 of "Flexible
Performant GEMM Kernels on GPUs" -- for every side, layout and padding."""
import numpy as np
import pytest
import torch

from dense_gemm_epilogues_gb300 import inputs as I

import parity_helpers as H


@pytest.mark.parametrize("side", ["left", "right"])
@pytest.mark.parametrize("layout", ["N", "T"])
@pytest.mark.parametrize("ab", ["f16", "s8"])
def test_dense_equivalent_matches_closed_form(side, layout, ab):
    dist = I.I8 if ab == "s8" else I.U11
    d_out = "s32" if ab == "s8" else "f32"
    p = I.DiagProblem("dh", ab, side, layout, 23, 17, pad_x=3, d=d_out, dist_diag=dist, dist_x=dist)
    dinp = I.generate_diag(p, 31)
    D = H.oracle_full(H.dense_inputs_of(dinp))
    x = dinp.x_logical.double()
    dg = dinp.diag.double()
    closed = dg[:, None] * x if side == "left" else x * dg[None, :]
    if ab == "s8":
        np.testing.assert_array_equal(D, closed.numpy().astype(np.int32))
    else:   # fp16 x fp16 products are exact in fp32
        np.testing.assert_array_equal(D, closed.float().numpy())


def test_storage_of_x_follows_its_layout():
    p = I.DiagProblem("dh2", "f32", "left", "N", 5, 4, pad_x=2)
    dinp = I.generate_diag(p, 32)
    assert p.ldx == 7 and dinp.X.shape == (4, 7)                 # column-major: N columns of ldx
    assert torch.equal(dinp.X[:, :5], dinp.x_logical.t())
    assert torch.all(torch.isnan(dinp.X[:, 5:]))                  # poisoned padding
    q = p.with_(layout_x="T")
    assert q.ldx == 6 and I.generate_diag(q, 32).X.shape == (5, 6)
    assert q.dense().K == 5 and p.with_(side="right").dense().K == 4
