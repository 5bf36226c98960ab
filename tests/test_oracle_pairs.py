"""Pins of the oracle's complex and dual-number GEMM (CPU only).

"Flexible Performant GEMM Kernels on GPUs", section 5.4: complex numbers
x + y i with i*i = -1, dual numbers x + y eps with eps*eps = 0, stored
interleaved.  The oracle is pinned by hand-worked products (tests/golden), by
numpy's complex128 matmul on small integers (exact), by the representation of
both number systems as 2 x 2 real matrices (complex: [[a, -b], [b, a]]; dual:
[[a, b], [0, a]]), under which the pair GEMM is a real block GEMM computed by
numpy in int64, and by the reduction to the real oracle when every unit part
is zero.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
from dense_gemm_epilogues_gb300 import inputs as I

HERE = os.path.dirname(os.path.abspath(__file__))
DT = {"f32": O.F32, "f16": O.F16, "bf16": O.BF16}
LAY = {"N": O.LAYOUT_N, "T": O.LAYOUT_T}
BIAS = {"none": O.BIAS_NONE, "col": O.BIAS_COL, "row": O.BIAS_ROW}
ACT = {"none": O.ACT_NONE, "relu": O.ACT_RELU}
UNIT = {"complex": O.UNIT_IMAGINARY, "dual": O.UNIT_DUAL}
LAYOUTS = ["NN", "NT", "TN", "TT"]
SMALL = I.Dist("small", -3, 3)


def run_pairs(inp: I.PairInputs, nthreads=None):
    p = inp.problem
    D = O.gemm_pairs(UNIT[p.unit], DT[p.ab], LAY[p.layout_a], LAY[p.layout_b], p.M, p.N, p.K,
                     p.alpha, inp.A, p.lda, inp.B, p.ldb, beta=p.beta,
                     c_dtype=DT[p.c] if p.c else O.F32, C=inp.C, ldc=p.ldc if p.c else 0,
                     bias_dtype=DT[p.bias] if p.bias else O.F32, bias=inp.bias,
                     bias_mode=BIAS[p.bias_mode], act=ACT[p.act], d_dtype=DT[p.d], ldd=p.ldd,
                     nthreads=nthreads, c_act=ACT[p.c_act])
    return D[:, :p.N]


def _golden():
    with open(os.path.join(HERE, "golden", "hand_worked_pairs.json")) as f:
        return json.load(f)["cases"]


def _with_values(p: I.PairProblem, a, b, c=None, bias=None) -> I.PairInputs:
    """Inputs of problem p holding the given logical pair matrices."""
    a = torch.tensor(a, dtype=torch.float64).to(I.TORCH_DTYPES[p.ab])
    b = torch.tensor(b, dtype=torch.float64).to(I.TORCH_DTYPES[p.ab])
    A = I._store_pairs(a, p.layout_a, p.lda, p.ab)
    B = I._store_pairs(b, p.layout_b, p.ldb, p.ab)
    C = None
    if c is not None:
        C = I._store_pairs(torch.tensor(c, dtype=torch.float64).to(I.TORCH_DTYPES[p.c]), "T",
                           p.ldc, p.c)
    bt = torch.tensor(bias, dtype=torch.float32) if bias is not None else None
    return I.PairInputs(A=A, B=B, C=C, bias=bt, problem=p, logical={"a": a, "b": b})


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("case", _golden(), ids=lambda c: c["name"])
def test_hand_worked_pairs(case, layout):
    p = I.PairProblem(case["name"], case["unit"], "f16", layout[0], layout[1], case["M"],
                      case["N"], case["K"], alpha=case.get("alpha", 1.0),
                      beta=case.get("beta", 0.0), c="f32" if "C" in case else None,
                      bias="f32" if "bias" in case else None,
                      bias_mode="col" if "bias" in case else "none", act=case.get("act", "none"),
                      pad_a=1, pad_b=2, pad_d=1)
    inp = _with_values(p, case["A"], case["B"], case.get("C"), case.get("bias"))
    np.testing.assert_array_equal(run_pairs(inp), np.array(case["D"], dtype=np.float32))


def _as_complex(x: torch.Tensor) -> np.ndarray:
    x = x.double().numpy()
    return x[..., 0] + 1j * x[..., 1]


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("ab", ["f16", "bf16", "f32"])
def test_complex_small_integers_match_numpy(layout, ab):
    """Small-integer data: every product and sum is exact, so the oracle must
    equal numpy's complex128 matmul exactly (alpha, beta, C included)."""
    p = I.PairProblem("cnp", "complex", ab, layout[0], layout[1], 13, 11, 17, alpha=2.0,
                      beta=-3.0, c="f32", dist_a=SMALL, dist_b=SMALL, dist_c=SMALL, pad_a=2,
                      pad_b=1, pad_c=3)
    inp = I.generate_pairs(p, 50)
    ref = 2.0 * (_as_complex(inp.logical["a"]) @ _as_complex(inp.logical["b"])) \
        - 3.0 * _as_complex(inp.logical["c"])
    got = run_pairs(inp).astype(np.float64)
    np.testing.assert_array_equal(got[..., 0], ref.real)
    np.testing.assert_array_equal(got[..., 1], ref.imag)


def _blocks(x: torch.Tensor, unit: str) -> np.ndarray:
    """Each pair (a, b) as a 2 x 2 integer block: complex [[a, -b], [b, a]],
    dual [[a, b], [0, a]]; a (rows x cols) pair matrix -> (2 rows x 2 cols)."""
    a = x[..., 0].long().numpy()
    b = x[..., 1].long().numpy()
    r, c = a.shape
    out = np.zeros((2 * r, 2 * c), dtype=np.int64)
    out[0::2, 0::2] = a
    out[1::2, 1::2] = a
    if unit == "complex":
        out[0::2, 1::2] = -b
        out[1::2, 0::2] = b
    else:
        out[0::2, 1::2] = b
    return out


@pytest.mark.parametrize("unit", ["complex", "dual"])
@pytest.mark.parametrize("layout", LAYOUTS)
def test_block_matrix_representation(unit, layout):
    """The pair GEMM equals the real block GEMM of the 2 x 2 representations
    (numpy int64 matmul); the product's pair is read off the first block row:
    real part at [0, 0], unit part at [1, 0] (complex) or [0, 1] (dual)."""
    p = I.PairProblem("blk", unit, "f16", layout[0], layout[1], 7, 9, 12, dist_a=SMALL,
                      dist_b=SMALL)
    inp = I.generate_pairs(p, 51)
    prod = _blocks(inp.logical["a"], unit) @ _blocks(inp.logical["b"], unit)
    got = run_pairs(inp).astype(np.float64)
    np.testing.assert_array_equal(got[..., 0], prod[0::2, 0::2])
    unit_part = prod[1::2, 0::2] if unit == "complex" else prod[0::2, 1::2]
    np.testing.assert_array_equal(got[..., 1], unit_part)
    # The blocks are closed under the product: the other entries agree too.
    np.testing.assert_array_equal(prod[1::2, 1::2], prod[0::2, 0::2])


@pytest.mark.parametrize("unit", ["complex", "dual"])
@pytest.mark.parametrize("ab", ["f16", "bf16"])
def test_zero_unit_parts_reduce_to_real_oracle(unit, ab):
    """With every unit part of A and B zero, the real parts are the real GEMM
    (bit for bit: the same fp64 sums in the same order) and the unit parts
    carry only beta * C + bias."""
    p = I.PairProblem("real", unit, ab, "T", "N", 21, 19, 33, alpha=1.5, beta=0.5, c="f32",
                      bias="f32", bias_mode="col", act="relu")
    inp = I.generate_pairs(p, 52)
    inp.A.view(-1, 2)[:, 1] = 0
    inp.B.view(-1, 2)[:, 1] = 0
    got = run_pairs(inp)
    Ar = inp.A[..., 0].contiguous()
    Br = inp.B[..., 0].contiguous()
    Cr = inp.C[..., 0].contiguous()
    real, _ = O.gemm(DT[ab], O.LAYOUT_T, O.LAYOUT_N, p.M, p.N, p.K, 1.5, Ar, p.lda, Br, p.ldb,
                     beta=0.5, c_dtype=O.F32, C=Cr, ldc=p.ldc, bias_dtype=O.F32,
                     bias=inp.bias[:, 0].contiguous(), bias_mode=O.BIAS_COL, act=O.ACT_RELU)
    np.testing.assert_array_equal(got[..., 0], real)
    expect_u = np.maximum(0.5 * inp.logical["c"][..., 1].double().numpy()
                          + inp.bias[:, 1].double().numpy()[None, :], 0.0).astype(np.float32)
    np.testing.assert_array_equal(got[..., 1], expect_u)


@pytest.mark.parametrize("unit", ["complex", "dual"])
def test_epilogue_per_part_row_bias_and_relu_on_c(unit):
    """Row bias pairs, ReLU on C and on D, each applied to the two parts apart."""
    p = I.PairProblem("epi", unit, "f16", "N", "T", 6, 5, 4, alpha=1.0, beta=2.0, c="f32",
                      bias="f32", bias_mode="row", act="relu", c_act="relu", dist_a=SMALL,
                      dist_b=SMALL, dist_c=SMALL, dist_bias=SMALL)
    inp = I.generate_pairs(p, 53)
    a, b = _as_complex(inp.logical["a"]), _as_complex(inp.logical["b"])
    if unit == "complex":
        prod = a @ b
    else:   # (a + b eps)(c + d eps) = ac + (ad + bc) eps
        prod = a.real @ b.real + 1j * (a.real @ b.imag + a.imag @ b.real)
    c = np.maximum(inp.logical["c"].double().numpy(), 0.0)
    bias = inp.bias.double().numpy()
    for part, val in ((0, prod.real), (1, prod.imag)):
        expect = np.maximum(val + 2.0 * c[..., part] + bias[:, part][:, None], 0.0)
        np.testing.assert_array_equal(run_pairs(inp)[..., part], expect.astype(np.float32))


def test_entries_match_full_and_16_bit_outputs():
    p = I.PairProblem("ent", "complex", "bf16", "T", "T", 30, 26, 40, beta=1.0, c="bf16", d="bf16")
    inp = I.generate_pairs(p, 54)
    full = run_pairs(inp)
    rows = np.array([0, 29, 7, 15, 29], dtype=np.int64)
    cols = np.array([0, 25, 13, 0, 1], dtype=np.int64)
    out = O.gemm_pairs_entries(O.UNIT_IMAGINARY, O.BF16, O.LAYOUT_T, O.LAYOUT_T, p.M, p.N, p.K,
                               1.0, inp.A, p.lda, inp.B, p.ldb, rows, cols, beta=1.0,
                               c_dtype=O.BF16, C=inp.C, ldc=p.ldc, d_dtype=O.BF16)
    np.testing.assert_array_equal(out, full[rows, cols])
    # and each part is the round-to-nearest-even bfloat16 of the fp32 result
    ref = run_pairs(I.PairInputs(inp.A, inp.B, inp.C, None, p.with_(d="f32")))
    np.testing.assert_array_equal(out[:, 0], [O.bf16_from_double(float(x)) for x in ref[rows, cols, 0]])


def test_invalid_pair_problems():
    A = np.zeros(8, dtype=np.int8)
    with pytest.raises(ValueError):   # integer parts are not supported
        O.gemm_pairs(O.UNIT_IMAGINARY, O.S8, O.LAYOUT_N, O.LAYOUT_N, 2, 2, 2, 1.0, A, 2, A, 2,
                     d_dtype=O.S32)
    F = np.zeros(8, dtype=np.float32)
    with pytest.raises(ValueError):   # unknown unit
        O.gemm_pairs(7, O.F32, O.LAYOUT_N, O.LAYOUT_N, 2, 2, 2, 1.0, F, 2, F, 2)
