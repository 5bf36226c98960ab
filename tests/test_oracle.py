"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these tests compares the oracle with itself: each expected value comes
from a hand-worked example, a closed form, an algebraic identity, a library
routine (numpy integer matmul, numpy's IEEE float16 conversion), or exact
rational arithmetic.  No GPU is needed.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from dense_gemm_epilogues_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

DT = {"f32": O.F32, "f16": O.F16, "bf16": O.BF16, "s8": O.S8, "s32": O.S32}
LAY = {"N": O.LAYOUT_N, "T": O.LAYOUT_T}
BIAS = {"none": O.BIAS_NONE, "col": O.BIAS_COL, "row": O.BIAS_ROW}
ACT = {"none": O.ACT_NONE, "relu": O.ACT_RELU}


def run_oracle(inp: I.Inputs, loop_order=0, nthreads=None):
    p = inp.problem
    D, ovf = O.gemm(DT[p.ab], LAY[p.layout_a], LAY[p.layout_b], p.M, p.N, p.K, p.alpha,
                    inp.A, p.lda, inp.B, p.ldb, beta=p.beta,
                    c_dtype=DT[p.c] if p.c else O.F32, C=inp.C, ldc=p.ldc if p.c else 0,
                    bias_dtype=DT[p.bias] if p.bias else O.F32, bias=inp.bias,
                    bias_mode=BIAS[p.bias_mode], act=ACT[p.act], d_dtype=DT[p.d], ldd=p.ldd,
                    loop_order=loop_order, nthreads=nthreads, c_act=ACT[p.c_act],
                    out_scale=p.out_scale, a_act=ACT[p.a_act], a_scale=p.a_scale,
                    b_act=ACT[p.b_act], b_scale=p.b_scale)
    return D[:, :p.N], ovf


def as_f64(D, dtype):
    return O.decode(D, DT[dtype])


def logical_f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy() if t.dtype != torch.int8 else t.to(torch.int64).numpy()


LAYOUTS = ["NN", "NT", "TN", "TT"]


# --------------------------------------------------------------------------
# Hand-worked examples (tests/golden/hand_worked.json)
# --------------------------------------------------------------------------

def _golden_cases():
    with open(os.path.join(GOLDEN, "hand_worked.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
@pytest.mark.parametrize("layout", LAYOUTS)
def test_hand_worked_examples(case, layout):
    a = torch.tensor(case["A"], dtype=torch.float64)
    b = torch.tensor(case["B"], dtype=torch.float64)
    M, K = a.shape
    N = b.shape[1]
    ab = case["ab"]
    td = I.TORCH_DTYPES[ab]
    A = I._store(a.to(td), layout[0], M if layout[0] == "N" else K, ab)
    B = I._store(b.to(td), layout[1], K if layout[1] == "N" else N, ab)
    lda = M if layout[0] == "N" else K
    ldb = K if layout[1] == "N" else N
    C = None
    if "C" in case:
        C = torch.tensor(case["C"], dtype=torch.float64).to(I.TORCH_DTYPES[case["c"]]).contiguous()
    bias = None
    if case["bias_mode"] != "none":
        bias = torch.tensor(case["bias"], dtype=torch.float64).to(
            I.TORCH_DTYPES[case["bias_dtype"]])
    D, ovf = O.gemm(DT[ab], LAY[layout[0]], LAY[layout[1]], M, N, K, case["alpha"], A, lda, B,
                    ldb, beta=case["beta"], c_dtype=DT[case["c"]], C=C, ldc=N,
                    bias_dtype=DT[case.get("bias_dtype", "f32")], bias=bias,
                    bias_mode=BIAS[case["bias_mode"]], act=ACT[case["act"]],
                    d_dtype=DT[case["d"]], c_act=ACT[case.get("c_act", "none")],
                    a_act=ACT[case.get("a_act", "none")], a_scale=case.get("a_scale", 1.0),
                    b_act=ACT[case.get("b_act", "none")], b_scale=case.get("b_scale", 1.0))
    assert ovf == 0
    if "D_bits" in case:
        assert D.tolist() == case["D_bits"]
    else:
        assert D.astype(np.float64).tolist() == case["D"]


# --------------------------------------------------------------------------
# Closed forms and identities
# --------------------------------------------------------------------------

@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("ab", ["f16", "bf16", "f32", "s8"])
def test_identity_A_gives_op_B(layout, ab):
    """A = I (M = K): D = op(B) exactly, in every layout."""
    n, N = 13, 9
    d = "s32" if ab == "s8" else "f32"
    p = I.Problem("id", ab, layout[0], layout[1], n, N, n, d=d,
                  dist_a=I.Dist("zeros"), dist_b=I.Dist("small", -100, 100), pad_a=3, pad_b=2)
    inp = I.generate(p, 1, keep_logical=True)
    eye = torch.eye(n, dtype=torch.float32).to(I.TORCH_DTYPES[ab])
    inp.A = I._store(eye, p.layout_a, p.lda, ab)
    D, _ = run_oracle(inp)
    np.testing.assert_array_equal(D.astype(np.float64), logical_f64(inp.logical["b"]))


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("ab", ["f16", "bf16", "f32", "s8"])
def test_all_ones_gives_K(layout, ab):
    """All-ones A and B: every entry of D equals K (checks ld/layout indexing,
    with padded leading dimensions whose padding is poisoned)."""
    M, N, K = 7, 11, 37
    d = "s32" if ab == "s8" else "f32"
    p = I.Problem("ones", ab, layout[0], layout[1], M, N, K, d=d, dist_a=I.Dist("ones"),
                  dist_b=I.Dist("ones"), pad_a=5, pad_b=3, pad_d=4)
    D, _ = run_oracle(I.generate(p, 2))
    assert np.all(D.astype(np.float64) == K)


def _numpy_expected(inp: I.Inputs) -> np.ndarray:
    """alpha * a @ b + beta * c + bias, then ReLU, in exact int64 (small ints)."""
    p = inp.problem
    a = inp.logical["a"].to(torch.int64).numpy() if p.ab == "s8" else \
        inp.logical["a"].to(torch.float64).numpy().astype(np.int64)
    b = inp.logical["b"].to(torch.int64).numpy() if p.ab == "s8" else \
        inp.logical["b"].to(torch.float64).numpy().astype(np.int64)
    v = int(p.alpha) * (a @ b)
    if p.beta != 0:
        c = inp.logical["c"].to(torch.float64).numpy().astype(np.int64)
        if p.c_act == "relu":
            c = np.maximum(c, 0)
        v = v + int(p.beta) * c
    if p.bias_mode == "col":
        v = v + inp.bias.to(torch.float64).numpy().astype(np.int64)[None, :]
    elif p.bias_mode == "row":
        v = v + inp.bias.to(torch.float64).numpy().astype(np.int64)[:, None]
    if p.act == "relu":
        v = np.maximum(v, 0)
    return v


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("ab", ["f16", "bf16", "f32", "s8"])
@pytest.mark.parametrize("epi", ["plain", "alpha_beta", "bias_col_relu", "bias_row_relu",
                                 "relu_on_c_and_d"])
def test_small_integers_match_numpy_int_matmul(layout, ab, epi):
    """Small-integer data makes every step exact, so the oracle must equal
    numpy's int64 matmul of the logical matrices bit for bit.  Non-square
    shapes catch a transposed operand; the epilogue variants catch a dropped
    term, a wrong sign and a row/column mix-up of the bias."""
    M, N, K = 19, 23, 29
    kw = dict(dist_a=I.Dist("small", -3, 3), dist_b=I.Dist("small", -3, 3), pad_a=1, pad_b=2)
    is_int = ab == "s8"
    cd = "s32" if is_int else "f32"
    if epi == "alpha_beta":
        kw.update(alpha=3.0, beta=-2.0, c=cd, dist_c=I.Dist("small", -50, 50), pad_c=3)
    elif epi == "bias_col_relu":
        kw.update(bias=cd, bias_mode="col", act="relu", dist_bias=I.Dist("small", -20, 20),
                  alpha=2.0, beta=1.0, c=cd, dist_c=I.Dist("small", -5, 5))
    elif epi == "bias_row_relu":
        kw.update(bias=cd, bias_mode="row", act="relu", dist_bias=I.Dist("small", -20, 20))
    elif epi == "relu_on_c_and_d":
        kw.update(bias=cd, bias_mode="col", act="relu", c_act="relu", alpha=1.0, beta=2.0, c=cd,
                  dist_c=I.Dist("small", -30, 30), dist_bias=I.Dist("small", -20, 20))
    p = I.Problem("small", ab, layout[0], layout[1], M, N, K, d=cd, **kw)
    inp = I.generate(p, 3, keep_logical=True)
    D, ovf = run_oracle(inp)
    assert ovf == 0
    np.testing.assert_array_equal(D.astype(np.int64), _numpy_expected(inp))


@pytest.mark.parametrize("ab", ["f16", "f32"])
def test_loop_orders_agree(ab):
    """The dot-product (i, j, k) order and the k-outermost outer-product order
    of the CUTLASS page add the same products in the same k order for every
    entry, so they agree bit for bit, on random data too."""
    p = I.Problem("lo", ab, "N", "T", 17, 13, 15, alpha=1.25, beta=-0.75, c="f32",
                  bias="f32", bias_mode="col", act="relu", pad_a=2)
    inp = I.generate(p, 4)
    D0, _ = run_oracle(inp, loop_order=0)
    D1, _ = run_oracle(inp, loop_order=1)
    np.testing.assert_array_equal(D0, D1)
    pi = I.Problem("lo8", "s8", "T", "T", 9, 10, 33, d="s32", dist_a=I.I8, dist_b=I.I8)
    inp = I.generate(pi, 5)
    np.testing.assert_array_equal(run_oracle(inp, 0)[0], run_oracle(inp, 1)[0])


def test_linearity_in_alpha_and_beta():
    """gemm(2*alpha) = 2*gemm(alpha) and gemm(alpha, beta, C) - gemm(alpha, 0) = beta*C,
    exact on small-integer data."""
    p = I.Problem("lin", "f16", "T", "N", 12, 10, 20, alpha=3.0, c="f32",
                  dist_a=I.Dist("small", -4, 4), dist_b=I.Dist("small", -4, 4),
                  dist_c=I.Dist("small", -9, 9))
    inp = I.generate(p, 6, keep_logical=True)
    D1, _ = run_oracle(inp)
    inp2 = I.Inputs(inp.A, inp.B, inp.C, None, p.with_(alpha=6.0))
    D2, _ = run_oracle(inp2)
    np.testing.assert_array_equal(D2, 2 * D1)
    inp3 = I.Inputs(inp.A, inp.B, inp.C, None, p.with_(beta=-2.5))
    D3, _ = run_oracle(inp3)
    np.testing.assert_array_equal(D3 - D1, np.float32(-2.5) * inp.C.numpy())


@pytest.mark.parametrize("layout", LAYOUTS)
def test_transpose_identity(layout):
    """D = op(A) op(B) equals (op(B)^T op(A)^T)^T: storing op(B)^T is the same
    storage as B with the other layout letter."""
    M, N, K = 9, 14, 11
    p = I.Problem("tr", "f32", layout[0], layout[1], M, N, K)
    inp = I.generate(p, 7)
    D, _ = run_oracle(inp)
    flip = {"N": "T", "T": "N"}
    Dt, _ = O.gemm(O.F32, LAY[flip[layout[1]]], LAY[flip[layout[0]]], N, M, K, 1.0,
                   inp.B, p.ldb, inp.A, p.lda, d_dtype=O.F32)
    np.testing.assert_array_equal(Dt.T, D)


def test_linearisation_offsets():
    """Column-major linearisation n*M + m (section 3.2, Figure 4): a matrix whose
    storage holds its own linear index reads back a(i, k) = i + k*lda."""
    M, K, lda = 5, 4, 7
    store = torch.arange(K * lda, dtype=torch.float32).reshape(K, lda)
    sel = torch.zeros((K, 1), dtype=torch.float32)   # B = e_k selects column k of A
    for k in range(K):
        sel.zero_()
        sel[k, 0] = 1.0
        D, _ = O.gemm(O.F32, O.LAYOUT_N, O.LAYOUT_N, M, 1, K, 1.0, store, lda, sel, K)
        assert D[:, 0].tolist() == [float(i + k * lda) for i in range(M)]


def test_diagonal_operand():
    """A = diag(d) gives D[i,j] = d_i * b(i,j) (the diagonal GEMM of section 5.2)."""
    n, N = 16, 8
    p = I.Problem("diag", "f32", "N", "T", n, N, n, dist_a=I.Dist("zeros"))
    inp = I.generate(p, 8, keep_logical=True)
    d = torch.linspace(-2, 3, n, dtype=torch.float32)
    inp.A = I._store(torch.diag(d), "N", n, "f32")
    D, _ = run_oracle(inp)
    expect = (d.double()[:, None] * inp.logical["b"].double()).float().numpy()
    np.testing.assert_array_equal(D, expect)


def test_diagonal_operand_right():
    """B = diag(d) gives D[i,j] = a(i,j) * d_j (section 5.2 with the diagonal on
    the right): column j of A scaled by d_j, in both layouts of A."""
    M, n = 9, 13
    d = torch.linspace(-1.5, 2.5, n, dtype=torch.float32)
    for la in ("N", "T"):
        p = I.Problem("diag_r", "f32", la, "N", M, n, n, dist_b=I.Dist("zeros"))
        inp = I.generate(p, 11, keep_logical=True)
        inp.B = I._store(torch.diag(d), "N", n, "f32")
        D, _ = run_oracle(inp)
        expect = (inp.logical["a"].double() * d.double()[None, :]).float().numpy()
        np.testing.assert_array_equal(D, expect)


def test_diagonal_operand_int8_with_c():
    """int8, A = diag(d): D = alpha*d_i*b(i,j) + beta*C[i,j], exact in int32."""
    n, N = 12, 7
    p = I.Problem("diag_i8", "s8", "N", "T", n, N, n, alpha=3.0, beta=-2.0, c="s32", d="s32",
                  dist_a=I.Dist("zeros"), dist_b=I.I8, dist_c=I.Dist("int", -1000, 1000))
    inp = I.generate(p, 12, keep_logical=True)
    d = torch.arange(-6, 6, dtype=torch.int64) * 21          # -126 .. 105
    inp.A = I._store(torch.diag(d).to(torch.int8), "N", n, "s8")
    D, _ = run_oracle(inp)
    expect = 3 * d[:, None] * inp.logical["b"].long() - 2 * inp.logical["c"].long()
    np.testing.assert_array_equal(D, expect.numpy().astype(np.int32))


def test_epilogue_only_when_A_is_zero():
    """A = 0: D = cast(beta*C + bias) and ReLU output is non-negative."""
    p = I.Problem("epi", "bf16", "T", "N", 10, 12, 8, beta=0.5, c="f32", d="bf16",
                  bias="f32", bias_mode="col", act="relu", dist_a=I.Dist("zeros"))
    inp = I.generate(p, 9)
    D, _ = run_oracle(inp)
    v = 0.5 * inp.C.double().numpy() + inp.bias.double().numpy()[None, :]
    v = np.maximum(v, 0.0)
    expect = np.array([[O.bf16_from_double(x) for x in row] for row in v], dtype=np.uint16)
    np.testing.assert_array_equal(D, expect)
    assert np.all(as_f64(D, "bf16") >= 0)


def test_beta_zero_ignores_C():
    """beta == 0: C is not read, so NaNs in C do not reach D (and C may be NULL)."""
    p = I.Problem("b0", "f16", "T", "N", 6, 6, 6, beta=0.0, c="f32")
    inp = I.generate(p, 10)
    inp.C.fill_(float("nan"))
    D, _ = run_oracle(inp)
    assert np.all(np.isfinite(D))
    inp.C = None
    D2, _ = run_oracle(I.Inputs(inp.A, inp.B, None, None, p.with_(c=None)))
    np.testing.assert_array_equal(D, D2)


# --------------------------------------------------------------------------
# Exact arithmetic (brute force on tiny inputs)
# --------------------------------------------------------------------------

def test_random_float_within_fp64_rounding_of_exact_sum():
    """Exact rational sum of the products vs the oracle's fp64 accumulation:
    the difference is within the standard bound K * 2^-53 * sum |a||b| (plus
    the final fp32 rounding of the output)."""
    M, N, K = 5, 4, 64
    p = I.Problem("exact", "f32", "T", "T", M, N, K, alpha=1.0)
    inp = I.generate(p, 11, keep_logical=True)
    D, _ = run_oracle(inp)
    a = inp.logical["a"].double().numpy()
    b = inp.logical["b"].double().numpy()
    for i in range(M):
        for j in range(N):
            exact = sum(Fraction(float(a[i, k])) * Fraction(float(b[k, j])) for k in range(K))
            mag = sum(abs(float(a[i, k]) * float(b[k, j])) for k in range(K))
            bound = K * 2.0 ** -53 * mag + abs(float(exact)) * 2.0 ** -24
            assert abs(float(D[i, j]) - float(exact)) <= bound


def test_int32_overflow_is_flagged():
    """|sum| = K * 16384 > 2^31 - 1 for K = 131073 (all -128): the oracle keeps the
    low 32 bits and reports the overflow."""
    K = 131073
    A = torch.full((1, K), -128, dtype=torch.int8)
    B = torch.full((K, 1), -128, dtype=torch.int8)
    D, ovf = O.gemm(O.S8, O.LAYOUT_T, O.LAYOUT_N, 1, 1, K, 1.0, A, K, B, K, d_dtype=O.S32)
    assert ovf == 1
    assert int(D[0, 0]) == ((K * 16384 + 2**31) % 2**32) - 2**31
    D, ovf = O.gemm(O.S8, O.LAYOUT_T, O.LAYOUT_N, 1, 1, 8192, 1.0, A, K, B, K, d_dtype=O.S32)
    assert ovf == 0 and int(D[0, 0]) == 8192 * 16384


# --------------------------------------------------------------------------
# Output casts (IEEE 754 round to nearest, ties to even)
# --------------------------------------------------------------------------

F16_CASES = [  # (value, expected bits) worked from the binary16 definition
    (1.0, 0x3C00), (-2.0, 0xC000), (65504.0, 0x7BFF), (65519.99, 0x7BFF), (65520.0, 0x7C00),
    (1 + 2**-11, 0x3C00), (1 + 3 * 2**-11, 0x3C02), (1 + 2**-11 + 2**-30, 0x3C01),
    (2.0**-14, 0x0400), (2.0**-24, 0x0001), (2.0**-25, 0x0000), (3 * 2.0**-25, 0x0002),
    (2.0**-14 - 2.0**-25, 0x0400), (0.1, 0x2E66), (-0.0, 0x8000), (float("inf"), 0x7C00),
]
BF16_CASES = [
    (1.0, 0x3F80), (1 + 2**-8, 0x3F80), (1 + 3 * 2**-8, 0x3F82), (1 + 2**-8 + 2**-40, 0x3F81),
    (-3.0, 0xC040), (2.0**-126, 0x0080), (2.0**-133, 0x0001), (2.0**-134, 0x0000),
    (0.1, 0x3DCD), (3.3895313892515355e38, 0x7F7F), (3.40e38, 0x7F80),
]


@pytest.mark.parametrize("x,bits", F16_CASES)
def test_f16_rounding_cases(x, bits):
    assert O.f16_from_double(x) == bits


@pytest.mark.parametrize("x,bits", BF16_CASES)
def test_bf16_rounding_cases(x, bits):
    assert O.bf16_from_double(x) == bits


def test_f16_encode_matches_numpy_and_decode_roundtrips():
    """numpy's float64 -> float16 conversion is IEEE round to nearest even."""
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-8, 5, 4000),
                         rng.uniform(-70000, 70000, 500)])
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([O.f16_from_double(float(x)) for x in xs], dtype=np.uint16)
    np.testing.assert_array_equal(got, ref)
    for b in range(0, 0x7C00, 7):
        assert O.f16_to_double(b) == float(np.uint16(b).view(np.float16))


def test_bf16_encode_matches_torch_on_float32_values():
    """For values exact in fp32, torch's float32 -> bfloat16 is one RNE step."""
    rng = np.random.default_rng(1)
    xs = (rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000)).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([O.bf16_from_double(float(x)) for x in xs], dtype=np.uint16)
    np.testing.assert_array_equal(got, ref)
    for b in range(0, 0x7F80, 97):
        want = torch.tensor([b], dtype=torch.int16).view(torch.bfloat16).double().item()
        assert O.bf16_to_double(b) == want


# --------------------------------------------------------------------------
# Entry sampling and argument checks
# --------------------------------------------------------------------------

def test_entries_match_full():
    p = I.Problem("ent", "bf16", "N", "N", 33, 21, 40, alpha=0.5, beta=2.0, c="bf16",
                  d="bf16", bias="f32", bias_mode="row", act="relu", pad_a=3)
    inp = I.generate(p, 12)
    D, _ = run_oracle(inp)
    rng = np.random.default_rng(2)
    rows = rng.integers(0, p.M, 100)
    cols = rng.integers(0, p.N, 100)
    out, _ = O.gemm_entries(O.BF16, O.LAYOUT_N, O.LAYOUT_N, p.M, p.N, p.K, p.alpha, inp.A,
                            p.lda, inp.B, p.ldb, rows, cols, beta=p.beta, c_dtype=O.BF16,
                            C=inp.C, ldc=p.ldc, bias_dtype=O.F32, bias=inp.bias,
                            bias_mode=O.BIAS_ROW, act=O.ACT_RELU, d_dtype=O.BF16)
    np.testing.assert_array_equal(out, D[rows, cols])


def test_invalid_arguments_rejected():
    A = np.zeros(64, dtype=np.float32)
    with pytest.raises(ValueError):   # lda < M for a column-major A
        O.gemm(O.F32, O.LAYOUT_N, O.LAYOUT_N, 8, 2, 2, 1.0, A, 4, A, 2)
    with pytest.raises(ValueError):   # beta != 0 without C
        O.gemm(O.F32, O.LAYOUT_T, O.LAYOUT_N, 2, 2, 2, 1.0, A, 2, A, 2, beta=1.0)
    with pytest.raises(ValueError):   # non-integral alpha on the int path
        O.gemm(O.S8, O.LAYOUT_T, O.LAYOUT_N, 2, 2, 2, 0.5, A, 2, A, 2, d_dtype=O.S32)


def test_k_zero_is_epilogue_of_beta_c():
    """K == 0: the product is an empty sum, so D = act(beta*C + bias) and A, B
    (and their leading dimensions) are not read."""
    p = I.Problem("k0", "f16", "T", "N", 5, 6, 0, alpha=3.0, beta=0.5, c="f32", bias="f32",
                  bias_mode="col", act="relu")
    inp = I.generate(p, 13)
    D, _ = run_oracle(inp)
    v = np.maximum(np.float64(0.5) * inp.C.double().numpy() + inp.bias.double().numpy()[None, :], 0)
    np.testing.assert_array_equal(D, v.astype(np.float32))


# ----------------------- int8 output (requantising cast) ---------------------
# Reading (the pages define no requantisation): q = saturate_int8(rne(fp32(v) *
# fp32(out_scale))) of the int32 epilogue result v, the product taken in fp32.

def _requant_case(values, scale):
    """An epilogue-only int8 problem whose int32 results are exactly `values`
    (A = 0, beta = 1, C = values), requantised with `scale`."""
    n = len(values)
    p = I.Problem("rq", "s8", "T", "N", 1, n, 4, beta=1.0, c="s32", d="s8", out_scale=scale,
                  dist_a=I.Dist("zeros"), dist_b=I.I8)
    inp = I.generate(p, 60)
    inp.C = torch.tensor([values], dtype=torch.int32)
    D, _ = run_oracle(inp)
    return D[0].tolist()


def test_requant_ties_round_to_even_and_saturate():
    # 5*0.5 = 2.5 -> 2, 7*0.5 = 3.5 -> 4, -5*0.5 = -2.5 -> -2, 3*0.5 = 1.5 -> 2,
    # 1000 -> 127, -1000 -> -128, 255*0.5 = 127.5 -> 128 -> saturates to 127.
    assert _requant_case([5, 7, -5, 3, 2000, -2000, 255], 0.5) == [2, 4, -2, 2, 127, -128, 127]


def test_requant_product_is_taken_in_fp32():
    """v = 3*2^23 - 1 is not an fp32 value: it converts to 3*2^23 (ties to even),
    so v * 2^-24 is 1.5 in fp32 and rounds to 2; in exact arithmetic it is just
    below 1.5 and would round to 1."""
    v = 3 * 2**23 - 1
    assert _requant_case([v, -v], 2.0**-24) == [2, -2]


def test_requant_matches_numpy_closed_form():
    """A random int8 GEMM with C, bias and ReLU: the int8 output equals numpy's
    int64 matmul, wrapped to int32, converted to float32, times the float32
    scale, rounded half to even (np.rint) and clipped."""
    p = I.Problem("rqnp", "s8", "N", "T", 23, 19, 41, alpha=2.0, beta=-1.0, c="s32", d="s8",
                  bias="s32", bias_mode="col", act="relu", out_scale=0.0123,
                  dist_a=I.I8, dist_b=I.I8, dist_c=I.Dist("int", -5000, 5000),
                  dist_bias=I.Dist("int", -3000, 3000))
    inp = I.generate(p, 61, keep_logical=True)
    D, _ = run_oracle(inp)
    a = inp.logical["a"].numpy().astype(np.int64)
    b = inp.logical["b"].numpy().astype(np.int64)
    c = inp.logical["c"].numpy().astype(np.int64)
    v = np.maximum(2 * (a @ b) - c + inp.bias.numpy().astype(np.int64)[None, :], 0)
    v32 = v.astype(np.int32)
    q = np.clip(np.rint(v32.astype(np.float32) * np.float32(0.0123)), -128, 127).astype(np.int8)
    np.testing.assert_array_equal(D, q)


# --------------------------------------------------------------------------
# Transforms of A and B after load ("Flexible Performant GEMM Kernels on GPUs",
# section 4.2, Figure 10): t(x) = act(scale * x), product in fp32, rounded
# back to a 16-bit operand's type.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("ab", ["f16", "bf16", "f32", "s8"])
@pytest.mark.parametrize("acts", [("relu", "none"), ("none", "relu"), ("relu", "relu")])
def test_transform_relu_matches_numpy_on_small_integers(layout, ab, acts):
    """Small integers stay exact through every step, so the oracle must equal
    numpy's int64 product of the rectified logical matrices."""
    M, N, K = 11, 13, 17
    cd = "s32" if ab == "s8" else "f32"
    p = I.Problem("t_relu", ab, layout[0], layout[1], M, N, K, d=cd, a_act=acts[0], b_act=acts[1],
                  alpha=2.0, beta=-1.0, c=cd, dist_c=I.Dist("small", -9, 9),
                  dist_a=I.Dist("small", -4, 4), dist_b=I.Dist("small", -4, 4), pad_a=1, pad_b=3)
    inp = I.generate(p, 41, keep_logical=True)
    a = inp.logical["a"].to(torch.float64).numpy().astype(np.int64)
    b = inp.logical["b"].to(torch.float64).numpy().astype(np.int64)
    c = inp.logical["c"].to(torch.float64).numpy().astype(np.int64)
    if acts[0] == "relu":
        a = np.maximum(a, 0)
    if acts[1] == "relu":
        b = np.maximum(b, 0)
    D, ovf = run_oracle(inp)
    assert ovf == 0
    np.testing.assert_array_equal(D.astype(np.int64), 2 * (a @ b) - c)


@pytest.mark.parametrize("ab", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("scales", [(2.0, 1.0), (1.0, 0.25), (-4.0, 0.5)])
def test_transform_power_of_two_scales_factor_out(ab, scales):
    """Scaling by powers of two is exact in every format, so the product of
    scaled operands is the product times sa * sb, bit for bit."""
    p = I.Problem("t_scale", ab, "N", "T", 9, 12, 21, dist_a=I.Dist("small", -8, 8),
                  dist_b=I.Dist("small", -8, 8))
    inp = I.generate(p, 42)
    base, _ = run_oracle(inp)
    scaled, _ = run_oracle(I.Inputs(inp.A, inp.B, inp.C, inp.bias,
                                    p.with_(a_scale=scales[0], b_scale=scales[1])))
    np.testing.assert_array_equal(scaled.astype(np.float64),
                                  base.astype(np.float64) * scales[0] * scales[1])


# Scales for which, on some fp16 x in [1, 2), rounding fp32(s) * x to fp32 first
# and then to fp16 differs from rounding the exact product to fp16 once (found by
# a search over random fp32 scales; the test below re-checks that they do).
DOUBLE_ROUNDING_SCALES = [0.9447439312934875, 0.7901661992073059]


@pytest.mark.parametrize("ab", ["f16", "bf16"])
def test_transform_takes_the_scale_in_fp32_then_rounds_to_the_operand_type(ab):
    """For every fp16 (bf16) value in [1, 2), a grid of other values, and several
    scales, the transformed element the sum uses is round_type(fp32(s) * fp32(x)),
    computed here with numpy's float32 product and numpy's float16 (torch's
    bfloat16) rounding.  A = the values as one column, B = 1, so D[i, 0] is t(A[i]).
    For fp16 the scales include ones where taking the product exactly (in fp64)
    and rounding once gives a different element, so the fp32 step is pinned."""
    mant = 1024 if ab == "f16" else 128
    grid = torch.cat([torch.arange(mant, 2 * mant, dtype=torch.float64) / mant,
                      torch.linspace(-7.3, 7.9, 211, dtype=torch.float64)])
    vals = grid.to(I.TORCH_DTYPES[ab])
    M = vals.numel()
    x32 = vals.to(torch.float32).numpy()
    differs = 0
    for s in [0.1, 1.0 / 3.0, -2.7182817, 0.7071068] + DOUBLE_ROUNDING_SCALES:
        p = I.Problem("t_round", ab, "T", "N", M, 1, 1, a_scale=s, a_act="relu")
        inp = I.Inputs(A=vals.reshape(M, 1).contiguous(), B=torch.ones(1, 1, dtype=vals.dtype),
                       C=None, bias=None, problem=p)
        D, _ = run_oracle(inp)
        prod = np.maximum(np.float32(s) * x32, np.float32(0.0))
        if ab == "f16":
            want = prod.astype(np.float16).astype(np.float64)
            once = np.maximum(np.float64(np.float32(s)) * x32.astype(np.float64), 0.0).astype(np.float16)
            differs += int(np.count_nonzero(once.astype(np.float64) != want))
        else:
            want = torch.from_numpy(prod).to(torch.bfloat16).to(torch.float64).numpy()
        np.testing.assert_array_equal(D[:, 0].astype(np.float64), want)
    if ab == "f16":
        assert differs > 0, "the scale grid no longer tells one rounding from two"


def test_transform_fp32_operand_keeps_the_fp32_product():
    """An fp32 operand is not narrowed: t(x) = fp32(s * x)."""
    x = np.array([[1.0], [3.0], [-0.1]], dtype=np.float32)
    s = 0.1
    p = I.Problem("t_f32", "f32", "T", "N", 3, 1, 1, a_scale=s)
    inp = I.Inputs(A=torch.from_numpy(x), B=torch.ones(1, 1), C=None, bias=None, problem=p)
    D, _ = run_oracle(inp)
    np.testing.assert_array_equal(D[:, 0], (np.float32(s) * x[:, 0]).astype(np.float32))


def test_transform_loop_orders_agree():
    p = I.Problem("t_lo", "bf16", "T", "N", 13, 11, 19, a_scale=0.3, a_act="relu", b_scale=-1.7,
                  alpha=1.5, beta=0.5, c="f32")
    inp = I.generate(p, 43)
    np.testing.assert_array_equal(run_oracle(inp, 0)[0], run_oracle(inp, 1)[0])
    pi = I.Problem("t_lo8", "s8", "N", "T", 9, 10, 33, d="s32", dist_a=I.I8, dist_b=I.I8,
                   a_act="relu", b_act="relu")
    inp = I.generate(pi, 44)
    np.testing.assert_array_equal(run_oracle(inp, 0)[0], run_oracle(inp, 1)[0])


def test_transform_arguments_rejected():
    A = np.zeros(4, np.int8)
    with pytest.raises(ValueError):   # a scale on int8 operands leaves the integers
        O.gemm(O.S8, O.LAYOUT_T, O.LAYOUT_N, 2, 2, 2, 1.0, A, 2, A, 2, d_dtype=O.S32, a_scale=2.0)
    Af = np.zeros(4, np.float32)
    with pytest.raises(ValueError):
        O.gemm(O.F32, O.LAYOUT_T, O.LAYOUT_N, 2, 2, 2, 1.0, Af, 2, Af, 2, b_scale=float("inf"))
    with pytest.raises(ValueError):
        O.gemm(O.F32, O.LAYOUT_T, O.LAYOUT_N, 2, 2, 2, 1.0, Af, 2, Af, 2, a_act=5)
