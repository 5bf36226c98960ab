"""Shared helpers of the parity tests: run a problem through the GPU library
(C ABI, device buffers with guard bands) and through the CPU oracle, and compare.

The tolerance for floating outputs, computed in fp64 from both outputs widened
to fp64:  max |D - D_ref| <= 1e-2 * (|D_ref| + 1) elementwise, and
||D - D_ref||_F / ||D_ref||_F <= 2e-3.  Integer outputs must be bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import dense_gemm_epilogues_gb300 as G
import oracle as O
from dense_gemm_epilogues_gb300 import inputs as I

OR_DT = {"f32": O.F32, "f16": O.F16, "bf16": O.BF16, "s8": O.S8, "s32": O.S32}
OR_LAY = {"N": O.LAYOUT_N, "T": O.LAYOUT_T}
OR_BIAS = {"none": O.BIAS_NONE, "col": O.BIAS_COL, "row": O.BIAS_ROW}
OR_ACT = {"none": O.ACT_NONE, "relu": O.ACT_RELU}
G_BIAS = {"none": G.GEMM_BIAS_NONE, "col": G.GEMM_BIAS_COL, "row": G.GEMM_BIAS_ROW}

ABS_TOL = 1e-2
FRO_TOL = 2e-3
GUARD_ROWS = 3
SENTINEL = {"f32": float.fromhex("0x1.5p+100"), "f16": 12345.0, "bf16": 1.5e30, "s32": 0x5A5A5A5A,
            "s8": 0x5A}


def _oracle_kwargs(p: I.Problem, inp: I.Inputs) -> dict:
    return dict(beta=p.beta, c_dtype=OR_DT[p.c] if p.c else O.F32, C=inp.C,
                ldc=p.ldc if p.c else 0, bias_dtype=OR_DT[p.bias] if p.bias else O.F32,
                bias=inp.bias, bias_mode=OR_BIAS[p.bias_mode], act=OR_ACT[p.act],
                d_dtype=OR_DT[p.d], c_act=OR_ACT[p.c_act], out_scale=p.out_scale,
                a_act=OR_ACT[p.a_act], a_scale=p.a_scale, b_act=OR_ACT[p.b_act], b_scale=p.b_scale)


def oracle_full(inp: I.Inputs) -> np.ndarray:
    p = inp.problem
    D, ovf = O.gemm(OR_DT[p.ab], OR_LAY[p.layout_a], OR_LAY[p.layout_b], p.M, p.N, p.K, p.alpha,
                    inp.A, p.lda, inp.B, p.ldb, ldd=p.N, **_oracle_kwargs(p, inp))
    assert ovf == 0, "inputs overflow int32; the library contract leaves that undefined"
    return D


def oracle_entries(inp: I.Inputs, rows, cols) -> np.ndarray:
    p = inp.problem
    out, ovf = O.gemm_entries(OR_DT[p.ab], OR_LAY[p.layout_a], OR_LAY[p.layout_b], p.M, p.N, p.K,
                              p.alpha, inp.A, p.lda, inp.B, p.ldb, rows, cols,
                              **_oracle_kwargs(p, inp))
    assert ovf == 0
    return out


def to_f64(x, dtype: str) -> np.ndarray:
    """Widen raw output (numpy bits for 16-bit types, or a torch tensor) to fp64."""
    if isinstance(x, torch.Tensor):
        return x.to(torch.float64).cpu().numpy()
    if dtype in ("f16", "bf16"):
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16))
        return t.view(I.TORCH_DTYPES[dtype]).to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def check_close(D_gpu: torch.Tensor, D_ref_raw: np.ndarray, d_dtype: str, what: str = ""):
    if d_dtype in ("s32", "s8"):
        got = D_gpu.cpu().numpy().astype(np.int64)
        ref = np.asarray(D_ref_raw).astype(np.int64)
        bad = np.argwhere(got != ref)
        assert bad.size == 0, f"{what}: {len(bad)} integer mismatches, first at {bad[:3].tolist()}"
        return
    got = to_f64(D_gpu, d_dtype)
    ref = to_f64(D_ref_raw, d_dtype)
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    err = np.abs(got - ref)
    lim = ABS_TOL * (np.abs(ref) + 1.0)
    worst = np.unravel_index(np.argmax(err - lim), err.shape) if err.size else None
    assert np.all(err <= lim), (f"{what}: elementwise bound violated at {worst}: "
                                f"got {got[worst]} ref {ref[worst]}")
    nref = np.linalg.norm(ref)
    if nref > 0:
        fro = np.linalg.norm(got - ref) / nref
        assert fro <= FRO_TOL, f"{what}: relative Frobenius error {fro:.3e} > {FRO_TOL}"


def _act(a: str) -> int:
    return G.GEMM_ACT_RELU if a == "relu" else G.GEMM_ACT_NONE


def epilogue_for(p: I.Problem, bias_ptr: int = 0, **overrides) -> G.gemm_epilogue_t:
    """The library's epilogue struct for a problem: bias, activations, output
    type, and the operand transforms of A and B after load."""
    kw = dict(out_scale=p.out_scale, a_act=_act(p.a_act), a_scale=p.a_scale, b_act=_act(p.b_act),
              b_scale=p.b_scale)
    kw.update(overrides)
    return G.make_epilogue(G.DTYPE_CODES[p.d], bias_ptr, G.DTYPE_CODES[p.bias] if p.bias else G.GEMM_F32,
                           G_BIAS[p.bias_mode], _act(p.act), _act(p.c_act), **kw)


class DeviceProblem:
    """Device copies of a problem's inputs, plus a guarded output buffer."""

    def __init__(self, inp: I.Inputs, device="cuda"):
        p = inp.problem
        self.inp, self.p = inp, p
        self.A = inp.A.to(device)
        self.B = inp.B.to(device)
        self.C = inp.C.to(device) if inp.C is not None else None
        self.bias = inp.bias.to(device) if inp.bias is not None else None
        rows = p.M + 2 * GUARD_ROWS
        self.Dbuf = torch.full((rows, p.ldd), SENTINEL[p.d], dtype=I.TORCH_DTYPES[p.d], device=device)
        self.D = self.Dbuf[GUARD_ROWS:GUARD_ROWS + p.M]

    def epilogue(self) -> G.gemm_epilogue_t:
        return epilogue_for(self.p, self.bias.data_ptr() if self.bias is not None else 0)

    def run(self, plan: G.Plan, stream=None):
        p = self.p
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        G.gemm_run(plan.handle, G.LAYOUT_CODES[p.layout_a], G.LAYOUT_CODES[p.layout_b], p.M, p.N,
                   p.K, p.alpha, self.A.data_ptr(), p.lda, self.B.data_ptr(), p.ldb, p.beta,
                   self.C.data_ptr() if self.C is not None else None, p.ldc if p.c else 0,
                   self.D.data_ptr(), p.ldd, self.epilogue(), stream)

    def check_guards(self):
        p = self.p
        s = torch.tensor(SENTINEL[p.d], dtype=I.TORCH_DTYPES[p.d])
        top = self.Dbuf[:GUARD_ROWS].cpu()
        bot = self.Dbuf[GUARD_ROWS + p.M:].cpu()
        pad = self.D[:, p.N:].cpu()
        for name, t in (("rows before D", top), ("rows after D", bot), ("padding of D", pad)):
            assert torch.all(t == s), f"kernel wrote into the {name}"

    def result(self) -> torch.Tensor:
        return self.D[:, :self.p.N]


def make_plan(p: I.Problem, kernel=None) -> G.Plan:
    c = p.c if p.c else ("s32" if p.ab == "s8" else "f32")
    plan = G.Plan(G.DTYPE_CODES[p.ab], G.DTYPE_CODES[c], torch.cuda.current_device())
    if kernel is not None:
        plan.set_kernel(kernel)
    return plan


def run_and_check_full(p: I.Problem, seed: int, kernel=None, expect_kernel=None) -> dict:
    inp = I.generate(p, seed)
    dp = DeviceProblem(inp)
    plan = make_plan(p, kernel)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    cfg = plan.last_config()
    if expect_kernel is not None:
        assert cfg["kernel"] == expect_kernel, f"ran {cfg['kernel_name']}"
    dp.check_guards()
    check_close(dp.result(), oracle_full(inp), p.d, p.name)
    plan.close()
    return cfg


def sample_entries(M: int, N: int, n: int, seed: int, tile_m=128, tile_n=256):
    """Random entries plus corners and tile-boundary rows/columns."""
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, M, n))
    cols = list(rng.integers(0, N, n))
    edge_r = sorted({0, M - 1, min(M - 1, tile_m - 1), min(M - 1, tile_m), M // 2, max(0, M - tile_m)})
    edge_c = sorted({0, N - 1, min(N - 1, tile_n - 1), min(N - 1, tile_n), N // 2, max(0, N - tile_n)})
    for r in edge_r:
        for c in edge_c:
            rows.append(r)
            cols.append(c)
    return np.array(rows, dtype=np.int64), np.array(cols, dtype=np.int64)


def boundary_entries(M: int, N: int, row_block: int = 128, col_block: int = 64):
    """Whole rows at both edges of every row block of D (the first and last row
    each CTA of a tile owns) and whole columns at both edges of every column
    block (the first and last column of each epilogue chunk), as (rows, cols)
    entry lists.  Every tile then has at least one whole row and one whole
    column of its outputs checked."""
    rs = sorted({r for t in range(0, M, row_block) for r in (t, min(t + row_block - 1, M - 1))})
    cs = sorted({c for t in range(0, N, col_block) for c in (t, min(t + col_block - 1, N - 1))})
    rows = np.concatenate([np.repeat(np.asarray(rs, dtype=np.int64), N),
                           np.tile(np.arange(M, dtype=np.int64), len(cs))])
    cols = np.concatenate([np.tile(np.arange(N, dtype=np.int64), len(rs)),
                           np.repeat(np.asarray(cs, dtype=np.int64), M)])
    return rows, cols


def tma_aligned(p: I.Problem, mult: int = 8) -> I.Problem:
    """Pad the leading dimensions of A and B up to a multiple of `mult` elements
    (16 bytes for 16-bit types), as the tensor-core kernels' TMA loads require.
    The logical sizes (and their ragged tails) are unchanged; the padding is
    poisoned by the input generator."""
    ra = (p.M if p.layout_a == "N" else p.K)
    rb = (p.K if p.layout_b == "N" else p.N)
    return p.with_(pad_a=p.pad_a + (-(ra + p.pad_a)) % mult, pad_b=p.pad_b + (-(rb + p.pad_b)) % mult)


# ------------------------- diagonal-operand GEMM -----------------------------

def dense_inputs_of(dinp: I.DiagInputs) -> I.Inputs:
    """The oracle's view of a diagonal-operand problem: the diagonal written out
    as a square dense matrix (zeros off the diagonal), x as the other operand."""
    p = dinp.problem
    dp = p.dense()
    n = p.n_diag
    square = torch.zeros((n, n), dtype=dinp.diag.dtype)
    idx = torch.arange(n)
    square[idx, idx] = dinp.diag
    sq = I._store(square, "N", n, p.ab)
    if p.side == "left":
        return I.Inputs(A=sq, B=dinp.X, C=dinp.C, bias=dinp.bias, problem=dp)
    return I.Inputs(A=dinp.X, B=sq, C=dinp.C, bias=dinp.bias, problem=dp)


class DeviceDiag:
    """Device copies of a diagonal-operand problem, plus a guarded output."""

    def __init__(self, dinp: I.DiagInputs, device="cuda"):
        p = dinp.problem
        self.inp, self.p = dinp, p
        self.diag = dinp.diag.to(device)
        self.X = dinp.X.to(device)
        self.C = dinp.C.to(device) if dinp.C is not None else None
        self.bias = dinp.bias.to(device) if dinp.bias is not None else None
        rows = p.M + 2 * GUARD_ROWS
        self.Dbuf = torch.full((rows, p.ldd), SENTINEL[p.d], dtype=I.TORCH_DTYPES[p.d], device=device)
        self.D = self.Dbuf[GUARD_ROWS:GUARD_ROWS + p.M]

    def epilogue(self) -> G.gemm_epilogue_t:
        p = self.p
        return G.make_epilogue(G.DTYPE_CODES[p.d],
                               self.bias.data_ptr() if self.bias is not None else 0,
                               G.DTYPE_CODES[p.bias] if p.bias else G.GEMM_F32,
                               G_BIAS[p.bias_mode],
                               G.GEMM_ACT_RELU if p.act == "relu" else G.GEMM_ACT_NONE,
                               G.GEMM_ACT_RELU if p.c_act == "relu" else G.GEMM_ACT_NONE)

    def run(self, plan: G.Plan, stream=None, C=None, D=None):
        p = self.p
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        C = self.C if C is None else C
        D = self.D if D is None else D
        G.gemm_run_diag(plan.handle, G.GEMM_SIDE_LEFT if p.side == "left" else G.GEMM_SIDE_RIGHT,
                        G.LAYOUT_CODES[p.layout_x], p.M, p.N, p.alpha, self.diag.data_ptr(),
                        self.X.data_ptr(), p.ldx, p.beta, C.data_ptr() if C is not None else None,
                        p.ldc if p.c else 0, D.data_ptr(), p.ldd, self.epilogue(), stream)

    def check_guards(self):
        p = self.p
        s = torch.tensor(SENTINEL[p.d], dtype=I.TORCH_DTYPES[p.d])
        for name, t in (("rows before D", self.Dbuf[:GUARD_ROWS]),
                        ("rows after D", self.Dbuf[GUARD_ROWS + p.M:]), ("padding of D", self.D[:, p.N:])):
            assert torch.all(t.cpu() == s), f"kernel wrote into the {name}"

    def result(self) -> torch.Tensor:
        return self.D[:, :self.p.N]


def make_diag_plan(p: I.DiagProblem) -> G.Plan:
    c = p.c if p.c else ("s32" if p.ab == "s8" else "f32")
    return G.Plan(G.DTYPE_CODES[p.ab], G.DTYPE_CODES[c], torch.cuda.current_device())


# --------------------------- complex / dual GEMM -----------------------------

OR_UNIT = {"complex": O.UNIT_IMAGINARY, "dual": O.UNIT_DUAL}
G_UNIT = {"complex": G.GEMM_UNIT_IMAGINARY, "dual": G.GEMM_UNIT_DUAL}


def _oracle_pair_kwargs(p: I.PairProblem, inp: I.PairInputs) -> dict:
    return dict(beta=p.beta, c_dtype=OR_DT[p.c] if p.c else O.F32, C=inp.C,
                ldc=p.ldc if p.c else 0, bias_dtype=OR_DT[p.bias] if p.bias else O.F32,
                bias=inp.bias, bias_mode=OR_BIAS[p.bias_mode], act=OR_ACT[p.act],
                d_dtype=OR_DT[p.d], c_act=OR_ACT[p.c_act])


def oracle_pairs_full(inp: I.PairInputs) -> np.ndarray:
    """(M, N, 2) output pairs (raw bits for 16-bit types)."""
    p = inp.problem
    return O.gemm_pairs(OR_UNIT[p.unit], OR_DT[p.ab], OR_LAY[p.layout_a], OR_LAY[p.layout_b],
                        p.M, p.N, p.K, p.alpha, inp.A, p.lda, inp.B, p.ldb, ldd=p.N,
                        **_oracle_pair_kwargs(p, inp))


def oracle_pairs_entries(inp: I.PairInputs, rows, cols) -> np.ndarray:
    p = inp.problem
    return O.gemm_pairs_entries(OR_UNIT[p.unit], OR_DT[p.ab], OR_LAY[p.layout_a],
                                OR_LAY[p.layout_b], p.M, p.N, p.K, p.alpha, inp.A, p.lda, inp.B,
                                p.ldb, rows, cols, **_oracle_pair_kwargs(p, inp))


class DevicePairs:
    """Device copies of a complex / dual problem, plus a guarded output."""

    def __init__(self, inp: I.PairInputs, device="cuda"):
        p = inp.problem
        self.inp, self.p = inp, p
        self.A = inp.A.to(device)
        self.B = inp.B.to(device)
        self.C = inp.C.to(device) if inp.C is not None else None
        self.bias = inp.bias.to(device) if inp.bias is not None else None
        self.Dbuf = torch.full((p.M + 2 * GUARD_ROWS, p.ldd, 2), SENTINEL[p.d],
                               dtype=I.TORCH_DTYPES[p.d], device=device)
        self.D = self.Dbuf[GUARD_ROWS:GUARD_ROWS + p.M]

    def epilogue(self) -> G.gemm_epilogue_t:
        p = self.p
        return G.make_epilogue(G.DTYPE_CODES[p.d],
                               self.bias.data_ptr() if self.bias is not None else 0,
                               G.DTYPE_CODES[p.bias] if p.bias else G.GEMM_F32,
                               G_BIAS[p.bias_mode],
                               G.GEMM_ACT_RELU if p.act == "relu" else G.GEMM_ACT_NONE,
                               G.GEMM_ACT_RELU if p.c_act == "relu" else G.GEMM_ACT_NONE)

    def run(self, plan: G.Plan, stream=None, A=None, B=None):
        p = self.p
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        A = self.A.data_ptr() if A is None else A
        B = self.B.data_ptr() if B is None else B
        G.gemm_run_complex(plan.handle, G_UNIT[p.unit], G.LAYOUT_CODES[p.layout_a],
                           G.LAYOUT_CODES[p.layout_b], p.M, p.N, p.K, p.alpha, A, p.lda, B, p.ldb,
                           p.beta, self.C.data_ptr() if self.C is not None else None,
                           p.ldc if p.c else 0, self.D.data_ptr(), p.ldd, self.epilogue(), stream)

    def check_guards(self):
        p = self.p
        s = torch.tensor(SENTINEL[p.d], dtype=I.TORCH_DTYPES[p.d])
        for name, t in (("rows before D", self.Dbuf[:GUARD_ROWS]),
                        ("rows after D", self.Dbuf[GUARD_ROWS + p.M:]), ("padding of D", self.D[:, p.N:])):
            assert torch.all(t.cpu() == s), f"kernel wrote into the {name}"

    def result(self) -> torch.Tensor:
        return self.D[:, :self.p.N]


def make_pair_plan(p: I.PairProblem) -> G.Plan:
    return G.Plan(G.DTYPE_CODES[p.ab], G.DTYPE_CODES[p.c or "f32"], torch.cuda.current_device())
