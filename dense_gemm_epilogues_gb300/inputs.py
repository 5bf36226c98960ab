"""Seeded synthetic inputs for the GEMM workloads.

This module draws random matrices and lays them out in memory; it holds none of
the GEMM's arithmetic.  Both the parity tests (GPU library vs CPU oracle) and
the benchmark draw their inputs here, so both sides read the same bytes.

Recipe: one CPU ``torch.Generator`` seeded per problem; values are drawn in the
order A, B, C, bias, each in logical row-major order (A is M x K, B is K x N,
C is M x N); floating values are drawn in fp32 and rounded once (round to
nearest even) to the storage type; the logical matrix is then written into its
storage layout (N = column-major, T = row-major) with an optional padded leading
dimension whose padding holds a poison value (NaN for floats, 127 for int8) so
that a kernel reading outside the logical matrix is caught.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import torch

TORCH_DTYPES = {
    "f32": torch.float32,
    "f16": torch.float16,
    "bf16": torch.bfloat16,
    "s8": torch.int8,
    "s32": torch.int32,
}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "s8": 1, "s32": 4}

BASE_SEED = 20261202


@dataclass(frozen=True)
class Dist:
    """A value distribution: 'uniform' on [lo, hi], 'normal' with std `std`,
    'int' uniform on the integers lo..hi inclusive, or 'small' uniform on the
    integers lo..hi (exactly representable in every input type)."""
    kind: str
    lo: float = -1.0
    hi: float = 1.0
    std: float = 1.0


U11 = Dist("uniform", -1.0, 1.0)
I8 = Dist("int", -128, 127)


@dataclass(frozen=True)
class Problem:
    name: str
    ab: str               # 'f16' | 'bf16' | 's8' | 'f32'
    layout_a: str         # 'N' | 'T'
    layout_b: str
    M: int
    N: int
    K: int
    alpha: float = 1.0
    beta: float = 0.0
    c: Optional[str] = None      # dtype of C (None: beta == 0, C not allocated)
    d: str = "f32"               # dtype of D
    bias: Optional[str] = None   # dtype of the bias vector
    bias_mode: str = "none"      # 'none' | 'col' | 'row'
    act: str = "none"            # 'none' | 'relu'
    c_act: str = "none"          # transform of C as it is read: 'none' | 'relu'
    out_scale: float = 1.0       # int8 output of an int8 problem: requantisation scale
    a_act: str = "none"          # transform of A as it is read: 'none' | 'relu' (after a_scale)
    a_scale: float = 1.0         # multiplier of A's elements as they are read
    b_act: str = "none"          # the same for B
    b_scale: float = 1.0
    dist_a: Dist = U11
    dist_b: Dist = U11
    dist_c: Dist = Dist("normal", std=1.0)
    dist_bias: Dist = Dist("normal", std=0.1)
    pad_a: int = 0               # extra leading-dimension elements (poisoned)
    pad_b: int = 0
    pad_c: int = 0
    pad_d: int = 0

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    @property
    def lda(self) -> int:
        return (self.M if self.layout_a == "N" else self.K) + self.pad_a

    @property
    def ldb(self) -> int:
        return (self.K if self.layout_b == "N" else self.N) + self.pad_b

    @property
    def ldc(self) -> int:
        return self.N + self.pad_c

    @property
    def ldd(self) -> int:
        return self.N + self.pad_d

    def with_(self, **kw) -> "Problem":
        return replace(self, **kw)


@dataclass
class Inputs:
    A: torch.Tensor                # storage (2-D, contiguous), host
    B: torch.Tensor
    C: Optional[torch.Tensor]
    bias: Optional[torch.Tensor]
    problem: Problem
    logical: dict = field(default_factory=dict)   # logical row-major copies (host)


def _draw(gen: torch.Generator, rows: int, cols: int, dist: Dist, dtype: str) -> torch.Tensor:
    shape = (rows, cols)
    if dist.kind == "uniform":
        x = torch.rand(shape, generator=gen, dtype=torch.float32) * (dist.hi - dist.lo) + dist.lo
    elif dist.kind == "normal":
        x = torch.randn(shape, generator=gen, dtype=torch.float32) * dist.std
    elif dist.kind in ("int", "small"):
        x = torch.randint(int(dist.lo), int(dist.hi) + 1, shape, generator=gen, dtype=torch.int64)
    elif dist.kind == "zeros":
        x = torch.zeros(shape, dtype=torch.float32)
    elif dist.kind == "ones":
        x = torch.ones(shape, dtype=torch.float32)
    else:
        raise ValueError(f"unknown distribution {dist.kind}")
    return x.to(TORCH_DTYPES[dtype])


def _poison(dtype: str):
    return 127 if dtype == "s8" else (2147483647 if dtype == "s32" else float("nan"))


def _store(logical: torch.Tensor, layout: str, ld: int, dtype: str) -> torch.Tensor:
    """Write a logical (rows x cols) matrix into column- ('N') or row-major ('T')
    storage with leading dimension ld.  Returns the 2-D storage tensor."""
    rows, cols = logical.shape
    if layout == "T":
        st = torch.full((rows, ld), _poison(dtype), dtype=TORCH_DTYPES[dtype]) if ld > cols \
            else torch.empty((rows, cols), dtype=TORCH_DTYPES[dtype])
        st[:, :cols] = logical
    else:
        st = torch.full((cols, ld), _poison(dtype), dtype=TORCH_DTYPES[dtype]) if ld > rows \
            else torch.empty((cols, rows), dtype=TORCH_DTYPES[dtype])
        st[:, :rows] = logical.t()
    return st.contiguous()


def generate(p: Problem, seed: int, keep_logical: bool = False) -> Inputs:
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    a = _draw(gen, p.M, p.K, p.dist_a, p.ab)
    b = _draw(gen, p.K, p.N, p.dist_b, p.ab)
    c = _draw(gen, p.M, p.N, p.dist_c, p.c) if p.c is not None else None
    nb = p.N if p.bias_mode == "col" else p.M
    bias = _draw(gen, 1, nb, p.dist_bias, p.bias).reshape(nb) if p.bias_mode != "none" else None
    A = _store(a, p.layout_a, p.lda, p.ab)
    B = _store(b, p.layout_b, p.ldb, p.ab)
    C = _store(c, "T", p.ldc, p.c) if c is not None else None
    logical = {"a": a, "b": b, "c": c} if keep_logical else {}
    return Inputs(A=A, B=B, C=C, bias=bias, problem=p, logical=logical)


@dataclass(frozen=True)
class DiagProblem:
    """A GEMM whose A (side 'left': A = diag(d), M x M) or B (side 'right':
    B = diag(d), N x N) is a diagonal matrix stored as its diagonal d alone.
    The other operand, x, is dense and seen as an M x N matrix stored in
    layout_x ('N' column-major, 'T' row-major) with leading dimension ldx."""
    name: str
    ab: str
    side: str                    # 'left' | 'right'
    layout_x: str
    M: int
    N: int
    alpha: float = 1.0
    beta: float = 0.0
    c: Optional[str] = None
    d: str = "f32"
    bias: Optional[str] = None
    bias_mode: str = "none"
    act: str = "none"
    c_act: str = "none"
    dist_diag: Dist = U11
    dist_x: Dist = U11
    dist_c: Dist = Dist("normal", std=1.0)
    dist_bias: Dist = Dist("normal", std=0.1)
    pad_x: int = 0
    pad_c: int = 0
    pad_d: int = 0

    @property
    def n_diag(self) -> int:
        return self.M if self.side == "left" else self.N

    @property
    def ldx(self) -> int:
        return (self.M if self.layout_x == "N" else self.N) + self.pad_x

    @property
    def ldc(self) -> int:
        return self.N + self.pad_c

    @property
    def ldd(self) -> int:
        return self.N + self.pad_d

    def dense(self) -> Problem:
        """The same GEMM with the diagonal as a square dense operand (stored
        column-major, leading dimension = its size): x is B (left) or A (right)."""
        common = dict(alpha=self.alpha, beta=self.beta, c=self.c, d=self.d, bias=self.bias,
                      bias_mode=self.bias_mode, act=self.act, c_act=self.c_act,
                      dist_c=self.dist_c, dist_bias=self.dist_bias, pad_c=self.pad_c,
                      pad_d=self.pad_d)
        if self.side == "left":
            return Problem(self.name, self.ab, "N", self.layout_x, self.M, self.N, self.M,
                           pad_b=self.pad_x, **common)
        return Problem(self.name, self.ab, self.layout_x, "N", self.M, self.N, self.N,
                       pad_a=self.pad_x, **common)

    def with_(self, **kw) -> "DiagProblem":
        return replace(self, **kw)


@dataclass
class DiagInputs:
    diag: torch.Tensor             # the n_diag diagonal entries (host)
    X: torch.Tensor                # storage of the dense operand (host)
    C: Optional[torch.Tensor]
    bias: Optional[torch.Tensor]
    problem: DiagProblem
    x_logical: Optional[torch.Tensor] = None


def generate_diag(p: DiagProblem, seed: int) -> DiagInputs:
    """Draw d, then x (logical M x N, row-major order), then C, then the bias."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    dg = _draw(gen, 1, p.n_diag, p.dist_diag, p.ab).reshape(p.n_diag)
    x = _draw(gen, p.M, p.N, p.dist_x, p.ab)
    c = _draw(gen, p.M, p.N, p.dist_c, p.c) if p.c is not None else None
    nb = p.N if p.bias_mode == "col" else p.M
    bias = _draw(gen, 1, nb, p.dist_bias, p.bias).reshape(nb) if p.bias_mode != "none" else None
    X = _store(x, p.layout_x, p.ldx, p.ab)
    C = _store(c, "T", p.ldc, p.c) if c is not None else None
    return DiagInputs(diag=dg, X=X, C=C, bias=bias, problem=p, x_logical=x)


@dataclass(frozen=True)
class PairProblem:
    """A GEMM over complex numbers (unit 'complex': x + y i, i*i = -1) or dual
    numbers (unit 'dual': x + y eps, eps*eps = 0).  Every matrix is stored
    interleaved: the pair of the element at storage offset e (in pairs) sits at
    scalar positions 2e (real part) and 2e + 1 (unit part).  Sizes and leading
    dimensions count pairs; alpha and beta are real."""
    name: str
    unit: str                    # 'complex' | 'dual'
    ab: str
    layout_a: str
    layout_b: str
    M: int
    N: int
    K: int
    alpha: float = 1.0
    beta: float = 0.0
    c: Optional[str] = None
    d: str = "f32"
    bias: Optional[str] = None
    bias_mode: str = "none"
    act: str = "none"
    c_act: str = "none"
    dist_a: Dist = U11
    dist_b: Dist = U11
    dist_c: Dist = Dist("normal", std=1.0)
    dist_bias: Dist = Dist("normal", std=0.1)
    pad_a: int = 0
    pad_b: int = 0
    pad_c: int = 0
    pad_d: int = 0

    @property
    def flops(self) -> float:
        """Real operations of the definition: 8 per complex multiply-add
        (4 multiplies, 4 adds), 6 per dual one (a c, a d + b c)."""
        return (8.0 if self.unit == "complex" else 6.0) * self.M * self.N * self.K

    @property
    def lda(self) -> int:
        return (self.M if self.layout_a == "N" else self.K) + self.pad_a

    @property
    def ldb(self) -> int:
        return (self.K if self.layout_b == "N" else self.N) + self.pad_b

    @property
    def ldc(self) -> int:
        return self.N + self.pad_c

    @property
    def ldd(self) -> int:
        return self.N + self.pad_d

    def with_(self, **kw) -> "PairProblem":
        return replace(self, **kw)


@dataclass
class PairInputs:
    A: torch.Tensor                # storage, shape (outer, ld, 2), host
    B: torch.Tensor
    C: Optional[torch.Tensor]      # (M, ldc, 2)
    bias: Optional[torch.Tensor]   # (n, 2)
    problem: PairProblem
    logical: dict = field(default_factory=dict)   # 'a', 'b', 'c': (rows, cols, 2)


def _store_pairs(logical: torch.Tensor, layout: str, ld: int, dtype: str) -> torch.Tensor:
    """Write a logical (rows x cols) matrix of pairs, shape (rows, cols, 2), into
    interleaved column- ('N') or row-major ('T') storage, shape (outer, ld, 2)."""
    rows, cols, _ = logical.shape
    if layout == "T":
        st = torch.full((rows, ld, 2), _poison(dtype), dtype=TORCH_DTYPES[dtype])
        st[:, :cols] = logical
    else:
        st = torch.full((cols, ld, 2), _poison(dtype), dtype=TORCH_DTYPES[dtype])
        st[:, :rows] = logical.transpose(0, 1)
    return st.contiguous()


def generate_pairs(p: PairProblem, seed: int) -> PairInputs:
    """Draw A, B, C, bias (each as real and unit parts of every element, in
    logical row-major order of the elements), then lay them out interleaved."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    a = _draw(gen, p.M, 2 * p.K, p.dist_a, p.ab).reshape(p.M, p.K, 2)
    b = _draw(gen, p.K, 2 * p.N, p.dist_b, p.ab).reshape(p.K, p.N, 2)
    c = _draw(gen, p.M, 2 * p.N, p.dist_c, p.c).reshape(p.M, p.N, 2) if p.c is not None else None
    nb = p.N if p.bias_mode == "col" else p.M
    bias = (_draw(gen, 1, 2 * nb, p.dist_bias, p.bias).reshape(nb, 2)
            if p.bias_mode != "none" else None)
    A = _store_pairs(a, p.layout_a, p.lda, p.ab)
    B = _store_pairs(b, p.layout_b, p.ldb, p.ab)
    C = _store_pairs(c, "T", p.ldc, p.c) if c is not None else None
    return PairInputs(A=A, B=B, C=C, bias=bias, problem=p, logical={"a": a, "b": b, "c": c})


def sha256_of(t: torch.Tensor) -> str:
    import hashlib
    return hashlib.sha256(t.contiguous().view(torch.uint8).numpy().tobytes()).hexdigest()


# ---------------------------------------------------------------------------
# The workloads (names say what they are, with their sizes).
# ---------------------------------------------------------------------------

def square_fp16_256() -> Problem:
    """M=N=K=256, A row-major / B column-major fp16 in U[-1,1], fp32 D = A*B."""
    return Problem("gemm_f16_tn_256", "f16", "T", "N", 256, 256, 256)


def square_fp16_8192(layout: str) -> Problem:
    """M=N=K=8192 fp16, fp32 C and D, alpha=1.5, beta=0.5, C ~ N(0,1)."""
    return Problem(f"gemm_f16_{layout.lower()}_8192_ab", "f16", layout[0], layout[1],
                   8192, 8192, 8192, alpha=1.5, beta=0.5, c="f32", d="f32")


def fc_bf16_8192x4096x11008() -> Problem:
    """X[8192,4096] bf16 ~ N(0,1) times W[4096,11008] bf16 ~ N(0,0.02), both
    row-major, + bias[11008] ~ N(0,0.1), ReLU, bf16 D."""
    return Problem("fc_bf16_8192x4096x11008_bias_relu", "bf16", "T", "T", 8192, 11008, 4096,
                   d="bf16", bias="f32", bias_mode="col", act="relu",
                   dist_a=Dist("normal", std=1.0), dist_b=Dist("normal", std=0.02),
                   dist_bias=Dist("normal", std=0.1))


def int8_8192() -> Problem:
    """M=N=K=8192 int8 (uniform integers in [-128,127]), A row-major / B
    column-major, int32 accumulate and output."""
    return Problem("gemm_s8_tn_8192", "s8", "T", "N", 8192, 8192, 8192, d="s32",
                   dist_a=I8, dist_b=I8)


def sgemm_4096_bias_relu() -> Problem:
    """fp32 SGEMM M=N=K=4096 (FFMA, no TF32), U[-1,1] inputs, bias ~ N(0,0.1), ReLU."""
    return Problem("sgemm_f32_tn_4096_bias_relu", "f32", "T", "N", 4096, 4096, 4096,
                   d="f32", bias="f32", bias_mode="col", act="relu")


def square_fp16(n: int) -> Problem:
    return Problem(f"gemm_f16_tn_{n}", "f16", "T", "N", n, n, n)


def skinny_fp16_16384x64x16384() -> Problem:
    return Problem("gemm_f16_tn_skinny_16384x64x16384", "f16", "T", "N", 16384, 64, 16384)


def diag_fp16_4096(layout_x: str = "N") -> DiagProblem:
    """A = diag(d) (4096 fp16 entries in U[-1,1]) times a dense 4096 x 4096 fp16
    B in U[-1,1], plus an fp32 C ~ N(0,1): D = A*B + C in fp32 (the mixed
    precision diagonal GEMM at N = 4096)."""
    return DiagProblem(f"diag_f16_left_{layout_x.lower()}_4096", "f16", "left", layout_x, 4096, 4096,
                       beta=1.0, c="f32", d="f32")


def pair_fp16_4096(unit: str) -> PairProblem:
    """Complex or dual GEMM D = A*B + C, M = N = K = 4096, fp16 A and B (both
    parts in U[-1,1]), fp32 C ~ N(0,1) and D, A and B column-major (N)."""
    return PairProblem(f"{'cgemm' if unit == 'complex' else 'dual_gemm'}_f16_nn_4096", unit, "f16",
                       "N", "N", 4096, 4096, 4096, beta=1.0, c="f32", d="f32")
