"""Seeded random parity sweep: problems drawn at random (shape, layouts, operand
and output types, alpha/beta, C type, bias mode, activations, operand transforms,
padding, forced kernel) and each compared with the fp64 oracle on the whole
output -- a net for combinations the targeted tests do not list.

Every draw is reproducible from its index (numpy's PCG64 seeded with the base
seed plus the index); the id of a failing case names it.
"""
import numpy as np
import pytest
import torch

import dense_gemm_epilogues_gb300 as G
from dense_gemm_epilogues_gb300 import inputs as I

import parity_helpers as H

pytestmark = pytest.mark.gpu

N_CASES = 200


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.load_library()
    yield
    torch.cuda.synchronize()


@pytest.fixture(autouse=True)
def _clean_env(monkeypatch):
    for v in ("GEMM_TC_CTA_GROUP", "GEMM_TC_BN", "GEMM_TC_SPLITK", "GEMM_STREAM_K", "GEMM_TC_TAIL_HALVES",
              "GEMM_XF_STAGE", "GEMM_TC_KROT", "GEMM_FFMA_TAIL"):
        monkeypatch.delenv(v, raising=False)


def draw(i: int):
    rng = np.random.default_rng(I.BASE_SEED * 1000 + i)
    ab = str(rng.choice(["f16", "bf16", "f16", "bf16", "s8", "f32"]))
    la, lb = str(rng.choice(["N", "T"])), str(rng.choice(["N", "T"]))
    M = int(rng.integers(1, 700))
    N = int(rng.integers(1, 700))
    K = int(rng.integers(1, 600))
    kw = {}
    if ab == "s8":
        kw.update(dist_a=I.I8, dist_b=I.I8, c="s32", d=str(rng.choice(["s32", "s32", "s8"])),
                  alpha=float(rng.integers(-3, 4)), beta=float(rng.integers(-2, 3)),
                  dist_c=I.Dist("int", -1000, 1000))
        if kw["d"] == "s8":
            kw["out_scale"] = float(rng.choice([0.001, 0.0003, 0.01]))
        if rng.random() < 0.4:
            kw.update(bias="s32", bias_mode=str(rng.choice(["col", "row"])), dist_bias=I.Dist("int", -500, 500))
        for op in ("a", "b"):
            if rng.random() < 0.3:
                kw[f"{op}_act"] = "relu"
    else:
        c_choices = ["f32"] if ab == "f32" else ["f32", "f16", "bf16"]
        d_choices = ["f32"] if ab == "f32" else ["f32", "f16", "bf16"]
        kw.update(alpha=float(rng.choice([1.0, 0.5, -1.25, 2.0])), d=str(rng.choice(d_choices)))
        if rng.random() < 0.6:
            kw.update(beta=float(rng.choice([0.5, -1.0, 1.0])), c=str(rng.choice(c_choices)))
            if rng.random() < 0.3:
                kw["c_act"] = "relu"
        if rng.random() < 0.5:
            kw.update(bias=str(rng.choice(["f32", "f16", "bf16"] if ab != "f32" else ["f32"])),
                      bias_mode=str(rng.choice(["col", "row"])))
        if rng.random() < 0.5:
            kw["act"] = "relu"
        for op in ("a", "b"):
            if rng.random() < 0.3:
                kw[f"{op}_act"] = str(rng.choice(["relu", "none"]))
                kw[f"{op}_scale"] = float(rng.choice([1.0, 0.5, -0.75, 0.1, 3.0]))
    if rng.random() < 0.3:
        kw.update(pad_a=int(rng.integers(0, 9)), pad_b=int(rng.integers(0, 9)))
    if rng.random() < 0.2:
        kw["pad_d"] = int(rng.integers(1, 5))
    p = I.Problem(f"fuzz{i}", ab, la, lb, M, N, K, **kw)
    aligned = rng.random() < 0.7
    if aligned and ab in ("f16", "bf16"):
        p = H.tma_aligned(p)
    elif aligned and ab == "s8":
        p = H.tma_aligned(p, 16)
    elif aligned and ab == "f32":
        p = H.tma_aligned(p, 4)
    # Forced kernel (else the selector decides) and, for the tensor cores, the path
    # of the operand transforms.
    kernel = None
    env = {}
    if ab in ("f16", "bf16"):
        kernel = rng.choice([None, None, G.GEMM_KERNEL_TC, G.GEMM_KERNEL_TC_PAIR, G.GEMM_KERNEL_SIMT])
        if kernel == G.GEMM_KERNEL_TC:
            env["GEMM_TC_BN"] = str(rng.choice([64, 128, 256]))
        env["GEMM_XF_STAGE"] = str(rng.choice(["0", "1"]))
    elif ab == "f32":
        kernel = rng.choice([None, G.GEMM_KERNEL_SIMT])
    else:
        kernel = rng.choice([None, None, G.GEMM_KERNEL_SIMT])
        if rng.random() < 0.5:
            env["GEMM_TC_CTA_GROUP"] = "2"
    return p, (None if kernel is None else int(kernel)), env


def _tc_feasible(p: I.Problem) -> bool:
    es = I.ELEM_BYTES[p.ab]
    return (p.lda * es) % 16 == 0 and (p.ldb * es) % 16 == 0


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_problem(i, monkeypatch):
    p, kernel, env = draw(i)
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    if kernel in (G.GEMM_KERNEL_TC, G.GEMM_KERNEL_TC_PAIR) and not _tc_feasible(p):
        kernel = None                      # the forced tensor-core kernel needs TMA-aligned operands
    if kernel == G.GEMM_KERNEL_TC_PAIR and (p.M <= 128 or p.N <= 128):
        kernel = G.GEMM_KERNEL_TC
    inp = I.generate(p, 500 + i)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p, kernel)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    cfg = plan.last_config()
    if kernel is not None:
        assert cfg["kernel"] == kernel, (cfg, p)
    dp.check_guards()
    H.check_close(dp.result(), H.oracle_full(inp), p.d, f"{p} kernel={cfg['kernel_name']} env={env}")
    plan.close()
