"""Parity at the full workload sizes, in the launch configuration the benchmark
times (default selector, same problem definitions and seeds).

The oracle recomputes sampled outputs one by one (random entries, corners and
tile-boundary rows/columns); the int8 workload is also checked on whole rows.
Guard bands around D must be untouched.
"""
import numpy as np
import pytest
import torch

import dense_gemm_epilogues_gb300 as G
from dense_gemm_epilogues_gb300 import inputs as I

import parity_helpers as H

pytestmark = pytest.mark.gpu

N_SAMPLES = 1500


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.load_library()
    yield
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kernel", [G.GEMM_KERNEL_TC, G.GEMM_KERNEL_TC_PAIR], ids=["cta1", "pair"])
@pytest.mark.parametrize("layout", ["NN", "TT"])
def test_square_fp16_8192_each_tensor_core_kernel(layout, kernel):
    """Both tensor-core kernels at the full size (the selector runs the pair kernel)."""
    p = I.square_fp16_8192(layout)
    inp = I.generate(p, I.BASE_SEED + 1)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p, kernel)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0 and plan.last_config()["kernel"] == kernel
    dp.check_guards()
    rows, cols = H.sample_entries(p.M, p.N, 600, 7, 256, 256)
    ref = H.oracle_entries(inp, rows, cols)
    got = dp.result()[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
    H.check_close(got, ref, p.d, p.name)
    plan.close()


TC_ANY = (G.GEMM_KERNEL_TC, G.GEMM_KERNEL_TC_PAIR)


def _check_sampled(p: I.Problem, seed: int, expect_kernel, extra_rows=()):
    inp = I.generate(p, seed)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    cfg = plan.last_config()
    allowed = expect_kernel if isinstance(expect_kernel, tuple) else (expect_kernel,)
    assert cfg["kernel"] in allowed, cfg
    dp.check_guards()
    rows, cols = H.sample_entries(p.M, p.N, N_SAMPLES, seed, cfg["bm"] or 128, cfg["bn"] or 128)
    for r in extra_rows:
        rows = np.concatenate([rows, np.full(p.N, r, dtype=np.int64)])
        cols = np.concatenate([cols, np.arange(p.N, dtype=np.int64)])
    ref = H.oracle_entries(inp, rows, cols)
    got = dp.result()[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
    H.check_close(got, ref, p.d, p.name)
    plan.close()
    return cfg


def test_square_fp16_256_full():
    p = I.square_fp16_256()
    cfg = H.run_and_check_full(p, I.BASE_SEED + 0)
    assert cfg["kernel"] in TC_ANY


@pytest.mark.parametrize("layout", ["NN", "NT", "TN", "TT"])
def test_square_fp16_8192_alpha_beta(layout):
    _check_sampled(I.square_fp16_8192(layout), I.BASE_SEED + 1, G.GEMM_KERNEL_TC_PAIR)


def test_fc_bf16_bias_relu():
    _check_sampled(I.fc_bf16_8192x4096x11008(), I.BASE_SEED + 2, G.GEMM_KERNEL_TC_PAIR)


def test_int8_8192_exact():
    _check_sampled(I.int8_8192(), I.BASE_SEED + 3, G.GEMM_KERNEL_TC_INT8, extra_rows=(0, 8191))


def test_sgemm_4096_bias_relu():
    _check_sampled(I.sgemm_4096_bias_relu(), I.BASE_SEED + 4, G.GEMM_KERNEL_FFMA)


@pytest.mark.parametrize("n", [512, 1024, 2048, 4096, 16384])
def test_square_fp16_sweep(n):
    _check_sampled(I.square_fp16(n), I.BASE_SEED + 5, TC_ANY)


def test_skinny_fp16():
    _check_sampled(I.skinny_fp16_16384x64x16384(), I.BASE_SEED + 6, TC_ANY)
