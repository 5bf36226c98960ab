"""Parity at the full workload sizes, in the launch configuration the benchmark
times (default selector, same problem definitions and seeds).

The 8192^3 fp16 TN GEMM and the 8192^3 int8 GEMM are compared with the oracle
on the whole output matrix.  The other layouts of the 8192^3 GEMM, the FC layer
and the square sweep are compared on whole rows at both edges of every
128-row block and whole columns at both edges of every 64-column block (every
CTA's rows of every tile, every epilogue chunk's columns, every half-tile unit
of a tail), plus random entries and corners.  Guard bands around D must be
untouched.
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


TC_ANY = (G.GEMM_KERNEL_TC, G.GEMM_KERNEL_TC_PAIR)


def _run(p: I.Problem, seed: int, expect_kernel, kernel=None):
    inp = I.generate(p, seed)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p, kernel)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    cfg = plan.last_config()
    allowed = expect_kernel if isinstance(expect_kernel, tuple) else (expect_kernel,)
    assert cfg["kernel"] in allowed, cfg
    dp.check_guards()
    plan.close()
    return inp, dp, cfg


def _check_whole(p: I.Problem, seed: int, expect_kernel):
    inp, dp, cfg = _run(p, seed, expect_kernel)
    got = dp.result().cpu()
    del dp
    torch.cuda.empty_cache()
    H.check_close(got, H.oracle_full(inp), p.d, p.name + " (whole matrix)")
    return cfg


def _check_boundaries(p: I.Problem, seed: int, expect_kernel, kernel=None, row_block=128, col_block=64):
    inp, dp, cfg = _run(p, seed, expect_kernel, kernel)
    rows, cols = H.boundary_entries(p.M, p.N, row_block, col_block)
    r2, c2 = H.sample_entries(p.M, p.N, N_SAMPLES, seed, cfg["bm"] or 128, cfg["bn"] or 128)
    rows, cols = np.concatenate([rows, r2]), np.concatenate([cols, c2])
    ref = H.oracle_entries(inp, rows, cols)
    got = dp.result()[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
    H.check_close(got, ref, p.d, p.name + " (block-edge rows and columns)")
    return cfg


def test_square_fp16_8192_tn_whole_matrix():
    cfg = _check_whole(I.square_fp16_8192("TN"), I.BASE_SEED + 1, G.GEMM_KERNEL_TC_PAIR)
    assert cfg["half_tiles"] > 0          # the tail's half-tile units are inside the checked matrix


def test_int8_8192_whole_matrix_exact():
    _check_whole(I.int8_8192(), I.BASE_SEED + 3, G.GEMM_KERNEL_TC_INT8)


@pytest.mark.parametrize("layout", ["NN", "NT", "TT"])
def test_square_fp16_8192_alpha_beta(layout):
    _check_boundaries(I.square_fp16_8192(layout), I.BASE_SEED + 1, G.GEMM_KERNEL_TC_PAIR)


@pytest.mark.parametrize("layout", ["NN", "TT"])
def test_square_fp16_8192_single_cta_kernel(layout):
    """The single-CTA tensor-core kernel at the full size (the selector runs pairs)."""
    _check_boundaries(I.square_fp16_8192(layout), I.BASE_SEED + 1, G.GEMM_KERNEL_TC, G.GEMM_KERNEL_TC)


def test_fc_bf16_bias_relu():
    _check_boundaries(I.fc_bf16_8192x4096x11008(), I.BASE_SEED + 2, G.GEMM_KERNEL_TC_PAIR)


def test_square_fp16_256_full():
    p = I.square_fp16_256()
    cfg = H.run_and_check_full(p, I.BASE_SEED + 0)
    assert cfg["kernel"] in TC_ANY


def test_sgemm_4096_bias_relu():
    _check_boundaries(I.sgemm_4096_bias_relu(), I.BASE_SEED + 4, G.GEMM_KERNEL_FFMA)


@pytest.mark.parametrize("n", [512, 1024, 2048, 4096])
def test_square_fp16_sweep_whole(n):
    p = I.square_fp16(n)
    cfg = H.run_and_check_full(p, I.BASE_SEED + 5)
    assert cfg["kernel"] in TC_ANY


def test_square_fp16_16384():
    _check_boundaries(I.square_fp16(16384), I.BASE_SEED + 5, TC_ANY)


def test_skinny_fp16_whole():
    p = I.skinny_fp16_16384x64x16384()
    cfg = H.run_and_check_full(p, I.BASE_SEED + 6)
    assert cfg["kernel"] in TC_ANY


def test_fc_relu_on_x_staged_at_full_size():
    """The FC layer with ReLU applied to X after load: X is re-read by 43 tile
    columns, so the selector stages the transform; whole rows and columns at
    both edges of every 256 x 256 pair tile against the oracle (its transformed
    path is slower, so the blocks are the pair tiles rather than 128 x 64)."""
    p = I.fc_bf16_8192x4096x11008().with_(name="fc_relu_x", a_act="relu")
    cfg = _check_boundaries(p, I.BASE_SEED + 2, G.GEMM_KERNEL_TC_PAIR, row_block=256, col_block=256)
    assert cfg["xf_staged"] == G.GEMM_XF_A


def test_skinny_relu_on_a_in_kernel():
    """The skinny GEMM with ReLU on A (A read by one tile column): the transform
    runs inside the kernel; block-edge rows and columns against the oracle."""
    p = I.skinny_fp16_16384x64x16384().with_(name="skinny_relu_a", a_act="relu", b_scale=0.5)
    cfg = _check_boundaries(p, I.BASE_SEED + 6, TC_ANY)
    assert cfg["xf_staged"] == 0
