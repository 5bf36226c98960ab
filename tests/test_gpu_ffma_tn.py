"""FFMA SGEMM in the TN case (A row-major, B column-major: both K-contiguous),
the layout of fp32 fully connected layers.

Checked element by element against the fp64 oracle: many K slices with a
ragged last one, ragged M and N over many tiles, every epilogue option, K
shorter than one slice, single rows and columns, batches, and bit-exact
small-integer data.
"""
import numpy as np
import pytest
import torch

import dense_gemm_epilogues_gb300 as G
from dense_gemm_epilogues_gb300 import inputs as I
import parity_helpers as H

pytestmark = pytest.mark.gpu


def test_ragged_m_n_k_full_epilogue():
    """1157 x 300 outputs (ragged in both), K = 1001: the last K slice holds one
    value; padded leading dimensions."""
    p = I.Problem("sgt1", "f32", "T", "N", 1157, 300, 1001, alpha=0.75, beta=-0.5, c="f32", d="bf16",
                  bias="f32", bias_mode="col", act="relu", pad_a=3, pad_b=3)
    H.run_and_check_full(p, 160, expect_kernel=G.GEMM_KERNEL_FFMA)


def test_row_bias_relu_on_c_f16_out():
    p = I.Problem("sgt2", "f32", "T", "N", 384, 520, 640, alpha=1.25, beta=1.0, c="f32", d="f16",
                  bias="f32", bias_mode="row", c_act="relu", act="relu")
    H.run_and_check_full(p, 161, expect_kernel=G.GEMM_KERNEL_FFMA)


@pytest.mark.parametrize("mnk", [(1, 1, 4), (7, 5, 20), (130, 129, 36), (64, 200, 96)],
                         ids=lambda s: "x".join(map(str, s)))
def test_short_k_and_tiny_shapes(mnk):
    """Single rows and columns, K of one or a few slices."""
    M, N, K = mnk
    p = I.Problem("sgt3", "f32", "T", "N", M, N, K, beta=0.5, c="f32")
    H.run_and_check_full(p, 162, expect_kernel=G.GEMM_KERNEL_FFMA)


def test_small_integers_bit_exact():
    """Products and sums of small integers are exact in fp32 in any order, so the
    result must equal the oracle bit for bit."""
    p = I.Problem("sgt4", "f32", "T", "N", 300, 260, 1000, alpha=2.0, beta=-1.0, c="f32",
                  dist_a=I.Dist("small", -3, 3), dist_b=I.Dist("small", -3, 3),
                  dist_c=I.Dist("small", -100, 100), bias="f32", bias_mode="col",
                  dist_bias=I.Dist("small", -50, 50), act="relu")
    inp = I.generate(p, 163)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert plan.last_config()["kernel"] == G.GEMM_KERNEL_FFMA
    np.testing.assert_array_equal(dp.result().cpu().numpy(), H.oracle_full(inp))
    dp.check_guards()
    plan.close()


def test_batched():
    from test_gpu_batched import run_batched
    p = I.Problem("sgt5", "f32", "T", "N", 200, 136, 264, alpha=0.5, beta=1.0, c="f32", bias="f32",
                  bias_mode="col", act="relu")
    assert run_batched(p, 3, 164)["kernel"] == G.GEMM_KERNEL_FFMA


# ----------------------------- split tail wave ------------------------------

def _slots():
    return 2 * torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("layout", ["TN", "NN", "NT", "TT"])
@pytest.mark.parametrize("tail", ["split", "whole"])
def test_split_tail_wave(layout, tail, monkeypatch):
    """Two CTAs per SM hold 2 x SMs tiles at a time; when the last wave holds at
    most half of that, its tiles are split over K into parts whose raw sums a
    reduction pass adds in K order before the epilogue.  Ragged M, N and K,
    full epilogue; the split and the unsplit run both against the oracle."""
    if tail == "whole":
        monkeypatch.setenv("GEMM_FFMA_TAIL", "0")
    else:
        monkeypatch.delenv("GEMM_FFMA_TAIL", raising=False)
    slots = _slots()
    tiles_n = 16
    tiles_m = (slots + 16 + tiles_n - 1) // tiles_n        # a few tiles past one full wave
    M, N = tiles_m * 128 - 36, tiles_n * 128 - 48     # multiples of 4: every layout stays on FFMA
    p = I.Problem("sgt_tail", "f32", layout[0], layout[1], M, N, 516, alpha=1.5, beta=-0.5, c="f32",
                  bias="f32", bias_mode="col", act="relu")
    cfg = H.run_and_check_full(p, 170, expect_kernel=G.GEMM_KERNEL_FFMA)
    rem = (tiles_m * tiles_n) % slots
    if tail == "split":
        assert cfg["sk_tiles"] == rem and cfg["split_k"] >= 2, cfg
        assert cfg["grid"] == tiles_m * tiles_n - rem + rem * cfg["split_k"]
    else:
        assert cfg["sk_tiles"] == 0 and cfg["grid"] == tiles_m * tiles_n


def test_split_tail_bit_exact_on_small_integers():
    """Small integers: every partial sum is exact, so the split tail gives the
    oracle's result bit for bit."""
    slots = _slots()
    M, N = ((slots + 8 + 15) // 16) * 128, 16 * 128
    p = I.Problem("sgt_tail_x", "f32", "T", "N", M, N, 768, alpha=2.0, beta=1.0, c="f32",
                  dist_a=I.Dist("small", -3, 3), dist_b=I.Dist("small", -3, 3),
                  dist_c=I.Dist("small", -100, 100))
    inp = I.generate(p, 171)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    cfg = plan.last_config()
    assert cfg["kernel"] == G.GEMM_KERNEL_FFMA and cfg["sk_tiles"] > 0, cfg
    np.testing.assert_array_equal(dp.result().cpu().numpy(), H.oracle_full(inp))
    plan.close()
