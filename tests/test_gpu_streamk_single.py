"""Single-CTA tensor-core kernel with stream-K: all CTAs share the tiles' K blocks.

Each CTA takes an equal contiguous range of the linear (tile, K block) space;
a CTA holding part of a tile publishes its raw fp32 partial and counts itself in
on the tile, and the last to arrive adds every part in K order and runs the
epilogue.  Checked element by element against the fp64 oracle: all layouts, the
full epilogue, ragged M, N and K, tiles shared by many CTAs, batches, repeated
launches and CUDA-graph replay (the arrival counters must return to zero).
"""
import pytest
import torch

import dense_gemm_epilogues_gb300 as G
from dense_gemm_epilogues_gb300 import inputs as I
import parity_helpers as H

pytestmark = pytest.mark.gpu

LAYOUTS = ["NN", "NT", "TN", "TT"]


@pytest.fixture
def single_sk(monkeypatch):
    monkeypatch.setenv("GEMM_TC_CTA_GROUP", "1")
    monkeypatch.setenv("GEMM_TC_SPLITK", "1")


def _check_sk(cfg):
    assert cfg["kernel"] == G.GEMM_KERNEL_TC and cfg["sk_tiles"] == cfg["tiles"] and cfg["split_k"] > 1, cfg


@pytest.mark.parametrize("layout", LAYOUTS)
def test_split_tiles_full_epilogue(layout, single_sk):
    p = H.tma_aligned(I.Problem("sk1", "bf16", layout[0], layout[1], 384, 640, 3072, alpha=0.75, beta=-0.5,
                                c="f32", d="bf16", bias="f32", bias_mode="col", act="relu"))
    _check_sk(H.run_and_check_full(p, 150))


def test_ragged_m_n_k(single_sk):
    """Ragged tiles in M and N and a partial last K block."""
    p = H.tma_aligned(I.Problem("sk1_ragged", "f16", "T", "N", 300, 200, 5000, alpha=1.25, beta=0.5, c="f16",
                                d="f32"))
    _check_sk(H.run_and_check_full(p, 151))


def test_many_ctas_per_tile(single_sk):
    """Few tiles, deep K: dozens of CTAs share each tile."""
    p = H.tma_aligned(I.Problem("sk1_deep", "f16", "T", "N", 256, 256, 8192, beta=0.0, d="f32"))
    cfg = H.run_and_check_full(p, 152)
    _check_sk(cfg)
    assert cfg["split_k"] >= 8, cfg


def test_skinny(single_sk):
    """The skinny shape class (N = 64, one tile column)."""
    p = H.tma_aligned(I.Problem("sk1_skinny", "f16", "T", "N", 16384, 64, 2048, beta=0.0, d="f32"))
    _check_sk(H.run_and_check_full(p, 153))


def test_batched(single_sk):
    from test_gpu_batched import run_batched
    p = H.tma_aligned(I.Problem("sk1_batched", "f16", "T", "N", 256, 384, 1536, alpha=0.5, beta=1.0, c="f32",
                                d="f16", pad_d=8))
    cfg = run_batched(p, 3, 154)
    _check_sk(cfg)


def test_repeated_launches_and_graph_replay(single_sk):
    """Counters go back to zero after every launch: plain repeats and replays of
    a captured CUDA graph all give the right result."""
    p = H.tma_aligned(I.Problem("sk1_rep", "f16", "T", "N", 512, 512, 4096, alpha=1.5, beta=0.5, c="f32",
                                d="f32"))
    inp = I.generate(p, 155)
    ref = H.oracle_full(inp)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p)
    for _ in range(3):
        dp.D.fill_(0)
        dp.run(plan)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        _check_sk(plan.last_config())
        H.check_close(dp.result(), ref, "f32", "stream-K repeat")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            dp.run(plan, stream=s.cuda_stream)
    torch.cuda.synchronize()
    for _ in range(3):
        dp.D.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        H.check_close(dp.result(), ref, "f32", "stream-K graph replay")
    dp.check_guards()
    plan.close()


def test_split_and_whole_tiles_both_match_the_oracle(monkeypatch):
    """The same problem with stream-K off and on: both within the oracle's
    tolerance (they differ only in the order of fp32 additions)."""
    monkeypatch.setenv("GEMM_TC_CTA_GROUP", "1")
    p = H.tma_aligned(I.Problem("sk1_onoff", "f16", "N", "T", 256, 512, 4096, beta=0.0, d="f32"))
    inp = I.generate(p, 156)
    out = {}
    for mode in ("0", "1"):
        monkeypatch.setenv("GEMM_TC_SPLITK", mode)
        dp = H.DeviceProblem(inp)
        plan = H.make_plan(p)
        dp.run(plan)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        assert (plan.last_config()["sk_tiles"] > 0) == (mode == "1")
        out[mode] = dp.result().clone()
        plan.close()
    ref = H.oracle_full(inp)
    H.check_close(out["1"], ref, "f32", "split")
    H.check_close(out["0"], ref, "f32", "whole")
