"""CTA-pair kernel: the tiles of a partial last wave run as two 256 x 128 halves.

With T output tiles over G CTA pairs, the last r = T mod G tiles, when 2r <= G,
become 2r units of half a tile's columns (an N = 128 MMA, 64 columns of B per
CTA), one per pair.  Every unit must produce exactly its columns: whole and
ragged tiles, a half lying entirely beyond N, all four operand layouts, and the
full epilogue.  Compared element by element with the fp64 oracle.
"""
import pytest
import torch

import dense_gemm_epilogues_gb300 as G
from dense_gemm_epilogues_gb300 import inputs as I
import parity_helpers as H

pytestmark = pytest.mark.gpu

LAYOUTS = ["NN", "NT", "TN", "TT"]


@pytest.fixture
def pairs(monkeypatch):
    monkeypatch.setenv("GEMM_TC_CTA_GROUP", "2")
    monkeypatch.delenv("GEMM_TC_TAIL_HALVES", raising=False)
    monkeypatch.delenv("GEMM_STREAM_K", raising=False)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_all_tiles_split_when_they_fit_half_the_pairs(layout, pairs):
    """3 x 5 tiles, far fewer than the pairs: every tile runs as two halves."""
    p = H.tma_aligned(I.Problem("halves_small", "f16", layout[0], layout[1], 768, 1280, 320, alpha=1.25,
                                beta=0.5, c="f32", d="f32"))
    cfg = H.run_and_check_full(p, 140, expect_kernel=G.GEMM_KERNEL_TC_PAIR)
    assert cfg["half_tiles"] == 15 and cfg["grid"] == 2 * 30, cfg


@pytest.mark.parametrize("layout", LAYOUTS)
def test_ragged_halves_with_full_epilogue(layout, pairs):
    """Ragged M and N: the last tile column holds 76 valid columns, so its second
    half lies wholly beyond N; bias, ReLU, beta*C and a bf16 cast."""
    p = H.tma_aligned(I.Problem("halves_ragged", "bf16", layout[0], layout[1], 600, 1100, 200, alpha=0.75,
                                beta=-0.5, c="f32", d="bf16", bias="f32", bias_mode="col", act="relu"))
    cfg = H.run_and_check_full(p, 141, expect_kernel=G.GEMM_KERNEL_TC_PAIR)
    assert cfg["half_tiles"] == 3 * 5, cfg


def test_tail_of_several_waves(pairs):
    """More tiles than pairs: whole tiles first, then the split tail (when the
    remainder is at most half the pairs on this device)."""
    p = H.tma_aligned(I.Problem("halves_waves", "f16", "T", "N", 2048, 3072, 128, beta=1.0, c="f16", d="f16"))
    cfg = H.run_and_check_full(p, 142, expect_kernel=G.GEMM_KERNEL_TC_PAIR)
    pairs_n = cfg["grid"] // 2
    r = cfg["tiles"] % pairs_n
    assert cfg["half_tiles"] == (r if 0 < 2 * r <= pairs_n else 0), cfg


def test_halves_off_gives_the_same_bits(pairs, monkeypatch):
    """The split changes which pair computes which columns, not the arithmetic:
    the same K order per element, so D is bit-identical with the split off."""
    p = H.tma_aligned(I.Problem("halves_bits", "bf16", "T", "N", 1024, 1536, 512, alpha=1.5, beta=0.5,
                                c="f32", d="f32", bias="f32", bias_mode="col", act="relu"))
    inp = I.generate(p, 143)
    out = {}
    for mode in ("1", "0"):
        monkeypatch.setenv("GEMM_TC_TAIL_HALVES", mode)
        dp = H.DeviceProblem(inp)
        plan = H.make_plan(p)
        dp.run(plan)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        cfg = plan.last_config()
        assert (cfg["half_tiles"] > 0) == (mode == "1"), cfg
        out[mode] = dp.result().clone()
        dp.check_guards()
        plan.close()
    H.check_close(out["1"], H.oracle_full(inp), p.d, p.name)
    assert torch.equal(out["1"], out["0"])


def test_batched_halves(pairs):
    """A strided batch whose tiles all fit as halves: each unit finds its problem."""
    from test_gpu_batched import run_batched
    p = H.tma_aligned(I.Problem("halves_batched", "f16", "T", "N", 512, 512, 256, alpha=0.5, beta=1.0,
                                c="f16", d="f16", pad_d=8))
    cfg = run_batched(p, 4, 144)
    assert cfg["kernel"] == G.GEMM_KERNEL_TC_PAIR and cfg["half_tiles"] == 4 * 2 * 2, cfg
