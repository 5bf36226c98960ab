"""GPU parity of the two-pair clusters of the CTA-pair kernel: clusters of four
CTAs on vertically adjacent 256 x 256 tiles that share B by TMA multicast
(gemm_config_t.cluster == 4).  Each cluster size is forced in turn through
GEMM_TC_CLUSTER and compared with the oracle element by element."""
import pytest
import torch

import dense_gemm_epilogues_gb300 as G
from dense_gemm_epilogues_gb300 import inputs as I

import parity_helpers as H

pytestmark = pytest.mark.gpu
LAYOUTS = ["NN", "NT", "TN", "TT"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.load_library()


@pytest.fixture(params=[4, 2], ids=["quad", "pair"])
def cluster(request, monkeypatch):
    monkeypatch.setenv("GEMM_TC_CLUSTER", str(request.param))
    monkeypatch.setenv("GEMM_TC_CTA_GROUP", "2")   # pairs even where the grid is under a wave
    return request.param


def _run(p, seed, cluster):
    cfg = H.run_and_check_full(p, seed, expect_kernel=G.GEMM_KERNEL_TC_PAIR)
    assert cfg["cluster"] == cluster and cfg["cta_group"] == 2
    return cfg


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("ab", ["f16", "bf16"])
def test_ragged_alpha_beta(layout, ab, cluster):
    """600 x 520 x 200: two super-tile rows (the second one half outside D),
    ragged columns and K."""
    p = H.tma_aligned(I.Problem("quad", ab, layout[0], layout[1], 600, 520, 200, alpha=1.5,
                                beta=-0.5, c="f32", bias="f32", bias_mode="col", act="relu",
                                pad_d=3))
    _run(p, 600, cluster)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_odd_tile_rows_leave_a_pair_outside(layout, cluster):
    """Three tile rows: the second pair of the last super-tile computes rows that
    lie entirely outside D (its loads read zeros, its stores are masked)."""
    p = H.tma_aligned(I.Problem("quad_odd", "f16", layout[0], layout[1], 700, 300, 136, beta=1.0,
                                c="f32"))
    _run(p, 610, cluster)


def test_many_super_tiles_persistent(cluster):
    """More super-tiles than clusters: each cluster walks several."""
    p = I.Problem("quad_many", "bf16", "T", "N", 4096, 3072, 192, beta=0.25, c="bf16", d="bf16")
    cfg = _run(p, 620, cluster)
    assert cfg["tiles"] > cfg["grid"] // 2


def test_small_integers_bit_exact(cluster):
    p = I.Problem("quad_exact", "f16", "N", "T", 1024, 768, 512, alpha=2.0, beta=1.0, c="f32",
                  dist_a=I.Dist("small", -3, 3), dist_b=I.Dist("small", -3, 3),
                  dist_c=I.Dist("small", -3, 3))
    inp = I.generate(p, 630)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0 and plan.last_config()["cluster"] == cluster
    dp.check_guards()
    import numpy as np
    np.testing.assert_array_equal(dp.result().cpu().numpy(), H.oracle_full(inp))
    plan.close()


def test_batched_super_tiles(cluster):
    """Strided batch: the problem index is the outer coordinate of the super-tiles."""
    import test_gpu_batched as TB
    p = H.tma_aligned(I.Problem("quad_bat", "f16", "T", "N", 520, 264, 128, beta=0.5, c="f32"))
    cfg = TB.run_batched(p, 3, 640)
    assert cfg["kernel"] == G.GEMM_KERNEL_TC_PAIR and cfg["cluster"] == cluster
