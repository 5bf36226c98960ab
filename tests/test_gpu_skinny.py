"""One tile column (N no wider than the single-CTA tile): every tile streams its
own rows of A over the whole of K and shares only B with the others.

Checked element by element against the fp64 oracle: a full wave of 128 x 64
tiles, a last stage holding a single K block, 128-wide tiles, ragged M and N,
the full epilogue and all four layouts.
"""
import pytest

import dense_gemm_epilogues_gb300 as G
from dense_gemm_epilogues_gb300 import inputs as I
import parity_helpers as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mnk_bn", [(16384, 64, 2048, 64), (3000, 40, 1064, 64), (1200, 128, 2112, 128)],
                         ids=lambda s: "x".join(map(str, s[:3])))
def test_single_tile_column(mnk_bn, monkeypatch):
    """128 tiles of 128 x 64 (a full wave, no stream-K); K = 1064: 17 K blocks, so
    the last stage of two slabs holds one; 128-wide tiles over K = 2112."""
    M, N, K, bn = mnk_bn
    monkeypatch.setenv("GEMM_TC_BN", str(bn))
    p = H.tma_aligned(I.Problem("skinny", "f16", "T", "N", M, N, K, alpha=1.25, beta=0.5, c="f32",
                                d="f32", bias="f32", bias_mode="col", act="relu"))
    cfg = H.run_and_check_full(p, 170, expect_kernel=G.GEMM_KERNEL_TC)
    assert cfg["sk_tiles"] == 0 and cfg["bn"] == bn and (p.N + bn - 1) // bn == 1, cfg


@pytest.mark.parametrize("layout", ["NN", "NT", "TN", "TT"])
def test_single_tile_column_all_layouts(layout):
    p = H.tma_aligned(I.Problem("skinny_lay", "bf16", layout[0], layout[1], 2000, 64, 2000, beta=-1.0,
                                c="bf16", d="bf16"))
    H.run_and_check_full(p, 171, expect_kernel=G.GEMM_KERNEL_TC)


@pytest.mark.parametrize("krot", ["on", "off"])
@pytest.mark.parametrize("layout", ["TN", "NT"])
def test_k_rotation_small_integers_bit_exact(krot, layout, monkeypatch):
    """With one tile column each tile starts its K loop at one of 8 evenly spaced
    K blocks and wraps around (a permutation of the K blocks: 19 blocks, the
    ragged last one landing mid-loop for most tiles).  Small integers keep every
    sum exact, so rotated and unrotated runs both equal the oracle bit for bit."""
    import numpy as np
    import torch
    monkeypatch.setenv("GEMM_TC_KROT", "1" if krot == "on" else "0")
    p = H.tma_aligned(I.Problem("skinny_rot", "f16", layout[0], layout[1], 128 * 12, 64, 64 * 18 + 40, alpha=2.0,
                                beta=1.0, c="f32", dist_a=I.Dist("small", -3, 3), dist_b=I.Dist("small", -3, 3),
                                dist_c=I.Dist("small", -50, 50)))
    inp = I.generate(p, 172)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0 and plan.last_config()["kernel"] == G.GEMM_KERNEL_TC
    np.testing.assert_array_equal(dp.result().cpu().numpy(), H.oracle_full(inp))
    plan.close()
