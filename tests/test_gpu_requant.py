"""GPU parity of the int8 requantising output of int8 problems (out_dtype
GEMM_S8: D = saturate_int8(round_half_even(fp32(v) * out_scale))) against the
oracle, bit for bit, on every kernel that finishes an int8 problem."""
import numpy as np
import pytest
import torch

import dense_gemm_epilogues_gb300 as G
from dense_gemm_epilogues_gb300 import inputs as I

import parity_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.load_library()


def _problem(layout, M, N, K, **kw):
    base = dict(alpha=1.0, beta=1.0, c="s32", d="s8", bias="s32", bias_mode="col", act="relu",
                out_scale=0.0173, dist_a=I.I8, dist_b=I.I8, dist_c=I.Dist("int", -20000, 20000),
                dist_bias=I.Dist("int", -2000, 2000), pad_d=5)
    base.update(kw)
    return H.tma_aligned(I.Problem("rq", "s8", layout[0], layout[1], M, N, K, **base))


@pytest.mark.parametrize("cta_group", ["1", "2"])
@pytest.mark.parametrize("layout", ["TN", "NT", "NN", "TT"])
def test_requant_tensor_core_kernels(layout, cta_group, monkeypatch):
    monkeypatch.setenv("GEMM_TC_CTA_GROUP", cta_group)
    cfg = H.run_and_check_full(_problem(layout, 300, 280, 1100), 800,
                               expect_kernel=G.GEMM_KERNEL_TC_INT8)
    assert cfg["cta_group"] == int(cta_group)


def test_requant_saturates_and_rounds_ties_on_the_gpu():
    """Large scale: most outputs saturate; small-integer C makes exact .5 ties."""
    p = _problem("TN", 256, 256, 64, out_scale=0.5, act="none", bias_mode="none", bias=None,
                 dist_a=I.Dist("int", -3, 3), dist_b=I.Dist("int", -3, 3),
                 dist_c=I.Dist("int", -400, 400))
    H.run_and_check_full(p, 801)


def test_requant_generic_kernel_and_row_bias():
    p = I.Problem("rq_gen", "s8", "T", "N", 77, 65, 33, beta=-2.0, c="s32", d="s8", bias="s32",
                  bias_mode="row", out_scale=-0.031, dist_a=I.I8, dist_b=I.I8,
                  dist_c=I.Dist("int", -3000, 3000), dist_bias=I.Dist("int", -500, 500), pad_a=3)
    assert H.run_and_check_full(p, 802)["kernel"] == G.GEMM_KERNEL_SIMT


def test_requant_diagonal_operand():
    p = I.DiagProblem("rq_diag", "s8", "left", "N", 130, 200, beta=1.0, c="s32", d="s8",
                      dist_diag=I.I8, dist_x=I.I8, dist_c=I.Dist("int", -3000, 3000))
    dinp = I.generate_diag(p, 803)
    dd = H.DeviceDiag(dinp)
    plan = H.make_diag_plan(p)
    G.gemm_run_diag(plan.handle, G.GEMM_SIDE_LEFT, G.GEMM_OP_N, p.M, p.N, p.alpha, dd.diag.data_ptr(),
                    dd.X.data_ptr(), p.ldx, p.beta, dd.C.data_ptr(), p.ldc, dd.D.data_ptr(), p.ldd,
                    G.make_epilogue(G.GEMM_S8, out_scale=0.02), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    dp = H.dense_inputs_of(dinp)
    ref = H.oracle_full(I.Inputs(dp.A, dp.B, dp.C, dp.bias, dp.problem.with_(out_scale=0.02)))
    H.check_close(dd.result(), ref, "s8", "diagonal int8 -> int8")
    plan.close()


def test_requant_host_entry():
    p = _problem("TN", 200, 160, 96, pad_d=0)
    inp = I.generate(p, 804)
    plan = H.make_plan(p)
    D = torch.zeros((p.M, p.ldd), dtype=torch.int8).pin_memory()
    bias = inp.bias.pin_memory()
    epi = G.make_epilogue(G.GEMM_S8, bias.data_ptr(), G.GEMM_S32, G.GEMM_BIAS_COL, G.GEMM_ACT_RELU,
                          out_scale=p.out_scale)
    G.gemm_run_host(plan.handle, G.GEMM_OP_T, G.GEMM_OP_N, p.M, p.N, p.K, p.alpha,
                    inp.A.pin_memory().data_ptr(), p.lda, inp.B.pin_memory().data_ptr(), p.ldb, p.beta,
                    inp.C.pin_memory().data_ptr(), p.ldc, D.data_ptr(), p.ldd, epi,
                    torch.cuda.current_stream().cuda_stream)
    H.check_close(D[:, :p.N], H.oracle_full(inp), "s8", "host int8 -> int8")
    plan.close()


def test_requant_rejects_non_finite_scale():
    plan = G.Plan(G.GEMM_S8, G.GEMM_S32, torch.cuda.current_device())
    A = torch.zeros(64 * 64, dtype=torch.int8, device="cuda")
    D = torch.zeros(64 * 64, dtype=torch.int8, device="cuda")
    with pytest.raises(G.GemmError) as e:
        G.gemm_run(plan.handle, G.GEMM_OP_T, G.GEMM_OP_N, 64, 64, 64, 1.0, A.data_ptr(), 64,
                   A.data_ptr(), 64, 0.0, None, 0, D.data_ptr(), 64,
                   G.make_epilogue(G.GEMM_S8, out_scale=float("nan")))
    assert e.value.status == G.GEMM_ERR_INVALID_ARG
    plan.close()
