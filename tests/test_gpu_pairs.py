"""GPU parity of gemm_run_complex (complex and dual-number GEMM on interleaved
storage, "Flexible Performant GEMM Kernels on GPUs", section 5.4) against the
oracle's pair GEMM, element by element."""
import numpy as np
import pytest
import torch

import dense_gemm_epilogues_gb300 as G
from dense_gemm_epilogues_gb300 import inputs as I

import parity_helpers as H

pytestmark = pytest.mark.gpu
SMALL = I.Dist("small", -3, 3)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.load_library()


def run_full(p: I.PairProblem, seed: int, exact=False, **run_kw) -> dict:
    inp = I.generate_pairs(p, seed)
    dp = H.DevicePairs(inp)
    plan = H.make_pair_plan(p)
    dp.run(plan, **run_kw)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    cfg = plan.last_config()
    dp.check_guards()
    ref = H.oracle_pairs_full(inp)
    if exact:
        np.testing.assert_array_equal(dp.result().cpu().numpy(), ref)
    else:
        H.check_close(dp.result(), ref, p.d, p.name)
    plan.close()
    return cfg


@pytest.mark.parametrize("unit", ["complex", "dual"])
@pytest.mark.parametrize("layout", ["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("ab", ["f16", "bf16"])
def test_pairs_tensor_cores(unit, layout, ab):
    """300 x 150 x 100 pairs: a real GEMM of 300 x 300 x 200, ragged in every
    dimension of the CTA-pair tiles; alpha, beta, C, bias pairs and ReLU."""
    p = I.PairProblem(f"{unit}_{ab}", unit, ab, layout[0], layout[1], 300, 150, 100, alpha=1.5,
                      beta=-0.5, c="f32", bias="f32", bias_mode="col", act="relu", pad_d=2)
    cfg = run_full(p, 500)
    assert cfg["kernel"] in (G.GEMM_KERNEL_TC, G.GEMM_KERNEL_TC_PAIR)


@pytest.mark.parametrize("unit", ["complex", "dual"])
@pytest.mark.parametrize("layout", ["NN", "TN", "NT", "TT"])
def test_pairs_small_integers_bit_exact(unit, layout):
    """Small-integer parts: every product and partial sum is exact in fp32, so
    the tensor-core result must equal the oracle bit for bit."""
    p = I.PairProblem("exact", unit, "f16", layout[0], layout[1], 136, 72, 200, alpha=2.0,
                      beta=1.0, c="f32", dist_a=SMALL, dist_b=SMALL, dist_c=SMALL)
    run_full(p, 510, exact=True)


def test_pairs_f32_on_cuda_cores_and_16_bit_outputs():
    cfg = run_full(I.PairProblem("c32", "complex", "f32", "T", "N", 130, 70, 50, beta=1.0, c="f32",
                                 c_act="relu"), 520)
    assert cfg["kernel"] in (G.GEMM_KERNEL_FFMA, G.GEMM_KERNEL_SIMT)
    run_full(I.PairProblem("c16", "dual", "bf16", "N", "T", 96, 64, 80, beta=0.5, c="bf16",
                           d="bf16"), 521)
    run_full(I.PairProblem("c16h", "complex", "f16", "T", "T", 64, 40, 48, beta=2.0, c="f16",
                           d="f16"), 522)


def test_pairs_unaligned_operands_are_staged():
    """lda = 101 pairs: a row-major A that TMA cannot address is copied to an
    aligned scratch first; B one scalar off a pair boundary takes the unaligned
    loads of the staging pass."""
    p = I.PairProblem("odd", "complex", "f16", "T", "N", 140, 90, 100, pad_a=1, beta=1.0, c="f32")
    inp = I.generate_pairs(p, 530)
    dp = H.DevicePairs(inp)
    Bshift = torch.empty(dp.B.numel() + 1, dtype=dp.B.dtype, device="cuda")
    Bshift[1:] = dp.B.reshape(-1)
    plan = H.make_pair_plan(p)
    dp.run(plan, B=Bshift.data_ptr() + Bshift.element_size())
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert plan.last_config()["kernel"] in (G.GEMM_KERNEL_TC, G.GEMM_KERNEL_TC_PAIR)
    dp.check_guards()
    H.check_close(dp.result(), H.oracle_pairs_full(inp), p.d, p.name)
    plan.close()


def test_pairs_k_zero_and_empty():
    run_full(I.PairProblem("k0", "complex", "f16", "T", "N", 33, 17, 0, beta=-2.0, c="f32",
                           bias="f32", bias_mode="col"), 540)
    plan = G.Plan(G.GEMM_F16, G.GEMM_F32, torch.cuda.current_device())
    G.gemm_run_complex(plan.handle, G.GEMM_UNIT_DUAL, G.GEMM_OP_T, G.GEMM_OP_N, 0, 8, 8, 1.0, None,
                       8, None, 8, 0.0, None, 0, None, 8)
    assert plan.last_config()["kernel"] == G.GEMM_KERNEL_NONE
    plan.close()


def test_pairs_argument_errors():
    X = torch.zeros(64 * 64 * 2, dtype=torch.float16, device="cuda")
    D = torch.zeros(64 * 64 * 2, dtype=torch.float32, device="cuda")
    plan = G.Plan(G.GEMM_F16, G.GEMM_F32, torch.cuda.current_device())
    args = [plan.handle, G.GEMM_UNIT_IMAGINARY, G.GEMM_OP_T, G.GEMM_OP_N, 64, 64, 64, 1.0,
            X.data_ptr(), 64, X.data_ptr(), 64, 0.0, None, 0, D.data_ptr(), 64]
    for i, bad, status in ((1, 5, G.GEMM_ERR_INVALID_ARG), (9, 10, G.GEMM_ERR_INVALID_ARG),
                           (15, None, G.GEMM_ERR_INVALID_ARG)):
        a = list(args)
        a[i] = bad
        with pytest.raises(G.GemmError) as e:
            G.gemm_run_complex(*a)
        assert e.value.status == status
    with pytest.raises(G.GemmError) as e:   # a row bias would need M pairs added per row
        G.gemm_run_complex(*args, G.make_epilogue(G.GEMM_F32, D.data_ptr(), G.GEMM_F32,
                                                  G.GEMM_BIAS_ROW))
    assert e.value.status == G.GEMM_ERR_UNSUPPORTED
    plan.close()
    p8 = G.Plan(G.GEMM_S8, G.GEMM_S32, torch.cuda.current_device())
    with pytest.raises(G.GemmError) as e:
        G.gemm_run_complex(p8.handle, G.GEMM_UNIT_IMAGINARY, G.GEMM_OP_T, G.GEMM_OP_N, 64, 64, 64,
                           1.0, X.data_ptr(), 64, X.data_ptr(), 64, 0.0, None, 0, D.data_ptr(), 64,
                           G.make_epilogue(G.GEMM_S32))
    assert e.value.status == G.GEMM_ERR_UNSUPPORTED
    p8.close()


@pytest.mark.parametrize("unit", ["complex", "dual"])
def test_pairs_full_size_sampled(unit):
    """The 4096-pair workload the benchmark times (column-major A and B, both
    staged), checked on sampled output pairs with tile edges."""
    p = I.pair_fp16_4096(unit)
    inp = I.generate_pairs(p, I.BASE_SEED + 30)
    dp = H.DevicePairs(inp)
    plan = H.make_pair_plan(p)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert plan.last_config()["kernel"] == G.GEMM_KERNEL_TC_PAIR
    dp.check_guards()
    rows, cols = H.sample_entries(p.M, p.N, 1200, 31, 256, 128)
    ref = H.oracle_pairs_entries(inp, rows, cols)
    got = dp.result()[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
    H.check_close(got, ref, p.d, p.name)
    plan.close()
