"""GPU parity of gemm_run_diag (one diagonal operand, stored as its diagonal)
against the oracle run on the same GEMM with the diagonal written out as a
dense square matrix ("Flexible Performant GEMM Kernels on GPUs", section 5.2)."""
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


def run_full(p: I.DiagProblem, seed: int) -> dict:
    dinp = I.generate_diag(p, seed)
    dd = H.DeviceDiag(dinp)
    plan = H.make_diag_plan(p)
    dd.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    cfg = plan.last_config()
    assert cfg["kernel"] == G.GEMM_KERNEL_DIAG
    dd.check_guards()
    H.check_close(dd.result(), H.oracle_full(H.dense_inputs_of(dinp)), p.d, p.name)
    plan.close()
    return cfg


FLOAT_EPI = [
    dict(),
    dict(alpha=1.25, beta=-0.5, c="f32", bias="f32", bias_mode="col", act="relu"),
    dict(alpha=0.75, beta=2.0, c="f16", d="bf16", bias="bf16", bias_mode="row", c_act="relu"),
]


@pytest.fixture(params=["tma", "registers"])
def diag_kernel(request, monkeypatch):
    """16-bit x with TMA-alignable operands takes the TMA-staged kernel by
    default; GEMM_DIAG_TMA=0 keeps the register kernel, so both are checked."""
    if request.param == "registers":
        monkeypatch.setenv("GEMM_DIAG_TMA", "0")
    else:
        monkeypatch.delenv("GEMM_DIAG_TMA", raising=False)
    return request.param


@pytest.mark.parametrize("side", ["left", "right"])
@pytest.mark.parametrize("layout", ["N", "T"])
@pytest.mark.parametrize("ab", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("epi", range(len(FLOAT_EPI)))
def test_diag_float(side, layout, ab, epi, diag_kernel):
    """200 x 136: 4 x 3 tiles of 64 x 64 with ragged last rows and columns."""
    if ab == "f32" and diag_kernel == "registers":
        pytest.skip("fp32 x always takes the register kernel (covered by the tma case)")
    kw = dict(FLOAT_EPI[epi])
    if ab == "f32" and kw.get("c"):
        kw["c"] = "f32"                    # fp32 plans take fp32 C only
    p = I.DiagProblem(f"diag_{ab}", ab, side, layout, 200, 136, **kw)
    cfg = run_full(p, 400 + epi)
    assert cfg["tiles"] == 4 * 3 and cfg["bm"] == 64 and cfg["bn"] == 64
    staged = ab != "f32" and diag_kernel == "tma"
    assert cfg["stages"] == (6 if staged else 1), cfg
    assert cfg["grid"] == (min(12, torch.cuda.get_device_properties(0).multi_processor_count) if staged
                           else cfg["grid"])


@pytest.mark.parametrize("side", ["left", "right"])
@pytest.mark.parametrize("layout", ["N", "T"])
@pytest.mark.parametrize("cd", [("f32", "f32"), ("bf16", "f16"), (None, "bf16")], ids=["f32C", "bf16C", "noC"])
def test_diag_tma_kernel_many_tiles(side, layout, cd):
    """The TMA-staged kernel on more tiles than CTAs (every CTA cycles its ring
    of stages several times), a ragged last tile row and column, every C type."""
    c, d = cd
    kw = dict(alpha=1.5, beta=0.5, c=c) if c else dict(alpha=1.5)
    p = I.DiagProblem("diag_tma_many", "bf16", side, layout, 64 * 40 + 16, 64 * 33 + 40, d=d,
                      bias="f32", bias_mode="col", act="relu", **kw)
    cfg = run_full(p, 440)
    assert cfg["stages"] == 6 and cfg["tiles"] == 41 * 34


@pytest.mark.parametrize("side", ["left", "right"])
@pytest.mark.parametrize("layout", ["N", "T"])
def test_diag_int8_exact(side, layout):
    p = I.DiagProblem("diag_s8", "s8", side, layout, 130, 200, alpha=3.0, beta=-2.0, c="s32",
                      d="s32", bias="s32", bias_mode="col", act="relu", dist_diag=I.I8,
                      dist_x=I.I8, dist_c=I.Dist("int", -50000, 50000),
                      dist_bias=I.Dist("int", -1000, 1000))
    run_full(p, 410)


@pytest.mark.parametrize("layout", ["N", "T"])
def test_diag_unaligned_rows_take_the_scalar_path(layout):
    """Odd leading dimensions (no aligned 8-element vectors) in x, C and D."""
    p = I.DiagProblem("diag_odd", "f16", "right", layout, 77, 70, beta=1.0, c="f32", pad_x=1,
                      pad_c=1, pad_d=1)
    run_full(p, 420)


def test_diag_unaligned_diagonal_pointer():
    """The diagonal starting one element past a 16-byte boundary."""
    p = I.DiagProblem("diag_off", "f16", "right", "T", 64, 96, beta=0.5, c="f32")
    dinp = I.generate_diag(p, 430)
    dd = H.DeviceDiag(dinp)
    buf = torch.zeros(p.N + 1, dtype=torch.float16, device="cuda")
    buf[1:] = dd.diag
    dd.diag = buf[1:]
    plan = H.make_diag_plan(p)
    dd.run(plan)
    torch.cuda.synchronize()
    H.check_close(dd.result(), H.oracle_full(H.dense_inputs_of(dinp)), p.d, p.name)
    plan.close()


def test_diag_tiny_shapes():
    for M, N in ((1, 1), (1, 9), (5, 3), (65, 1)):
        for side in ("left", "right"):
            run_full(I.DiagProblem("diag_tiny", "bf16", side, "N", M, N, beta=1.0, c="bf16",
                                   d="bf16"), 440 + M + N)


def test_diag_in_place_c_equals_d():
    p = I.DiagProblem("diag_inplace", "f16", "left", "T", 150, 100, alpha=2.0, beta=-1.0, c="f32",
                      d="f32")
    dinp = I.generate_diag(p, 450)
    ref = H.oracle_full(H.dense_inputs_of(dinp))
    dd = H.DeviceDiag(dinp)
    CD = dd.C.clone()
    plan = H.make_diag_plan(p)
    dd.run(plan, C=CD, D=CD)
    torch.cuda.synchronize()
    H.check_close(CD, ref, "f32", "in place")
    plan.close()


def test_diag_persistent_grid_at_the_full_size():
    """4096 x 4096 fp16 with fp32 C, D = diag(d) * B + C (both layouts of B):
    more tiles than resident CTAs, so every CTA walks several tiles.  Sampled
    entries (with tile edges) against the oracle."""
    for layout in ("N", "T"):
        p = I.diag_fp16_4096(layout)
        dinp = I.generate_diag(p, I.BASE_SEED + 20)
        dd = H.DeviceDiag(dinp)
        plan = H.make_diag_plan(p)
        dd.run(plan)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        cfg = plan.last_config()
        assert cfg["kernel"] == G.GEMM_KERNEL_DIAG and cfg["tiles"] == 64 * 64 and cfg["grid"] < 64 * 64
        dd.check_guards()
        rows, cols = H.sample_entries(p.M, p.N, 4000, 21, 64, 64)
        ref = H.oracle_entries(H.dense_inputs_of(dinp), rows, cols)
        got = dd.result()[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
        H.check_close(got, ref, p.d, p.name)
        plan.close()


def test_diag_argument_errors():
    plan = G.Plan(G.GEMM_F16, G.GEMM_F32, torch.cuda.current_device())
    X = torch.zeros(64 * 64, dtype=torch.float16, device="cuda")
    D = torch.zeros(64 * 64, dtype=torch.float32, device="cuda")
    ok = (plan.handle, G.GEMM_SIDE_LEFT, G.GEMM_OP_N, 64, 64, 1.0, X.data_ptr(), X.data_ptr(), 64, 0.0,
          None, 0, D.data_ptr(), 64)
    G.gemm_run_diag(*ok)
    torch.cuda.synchronize()
    for i, bad, status in ((1, 2, G.GEMM_ERR_INVALID_ARG),          # side
                           (8, 63, G.GEMM_ERR_INVALID_ARG),         # ldx < M, column-major x
                           (6, None, G.GEMM_ERR_INVALID_ARG),       # no diagonal
                           (9, 1.0, G.GEMM_ERR_INVALID_ARG)):       # beta != 0 without C
        args = list(ok)
        args[i] = bad
        with pytest.raises(G.GemmError) as e:
            G.gemm_run_diag(*args)
        assert e.value.status == status
    args = list(ok)
    args[3] = 0
    G.gemm_run_diag(*args)                                         # M == 0: nothing launched
    assert plan.last_config()["kernel"] == G.GEMM_KERNEL_NONE
    plan.close()
    p8 = G.Plan(G.GEMM_S8, G.GEMM_S32, torch.cuda.current_device())
    with pytest.raises(G.GemmError) as e:
        G.gemm_run_diag(p8.handle, G.GEMM_SIDE_RIGHT, G.GEMM_OP_T, 64, 64, 0.5, X.data_ptr(),
                        X.data_ptr(), 64, 0.0, None, 0, D.data_ptr(), 64,
                        G.make_epilogue(G.GEMM_S32))
    assert e.value.status == G.GEMM_ERR_UNSUPPORTED
    p8.close()


def test_diag_tma_kernel_bounded_wait_reports_timeout():
    """A wait bound far below the kernel's run time makes the TMA-staged kernel's
    waits expire: it records GEMM_ERR_TIMEOUT, its producer drains the copies in
    flight, and the same context then runs the problem correctly."""
    p = I.DiagProblem("diag_tmo", "f16", "left", "T", 4096, 4096, beta=0.5, c="f32")
    dinp = I.generate_diag(p, 450)
    dd = H.DeviceDiag(dinp)
    plan = H.make_diag_plan(p)
    G.gemm_plan_set_timeout(plan.handle, 200)       # 200 ns
    dd.run(plan)
    torch.cuda.synchronize()
    assert plan.last_config()["stages"] == 6
    assert plan.device_status() == G.GEMM_ERR_TIMEOUT
    G.gemm_plan_set_timeout(plan.handle, 4_000_000_000)
    dd.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    rows, cols = H.sample_entries(p.M, p.N, 2000, 451, 64, 64)
    got = dd.result()[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
    H.check_close(got, H.oracle_entries(H.dense_inputs_of(dinp), rows, cols), p.d, "after timeout")
    plan.close()
