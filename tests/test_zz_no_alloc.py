"""The allocation-free int8 entry point, gemm_run_s8_noalloc.

Some callers cannot allocate device memory when they call the GEMM: their
device memory was reserved up front by a framework's memory pool, or their loop
cannot afford cudaMalloc/cudaFree and the synchronisation those imply.
gemm_run_s8_noalloc serves them from a fixed staging array that the library
holds on each device.  These tests call it through the C ABI and check its
output against the plan-based entry point (gemm_run) and against the oracle on
the same inputs -- bit for bit, the tolerance every int8 test here uses -- on
two calls in a row (the second call reuses the array the first one left
filled, with other shapes and layouts); check that a problem too large for the
array is refused before anything is launched; and check that an in-kernel wait
that runs out is reported through the library's own error word
(gemm_noalloc_device_status), after which the same context computes the next
call correctly.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test.  It needs no state from them.
"""
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


def _noalloc_run(dp: H.DeviceProblem, status_ptr=None):
    p = dp.p
    G.gemm_run_s8_noalloc(G.LAYOUT_CODES[p.layout_a], G.LAYOUT_CODES[p.layout_b], p.M, p.N, p.K,
                          p.alpha, dp.A.data_ptr(), p.lda, dp.B.data_ptr(), p.ldb, p.beta,
                          dp.C.data_ptr() if dp.C is not None else None, p.ldc if p.c else 0,
                          dp.D.data_ptr(), p.ldd, dp.epilogue(), status_ptr,
                          torch.cuda.current_stream().cuda_stream)


PROBLEMS = [
    H.tma_aligned(I.Problem("noalloc_1", "s8", "T", "N", 1000, 776, 1544, d="s32",
                            dist_a=I.I8, dist_b=I.I8)),
    H.tma_aligned(I.Problem("noalloc_2", "s8", "N", "T", 520, 1032, 2056, alpha=2.0, beta=-3.0,
                            c="s32", d="s32", bias="s32", bias_mode="col", act="relu",
                            dist_a=I.I8, dist_b=I.I8, dist_c=I.Dist("int", -1000, 1000),
                            dist_bias=I.Dist("int", -500, 500))),
]


def test_noalloc_matches_gemm_run_and_oracle_on_two_calls_in_a_row():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert G.gemm_noalloc_device_status() == 0      # also clears what an earlier test left
    for call, p in enumerate(PROBLEMS):
        inp = I.generate(p, 300 + call)
        ref = H.DeviceProblem(inp)
        plan = H.make_plan(p)
        ref.run(plan)                                  # the existing entry point
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        assert plan.last_config()["kernel"] == G.GEMM_KERNEL_TC_INT8
        plan.close()

        got = H.DeviceProblem(inp)
        _noalloc_run(got, status.data_ptr() if call == 1 else None)
        torch.cuda.synchronize()
        got.check_guards()
        H.check_close(got.result(), ref.result().cpu().numpy(), "s32", f"no-alloc call {call + 1}")
        H.check_close(got.result(), H.oracle_full(inp), "s32", f"no-alloc call {call + 1} vs oracle")
    assert int(status.item()) == 0
    assert G.gemm_noalloc_device_status() == 0


def test_noalloc_refuses_problems_beyond_its_scratch():
    p = I.Problem("noalloc_big", "s8", "T", "N", 4096, 4096, 4096, d="s32")
    need = 2 * (p.M * p.K + p.N * p.K)
    assert need > G.NOALLOC_SCRATCH_BYTES
    D = torch.empty((p.M, p.N), dtype=torch.int32, device="cuda")
    A = torch.zeros((p.M, p.K), dtype=torch.int8, device="cuda")
    B = torch.zeros((p.N, p.K), dtype=torch.int8, device="cuda")
    with pytest.raises(G.GemmError) as e:
        G.gemm_run_s8_noalloc(G.GEMM_OP_T, G.GEMM_OP_N, p.M, p.N, p.K, 1.0, A.data_ptr(), p.K,
                              B.data_ptr(), p.K, 0.0, None, 0, D.data_ptr(), p.N,
                              G.make_epilogue(G.GEMM_S32), None,
                              torch.cuda.current_stream().cuda_stream)
    assert e.value.status == G.GEMM_ERR_UNSUPPORTED


def test_noalloc_expired_wait_is_reported_and_context_survives():
    """A wait bound far below a tile's run time makes the kernel's bounded waits
    expire: the kernel records GEMM_ERR_TIMEOUT in the library's word and winds
    down; gemm_noalloc_device_status reports it once, and with the default bound
    restored the next call is exact again."""
    p = PROBLEMS[0]
    inp = I.generate(p, 310)
    dp = H.DeviceProblem(inp)
    assert G.gemm_noalloc_device_status() == 0
    try:
        G.gemm_noalloc_set_timeout(200)              # 200 ns
        _noalloc_run(dp)
        torch.cuda.synchronize()
    finally:
        G.gemm_noalloc_set_timeout(4_000_000_000)
    assert G.gemm_noalloc_device_status() == G.GEMM_ERR_TIMEOUT
    assert G.gemm_noalloc_device_status() == 0       # read once, then cleared
    _noalloc_run(dp)
    torch.cuda.synchronize()
    assert G.gemm_noalloc_device_status() == 0
    dp.check_guards()
    H.check_close(dp.result(), H.oracle_full(inp), "s32", "no-alloc after an expired wait")


def test_noalloc_operand_transforms():
    """The operand transform of int8 problems (ReLU on A and/or B) applies here as
    for gemm_run: in the staging pass, exact."""
    p = PROBLEMS[0].with_(name="noalloc_relu", a_act="relu", b_act="relu")
    inp = I.generate(p, 320)
    dp = H.DeviceProblem(inp)
    assert G.gemm_noalloc_device_status() == 0
    _noalloc_run(dp)
    torch.cuda.synchronize()
    assert G.gemm_noalloc_device_status() == 0
    dp.check_guards()
    H.check_close(dp.result(), H.oracle_full(inp), "s32", "no-alloc with ReLU on A and B")
