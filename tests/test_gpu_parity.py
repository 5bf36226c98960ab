"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Small and ragged problems are compared element by element on the full output;
every kernel (tensor-core fp16/bf16, exact int8, FFMA SGEMM, generic CUDA-core)
and every layout, epilogue and output type is covered, plus guard bands around
D, in-place C == D, empty and K == 0 problems, host-buffer entry and the
bounded-wait status.
"""
import numpy as np
import pytest
import torch

import dense_gemm_epilogues_gb300 as G
from dense_gemm_epilogues_gb300 import inputs as I

import parity_helpers as H

pytestmark = pytest.mark.gpu

LAYOUTS = ["NN", "NT", "TN", "TT"]
TC_KERNELS = [G.GEMM_KERNEL_TC, G.GEMM_KERNEL_TC_PAIR]
TC_IDS = ["cta1", "pair"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.load_library()
    yield
    torch.cuda.synchronize()


# ------------------------------- tensor cores --------------------------------

@pytest.mark.parametrize("kernel", TC_KERNELS, ids=TC_IDS)
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("ab", ["f16", "bf16"])
def test_tc_ragged_alpha_beta(layout, ab, kernel):
    """Several tiles with ragged M, N, K tails; alpha/beta with fp32 C; both
    tensor-core kernels (one CTA per tile, CTA pairs)."""
    p = H.tma_aligned(I.Problem("tc_ab", ab, layout[0], layout[1], 300, 520, 200, alpha=1.5,
                                  beta=0.5, c="f32"))
    H.run_and_check_full(p, 101, kernel=kernel, expect_kernel=kernel)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_selector_picks_pair_kernel_when_it_is_faster(layout):
    """72 pair tiles (one wave) and K = 7680: the pairs' better per-wave rate
    outweighs their higher fixed cost, so the selector runs pairs.  Sampled
    outputs (with tile edges) against the oracle."""
    p = H.tma_aligned(I.Problem("tc_auto", "f16", layout[0], layout[1], 2048, 2304, 7680, beta=0.5,
                                c="f32"))
    inp = I.generate(p, 120)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0 and plan.last_config()["kernel"] == G.GEMM_KERNEL_TC_PAIR
    dp.check_guards()
    rows, cols = H.sample_entries(p.M, p.N, 800, 120, 256, 256)
    got = dp.result()[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
    H.check_close(got, H.oracle_entries(inp, rows, cols), p.d, p.name)
    plan.close()


@pytest.mark.parametrize("layout", LAYOUTS)
def test_selector_picks_single_cta_below_a_wave_of_pairs(layout):
    """6 pair tiles would leave most SMs idle: the single-CTA kernel's finer grid runs."""
    p = H.tma_aligned(I.Problem("tc_small", "f16", layout[0], layout[1], 520, 300, 136))
    H.run_and_check_full(p, 121, expect_kernel=G.GEMM_KERNEL_TC)


@pytest.mark.parametrize("kernel", TC_KERNELS, ids=TC_IDS)
@pytest.mark.parametrize("layout", LAYOUTS)
def test_tc_bias_relu_bf16_out(layout, kernel):
    p = H.tma_aligned(I.Problem("tc_fc", "bf16", layout[0], layout[1], 257, 384, 320, d="bf16",
                                bias="f32", bias_mode="col", act="relu",
                                dist_a=I.Dist("normal", std=1.0), dist_b=I.Dist("normal", std=0.05)))
    H.run_and_check_full(p, 102, kernel=kernel, expect_kernel=kernel)


@pytest.mark.parametrize("kernel", TC_KERNELS, ids=TC_IDS)
@pytest.mark.parametrize("n", [64, 96, 128, 129, 200])
def test_tc_narrow_n_tiles(n, kernel):
    """N <= 128 selects 128-wide single-CTA tiles; forcing the pair kernel there
    leaves the second CTA's half of B entirely out of bounds (zero-filled)."""
    p = H.tma_aligned(I.Problem("tc_n", "f16", "T", "N", 256, n, 192))
    H.run_and_check_full(p, 103, kernel=kernel, expect_kernel=kernel)


@pytest.mark.parametrize("kernel", TC_KERNELS, ids=TC_IDS)
@pytest.mark.parametrize("c,d", [("f16", "f16"), ("bf16", "f32"), ("f32", "bf16"), ("f32", "f16")])
def test_tc_c_and_d_types(c, d, kernel):
    ab = "bf16" if "bf16" in (c, d) else "f16"
    p = H.tma_aligned(I.Problem("tc_cd", ab, "N", "T", 200, 300, 136, alpha=-0.75, beta=1.25, c=c,
                                d=d, bias="bf16" if ab == "bf16" else "f16", bias_mode="row",
                                act="relu"))
    H.run_and_check_full(p, 104, kernel=kernel, expect_kernel=kernel)


@pytest.mark.parametrize("kernel", TC_KERNELS, ids=TC_IDS)
@pytest.mark.parametrize("layout", LAYOUTS)
def test_tc_padded_leading_dims(layout, kernel):
    """Leading dimensions larger than the logical extent (poisoned padding, 16-byte
    multiples) and a padded, unaligned-width D."""
    p = H.tma_aligned(I.Problem("tc_pad", "f16", layout[0], layout[1], 190, 270, 150, beta=1.0,
                                c="f32", pad_a=8, pad_b=16, pad_c=3, pad_d=5))
    H.run_and_check_full(p, 105, kernel=kernel, expect_kernel=kernel)


@pytest.mark.parametrize("kernel", TC_KERNELS, ids=TC_IDS)
@pytest.mark.parametrize("layout", LAYOUTS)
def test_tc_small_integers_bit_exact(layout, kernel):
    """Small-integer data is exact in every step, so the tensor-core result must
    equal the oracle bit for bit (fp32 out)."""
    p = H.tma_aligned(I.Problem("tc_exact", "f16", layout[0], layout[1], 260, 300, 520, alpha=2.0,
                                beta=-1.0, c="f32", dist_a=I.Dist("small", -3, 3),
                                dist_b=I.Dist("small", -3, 3), dist_c=I.Dist("small", -100, 100),
                                bias="f32", bias_mode="col", dist_bias=I.Dist("small", -50, 50),
                                act="relu"))
    inp = I.generate(p, 106)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p, kernel)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert plan.last_config()["kernel"] == kernel
    np.testing.assert_array_equal(dp.result().cpu().numpy(), H.oracle_full(inp))
    dp.check_guards()


@pytest.mark.parametrize("kernel", TC_KERNELS, ids=TC_IDS)
def test_tc_in_place_c_equals_d(kernel):
    p = I.Problem("inplace", "f16", "T", "N", 150, 260, 96, alpha=1.0, beta=2.0, c="f32")
    inp = I.generate(p, 107)
    ref = H.oracle_full(inp)
    plan = H.make_plan(p, kernel)
    A, B = inp.A.cuda(), inp.B.cuda()
    CD = inp.C.cuda()
    G.gemm_run(plan.handle, G.GEMM_OP_T, G.GEMM_OP_N, p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda,
               B.data_ptr(), p.ldb, p.beta, CD.data_ptr(), p.ldc, CD.data_ptr(), p.ldc,
               G.make_epilogue(G.GEMM_F32), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    H.check_close(CD, ref, "f32", "in-place")


@pytest.mark.parametrize("kernel", TC_KERNELS, ids=TC_IDS)
def test_tc_many_tiles_persistent_loop(kernel):
    """More tiles than CTAs (pairs): each walks several tiles (both accumulator buffers)."""
    p = I.Problem("tc_many", "f16", "T", "N", 3072, 2560, 64, beta=0.5, c="f32")
    cfg = H.run_and_check_full(p, 108, kernel=kernel, expect_kernel=kernel)
    assert cfg["tiles"] > cfg["grid"] // cfg["cta_group"]


# ---------------------------------- int8 -------------------------------------

@pytest.fixture(params=[1, 2], ids=["cta1", "pair"])
def cta_group(request, monkeypatch):
    """Run the exact int8 path on single-CTA tiles (GEMM_TC_CTA_GROUP=1) or on
    CTA pairs (GEMM_TC_CTA_GROUP=2; the selector's choice for grids of a wave or more)."""
    monkeypatch.setenv("GEMM_TC_CTA_GROUP", str(request.param))
    return request.param


@pytest.mark.parametrize("layout", LAYOUTS)
def test_int8_exact_ragged(layout, cta_group):
    """K = 1100 spans a full exact 1024-chunk and a tail; bit-exact int32."""
    p = H.tma_aligned(I.Problem("i8", "s8", layout[0], layout[1], 260, 390, 1100, d="s32",
                                dist_a=I.I8, dist_b=I.I8))
    cfg = H.run_and_check_full(p, 109, expect_kernel=G.GEMM_KERNEL_TC_INT8)
    assert cfg["cta_group"] == cta_group


def test_int8_adversarial_extremes_exact(cta_group):
    """All -128: every partial sum is 16384*k, far beyond fp32's exact range at
    K = 4096 (2^26), so a single fp32 accumulator would be wrong; each 1024-deep
    chunk reaches exactly 2^24, the largest sum the chunking allows."""
    p = I.Problem("i8max", "s8", "T", "N", 130, 140, 4096, d="s32",
                  dist_a=I.Dist("int", -128, -128), dist_b=I.Dist("int", -128, -128))
    cfg = H.run_and_check_full(p, 110, expect_kernel=G.GEMM_KERNEL_TC_INT8)
    assert cfg["cta_group"] == cta_group


def test_int8_many_tiles_and_chunks(cta_group):
    """More tiles than CTA pairs and several exact chunks per tile."""
    p = I.Problem("i8many", "s8", "T", "N", 2304, 2560, 1600, d="s32", dist_a=I.I8, dist_b=I.I8)
    cfg = H.run_and_check_full(p, 121, expect_kernel=G.GEMM_KERNEL_TC_INT8)
    assert cfg["cta_group"] == cta_group and cfg["tiles"] > cfg["grid"] // cfg["cta_group"]


def test_int8_alpha_beta_bias_relu(cta_group):
    p = H.tma_aligned(I.Problem("i8epi", "s8", "N", "T", 200, 136, 700, alpha=3.0, beta=-2.0,
                                c="s32", d="s32", bias="s32", bias_mode="col", act="relu",
                                dist_a=I.I8, dist_b=I.I8, dist_c=I.Dist("int", -100000, 100000),
                                dist_bias=I.Dist("int", -5000, 5000)))
    H.run_and_check_full(p, 111, expect_kernel=G.GEMM_KERNEL_TC_INT8)


# ---------------------------------- FFMA -------------------------------------

@pytest.mark.parametrize("layout", LAYOUTS)
def test_ffma_sgemm_bias_relu(layout):
    p = I.Problem("sg", "f32", layout[0], layout[1], 300, 260, 100, alpha=1.0, beta=0.5, c="f32",
                  bias="f32", bias_mode="col", act="relu")
    H.run_and_check_full(p, 112, expect_kernel=G.GEMM_KERNEL_FFMA)


def test_ffma_ragged_k_and_padding():
    p = I.Problem("sg2", "f32", "T", "N", 129, 131, 37, pad_a=3, pad_b=1, d="bf16")
    # lda = 40, ldb = 38: ldb is not a multiple of 4 -> generic path; force FFMA fails
    inp = I.generate(p, 113)
    plan = H.make_plan(p, G.GEMM_KERNEL_FFMA)
    dp = H.DeviceProblem(inp)
    with pytest.raises(G.GemmError) as e:
        dp.run(plan)
    assert e.value.status == G.GEMM_ERR_ALIGNMENT
    p2 = p.with_(pad_b=3)   # ldb = 40
    H.run_and_check_full(p2, 113, expect_kernel=G.GEMM_KERNEL_FFMA)


# ------------------------------ generic kernel -------------------------------

@pytest.mark.parametrize("ab", ["f16", "bf16", "s8", "f32"])
def test_generic_kernel_unaligned(ab):
    """Odd leading dimensions that TMA cannot describe run on the generic kernel."""
    d = "s32" if ab == "s8" else "f32"
    kw = dict(dist_a=I.I8, dist_b=I.I8) if ab == "s8" else {}
    p = I.Problem("gen", ab, "T", "N", 45, 37, 29, d=d, pad_a=1, pad_b=2, **kw)
    H.run_and_check_full(p, 114, expect_kernel=G.GEMM_KERNEL_SIMT)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_forced_generic_matches(layout):
    p = I.Problem("gen2", "bf16", layout[0], layout[1], 70, 90, 33, alpha=0.5, beta=-1.0,
                  c="bf16", d="f16", bias="f32", bias_mode="row", act="relu")
    H.run_and_check_full(p, 115, kernel=G.GEMM_KERNEL_SIMT, expect_kernel=G.GEMM_KERNEL_SIMT)


def test_k_zero_is_epilogue_of_beta_c():
    p = I.Problem("k0", "f16", "T", "N", 33, 47, 0, alpha=3.0, beta=0.5, c="f32", bias="f32",
                  bias_mode="col", act="relu")
    H.run_and_check_full(p, 116, expect_kernel=G.GEMM_KERNEL_SIMT)


def test_empty_problems_are_noops():
    for M, N in ((0, 16), (16, 0)):
        p = I.Problem("empty", "f16", "T", "N", M, N, 8)
        inp = I.generate(p, 117)
        dp = H.DeviceProblem(inp)
        plan = H.make_plan(p)
        dp.run(plan)
        torch.cuda.synchronize()
        assert plan.last_config()["kernel"] == G.GEMM_KERNEL_NONE
        dp.check_guards()


# ------------------------------ host entry point -----------------------------

def test_run_host_buffers():
    p = I.Problem("host", "bf16", "T", "T", 300, 280, 96, beta=0.25, c="f32", d="bf16",
                  bias="f32", bias_mode="col", act="relu", pad_d=5)
    inp = I.generate(p, 118)
    ref = H.oracle_full(inp)
    plan = H.make_plan(p)
    A = inp.A.pin_memory()
    B = inp.B.pin_memory()
    C = inp.C.pin_memory()
    bias = inp.bias.pin_memory()
    D = torch.full((p.M, p.ldd), 7.0, dtype=torch.bfloat16).pin_memory()
    epi = G.make_epilogue(G.GEMM_BF16, bias.data_ptr(), G.GEMM_F32, G.GEMM_BIAS_COL, G.GEMM_ACT_RELU)
    G.gemm_run_host(plan.handle, G.GEMM_OP_T, G.GEMM_OP_T, p.M, p.N, p.K, p.alpha, A.data_ptr(),
                    p.lda, B.data_ptr(), p.ldb, p.beta, C.data_ptr(), p.ldc, D.data_ptr(), p.ldd,
                    epi, torch.cuda.current_stream().cuda_stream)
    H.check_close(D[:, :p.N], ref, "bf16", "host entry")
    assert torch.all(D[:, p.N:] == 7.0), "the host entry wrote into the padding of D"


# ------------------------------- bounded waits -------------------------------

def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait bound far below a tile's run time makes the tensor-core kernel's
    waits expire: the kernel records GEMM_ERR_TIMEOUT, winds down and returns;
    the same context then runs the problem correctly."""
    p = I.Problem("tmo", "f16", "T", "N", 512, 512, 4096)
    inp = I.generate(p, 119)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p)
    G.gemm_plan_set_timeout(plan.handle, 200)       # 200 ns
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == G.GEMM_ERR_TIMEOUT
    G.gemm_plan_set_timeout(plan.handle, 4_000_000_000)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    H.check_close(dp.result(), H.oracle_full(inp), "f32", "after timeout")


# ------------------------------ stream-K tail --------------------------------

SK_SHAPES = [(1536, 1536, 2048), (2560, 2560, 512), (1000, 1800, 2000), (2304, 4352, 640)]


@pytest.mark.parametrize("stream_k", ["on", "off"])
@pytest.mark.parametrize("shape", SK_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_pair_stream_k_tail(shape, stream_k, monkeypatch):
    """Tiles of the last wave split over all CTA pairs by K blocks (up to four
    segments per tile here); the owning pair adds the published partials before
    the full epilogue (alpha, beta*C, bias, ReLU, bf16 cast)."""
    monkeypatch.setenv("GEMM_STREAM_K", "1" if stream_k == "on" else "0")
    monkeypatch.setenv("GEMM_TC_CTA_GROUP", "2")
    M, N, K = shape
    p = H.tma_aligned(I.Problem("sk", "bf16", "T", "N", M, N, K, alpha=0.75, beta=-0.5, c="f32",
                                d="bf16", bias="f32", bias_mode="col", act="relu"))
    cfg = H.run_and_check_full(p, 130, expect_kernel=G.GEMM_KERNEL_TC_PAIR)
    assert (cfg["sk_tiles"] > 0) == (stream_k == "on"), cfg


@pytest.mark.parametrize("layout", LAYOUTS)
def test_pair_stream_k_repeated_launches(layout, monkeypatch):
    """Several launches on one plan reuse the partial slots and flags (each
    launch publishes a new epoch); every result must still be right."""
    monkeypatch.setenv("GEMM_STREAM_K", "1")
    p = H.tma_aligned(I.Problem("sk_rep", "f16", layout[0], layout[1], 1280, 1536, 1536,
                                alpha=1.25, beta=1.0, c="f32"))
    inp = I.generate(p, 131)
    ref = H.oracle_full(inp)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p)
    for _ in range(3):
        dp.D.fill_(0)
        dp.run(plan)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        cfg = plan.last_config()
        assert cfg["kernel"] == G.GEMM_KERNEL_TC_PAIR and cfg["sk_tiles"] > 0
        H.check_close(dp.result(), ref, "f32", "stream-K repeat")
    dp.check_guards()


def test_pair_stream_k_off_inside_cuda_graphs(monkeypatch):
    """The pair kernel's stream-K uses a per-launch epoch chosen on the host, which
    a graph would replay unchanged: a captured launch runs without stream-K, and
    every replay is right."""
    monkeypatch.setenv("GEMM_STREAM_K", "1")
    p = H.tma_aligned(I.Problem("sk_graph", "f16", "T", "N", 1280, 1536, 1536, alpha=1.25, beta=1.0, c="f32"))
    inp = I.generate(p, 132)
    ref = H.oracle_full(inp)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.last_config()["sk_tiles"] > 0
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            dp.run(plan, stream=s.cuda_stream)
    torch.cuda.synchronize()
    assert plan.last_config()["sk_tiles"] == 0
    for _ in range(3):
        dp.D.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        H.check_close(dp.result(), ref, "f32", "stream-K under graph replay")
    dp.check_guards()
    plan.close()


# ------------------------- transform of C as it is read ----------------------

@pytest.mark.parametrize("kernel,ab", [(G.GEMM_KERNEL_TC_PAIR, "f16"), (G.GEMM_KERNEL_TC, "bf16"),
                                       (G.GEMM_KERNEL_TC_INT8, "s8"), (G.GEMM_KERNEL_FFMA, "f32"),
                                       (G.GEMM_KERNEL_SIMT, "f16")],
                         ids=["pair", "cta1", "int8", "ffma", "simt"])
def test_bias_relu_on_c_and_d(kernel, ab):
    """The last row of the paper's fusion table: bias, ReLU on C (as it is read)
    and ReLU on D, in one kernel."""
    is_int = ab == "s8"
    cd = "s32" if is_int else "f32"
    kw = dict(dist_a=I.I8, dist_b=I.I8, dist_c=I.Dist("int", -200000, 200000),
              dist_bias=I.Dist("int", -3000, 3000)) if is_int else {}
    beta = 2.0 if is_int else 1.5      # the int8 path takes integral alpha and beta
    p = H.tma_aligned(I.Problem("relu_c", ab, "T", "N", 300, 264, 320, alpha=1.0, beta=beta, c=cd,
                                d=cd, bias=cd, bias_mode="col", act="relu", c_act="relu", **kw))
    H.run_and_check_full(p, 140, kernel=kernel, expect_kernel=kernel)
