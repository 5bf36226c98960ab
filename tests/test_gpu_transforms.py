"""GPU parity of the operand transforms after load: every element of A (of B)
enters the product as t(x) = act(scale * x), the product in fp32, then ReLU,
then (16-bit operands) rounded back to the operand's type -- the transforms
that "Flexible Performant GEMM Kernels on GPUs" applies after each load and
before the multiply-accumulate (section 4.2, "Transforms", Figure 10).

Each kernel runs them its own way (the tensor-core kernels either on the
staged shared-memory tiles, with extra transform warps, or through a transform
pass over the operand into scratch before the GEMM -- both forced in turn with
GEMM_XF_STAGE; the CUDA-core kernels as the elements are loaded; int8 problems
in the fp16 staging pass), so each is compared with the oracle, element by
element, on ragged multi-tile problems in every layout, and bit for bit on
small-integer data where every step is exact.
"""
import numpy as np
import pytest
import torch

import dense_gemm_epilogues_gb300 as G
from dense_gemm_epilogues_gb300 import inputs as I

import parity_helpers as H

pytestmark = pytest.mark.gpu

LAYOUTS = ["NN", "NT", "TN", "TT"]
# (a_act, a_scale, b_act, b_scale): A alone, B alone, both (a negative scale
# under ReLU keeps only the negative elements); "odd": scales that fp16 cannot
# hold exactly (fp16 operands then take the fp32 product path in the kernels).
WHICH = {
    "A": ("relu", 1.75, "none", 1.0),
    "B": ("none", 1.0, "relu", -0.625),
    "AB": ("relu", -1.5, "relu", 0.75),
    "odd": ("none", 0.1, "relu", 1.0 / 3.0),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.load_library()
    yield
    torch.cuda.synchronize()


@pytest.fixture
def clean_env(monkeypatch):
    for v in ("GEMM_TC_CTA_GROUP", "GEMM_TC_BN", "GEMM_TC_SPLITK", "GEMM_STREAM_K", "GEMM_TC_TAIL_HALVES",
              "GEMM_XF_STAGE"):
        monkeypatch.delenv(v, raising=False)
    return monkeypatch


@pytest.fixture(params=["in_kernel", "staged"])
def xf_path(request, clean_env):
    """Where the tensor-core path applies the transforms: on the staged tiles
    inside the GEMM kernel, or in a staging pass before it."""
    clean_env.setenv("GEMM_XF_STAGE", "1" if request.param == "staged" else "0")
    return request.param


def _check_path(cfg: dict, p: I.Problem, path: str):
    want = 0
    if path == "staged":
        want = ((G.GEMM_XF_A if (p.a_act != "none" or p.a_scale != 1.0) else 0) |
                (G.GEMM_XF_B if (p.b_act != "none" or p.b_scale != 1.0) else 0))
    assert cfg["xf_staged"] == want, cfg


def _xf(p: I.Problem, which: str) -> I.Problem:
    a_act, a_scale, b_act, b_scale = WHICH[which]
    return p.with_(a_act=a_act, a_scale=a_scale, b_act=b_act, b_scale=b_scale)


# ------------------------------- tensor cores --------------------------------

@pytest.mark.parametrize("which", list(WHICH))
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("ab", ["f16", "bf16"])
def test_pair_kernel_transforms(layout, ab, which, clean_env, xf_path):
    """CTA pairs: 2 x 3 tiles with ragged M and N, K = 264 (five K blocks: the
    last stage holds one, the last block 8 deep), alpha/beta with fp32 C."""
    clean_env.setenv("GEMM_TC_TAIL_HALVES", "0")
    p = H.tma_aligned(_xf(I.Problem("xf_pair", ab, layout[0], layout[1], 300, 520, 264, alpha=1.25, beta=0.5,
                                    c="f32"), which))
    cfg = H.run_and_check_full(p, 301, kernel=G.GEMM_KERNEL_TC_PAIR, expect_kernel=G.GEMM_KERNEL_TC_PAIR)
    _check_path(cfg, p, xf_path)


@pytest.mark.parametrize("which", list(WHICH))
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("bn", [64, 128, 256])
def test_single_cta_kernel_transforms(layout, bn, which, clean_env, xf_path):
    """One CTA per tile, every tile width (their stages hold one or two K
    blocks; K = 392 is seven blocks, the last stage of two-block tiles holds
    one), ragged edges, bias + ReLU and a bf16 output."""
    clean_env.setenv("GEMM_TC_BN", str(bn))
    p = H.tma_aligned(_xf(I.Problem("xf_cta1", "bf16", layout[0], layout[1], 270, 330, 392, d="bf16",
                                    bias="f32", bias_mode="col", act="relu"), which))
    cfg = H.run_and_check_full(p, 302, kernel=G.GEMM_KERNEL_TC, expect_kernel=G.GEMM_KERNEL_TC)
    assert cfg["bn"] == bn and cfg["sk_tiles"] == 0
    _check_path(cfg, p, xf_path)


@pytest.mark.parametrize("kernel", [G.GEMM_KERNEL_TC, G.GEMM_KERNEL_TC_PAIR], ids=["cta1", "pair"])
@pytest.mark.parametrize("layout", LAYOUTS)
def test_tensor_core_transforms_bit_exact_on_small_integers(layout, kernel, clean_env, xf_path):
    """Small integers, power-of-two scales and ReLU: every transformed value,
    product and sum is exact, so D must equal the oracle bit for bit."""
    p = H.tma_aligned(I.Problem("xf_exact", "f16", layout[0], layout[1], 260, 300, 392, alpha=2.0, beta=-1.0,
                                c="f32", dist_a=I.Dist("small", -3, 3), dist_b=I.Dist("small", -3, 3),
                                dist_c=I.Dist("small", -100, 100), a_act="relu", a_scale=4.0,
                                b_act="relu", b_scale=-0.5))
    inp = I.generate(p, 303)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p, kernel)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0 and plan.last_config()["kernel"] == kernel
    _check_path(plan.last_config(), p, xf_path)
    np.testing.assert_array_equal(dp.result().cpu().numpy(), H.oracle_full(inp))
    dp.check_guards()
    plan.close()


@pytest.mark.parametrize("layout", LAYOUTS)
def test_pair_tail_halves_with_transforms(layout, clean_env, xf_path):
    """A pair tail split into 256 x 128 halves (K-major B: 64-row boxes at the
    start of each slab; MN-major B: one 64-wide box), ragged N, transforms on
    both operands."""
    clean_env.setenv("GEMM_TC_CTA_GROUP", "2")
    p = H.tma_aligned(_xf(I.Problem("xf_halves", "f16", layout[0], layout[1], 600, 1100, 200, alpha=0.75,
                                    beta=-0.5, c="f32", d="f16"), "AB"))
    cfg = H.run_and_check_full(p, 304, expect_kernel=G.GEMM_KERNEL_TC_PAIR)
    assert cfg["half_tiles"] == 3 * 5, cfg
    _check_path(cfg, p, xf_path)


@pytest.mark.parametrize("ab", ["f16", "bf16"])
def test_identity_transform_gives_the_same_bits(ab, clean_env):
    """load_xf set with act none and scale 1 is the identity: the result equals
    the untransformed run bit for bit."""
    p = H.tma_aligned(I.Problem("xf_ident", ab, "T", "N", 384, 640, 512, alpha=1.5, beta=0.5, c="f32"))
    inp = I.generate(p, 305)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p)
    stream = torch.cuda.current_stream().cuda_stream
    args = (plan.handle, G.GEMM_OP_T, G.GEMM_OP_N, p.M, p.N, p.K, p.alpha, dp.A.data_ptr(), p.lda,
            dp.B.data_ptr(), p.ldb, p.beta, dp.C.data_ptr(), p.ldc, dp.D.data_ptr(), p.ldd)
    G.gemm_run(*args, H.epilogue_for(p), stream)
    plain = dp.result().clone()
    G.gemm_run(*args, H.epilogue_for(p, load_xf=G.GEMM_XF_A | G.GEMM_XF_B), stream)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert torch.equal(plain, dp.result())
    plan.close()


def test_transform_changes_result_only_through_the_operands(clean_env):
    """ReLU on A with every element of A negative gives t_A = 0: D is then
    beta*C + bias exactly (the MMA adds exact zeros)."""
    p = H.tma_aligned(I.Problem("xf_zero", "f16", "T", "N", 256, 512, 256, alpha=3.0, beta=0.5, c="f32",
                                bias="f32", bias_mode="col", dist_a=I.Dist("uniform", -2.0, -0.5),
                                a_act="relu"))
    inp = I.generate(p, 306)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    ref = H.oracle_full(inp)
    want = (0.5 * inp.C[:, :p.N].double() + inp.bias.double()[None, :]).float().numpy()
    np.testing.assert_array_equal(ref, want)            # the oracle's own reading
    np.testing.assert_array_equal(dp.result().cpu().numpy(), ref)
    plan.close()


# --------------------------- batched and host entry ---------------------------

@pytest.mark.parametrize("kernel", [G.GEMM_KERNEL_TC, G.GEMM_KERNEL_TC_PAIR], ids=["cta1", "pair"])
@pytest.mark.parametrize("share_b", [False, True], ids=["own_b", "shared_b"])
def test_batched_transforms(kernel, share_b, clean_env, xf_path):
    """Three problems in one call, each against the oracle on its own; a shared
    B (stride 0) is transformed once when staged."""
    from test_gpu_batched import run_batched
    p = H.tma_aligned(_xf(I.Problem("xf_bat", "f16", "N", "T", 300, 264, 200, alpha=1.25, beta=-0.5, c="f32",
                                    bias="f32", bias_mode="col", act="relu", pad_d=3), "AB"))
    cfg = run_batched(p, 3, 307, share_b=share_b, kernel=kernel)
    _check_path(cfg, p, xf_path)


def test_host_entry_transforms(clean_env, xf_path):
    p = I.Problem("xf_host", "bf16", "T", "T", 300, 280, 96, beta=0.25, c="f32", d="bf16", bias="f32",
                  bias_mode="col", act="relu", a_act="relu", a_scale=0.5, b_scale=2.0)
    inp = I.generate(p, 308)
    plan = H.make_plan(p)
    A, B, C, bias = (t.pin_memory() for t in (inp.A, inp.B, inp.C, inp.bias))
    D = torch.full((p.M, p.ldd), 7.0, dtype=torch.bfloat16).pin_memory()
    G.gemm_run_host(plan.handle, G.GEMM_OP_T, G.GEMM_OP_T, p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda,
                    B.data_ptr(), p.ldb, p.beta, C.data_ptr(), p.ldc, D.data_ptr(), p.ldd,
                    H.epilogue_for(p, bias.data_ptr()), torch.cuda.current_stream().cuda_stream)
    H.check_close(D[:, :p.N], H.oracle_full(inp), "bf16", "host entry with transforms")
    plan.close()


# --------------------------------- CUDA cores ---------------------------------

@pytest.mark.parametrize("which", list(WHICH))
@pytest.mark.parametrize("layout", LAYOUTS)
def test_ffma_transforms(layout, which, clean_env):
    p = _xf(I.Problem("xf_ffma", "f32", layout[0], layout[1], 200, 264, 132, alpha=0.5, beta=1.0, c="f32",
                      bias="f32", bias_mode="col", act="relu"), which)
    H.run_and_check_full(p, 309, expect_kernel=G.GEMM_KERNEL_FFMA)


@pytest.mark.parametrize("ab", ["f16", "bf16", "f32"])
def test_generic_kernel_transforms(ab, clean_env):
    """The generic kernel (forced): the 16-bit round trip of the transformed
    value happens per element as it is loaded."""
    p = _xf(I.Problem("xf_simt", ab, "N", "T", 70, 90, 45, beta=0.5, c="f32"), "AB")
    H.run_and_check_full(p, 310, kernel=G.GEMM_KERNEL_SIMT, expect_kernel=G.GEMM_KERNEL_SIMT)


# ------------------------------------ int8 ------------------------------------

@pytest.mark.parametrize("which", ["A", "B", "AB"])
@pytest.mark.parametrize("cta_group", [1, 2])
def test_int8_relu_on_load_exact(which, cta_group, clean_env):
    """int8 operands take the activation only, applied in the fp16 staging pass;
    the result is exact, so it must equal the oracle bit for bit."""
    clean_env.setenv("GEMM_TC_CTA_GROUP", str(cta_group))
    acts = {"A": ("relu", "none"), "B": ("none", "relu"), "AB": ("relu", "relu")}[which]
    p = I.Problem("xf_s8", "s8", "T", "N", 520, 600, 1096, c="s32", d="s32", dist_a=I.I8, dist_b=I.I8,
                  a_act=acts[0], b_act=acts[1])
    cfg = H.run_and_check_full(p, 311, expect_kernel=G.GEMM_KERNEL_TC_INT8)
    assert cfg["cta_group"] == cta_group


def test_int8_relu_on_load_generic_kernel(clean_env):
    p = I.Problem("xf_s8_simt", "s8", "N", "T", 33, 47, 71, alpha=2.0, beta=-1.0, c="s32", d="s32",
                  dist_a=I.I8, dist_b=I.I8, dist_c=I.Dist("int", -1000, 1000), a_act="relu", b_act="relu")
    H.run_and_check_full(p, 312, kernel=G.GEMM_KERNEL_SIMT, expect_kernel=G.GEMM_KERNEL_SIMT)


# ------------------------------- argument errors -------------------------------

def test_paths_without_transforms_refuse_them(clean_env):
    """The diagonal and complex entry points have no operand transforms: they
    refuse a request for one rather than ignore it."""
    dev = torch.zeros(4096, dtype=torch.float16, device="cuda")
    out = torch.zeros(4096, dtype=torch.float32, device="cuda")
    plan = G.Plan(G.GEMM_F16, G.GEMM_F32, torch.cuda.current_device())
    epi = G.make_epilogue(G.GEMM_F32, a_act=G.GEMM_ACT_RELU)
    stream = torch.cuda.current_stream().cuda_stream
    with pytest.raises(G.GemmError) as e:
        G.gemm_run_diag(plan.handle, G.GEMM_SIDE_LEFT, G.GEMM_OP_T, 16, 16, 1.0, dev.data_ptr(),
                        dev.data_ptr(), 16, 0.0, None, 0, out.data_ptr(), 16, epi, stream)
    assert e.value.status == G.GEMM_ERR_UNSUPPORTED
    with pytest.raises(G.GemmError) as e:
        G.gemm_run_complex(plan.handle, G.GEMM_UNIT_IMAGINARY, G.GEMM_OP_T, G.GEMM_OP_N, 8, 8, 8, 1.0,
                           dev.data_ptr(), 16, dev.data_ptr(), 16, 0.0, None, 0, out.data_ptr(), 16, epi, stream)
    assert e.value.status == G.GEMM_ERR_UNSUPPORTED
    plan.close()


@pytest.mark.parametrize("kernel", [G.GEMM_KERNEL_TC, G.GEMM_KERNEL_TC_PAIR], ids=["cta1", "pair"])
def test_transform_warps_bounded_wait_reports_timeout(kernel, clean_env):
    """With the transforms inside the kernel and a 200 ns wait bound, the waits
    of the transform warps and of the MMA thread expire: the kernel records
    GEMM_ERR_TIMEOUT and winds down; the context then runs correctly."""
    clean_env.setenv("GEMM_XF_STAGE", "0")
    p = I.Problem("xf_tmo", "f16", "T", "N", 512, 512, 4096, a_act="relu", b_scale=0.5)
    inp = I.generate(p, 313)
    dp = H.DeviceProblem(inp)
    plan = H.make_plan(p, kernel)
    G.gemm_plan_set_timeout(plan.handle, 200)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == G.GEMM_ERR_TIMEOUT
    G.gemm_plan_set_timeout(plan.handle, 4_000_000_000)
    dp.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0 and plan.last_config()["xf_staged"] == 0
    H.check_close(dp.result(), H.oracle_full(inp), "f32", "after timeout")
    plan.close()


def test_matmul_helper_transforms_equal_pretransformed_operands(clean_env):
    """The Python helper's operand transforms: relu(0.5 * a) and relu(b) given as
    transforms give the same bits as the product of the operands transformed
    beforehand in fp16 (one rounding of the exact fp16 product either way)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(314)
    a = torch.randn(1024, 512, device="cuda", generator=g).half()
    b = torch.randn(512, 768, device="cuda", generator=g).half()
    got = G.matmul(a, b, a_relu=True, a_scale=0.5, b_relu=True)
    want = G.matmul(torch.relu(a * 0.5), torch.relu(b))
    torch.cuda.synchronize()
    assert torch.equal(got, want)
