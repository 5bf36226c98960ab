"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/gemm.h declares, validates arguments and selects
kernels as documented.  No compute call is made."""
import os
import ctypes
import re

import pytest

import dense_gemm_epilogues_gb300 as G

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm.h")

P = 1 << 20   # a 16-byte aligned fake device address (never dereferenced)


@pytest.fixture(scope="module", autouse=True)
def lib():
    from dense_gemm_epilogues_gb300 import build
    build.build()
    return G.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(gemm_[a-z_0-9]+)\s*\(", text,
                                 flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"{n} declared in gemm.h but not exported"
    assert set(names) == set(G.EXPORTED)


def test_abi_version_and_status_strings():
    assert G.gemm_abi_version() == 109
    for s in range(6):
        assert G.gemm_status_string(s).startswith("GEMM_")
    assert "unknown" in G.gemm_status_string(99)


def _v(ab=G.GEMM_F16, c=G.GEMM_F32, la=G.GEMM_OP_T, lb=G.GEMM_OP_N, M=64, N=64, K=64, alpha=1.0,
       A=P, lda=64, B=P, ldb=64, beta=0.0, C=None, ldc=0, D=P, ldd=64, epi=None):
    return G.gemm_validate(ab, c, la, lb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd, epi)


def test_validation_accepts_a_plain_problem():
    assert _v() == G.GEMM_OK


@pytest.mark.parametrize("kw,status", [
    (dict(M=-1), G.GEMM_ERR_INVALID_ARG),
    (dict(la=2), G.GEMM_ERR_INVALID_ARG),
    (dict(la=G.GEMM_OP_N, lda=63), G.GEMM_ERR_INVALID_ARG),         # lda < M for column-major A
    (dict(lda=63), G.GEMM_ERR_INVALID_ARG),                          # lda < K for row-major A
    (dict(lb=G.GEMM_OP_T, ldb=10), G.GEMM_ERR_INVALID_ARG),          # ldb < N for row-major B
    (dict(ldd=10), G.GEMM_ERR_INVALID_ARG),
    (dict(D=None), G.GEMM_ERR_INVALID_ARG),
    (dict(A=None), G.GEMM_ERR_INVALID_ARG),
    (dict(beta=1.0), G.GEMM_ERR_INVALID_ARG),                         # C missing
    (dict(beta=1.0, C=P, ldc=8), G.GEMM_ERR_INVALID_ARG),             # ldc < N
    (dict(beta=1.0, C=P, ldc=128, D=P, ldd=64), G.GEMM_ERR_INVALID_ARG),  # C == D, ldc != ldd
    (dict(ab=G.GEMM_S8, c=G.GEMM_F32), G.GEMM_ERR_INVALID_ARG),       # type pair
    (dict(ab=G.GEMM_F32, c=G.GEMM_F16), G.GEMM_ERR_INVALID_ARG),
    (dict(ab=G.GEMM_S8, c=G.GEMM_S32, alpha=0.5, epi=G.make_epilogue(G.GEMM_S32)),
     G.GEMM_ERR_UNSUPPORTED),                                        # non-integral alpha on int8
    (dict(epi=G.make_epilogue(G.GEMM_S32)), G.GEMM_ERR_INVALID_ARG),  # int output for fp16 inputs
    (dict(epi=G.make_epilogue(G.GEMM_F32, 0, G.GEMM_F32, G.GEMM_BIAS_COL)),
     G.GEMM_ERR_INVALID_ARG),                                        # bias mode without bias
    (dict(epi=G.make_epilogue(G.GEMM_F32, P, G.GEMM_S8, G.GEMM_BIAS_COL)),
     G.GEMM_ERR_INVALID_ARG),                                        # bias type
    (dict(M=1 << 31), G.GEMM_ERR_UNSUPPORTED),
    (dict(epi=G.make_epilogue(G.GEMM_F32, c_act=7)), G.GEMM_ERR_INVALID_ARG),
    # operand transforms
    (dict(epi=G.make_epilogue(G.GEMM_F32, load_xf=4)), G.GEMM_ERR_INVALID_ARG),      # unknown operand bit
    (dict(epi=G.make_epilogue(G.GEMM_F32, a_act=5)), G.GEMM_ERR_INVALID_ARG),        # unknown activation
    (dict(epi=G.make_epilogue(G.GEMM_F32, b_act=2)), G.GEMM_ERR_INVALID_ARG),
    (dict(epi=G.make_epilogue(G.GEMM_F32, a_scale=float("nan"))), G.GEMM_ERR_INVALID_ARG),
    (dict(epi=G.make_epilogue(G.GEMM_F32, b_scale=float("inf"))), G.GEMM_ERR_INVALID_ARG),
    (dict(ab=G.GEMM_S8, c=G.GEMM_S32, epi=G.make_epilogue(G.GEMM_S32, a_scale=2.0)),
     G.GEMM_ERR_UNSUPPORTED),                                        # int8 operands: activation only
])
def test_validation_rejects(kw, status):
    assert _v(**kw) == status


@pytest.mark.parametrize("kw", [
    dict(epi=G.make_epilogue(G.GEMM_F32, a_act=G.GEMM_ACT_RELU, a_scale=-2.5, b_scale=0.5)),
    dict(ab=G.GEMM_BF16, epi=G.make_epilogue(G.GEMM_BF16, b_act=G.GEMM_ACT_RELU)),
    dict(ab=G.GEMM_F32, epi=G.make_epilogue(G.GEMM_F32, a_scale=3.0)),
    dict(ab=G.GEMM_S8, c=G.GEMM_S32, epi=G.make_epilogue(G.GEMM_S32, a_act=G.GEMM_ACT_RELU,
                                                          b_act=G.GEMM_ACT_RELU)),
    # fields of an operand whose bit is clear are ignored
    dict(epi=G.make_epilogue(G.GEMM_F32, a_act=9, a_scale=float("nan"), load_xf=G.GEMM_XF_B)),
])
def test_validation_accepts_operand_transforms(kw):
    assert _v(**kw) == G.GEMM_OK


def test_epilogue_struct_matches_the_header():
    """The binding's struct has the header's fields in order (offsets of a C
    struct of ints, floats and one pointer on an LP64 target)."""
    E = G.gemm_epilogue_t
    names = [n for n, _ in E._fields_]
    assert names == ["bias", "bias_dtype", "bias_mode", "act", "out_dtype", "c_act", "out_scale", "load_xf",
                     "a_act", "a_scale", "b_act", "b_scale"]
    assert E.load_xf.offset == 32 and E.b_scale.offset == 48 and ctypes.sizeof(E) == 56
    e = G.make_epilogue(G.GEMM_F32, b_act=G.GEMM_ACT_RELU)
    assert e.load_xf == G.GEMM_XF_B and e.a_scale == 1.0
    assert G.make_epilogue(G.GEMM_F32).load_xf == 0


def test_validation_edge_cases_accepted():
    assert _v(M=0, D=None, A=None, B=None) == G.GEMM_OK           # empty: nothing is touched
    assert _v(K=0, A=None, B=None) == G.GEMM_OK                   # K == 0: D = epi(beta*C)
    assert _v(beta=1.0, C=P, ldc=64, D=P, ldd=64) == G.GEMM_OK    # in-place C == D
    assert _v(ab=G.GEMM_S8, c=G.GEMM_S32, alpha=3.0, beta=-2.0, C=P, ldc=64,
              epi=G.make_epilogue(G.GEMM_S32)) == G.GEMM_OK


def _sel(ab=G.GEMM_F16, c=G.GEMM_F32, la=G.GEMM_OP_T, lb=G.GEMM_OP_N, M=8192, N=8192, K=8192,
         A=P, lda=None, B=P, ldb=None, epi=None, sms=152):
    lda = lda if lda is not None else (K if la == G.GEMM_OP_T else M)
    ldb = ldb if ldb is not None else (K if lb == G.GEMM_OP_N else N)
    if epi is None and ab == G.GEMM_S8:
        epi = G.make_epilogue(G.GEMM_S32)
    return G.gemm_select(ab, c, la, lb, M, N, K, A, lda, B, ldb, None, 0, P, N, 0.0, epi, sms)


def test_selector_large_square_uses_256x256_pair_tiles():
    cfg = _sel()
    assert cfg["kernel"] == G.GEMM_KERNEL_TC_PAIR and cfg["cta_group"] == 2
    assert (cfg["bm"], cfg["bn"], cfg["bk"]) == (256, 256, 128)
    assert cfg["tiles"] == 32 * 32 and cfg["grid"] == 152 and cfg["raster"] == 8
    # 1024 tiles over 76 pairs: the last 36 (at most half the pairs) run as 72 half tiles.
    assert cfg["half_tiles"] == 36


def test_selector_single_cta_when_one_dimension_fits_one_tile():
    cfg = _sel(M=128, N=8192)
    assert cfg["kernel"] == G.GEMM_KERNEL_TC and cfg["bm"] == 128


@pytest.mark.parametrize("la,lb", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_selector_all_layouts_on_tensor_cores(la, lb):
    assert _sel(la=la, lb=lb)["kernel"] == G.GEMM_KERNEL_TC_PAIR


def test_selector_narrow_and_small_shapes():
    assert _sel(N=64, M=16384, K=16384)["bn"] == 64   # one 64-wide tile column
    cfg = _sel(M=512, N=512, K=512)   # 4 pair tiles: less than a wave of pairs
    assert cfg["kernel"] == G.GEMM_KERNEL_TC and cfg["bm"] == 128
    cfg = _sel(M=2560, N=2048, K=512)  # 80 pair tiles on 76 pairs: a second, nearly empty wave
    assert cfg["kernel"] == G.GEMM_KERNEL_TC
    cfg = _sel(M=8192, N=8192, K=1024)  # 1024 pair tiles: 13.5 waves
    assert cfg["kernel"] == G.GEMM_KERNEL_TC_PAIR and cfg["tiles"] == 1024


def test_selector_misaligned_operands_use_generic_kernel():
    assert _sel(A=P + 2)["kernel"] == G.GEMM_KERNEL_SIMT
    assert _sel(M=100, N=100, K=100, lda=101)["kernel"] == G.GEMM_KERNEL_SIMT
    assert _sel(K=0)["kernel"] == G.GEMM_KERNEL_SIMT
    assert _sel(M=0)["kernel"] == G.GEMM_KERNEL_NONE


def test_selector_int8_and_fp32_paths():
    cfg = _sel(ab=G.GEMM_S8, c=G.GEMM_S32)
    assert cfg["kernel"] == G.GEMM_KERNEL_TC_INT8 and cfg["cta_group"] == 2 and cfg["k_chunk"] == 1024
    cfg = _sel(ab=G.GEMM_S8, c=G.GEMM_S32, N=128)
    assert cfg["kernel"] == G.GEMM_KERNEL_TC_INT8 and cfg["bn"] == 128 and cfg["cta_group"] == 1
    assert _sel(ab=G.GEMM_S8, c=G.GEMM_S32, M=64, N=64, K=60)["kernel"] == G.GEMM_KERNEL_SIMT
    cfg = _sel(ab=G.GEMM_F32, c=G.GEMM_F32, M=4096, N=4096, K=4096)
    assert cfg["kernel"] == G.GEMM_KERNEL_FFMA and cfg["tiles"] == 32 * 32


def test_plan_create_without_gpu_reports_cuda_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(G.GemmError) as e:
        G.gemm_plan_create(G.GEMM_F16, G.GEMM_F32, 0)
    assert e.value.status == G.GEMM_ERR_CUDA
    with pytest.raises(G.GemmError) as e:
        G.gemm_plan_create(G.GEMM_S8, G.GEMM_F32, 0)
    assert e.value.status == G.GEMM_ERR_INVALID_ARG
