"""The selector's choice for every workload of the benchmark (host only, no GPU).

Each line is the kernel and tile the measurements picked for that workload on a
152-SM GB300 (76 co-resident CTA pairs); a change of the cost model that moves
one of them must be re-measured.
"""
import pytest

import dense_gemm_epilogues_gb300 as G
from dense_gemm_epilogues_gb300 import inputs as I

P = 1 << 20   # a 16-byte aligned fake device address (never dereferenced)


@pytest.fixture(scope="module", autouse=True)
def lib():
    from dense_gemm_epilogues_gb300 import build
    build.build()
    return G.load_library()


def select(p: I.Problem) -> dict:
    ab = G.DTYPE_CODES[p.ab]
    c = G.DTYPE_CODES[p.c] if p.c else (G.GEMM_S32 if p.ab == "s8" else G.GEMM_F32)
    epi = G.make_epilogue(G.DTYPE_CODES[p.d], a_act=G.GEMM_ACT_RELU if p.a_act == "relu" else G.GEMM_ACT_NONE,
                          a_scale=p.a_scale, b_act=G.GEMM_ACT_RELU if p.b_act == "relu" else G.GEMM_ACT_NONE,
                          b_scale=p.b_scale)
    return G.gemm_select(ab, c, G.LAYOUT_CODES[p.layout_a], G.LAYOUT_CODES[p.layout_b], p.M, p.N, p.K,
                         P, p.lda, P, p.ldb, P if p.c else None, p.ldc if p.c else 0, P, p.ldd,
                         p.beta, epi, 152)


@pytest.mark.parametrize("layout", ["NN", "NT", "TN", "TT"])
def test_headline_8192_on_cta_pairs(layout):
    cfg = select(I.square_fp16_8192(layout))
    assert cfg["kernel"] == G.GEMM_KERNEL_TC_PAIR and (cfg["bm"], cfg["bn"]) == (256, 256)
    assert cfg["grid"] == 152 and cfg["half_tiles"] == 36 and cfg["sk_tiles"] == 0


@pytest.mark.parametrize("make,kernel,tile", [
    (I.fc_bf16_8192x4096x11008, G.GEMM_KERNEL_TC_PAIR, (256, 256)),
    (I.int8_8192, G.GEMM_KERNEL_TC_INT8, (256, 256)),
    (I.sgemm_4096_bias_relu, G.GEMM_KERNEL_FFMA, (128, 128)),
    (I.skinny_fp16_16384x64x16384, G.GEMM_KERNEL_TC, (128, 64)),
    (I.square_fp16_256, G.GEMM_KERNEL_TC, (128, 64)),
], ids=["fc", "int8", "sgemm", "skinny", "256"])
def test_workload_kernels(make, kernel, tile):
    cfg = select(make())
    assert cfg["kernel"] == kernel and (cfg["bm"], cfg["bn"]) == tile, cfg
    if kernel == G.GEMM_KERNEL_FFMA:
        # 1024 tiles on 2 x 152 CTA slots: a last wave of 112 tiles, split over K in two.
        assert cfg["sk_tiles"] == 112 and cfg["split_k"] == 2 and cfg["grid"] == 912 + 224, cfg
    else:
        assert cfg["sk_tiles"] == 0


@pytest.mark.parametrize("n,kernel,bn", [(512, G.GEMM_KERNEL_TC, 64), (1024, G.GEMM_KERNEL_TC, 64),
                                          (2048, G.GEMM_KERNEL_TC, 256), (4096, G.GEMM_KERNEL_TC_PAIR, 256),
                                          (16384, G.GEMM_KERNEL_TC_PAIR, 256)])
def test_square_sweep(n, kernel, bn):
    cfg = select(I.square_fp16(n))
    assert cfg["kernel"] == kernel and cfg["bn"] == bn, cfg


def test_operand_transforms_in_the_kernel_run_whole_tiles(monkeypatch):
    """1024 x 1024 x 8192 takes single-CTA stream-K; with an operand transform
    kept inside the kernel the same shape runs whole tiles (the transform
    instances have no stream-K); staged, it keeps stream-K."""
    p = I.square_fp16(1024).with_(K=8192)
    assert select(p)["sk_tiles"] > 0
    cfg = select(p.with_(a_act="relu"))
    assert cfg["xf_staged"] == G.GEMM_XF_A and cfg["sk_tiles"] > 0, cfg
    monkeypatch.setenv("GEMM_XF_STAGE", "0")
    cfg = select(p.with_(a_act="relu"))
    assert cfg["kernel"] == G.GEMM_KERNEL_TC and cfg["sk_tiles"] == 0 and cfg["split_k"] == 1, cfg
    assert cfg["xf_staged"] == 0


@pytest.mark.parametrize("make,a_act,b_scale,staged", [
    (I.fc_bf16_8192x4096x11008, "relu", 1.0, G.GEMM_XF_A),            # X re-read by 43 tile columns
    (lambda: I.square_fp16_8192("TN"), "relu", 0.5, G.GEMM_XF_A | G.GEMM_XF_B),
    (I.skinny_fp16_16384x64x16384, "relu", 0.5, 0),                   # A read by one tile column; B 2 MiB
    (I.square_fp16_256, "relu", 0.5, 0),                                # operands under 4 MiB
], ids=["fc", "8192", "skinny", "256"])
def test_where_operand_transforms_run(make, a_act, b_scale, staged):
    """Operands that many tiles re-read (and that are not tiny) are transformed
    once by a staging pass; the rest inside the GEMM kernel."""
    cfg = select(make().with_(a_act=a_act, b_scale=b_scale))
    assert cfg["xf_staged"] == staged, cfg
