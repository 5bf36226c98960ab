"""Parity of every epilogue path of the tensor-core kernels against the fp64 oracle.

The float epilogue dispatches each warp's chunks to one of several loops:
- three loops specialised on D's type for the plain epilogue (no C, bias or ReLU);
- six for an fp32 column bias with or without ReLU and no C;
- one for fp32 C and D with no bias or ReLU;
- the general per-chunk path for everything else.

A specialised loop runs only when the warp's columns lie inside D and D's rows
take 16-byte vector stores. Otherwise the general path runs, and so do partial
last tile columns and unaligned rows. Each case below runs once with N a multiple
of the tile width and once with a ragged last tile column, so that one launch
mixes both paths. It runs on the single-CTA kernel (64- and 256-wide tiles) and
on the CTA-pair kernel. The near-miss cases (16-bit bias, row bias, ReLU on C,
16-bit C, odd D pitch) pin the general path's conditions.
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
    yield
    torch.cuda.synchronize()


@pytest.fixture(autouse=True)
def _clean_env(monkeypatch):
    for v in ("GEMM_TC_CTA_GROUP", "GEMM_TC_BN", "GEMM_TC_SPLITK", "GEMM_STREAM_K", "GEMM_TC_TAIL_HALVES",
              "GEMM_XF_STAGE", "GEMM_TC_KROT", "GEMM_FFMA_TAIL"):
        monkeypatch.delenv(v, raising=False)


# (name, Problem keyword arguments): the specialised loops first, then near misses.
CASES = [
    ("plain_f32", dict(d="f32")),
    ("plain_f16", dict(d="f16")),
    ("plain_bf16_alpha", dict(d="bf16", alpha=-1.25)),
    ("bias_relu_bf16", dict(d="bf16", bias="f32", bias_mode="col", act="relu")),
    ("bias_relu_f16", dict(d="f16", bias="f32", bias_mode="col", act="relu")),
    ("bias_relu_f32", dict(d="f32", bias="f32", bias_mode="col", act="relu")),
    ("bias_bf16_no_relu", dict(d="bf16", bias="f32", bias_mode="col")),
    ("c32", dict(d="f32", c="f32", beta=0.5, alpha=1.5)),
    ("c32_beta_neg", dict(d="f32", c="f32", beta=-1.0)),
    # the general path
    ("bias_f16_relu", dict(d="bf16", bias="f16", bias_mode="col", act="relu")),
    ("bias_row_relu", dict(d="f16", bias="f32", bias_mode="row", act="relu")),
    ("relu_only", dict(d="f16", act="relu")),
    ("c32_c_relu", dict(d="f32", c="f32", beta=0.5, c_act="relu")),
    ("c16_d32", dict(d="f32", c="f16", beta=0.5)),
    ("c32_d_bf16", dict(d="bf16", c="f32", beta=0.5)),
    ("c32_bias", dict(d="f32", c="f32", beta=0.5, bias="f32", bias_mode="col")),
    ("plain_f16_odd_pitch", dict(d="f16", pad_d=1)),
    ("plain_f32_padded_pitch", dict(d="f32", pad_d=4)),
]

KERNELS = [
    ("tc_bn256", G.GEMM_KERNEL_TC, {"GEMM_TC_BN": "256"}),
    ("tc_bn64", G.GEMM_KERNEL_TC, {"GEMM_TC_BN": "64"}),
    ("pair", G.GEMM_KERNEL_TC_PAIR, {}),
]


@pytest.mark.parametrize("n", [768, 720])
@pytest.mark.parametrize("kname,kernel,env", KERNELS, ids=[k[0] for k in KERNELS])
@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_epilogue_path(name, kw, kname, kernel, env, n, monkeypatch):
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    p = H.tma_aligned(I.Problem(f"epi_{name}", "f16", "T", "N", 640, n, 320, **kw))
    seed = 9000 + sum(ord(ch) for ch in name) + n
    cfg = H.run_and_check_full(p, seed, kernel=kernel, expect_kernel=kernel)
    if kernel == G.GEMM_KERNEL_TC:
        assert cfg["bn"] == int(env["GEMM_TC_BN"])


@pytest.mark.parametrize("kernel", [G.GEMM_KERNEL_TC, G.GEMM_KERNEL_TC_PAIR], ids=["tc", "pair"])
@pytest.mark.parametrize("case", ["plain_f16", "bias_relu_bf16", "c32"])
def test_epilogue_paths_batched(case, kernel):
    """Strided batches through the specialised loops: each problem's D, C and
    bias are found from its problem index."""
    from test_gpu_batched import run_batched
    kw = dict(CASES)[case]
    p = H.tma_aligned(I.Problem(f"epi_batched_{case}", "f16", "T", "N", 256, 512, 192, **kw))
    cfg = run_batched(p, 3, 9600, kernel=kernel)
    assert cfg["kernel"] == kernel
