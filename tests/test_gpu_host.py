"""GPU parity of gemm_run_host on problems large enough for its row-panel copy
pipeline (inputs copied in by row panels on one stream, each panel's GEMM on the
caller's stream, D copied out on a third): every element against the oracle."""
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


def _host_run(p, inp, pinned=True, in_place=False):
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t.clone())
    A, B = pin(inp.A), pin(inp.B)
    C = pin(inp.C) if inp.C is not None else None
    bias = pin(inp.bias) if inp.bias is not None else None
    D = C if in_place else pin(torch.full((p.M, p.ldd), H.SENTINEL[p.d], dtype=I.TORCH_DTYPES[p.d]))
    epi = G.make_epilogue(G.DTYPE_CODES[p.d], bias.data_ptr() if bias is not None else 0,
                          G.DTYPE_CODES[p.bias] if p.bias else G.GEMM_F32, H.G_BIAS[p.bias_mode],
                          G.GEMM_ACT_RELU if p.act == "relu" else G.GEMM_ACT_NONE)
    plan = H.make_plan(p)
    G.gemm_run_host(plan.handle, G.LAYOUT_CODES[p.layout_a], G.LAYOUT_CODES[p.layout_b], p.M, p.N,
                    p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                    C.data_ptr() if C is not None else None, p.ldc if p.c else 0, D.data_ptr(),
                    p.ldd, epi, torch.cuda.current_stream().cuda_stream)
    assert plan.device_status() == 0
    plan.close()
    return D


@pytest.mark.parametrize("layout", ["TN", "NT", "NN"])
def test_host_panels_alpha_beta_row_bias(layout):
    """5000 x 2048 x 512: four row panels (1280 rows, the last 1160); column-major
    A takes strided panel copies; a row bias follows its panel."""
    p = I.Problem("host_pan", "f16", layout[0], layout[1], 5000, 2048, 512, alpha=1.5, beta=-0.5,
                  c="f32", bias="f32", bias_mode="row", act="relu", pad_a=8, pad_d=4)
    inp = I.generate(p, 700)
    D = _host_run(p, inp)
    H.check_close(D[:, :p.N], H.oracle_full(inp), p.d, p.name)
    assert torch.all(D[:, p.N:] == H.SENTINEL[p.d]), "write into the padding of D"


def test_host_panels_in_place_and_pageable():
    """C and D the same host buffer (each panel's C is read before its D lands),
    and pageable host memory (the copies stay correct, only slower)."""
    p = I.Problem("host_inpl", "bf16", "T", "N", 4096, 2304, 256, beta=2.0, c="f32", d="f32")
    inp = I.generate(p, 710)
    ref = H.oracle_full(inp)
    D = _host_run(p, inp, pinned=False, in_place=True)
    H.check_close(D[:, :p.N], ref, p.d, p.name)


def test_host_panels_int8_exact():
    p = H.tma_aligned(I.Problem("host_i8", "s8", "T", "N", 4096, 4096, 264, d="s32", dist_a=I.I8,
                                dist_b=I.I8))
    inp = I.generate(p, 720)
    D = _host_run(p, inp)
    H.check_close(D[:, :p.N], H.oracle_full(inp), "s32", p.name)


def test_gemm_log_prints_the_configuration():
    """GEMM_LOG=1 (read once per process): every launch prints the configuration
    it runs to stderr -- checked in a child process."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import torch, dense_gemm_epilogues_gb300 as G\n"
            "a = torch.randn(1024, 512, device='cuda', dtype=torch.float16)\n"
            "b = torch.randn(512, 768, device='cuda', dtype=torch.float16)\n"
            "G.matmul(a, b); torch.cuda.synchronize()\n")
    env = dict(os.environ, GEMM_LOG="1", PYTHONPATH=root)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = [l for l in r.stderr.splitlines() if l.startswith("gemm: run ")]
    assert len(line) == 1 and "M=1024 N=768 K=512" in line[0] and "kernel=tc" in line[0], r.stderr
