"""GPU parity of gemm_run_strided_batched: a batch of independent problems in one
call, each compared element by element with the oracle run on that problem
alone (a batched GEMM is, by definition, the independent GEMMs)."""
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


def _stack(ts, gap):
    """Stack equally shaped 2-D storage tensors into one buffer, `gap` poisoned
    elements after each; returns (device tensor, element stride)."""
    flat = [t.reshape(-1) for t in ts]
    n = flat[0].numel()
    stride = n + gap
    fill = 127 if ts[0].dtype == torch.int8 else (0 if ts[0].dtype == torch.int32 else float("nan"))
    buf = torch.full((len(ts) * stride,), fill, dtype=ts[0].dtype)
    for z, f in enumerate(flat):
        buf[z * stride: z * stride + n] = f
    return buf.cuda(), stride


def run_batched(p: I.Problem, batch: int, seed: int, share_b=False, gap=8, kernel=None):
    inps = [I.generate(p, seed + z) for z in range(batch)]
    if share_b:
        for inp in inps:
            inp.B = inps[0].B
    A, sa = _stack([x.A for x in inps], gap)
    if share_b:
        B, sb = inps[0].B.cuda(), 0
    else:
        B, sb = _stack([x.B for x in inps], gap)
    C, sc = (_stack([x.C for x in inps], gap) if p.c else (None, 0))
    bias, sbias = (_stack([x.bias.reshape(1, -1) for x in inps], 0) if p.bias else (None, 0))
    sd = p.M * p.ldd + 16
    s = H.SENTINEL[p.d]
    Dbuf = torch.full((batch * sd,), s, dtype=I.TORCH_DTYPES[p.d], device="cuda")
    plan = H.make_plan(p, kernel)
    epi = H.epilogue_for(p, bias.data_ptr() if bias is not None else 0)
    G.gemm_run_strided_batched(plan.handle, G.LAYOUT_CODES[p.layout_a], G.LAYOUT_CODES[p.layout_b],
                               p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, sa, B.data_ptr(), p.ldb,
                               sb, p.beta, C.data_ptr() if C is not None else None,
                               p.ldc if p.c else 0, sc, Dbuf.data_ptr(), p.ldd, sd, batch, epi,
                               sbias, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    cfg = plan.last_config()
    for z, inp in enumerate(inps):
        Dz = Dbuf[z * sd: z * sd + p.M * p.ldd].view(p.M, p.ldd)
        H.check_close(Dz[:, :p.N], H.oracle_full(inp), p.d, f"{p.name} problem {z}")
        pad = Dbuf[z * sd + p.M * p.ldd: (z + 1) * sd]
        assert torch.all(pad.cpu() == torch.tensor(s, dtype=pad.dtype)), "write past a problem's D"
        if p.ldd > p.N:
            assert torch.all(Dz[:, p.N:].cpu() == torch.tensor(s, dtype=pad.dtype))
    plan.close()
    return cfg


@pytest.mark.parametrize("layout", ["NN", "NT", "TN", "TT"])
def test_batched_pair_kernel_alpha_beta_bias(layout, monkeypatch):
    monkeypatch.setenv("GEMM_TC_CTA_GROUP", "2")   # pairs, although 20 tiles are less than a wave
    p = H.tma_aligned(I.Problem("bat", "f16", layout[0], layout[1], 300, 264, 200, alpha=1.25,
                                beta=-0.5, c="f32", bias="f32", bias_mode="col", act="relu",
                                pad_d=3))
    cfg = run_batched(p, 5, 200)
    assert cfg["kernel"] == G.GEMM_KERNEL_TC_PAIR and cfg["tiles"] == 5 * 2 * 2


def test_batched_shared_weights_single_cta_bf16():
    """stride_b = 0: every problem multiplies by the same B (shared weights)."""
    p = H.tma_aligned(I.Problem("bat_w", "bf16", "T", "T", 200, 96, 320, d="bf16", bias="f32",
                                bias_mode="col"))
    cfg = run_batched(p, 7, 210, share_b=True)
    assert cfg["kernel"] == G.GEMM_KERNEL_TC
    assert cfg["tiles"] == 7 * 2 * ((96 + cfg["bn"] - 1) // cfg["bn"])   # 2 tile rows of 128 per problem


@pytest.mark.parametrize("cta_group", ["1", "2"])
def test_batched_int8_exact(cta_group, monkeypatch):
    monkeypatch.setenv("GEMM_TC_CTA_GROUP", cta_group)
    p = H.tma_aligned(I.Problem("bat_i8", "s8", "T", "N", 272, 288, 1100, alpha=2.0, beta=-1.0,
                                c="s32", d="s32", dist_a=I.I8, dist_b=I.I8,
                                dist_c=I.Dist("int", -1000, 1000)))
    cfg = run_batched(p, 3, 220, gap=16)
    assert cfg["kernel"] == G.GEMM_KERNEL_TC_INT8 and cfg["cta_group"] == int(cta_group)


def test_batched_ffma_and_generic():
    p = I.Problem("bat_f32", "f32", "N", "T", 152, 140, 72, beta=1.0, c="f32", bias="f32",
                  bias_mode="row", act="relu", c_act="relu")
    assert run_batched(p, 4, 230)["kernel"] == G.GEMM_KERNEL_FFMA
    q = I.Problem("bat_gen", "f16", "T", "N", 45, 37, 29, pad_a=1, pad_b=2)
    assert run_batched(q, 4, 240)["kernel"] == G.GEMM_KERNEL_SIMT


def test_batched_unaligned_stride_runs_per_problem():
    """A batch stride that is not a 16-byte multiple cannot be a TMA dimension:
    the call runs one launch per problem.  Here the later problems start off a
    16-byte boundary, so they run on the generic kernel; last_config shows the
    last problem's launch (one problem's 16 x 16 tiles)."""
    p = H.tma_aligned(I.Problem("bat_odd", "f16", "T", "N", 256, 256, 128, beta=0.5, c="f32"))
    cfg = run_batched(p, 3, 250, gap=3)
    assert cfg["kernel"] == G.GEMM_KERNEL_SIMT and cfg["tiles"] == 16 * 16


def test_batched_edge_cases():
    p = I.Problem("bat_e", "f16", "T", "N", 64, 64, 64)
    plan = H.make_plan(p)
    D = torch.zeros(64 * 64 * 2, dtype=torch.float32, device="cuda")
    A = torch.zeros(64 * 64 * 2, dtype=torch.float16, device="cuda")
    args = (plan.handle, G.GEMM_OP_T, G.GEMM_OP_N, 64, 64, 64, 1.0, A.data_ptr(), 64, 4096,
            A.data_ptr(), 64, 4096, 0.0, None, 0, 0, D.data_ptr(), 64)
    G.gemm_run_strided_batched(*args, 4096, 0, G.make_epilogue(G.GEMM_F32), 0)   # batch 0: no-op
    with pytest.raises(G.GemmError) as e:   # outputs of the two problems would overlap
        G.gemm_run_strided_batched(*args, 100, 2, G.make_epilogue(G.GEMM_F32), 0)
    assert e.value.status == G.GEMM_ERR_INVALID_ARG
    with pytest.raises(G.GemmError):
        G.gemm_run_strided_batched(*args, 4096, -1, G.make_epilogue(G.GEMM_F32), 0)
    plan.close()
