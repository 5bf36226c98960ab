"""GB300 (sm_103a) generalized GEMM with fused epilogues.

    D = epilogue(alpha * op(A) * op(B) + beta * C),  epilogue = bias, ReLU, cast

This package is a thin ctypes binding of ``libgemm.so`` (C ABI in
``include/gemm.h``): the functions below carry the C names and only marshal
arguments.  Every step of the computation runs in the library's CUDA kernels.
There is no CPU fallback: if the library is missing, loading fails loudly.

PyTorch is used only for device memory and streams (the ``matmul`` helper reads
pointers, strides and the current stream from tensors).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgemm.so")

# ---- enums (include/gemm.h) ----
GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_UNSUPPORTED, GEMM_ERR_ALIGNMENT, GEMM_ERR_CUDA, GEMM_ERR_TIMEOUT = range(6)
GEMM_OP_N, GEMM_OP_T = 0, 1
GEMM_F32, GEMM_F16, GEMM_BF16, GEMM_S8, GEMM_S32 = range(5)
GEMM_ACT_NONE, GEMM_ACT_RELU = 0, 1
GEMM_BIAS_NONE, GEMM_BIAS_COL, GEMM_BIAS_ROW = 0, 1, 2
(GEMM_KERNEL_AUTO, GEMM_KERNEL_NONE, GEMM_KERNEL_TC, GEMM_KERNEL_TC_INT8, GEMM_KERNEL_FFMA,
 GEMM_KERNEL_SIMT, GEMM_KERNEL_TC_PAIR, GEMM_KERNEL_DIAG) = range(8)
GEMM_SIDE_LEFT, GEMM_SIDE_RIGHT = 0, 1
GEMM_UNIT_IMAGINARY, GEMM_UNIT_DUAL = 0, 1

KERNEL_NAMES = {GEMM_KERNEL_AUTO: "auto", GEMM_KERNEL_NONE: "none", GEMM_KERNEL_TC: "tc",
                GEMM_KERNEL_TC_INT8: "tc_int8", GEMM_KERNEL_FFMA: "ffma", GEMM_KERNEL_SIMT: "simt",
                GEMM_KERNEL_TC_PAIR: "tc_pair", GEMM_KERNEL_DIAG: "diag"}
DTYPE_CODES = {"f32": GEMM_F32, "f16": GEMM_F16, "bf16": GEMM_BF16, "s8": GEMM_S8, "s32": GEMM_S32}
LAYOUT_CODES = {"N": GEMM_OP_N, "T": GEMM_OP_T}

# Every entry point declared in include/gemm.h.
EXPORTED = ["gemm_plan_create", "gemm_plan_destroy", "gemm_run", "gemm_run_host", "gemm_validate",
            "gemm_select", "gemm_plan_set_kernel", "gemm_plan_last_config", "gemm_plan_device_status",
            "gemm_plan_set_timeout", "gemm_status_string", "gemm_abi_version",
            "gemm_run_s8_noalloc", "gemm_noalloc_device_status", "gemm_noalloc_set_timeout",
            "gemm_run_strided_batched", "gemm_run_diag", "gemm_run_complex"]


GEMM_XF_A, GEMM_XF_B = 1, 2


class gemm_epilogue_t(ctypes.Structure):
    _fields_ = [("bias", ctypes.c_void_p), ("bias_dtype", ctypes.c_int), ("bias_mode", ctypes.c_int),
                ("act", ctypes.c_int), ("out_dtype", ctypes.c_int), ("c_act", ctypes.c_int),
                ("out_scale", ctypes.c_float), ("load_xf", ctypes.c_uint32),
                ("a_act", ctypes.c_int), ("a_scale", ctypes.c_float),
                ("b_act", ctypes.c_int), ("b_scale", ctypes.c_float)]


class gemm_config_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("kernel", "bm", "bn", "bk", "stages", "cta_group", "split_k", "raster", "grid",
                 "k_chunk", "tiles", "sk_tiles", "cluster", "half_tiles", "xf_staged")]

    def as_dict(self) -> dict:
        d = {n: getattr(self, n) for n, _ in self._fields_}
        d["kernel_name"] = KERNEL_NAMES.get(self.kernel, "?")
        return d


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gemm_status_string(status)}")


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libgemm.so.  Raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libgemm.so not found at {path}: build it with "
                           "`python -m dense_gemm_epilogues_gb300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    i64, dbl, vp, ci = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
    run_args = [vp, ci, ci, i64, i64, i64, dbl, vp, i64, vp, i64, dbl, vp, i64, vp, i64,
                ctypes.POINTER(gemm_epilogue_t), vp]
    lib.gemm_plan_create.argtypes = [ctypes.POINTER(vp), ci, ci, ci]
    lib.gemm_plan_destroy.argtypes = [vp]
    lib.gemm_run.argtypes = run_args
    lib.gemm_run_host.argtypes = run_args
    lib.gemm_validate.argtypes = [ci, ci, ci, ci, i64, i64, i64, dbl, vp, i64, vp, i64, dbl, vp, i64,
                                  vp, i64, ctypes.POINTER(gemm_epilogue_t)]
    lib.gemm_select.argtypes = [ci, ci, ci, ci, i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64,
                                dbl, ctypes.POINTER(gemm_epilogue_t), ci,
                                ctypes.POINTER(gemm_config_t)]
    lib.gemm_plan_set_kernel.argtypes = [vp, ci]
    lib.gemm_plan_last_config.argtypes = [vp, ctypes.POINTER(gemm_config_t)]
    lib.gemm_plan_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32)]
    lib.gemm_plan_set_timeout.argtypes = [vp, ctypes.c_uint64]
    lib.gemm_status_string.argtypes = [ci]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_abi_version.argtypes = []
    lib.gemm_run_strided_batched.argtypes = [vp, ci, ci, i64, i64, i64, dbl, vp, i64, i64, vp, i64, i64,
                                             dbl, vp, i64, i64, vp, i64, i64, i64,
                                             ctypes.POINTER(gemm_epilogue_t), i64, vp]
    lib.gemm_run_s8_noalloc.argtypes = [ci, ci, i64, i64, i64, dbl, vp, i64, vp, i64, dbl, vp, i64,
                                        vp, i64, ctypes.POINTER(gemm_epilogue_t), vp, vp]
    lib.gemm_noalloc_device_status.argtypes = [ctypes.POINTER(ctypes.c_int32), vp]
    lib.gemm_noalloc_set_timeout.argtypes = [ctypes.c_uint64]
    lib.gemm_run_diag.argtypes = [vp, ci, ci, i64, i64, dbl, vp, vp, i64, dbl, vp, i64, vp, i64,
                                  ctypes.POINTER(gemm_epilogue_t), vp]
    lib.gemm_run_complex.argtypes = [vp, ci, ci, ci, i64, i64, i64, dbl, vp, i64, vp, i64, dbl, vp, i64,
                                     vp, i64, ctypes.POINTER(gemm_epilogue_t), vp]
    for name in EXPORTED:
        if name not in ("gemm_status_string", "gemm_abi_version"):
            getattr(lib, name).restype = ci
    lib.gemm_abi_version.restype = ci
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != GEMM_OK:
        raise GemmError(status, where)


def _epi_ptr(epi: Optional[gemm_epilogue_t]):
    return ctypes.byref(epi) if epi is not None else None


def make_epilogue(out_dtype: int, bias: int = 0, bias_dtype: int = GEMM_F32,
                  bias_mode: int = GEMM_BIAS_NONE, act: int = GEMM_ACT_NONE,
                  c_act: int = GEMM_ACT_NONE, out_scale: float = 1.0,
                  a_act: int = GEMM_ACT_NONE, a_scale: float = 1.0,
                  b_act: int = GEMM_ACT_NONE, b_scale: float = 1.0,
                  load_xf: Optional[int] = None) -> gemm_epilogue_t:
    """The C struct.  load_xf defaults to the operands whose transform is not
    the identity (act none, scale 1); pass it to force a transform on or off."""
    if load_xf is None:
        load_xf = ((GEMM_XF_A if (a_act != GEMM_ACT_NONE or a_scale != 1.0) else 0) |
                   (GEMM_XF_B if (b_act != GEMM_ACT_NONE or b_scale != 1.0) else 0))
    return gemm_epilogue_t(bias or None, bias_dtype, bias_mode, act, out_dtype, c_act, out_scale,
                           load_xf, a_act, a_scale, b_act, b_scale)


# ---- C entry points, same names ----

def gemm_status_string(status: int) -> str:
    return load_library().gemm_status_string(status).decode()


def gemm_abi_version() -> int:
    return load_library().gemm_abi_version()


def gemm_plan_create(ab_dtype: int, c_dtype: int, device: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(load_library().gemm_plan_create(ctypes.byref(h), ab_dtype, c_dtype, device), "gemm_plan_create")
    return h.value


def gemm_plan_destroy(plan: int) -> None:
    _check(load_library().gemm_plan_destroy(plan), "gemm_plan_destroy")


def gemm_run(plan, layout_a, layout_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd,
             epi: Optional[gemm_epilogue_t] = None, stream: int = 0) -> None:
    _check(load_library().gemm_run(plan, layout_a, layout_b, M, N, K, alpha, A, lda, B, ldb, beta,
                                   C, ldc, D, ldd, _epi_ptr(epi), stream), "gemm_run")


def gemm_run_host(plan, layout_a, layout_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd,
                  epi: Optional[gemm_epilogue_t] = None, stream: int = 0) -> None:
    _check(load_library().gemm_run_host(plan, layout_a, layout_b, M, N, K, alpha, A, lda, B, ldb,
                                        beta, C, ldc, D, ldd, _epi_ptr(epi), stream), "gemm_run_host")


def gemm_run_strided_batched(plan, layout_a, layout_b, M, N, K, alpha, A, lda, stride_a, B, ldb,
                             stride_b, beta, C, ldc, stride_c, D, ldd, stride_d, batch,
                             epi: Optional[gemm_epilogue_t] = None, stride_bias: int = 0,
                             stream: int = 0) -> None:
    _check(load_library().gemm_run_strided_batched(plan, layout_a, layout_b, M, N, K, alpha, A, lda,
                                                   stride_a, B, ldb, stride_b, beta, C, ldc,
                                                   stride_c, D, ldd, stride_d, batch,
                                                   _epi_ptr(epi), stride_bias, stream),
           "gemm_run_strided_batched")


def gemm_run_diag(plan, side, layout_x, M, N, alpha, diag, X, ldx, beta, C, ldc, D, ldd,
                  epi: Optional[gemm_epilogue_t] = None, stream: int = 0) -> None:
    _check(load_library().gemm_run_diag(plan, side, layout_x, M, N, alpha, diag, X, ldx, beta, C, ldc,
                                        D, ldd, _epi_ptr(epi), stream), "gemm_run_diag")


def gemm_run_complex(plan, unit, layout_a, layout_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                     D, ldd, epi: Optional[gemm_epilogue_t] = None, stream: int = 0) -> None:
    _check(load_library().gemm_run_complex(plan, unit, layout_a, layout_b, M, N, K, alpha, A, lda, B,
                                           ldb, beta, C, ldc, D, ldd, _epi_ptr(epi), stream),
           "gemm_run_complex")


def gemm_run_s8_noalloc(layout_a, layout_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd,
                        epi: Optional[gemm_epilogue_t] = None, status: Optional[int] = None,
                        stream: int = 0) -> None:
    """int8 GEMM on the current device with no device allocation (library-held
    fixed scratch; see include/gemm.h).  `status`: optional device address of a
    caller-owned int32 error word."""
    _check(load_library().gemm_run_s8_noalloc(layout_a, layout_b, M, N, K, alpha, A, lda, B, ldb,
                                              beta, C, ldc, D, ldd, _epi_ptr(epi), status, stream),
           "gemm_run_s8_noalloc")


def gemm_noalloc_device_status(stream: int = 0) -> int:
    """Read and clear the library's error word of gemm_run_s8_noalloc on the
    current device (after synchronising `stream`)."""
    code = ctypes.c_int32(0)
    _check(load_library().gemm_noalloc_device_status(ctypes.byref(code), stream),
           "gemm_noalloc_device_status")
    return code.value


def gemm_noalloc_set_timeout(timeout_ns: int) -> None:
    _check(load_library().gemm_noalloc_set_timeout(timeout_ns), "gemm_noalloc_set_timeout")


NOALLOC_SCRATCH_BYTES = 32 << 20


def gemm_validate(ab_dtype, c_dtype, layout_a, layout_b, M, N, K, alpha, A, lda, B, ldb, beta, C,
                  ldc, D, ldd, epi: Optional[gemm_epilogue_t] = None) -> int:
    """Returns the status code (does not raise)."""
    return load_library().gemm_validate(ab_dtype, c_dtype, layout_a, layout_b, M, N, K, alpha, A,
                                        lda, B, ldb, beta, C, ldc, D, ldd, _epi_ptr(epi))


def gemm_select(ab_dtype, c_dtype, layout_a, layout_b, M, N, K, A, lda, B, ldb, C, ldc, D, ldd,
                beta, epi: Optional[gemm_epilogue_t], sm_count: int) -> dict:
    cfg = gemm_config_t()
    _check(load_library().gemm_select(ab_dtype, c_dtype, layout_a, layout_b, M, N, K, A, lda, B, ldb,
                                      C, ldc, D, ldd, beta, _epi_ptr(epi), sm_count,
                                      ctypes.byref(cfg)), "gemm_select")
    return cfg.as_dict()


def gemm_plan_set_kernel(plan: int, kernel: int) -> None:
    _check(load_library().gemm_plan_set_kernel(plan, kernel), "gemm_plan_set_kernel")


def gemm_plan_last_config(plan: int) -> dict:
    cfg = gemm_config_t()
    _check(load_library().gemm_plan_last_config(plan, ctypes.byref(cfg)), "gemm_plan_last_config")
    return cfg.as_dict()


def gemm_plan_device_status(plan: int, stream: int = 0) -> int:
    code = ctypes.c_int32(0)
    _check(load_library().gemm_plan_device_status(plan, stream, ctypes.byref(code)),
           "gemm_plan_device_status")
    return code.value


def gemm_plan_set_timeout(plan: int, timeout_ns: int) -> None:
    _check(load_library().gemm_plan_set_timeout(plan, timeout_ns), "gemm_plan_set_timeout")


# ---- torch-tensor convenience (marshalling only) ----

_TORCH_CODES = None


def _torch_code(t) -> int:
    global _TORCH_CODES
    import torch
    if _TORCH_CODES is None:
        _TORCH_CODES = {torch.float32: GEMM_F32, torch.float16: GEMM_F16, torch.bfloat16: GEMM_BF16,
                        torch.int8: GEMM_S8, torch.int32: GEMM_S32}
    return _TORCH_CODES[t.dtype]


def layout_of(t) -> tuple:
    """(layout code, leading dimension) of a 2-D tensor view: row-major (T) when
    its column stride is 1, column-major (N) when its row stride is 1."""
    r, c = t.shape
    if t.stride(1) == 1 and (r <= 1 or t.stride(0) >= max(c, 1)):
        return GEMM_OP_T, max(t.stride(0), c, 1)
    if t.stride(0) == 1 and (c <= 1 or t.stride(1) >= max(r, 1)):
        return GEMM_OP_N, max(t.stride(1), r, 1)
    raise ValueError("operand must have unit stride along one dimension")


class Plan:
    """Owns a gemm_plan_t for one (A/B type, C type, device)."""

    def __init__(self, ab_dtype: int, c_dtype: int, device: int = 0):
        self.handle = gemm_plan_create(ab_dtype, c_dtype, device)
        self.ab_dtype, self.c_dtype, self.device = ab_dtype, c_dtype, device

    def close(self):
        if getattr(self, "handle", None):
            gemm_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_kernel(self, kernel: int):
        gemm_plan_set_kernel(self.handle, kernel)

    def last_config(self) -> dict:
        return gemm_plan_last_config(self.handle)

    def device_status(self, stream: int = 0) -> int:
        return gemm_plan_device_status(self.handle, stream)


def matmul(a, b, *, c=None, alpha: float = 1.0, beta: float = 0.0, bias=None,
           bias_mode: int = GEMM_BIAS_COL, relu: bool = False, out=None, out_dtype=None,
           plan: Optional[Plan] = None, stream=None, c_relu: bool = False,
           a_relu: bool = False, a_scale: float = 1.0, b_relu: bool = False, b_scale: float = 1.0):
    """D = epilogue(alpha * t_A(a) @ t_B(b) + beta * c_act(c)) on the GPU for CUDA tensors.

    a: M x K view, b: K x N view (each with unit stride along one dimension;
    the stride decides N/T).  c, out: row-major M x N.  relu / c_relu: ReLU on
    the result / on c as it is read.  a_relu, a_scale (b_relu, b_scale): the
    operand transform t(x) = relu?(scale * x) applied to a (b) after load.
    Returns `out`."""
    import torch
    M, K = a.shape
    K2, N = b.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    la, lda = layout_of(a)
    lb, ldb = layout_of(b)
    c_code = _torch_code(c) if c is not None else (GEMM_S32 if a.dtype == torch.int8 else GEMM_F32)
    if out is None:
        od = out_dtype if out_dtype is not None else (c.dtype if c is not None else
                                                      (torch.int32 if a.dtype == torch.int8 else torch.float32))
        out = torch.empty((M, N), dtype=od, device=a.device)
    if out.stride(1) != 1:
        raise ValueError("out must be row-major")
    if plan is None:
        plan = Plan(_torch_code(a), c_code, a.device.index or 0)
    if stream is None:
        stream = torch.cuda.current_stream(a.device).cuda_stream
    epi = make_epilogue(_torch_code(out), bias.data_ptr() if bias is not None else 0,
                        _torch_code(bias) if bias is not None else GEMM_F32,
                        bias_mode if bias is not None else GEMM_BIAS_NONE,
                        GEMM_ACT_RELU if relu else GEMM_ACT_NONE,
                        GEMM_ACT_RELU if c_relu else GEMM_ACT_NONE,
                        a_act=GEMM_ACT_RELU if a_relu else GEMM_ACT_NONE, a_scale=a_scale,
                        b_act=GEMM_ACT_RELU if b_relu else GEMM_ACT_NONE, b_scale=b_scale)
    cp, ldc = (c.data_ptr(), c.stride(0)) if (c is not None and beta != 0.0) else (None, 0)
    gemm_run(plan.handle, la, lb, M, N, K, alpha, a.data_ptr(), lda, b.data_ptr(), ldb, beta, cp,
             ldc, out.data_ptr(), out.stride(0), epi, stream)
    return out
