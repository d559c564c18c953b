"""Python binding of libgf.so, the fused GEMM + epilogue library for GB300.

Argument marshalling only: every step of the path runs in the CUDA kernels
behind the C ABI declared in ``include/gf.h``. The functions keep the C names
(``gf_matmul_plan``, ``gf_matmul_execute``, ``gf_plan_free`` ...) and take
either torch tensors (device memory) or raw integer device pointers. There is
no CPU fallback: importing works without a GPU, but the library must be built
(``build()``) and every call fails loudly when it is missing.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB, build

__all__ = [
    "GF_OK", "GF_ERR_INVALID_VALUE", "GF_ERR_UNSUPPORTED", "GF_ERR_NO_DEVICE", "GF_ERR_CUDA",
    "GF_ERR_OUT_OF_MEMORY", "GF_ERR_DEVICE_TIMEOUT",
    "GF_F16", "GF_BF16",
    "GF_EPILOG_NONE", "GF_EPILOG_RELU_BIAS", "GF_EPILOG_RELU_AUX_BIAS", "GF_EPILOG_DRELU_BGRAD",
    "GF_EPILOG_BIAS", "GF_EPILOG_GELU_BIAS", "GF_EPILOG_GELU_AUX_BIAS", "GF_EPILOG_DGELU_BGRAD",
    "GF_BIAS_COL", "GF_BIAS_ROW", "GF_B_KN", "GF_B_NK", "GF_BGRAD_TWO_PASS", "GF_BGRAD_ATOMIC",
    "GF_OPT_BGRAD_MODE", "GF_OPT_WAIT_LIMIT_US", "GF_OPT_TILE_N", "GF_OPT_FAULT_DROP_LOAD",
    "GF_OPT_KERNEL", "GF_OPT_GROUP_M", "GF_OPT_L2_HINTS", "GF_OPT_SCHEDULE", "GF_OPT_SPLIT_K",
    "GF_OPT_PDL", "GF_OPT_RASTER",
    "GfError", "Plan", "build", "lib", "gf_matmul_plan", "gf_matmul_plan_ex",
    "gf_matmul_execute", "gf_plan_status", "gf_plan_set_option", "gf_plan_describe",
    "gf_plan_free", "gf_status_string", "gf_last_error", "gf_drelu_bgrad_noalloc",
    "gf_noalloc_status",
    "gf_swiglu_plan", "gf_swiglu_execute", "gf_dswiglu_plan", "gf_dswiglu_execute",
    "GF_NOALLOC_MAX_PARTIALS",
]

# gf_status
GF_OK, GF_ERR_INVALID_VALUE, GF_ERR_UNSUPPORTED, GF_ERR_NO_DEVICE = 0, 1, 2, 3
GF_ERR_CUDA, GF_ERR_OUT_OF_MEMORY, GF_ERR_DEVICE_TIMEOUT = 4, 5, 6
# gf_dtype
GF_F16, GF_BF16 = 0, 1
# gf_epilog
GF_EPILOG_NONE, GF_EPILOG_RELU_BIAS, GF_EPILOG_RELU_AUX_BIAS = 0, 1, 2
GF_EPILOG_DRELU_BGRAD, GF_EPILOG_BIAS = 3, 4
GF_EPILOG_GELU_BIAS, GF_EPILOG_GELU_AUX_BIAS, GF_EPILOG_DGELU_BGRAD = 5, 6, 7
# gf_bias_axis, gf_b_layout, gf_bgrad_mode
GF_BIAS_COL, GF_BIAS_ROW = 0, 1
GF_B_KN, GF_B_NK = 0, 1
GF_BGRAD_TWO_PASS, GF_BGRAD_ATOMIC = 0, 1
# gf_option
GF_OPT_BGRAD_MODE, GF_OPT_WAIT_LIMIT_US, GF_OPT_TILE_N, GF_OPT_FAULT_DROP_LOAD = 0, 1, 2, 3
GF_OPT_KERNEL, GF_OPT_GROUP_M, GF_OPT_L2_HINTS, GF_OPT_SCHEDULE = 4, 5, 6, 7
GF_OPT_SPLIT_K, GF_OPT_PDL, GF_OPT_RASTER = 8, 9, 10
# fp32 partial sums the allocation-free DRELU_BGRAD entry point can hold
GF_NOALLOC_MAX_PARTIALS = 2097152


class GfError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {gf_status_string(status)}")


_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int


def lib(path: str | None = None):
    """Load libgf.so (built in-tree by ``build()``); raise if it is missing."""
    global _lib
    if _lib is None:
        p = path or LIB
        if not os.path.exists(p):
            raise RuntimeError(
                f"libgf.so not found at {p}: build it with gemm_epilogue_tmem_gb300.build()")
        L = ctypes.CDLL(p)
        L.gf_matmul_plan.restype = _P
        L.gf_matmul_plan.argtypes = [_I64, _I64, _I64, _I32, _I32, _I32]
        L.gf_matmul_plan_ex.restype = _P
        L.gf_matmul_plan_ex.argtypes = [_I64, _I64, _I64, _I32, _I32, _I32, _I32]
        L.gf_matmul_execute.restype = _I32
        L.gf_matmul_execute.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P]
        L.gf_plan_status.restype = _I32
        L.gf_plan_status.argtypes = [_P, _P]
        L.gf_plan_set_option.restype = _I32
        L.gf_plan_set_option.argtypes = [_P, _I32, _I64]
        L.gf_plan_describe.restype = _I32
        L.gf_plan_describe.argtypes = [_P, _P, _P, _P, _P, _P]
        L.gf_plan_k_splits.restype = _I32
        L.gf_plan_k_splits.argtypes = [_P, _P]
        L.gf_plan_launches.restype = _I32
        L.gf_plan_launches.argtypes = [_P, _P]
        L.gf_plan_free.restype = None
        L.gf_plan_free.argtypes = [_P]
        L.gf_status_string.restype = ctypes.c_char_p
        L.gf_status_string.argtypes = [_I32]
        L.gf_last_error.restype = _I32
        L.gf_last_error.argtypes = []
        L.gf_swiglu_plan.restype = _P
        L.gf_swiglu_plan.argtypes = [_I64, _I64, _I64, _I32, _I32]
        L.gf_swiglu_execute.restype = _I32
        L.gf_swiglu_execute.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P]
        L.gf_dswiglu_plan.restype = _P
        L.gf_dswiglu_plan.argtypes = [_I64, _I64, _I64, _I32]
        L.gf_dswiglu_execute.restype = _I32
        L.gf_dswiglu_execute.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P]
        L.gf_matmul_autotune.restype = _I32
        L.gf_matmul_autotune.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I32]
        L.gf_drelu_bgrad_noalloc.restype = _I32
        L.gf_drelu_bgrad_noalloc.argtypes = [_I64, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _P, _P]
        L.gf_noalloc_status.restype = _I32
        L.gf_noalloc_status.argtypes = [_P]
        _lib = L
    return _lib


def _ptr(x) -> int | None:
    """torch tensor / int / None -> device address (or NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """Owns a gf_plan* and frees it when collected (or on ``free()``)."""

    def __init__(self, handle: int, m: int, n: int, k: int, dtype: int, epilog: int,
                 bias_axis: int, b_layout: int):
        self.handle = handle
        self.m, self.n, self.k = m, n, k
        self.dtype, self.epilog, self.bias_axis, self.b_layout = dtype, epilog, bias_axis, b_layout

    def free(self) -> None:
        if self.handle:
            lib().gf_plan_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def gf_status_string(status: int) -> str:
    return lib().gf_status_string(status).decode()


def gf_last_error() -> int:
    return int(lib().gf_last_error())


def gf_matmul_plan_ex(m: int, n: int, k: int, dtype: int, epilog: int, bias_axis: int = GF_BIAS_COL,
                      b_layout: int = GF_B_KN) -> Plan:
    h = lib().gf_matmul_plan_ex(m, n, k, dtype, epilog, bias_axis, b_layout)
    if not h:
        raise GfError(gf_last_error(), "gf_matmul_plan_ex")
    return Plan(h, m, n, k, dtype, epilog, bias_axis, b_layout)


def gf_matmul_plan(m: int, n: int, k: int, dtype: int, epilog: int,
                   bias_axis: int = GF_BIAS_COL) -> Plan:
    h = lib().gf_matmul_plan(m, n, k, dtype, epilog, bias_axis)
    if not h:
        raise GfError(gf_last_error(), "gf_matmul_plan")
    return Plan(h, m, n, k, dtype, epilog, bias_axis, GF_B_KN)


def gf_matmul_execute(plan: Plan, A, B, bias=None, out=None, aux_in=None, aux_out=None,
                      bgrad=None, stream=None) -> None:
    """Enqueue the planned GEMM + epilogue; raises GfError on a non-OK status."""
    rc = lib().gf_matmul_execute(plan.handle, _ptr(A), _ptr(B), _ptr(bias), _ptr(out),
                                 _ptr(aux_in), _ptr(aux_out), _ptr(bgrad), _stream(stream))
    if rc != GF_OK:
        raise GfError(rc, "gf_matmul_execute")


def gf_matmul_autotune(plan: Plan, A, B, bias=None, out=None, aux_in=None, aux_out=None,
                       bgrad=None, stream=None, reps: int = 3) -> dict:
    """Time the library's kernel/tile/schedule candidates on these buffers,
    keep the fastest in the plan and return its description."""
    rc = lib().gf_matmul_autotune(plan.handle, _ptr(A), _ptr(B), _ptr(bias), _ptr(out),
                                  _ptr(aux_in), _ptr(aux_out), _ptr(bgrad), _stream(stream), reps)
    if rc != GF_OK:
        raise GfError(rc, "gf_matmul_autotune")
    return gf_plan_describe(plan)


def gf_swiglu_plan(m: int, n: int, k: int, dtype: int, save_gu: bool = False) -> Plan:
    """Gate+up SwiGLU forward plan: h[m, n] = silu(x Wg^T) * (x Wu^T), x [m, k]."""
    h = lib().gf_swiglu_plan(m, n, k, dtype, 1 if save_gu else 0)
    if not h:
        raise GfError(gf_last_error(), "gf_swiglu_plan")
    return Plan(h, m, n, k, dtype, -1, GF_BIAS_COL, GF_B_NK)


def gf_swiglu_execute(plan: Plan, x, Wg, Wu, h, g_out=None, u_out=None, stream=None) -> None:
    rc = lib().gf_swiglu_execute(plan.handle, _ptr(x), _ptr(Wg), _ptr(Wu), _ptr(h), _ptr(g_out),
                                 _ptr(u_out), _stream(stream))
    if rc != GF_OK:
        raise GfError(rc, "gf_swiglu_execute")


def gf_dswiglu_plan(m: int, n: int, k: int, dtype: int) -> Plan:
    """dSwiGLU backward plan: dh = dout Wd with the dSwiGLU as its epilogue."""
    h = lib().gf_dswiglu_plan(m, n, k, dtype)
    if not h:
        raise GfError(gf_last_error(), "gf_dswiglu_plan")
    return Plan(h, m, n, k, dtype, -2, GF_BIAS_COL, GF_B_KN)


def gf_dswiglu_execute(plan: Plan, dout, Wd, g, u, d_gate, d_up, stream=None) -> None:
    rc = lib().gf_dswiglu_execute(plan.handle, _ptr(dout), _ptr(Wd), _ptr(g), _ptr(u),
                                  _ptr(d_gate), _ptr(d_up), _stream(stream))
    if rc != GF_OK:
        raise GfError(rc, "gf_dswiglu_execute")


def gf_plan_status(plan: Plan, stream=None) -> int:
    """Synchronise the stream and return the plan's status (GF_OK, GF_ERR_DEVICE_TIMEOUT ...)."""
    return int(lib().gf_plan_status(plan.handle, _stream(stream)))


def gf_plan_set_option(plan: Plan, option: int, value: int) -> None:
    rc = lib().gf_plan_set_option(plan.handle, option, value)
    if rc != GF_OK:
        raise GfError(rc, "gf_plan_set_option")


def gf_plan_describe(plan: Plan) -> dict:
    vals = [ctypes.c_int32() for _ in range(4)]
    ws = ctypes.c_int64()
    rc = lib().gf_plan_describe(plan.handle, *(ctypes.byref(v) for v in vals), ctypes.byref(ws))
    if rc != GF_OK:
        raise GfError(rc, "gf_plan_describe")
    ks = ctypes.c_int32()
    rc = lib().gf_plan_k_splits(plan.handle, ctypes.byref(ks))
    if rc != GF_OK:
        raise GfError(rc, "gf_plan_k_splits")
    nl = ctypes.c_int32()
    rc = lib().gf_plan_launches(plan.handle, ctypes.byref(nl))
    if rc != GF_OK:
        raise GfError(rc, "gf_plan_launches")
    return {"tile_m": vals[0].value, "tile_n": vals[1].value, "stages": vals[2].value,
            "grid": vals[3].value, "workspace_bytes": ws.value, "k_splits": ks.value,
            "launches": nl.value}


def gf_plan_free(plan: Plan) -> None:
    plan.free()


def gf_drelu_bgrad_noalloc(m: int, n: int, k: int, dtype: int, b_layout: int, A, B, out, aux_in,
                           bgrad, stream=None) -> None:
    """DRELU_BGRAD without any device allocation (fixed scratch inside the
    library; see include/gf.h). Raises GfError on a non-OK status."""
    rc = lib().gf_drelu_bgrad_noalloc(m, n, k, dtype, b_layout, _ptr(A), _ptr(B), _ptr(out),
                                      _ptr(aux_in), _ptr(bgrad), _stream(stream))
    if rc != GF_OK:
        raise GfError(rc, "gf_drelu_bgrad_noalloc")


def gf_noalloc_status(stream=None) -> int:
    """Synchronise the stream and return the status of the most recent
    gf_drelu_bgrad_noalloc on this device (GF_OK, GF_ERR_DEVICE_TIMEOUT ...)."""
    return int(lib().gf_noalloc_status(_stream(stream)))
