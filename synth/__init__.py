"""Seeded synthetic inputs for the fused GEMM + epilogue tests and benchmark.

This module is the one thing the CPU oracle and the CUDA path share: it makes
inputs and holds none of the method's arithmetic. The generator is defined in
``synth_hash.h`` (SplitMix64 counter hash; N(0, sigma) as a scaled Irwin-Hall
sum of eight 16-bit uniforms; Bernoulli(1/2) mask words) and has a host filler
(``libsynth_host.so``, plain C) and a device filler (``libsynth_cuda.so``) that
produce identical bits, so any row of a large device tensor can be regenerated
alone on the host.

The workload recipes below restate the shapes and spreads of the workloads on
the pages (fp16 (65536,16384)x(16384,8192) linear layer pair on "Fusing Matmul
Epilogs with nvmath-python", section "Suitable evaluation scenarios"; the
(m,n,k) = (1024,512,2048) RELU_BIAS example with a (m,1) bias on the
nvmath-python/cuBLASLt page, step 1; the SwiGLU MLP shape H=5120, I=17408 with
0.02-scaled weights in gemm_swiglu_mlp_fusion.py, ``_demo``).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(_HERE, "libsynth_host.so")
CUDA_LIB = os.path.join(_HERE, "libsynth_cuda.so")

F16, BF16, F32 = 0, 1, 2

# fixed tensor ids, one per role
TID_A, TID_B, TID_BIAS, TID_DY, TID_MASK = 1, 2, 3, 4, 5
TID_W2, TID_B2 = 6, 7
TID_WG, TID_WU, TID_WD, TID_DOUT = 8, 9, 10, 11
TID_PREACT = 12
TID_G_SAVED, TID_U_SAVED = 13, 14
TID_SAMPLE = 100
TID_SAMPLE_COL = 101  # sampled columns (bias-gradient checks)


def build_host(force: bool = False) -> str:
    src = [os.path.join(_HERE, "synth_host.c")]
    if force or not os.path.exists(HOST_LIB) or os.path.getmtime(HOST_LIB) < max(
        os.path.getmtime(p) for p in src + [os.path.join(_HERE, "synth_hash.h")]
    ):
        subprocess.check_call(
            ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", HOST_LIB, *src, "-lm"]
        )
    return HOST_LIB


def cuda_build_cmd() -> list[str]:
    return [
        "nvcc", "-O3", "-shared", "-Xcompiler", "-fPIC,-ffp-contract=off",
        "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
        "-o", CUDA_LIB,
        os.path.join(_HERE, "synth_cuda.cu"), os.path.join(_HERE, "synth_host.c"),
    ]


def build_cuda(force: bool = False) -> str:
    srcs = [os.path.join(_HERE, f) for f in ("synth_cuda.cu", "synth_host.c", "synth_hash.h")]
    if force or not os.path.exists(CUDA_LIB) or os.path.getmtime(CUDA_LIB) < max(
        os.path.getmtime(p) for p in srcs
    ):
        subprocess.check_call(cuda_build_cmd())
    return CUDA_LIB


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        lib = ctypes.CDLL(build_host())
        lib.synth_scale.restype = ctypes.c_float
        lib.synth_scale.argtypes = [ctypes.c_double]
        lib.synth_fill_normal.restype = None
        lib.synth_fill_normal.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_uint64, ctypes.c_uint32, ctypes.c_double,
        ]
        lib.synth_fill_mask_words.restype = None
        lib.synth_fill_mask_words.argtypes = [
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_uint64, ctypes.c_uint32,
        ]
        lib.synth_sample_rows.restype = None
        lib.synth_sample_rows.argtypes = [
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
        ]
        lib.synth_hash.restype = ctypes.c_uint64
        lib.synth_hash.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64]
        lib.synth_mix.restype = ctypes.c_uint64
        lib.synth_mix.argtypes = [ctypes.c_uint64]
        lib.synth_irwin_hall.restype = ctypes.c_int32
        lib.synth_irwin_hall.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64]
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        lib = ctypes.CDLL(build_cuda())
        lib.synth_dev_fill_normal.restype = ctypes.c_int
        lib.synth_dev_fill_normal.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
            ctypes.c_uint32, ctypes.c_double, ctypes.c_void_p,
        ]
        lib.synth_dev_fill_mask_words.restype = ctypes.c_int
        lib.synth_dev_fill_mask_words.argtypes = [
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
            ctypes.c_void_p,
        ]
        _dev = lib
    return _dev


# ---------------------------------------------------------------- host side
def hash64(seed: int, tensor_id: int, index: int) -> int:
    return int(_host_lib().synth_hash(seed, tensor_id, index))


def mix64(z: int) -> int:
    return int(_host_lib().synth_mix(z))


def irwin_hall(seed: int, tensor_id: int, element: int) -> int:
    return int(_host_lib().synth_irwin_hall(seed, tensor_id, element))


def scale(sigma: float) -> float:
    return float(_host_lib().synth_scale(sigma))


def normal(shape, dtype: int, seed: int, tensor_id: int, sigma: float, rows=None) -> np.ndarray:
    """Host draw of a [R, C] tensor (or of the given logical rows of it).

    fp16 -> np.float16 array; bf16 -> np.uint16 array of bf16 bits;
    fp32 -> np.float32 array.
    """
    if len(shape) == 1:
        shape = (1, shape[0])
        squeeze = True
    else:
        squeeze = False
    R, C = shape
    if rows is not None:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        assert rows.ndim == 1 and (rows.size == 0 or (rows.min() >= 0 and rows.max() < R))
        n = rows.size
    else:
        n = R
    np_dtype = {F16: np.float16, BF16: np.uint16, F32: np.float32}[dtype]
    out = np.empty((n, C), dtype=np_dtype)
    _host_lib().synth_fill_normal(
        out.ctypes.data, dtype, C, rows.ctypes.data if rows is not None else None, n,
        seed, tensor_id, sigma,
    )
    return out.reshape(C) if squeeze else out


def mask_words(M: int, N: int, seed: int, tensor_id: int = TID_MASK, word_rows=None) -> np.ndarray:
    """Host draw of the Bernoulli(1/2) column-word mask, uint32 [ceil(M/32), N]."""
    nw_total = (M + 31) // 32
    if word_rows is not None:
        word_rows = np.ascontiguousarray(np.asarray(word_rows, dtype=np.int64))
        assert word_rows.size == 0 or (word_rows.min() >= 0 and word_rows.max() < nw_total)
        n = word_rows.size
    else:
        n = nw_total
    out = np.empty((n, N), dtype=np.uint32)
    _host_lib().synth_fill_mask_words(
        out.ctypes.data, M, N, word_rows.ctypes.data if word_rows is not None else None, n,
        seed, tensor_id,
    )
    return out


def sample_rows(M: int, count: int, seed: int) -> np.ndarray:
    """Sorted distinct rows drawn as h(t) mod M, t = 0..count-1."""
    out = np.empty(count, dtype=np.int64)
    _host_lib().synth_sample_rows(out.ctypes.data, count, M, seed, TID_SAMPLE)
    return np.unique(out)


def sample_cols(N: int, count: int, seed: int) -> np.ndarray:
    """Sorted distinct columns drawn as h(t) mod N from their own stream."""
    out = np.empty(count, dtype=np.int64)
    _host_lib().synth_sample_rows(out.ctypes.data, count, N, seed, TID_SAMPLE_COL)
    return np.unique(out)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


# -------------------------------------------------------------- device side
def dev_normal(tensor, dtype: int, seed: int, tensor_id: int, sigma: float, stream=0) -> None:
    """Fill a contiguous CUDA tensor (viewed as [rows, cols]) in place."""
    assert tensor.is_cuda and tensor.is_contiguous()
    cols = tensor.shape[-1] if tensor.dim() > 0 else 1
    rows = tensor.numel() // max(cols, 1)
    rc = _dev_lib().synth_dev_fill_normal(
        tensor.data_ptr(), dtype, rows, cols, seed, tensor_id, sigma, stream
    )
    if rc != 0:
        raise RuntimeError(f"synth_dev_fill_normal failed with CUDA error {rc}")


def dev_mask_words(tensor, M: int, N: int, seed: int, tensor_id: int = TID_MASK, stream=0) -> None:
    assert tensor.is_cuda and tensor.is_contiguous() and tensor.numel() == ((M + 31) // 32) * N
    rc = _dev_lib().synth_dev_fill_mask_words(tensor.data_ptr(), M, N, seed, tensor_id, stream)
    if rc != 0:
        raise RuntimeError(f"synth_dev_fill_mask_words failed with CUDA error {rc}")


# ------------------------------------------------------------------ recipes
@dataclass(frozen=True)
class Tensor:
    name: str
    shape: tuple
    tensor_id: int
    sigma: float = 1.0
    kind: str = "normal"  # "normal" | "mask"


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: int
    seeds: tuple
    tensors: dict = field(default_factory=dict)
    note: str = ""


def _t(name, shape, tid, sigma=1.0, kind="normal"):
    return name, Tensor(name, tuple(shape), tid, sigma, kind)


MLP_TINY = Workload(
    "mlp2_relu_tiny", F16, (0,),
    dict([
        _t("X", (256, 512), TID_A),
        _t("W1", (512, 384), TID_B, 1 / math.sqrt(512)),
        _t("b1", (384,), TID_BIAS, 0.1),
        _t("W2", (384, 128), TID_W2, 1 / math.sqrt(384)),
        _t("b2", (128,), TID_B2, 0.1),
        _t("dY", (256, 128), TID_DY),
    ]),
    "2-layer ReLU MLP step: layer-1 forward RELU_AUX_BIAS, backward DRELU_BGRAD of G = dY W2^T",
)

RELU_BIAS_ROW = Workload(
    "relu_bias_rowbias_1024x512x2048", F16, (0, 1, 2, 3, 4),
    dict([
        _t("A", (1024, 2048), TID_A),
        _t("B", (2048, 512), TID_B),
        _t("bias", (1024,), TID_BIAS),
    ]),
    "single RELU_BIAS GEMM with a per-row (m,1) bias",
)

LINEAR_PAIR_LARGE = Workload(
    "linear_pair_65536x16384x8192", F16, (0,),
    dict([
        _t("X", (65536, 16384), TID_A),
        _t("W", (16384, 8192), TID_B, 1 / 128),
        _t("bias", (8192,), TID_BIAS, 0.1),
        _t("dY", (65536, 8192), TID_DY),
        _t("mask", (65536, 16384), TID_MASK, kind="mask"),
    ]),
    "forward RELU_AUX_BIAS X.W + bias; backward DRELU_BGRAD dY.W^T with a Bernoulli(1/2) mask",
)

GELU_BIAS = Workload(
    "gelu_bias_8192x16384x4096", BF16, (0,),
    dict([
        _t("X", (8192, 4096), TID_A),
        _t("W", (4096, 16384), TID_B, 1 / 64),
        _t("bias", (16384,), TID_BIAS, 0.1),
        _t("dY", (8192, 16384), TID_DY),
        _t("preact", (8192, 4096), TID_PREACT),
    ]),
    "forward GELU_AUX_BIAS; backward DGELU_BGRAD of dY.W^T against a synthetic pre-activation",
)


def swiglu(M: int) -> Workload:
    return Workload(
        f"swiglu_mlp_M{M}_H5120_I17408", BF16, (0,),
        dict([
            _t("x", (M, 5120), TID_A),
            _t("Wg", (17408, 5120), TID_WG, 0.02),
            _t("Wu", (17408, 5120), TID_WU, 0.02),
            _t("Wd", (5120, 17408), TID_WD, 0.02),
            _t("dout", (M, 5120), TID_DOUT),
        ]),
        "gate+up SwiGLU forward, down GEMM, dSwiGLU backward epilogue",
    )
