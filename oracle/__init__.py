"""CPU oracle of the fused GEMM + epilogue path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The product library (``gemm_epilogue_tmem_gb300``)
never does, and the two share no code: the oracle is plain C in ``oracle.c``
(one function per step of the method) composed here in the order the pages
give the steps.

Sources:
 [P1] "Fusing Matmul Epilogs with nvmath-python": "The problem addressed by
      fused epilogs" (product, bias per output column, ReLU); "Forward-pass
      capabilities in the source" (RELU_BIAS; RELU_AUX_BIAS returns the
      bit-encoded relu_aux mask); "Backward-pass path shown in the example"
      (DRELU_BGRAD = product with the transposed weight, mask applied, then the
      column-wise sum over the batch as the bias gradient).
 [P2] "nvmath-python 封装 cuBLASLt ..." step 1 (fp16 operands, (m,1) bias),
      step 2 (COMPUTE_32F_FAST_16F: fp32 accumulation).

Readings the pages leave open (listed with the rest in the design notes):
relu_aux is packed as column words (bit i%32 of word [i/32][j] is z[i][j] > 0,
padding bits 0); the mask is taken on the fp32 pre-activation, strictly > 0;
the bias gradient sums the fp32 masked product in double; outputs are rounded
to nearest even.

Pins: every function here is checked in ``tests/test_oracle_pins.py`` against
hand-worked examples (``tests/golden/``), library routines (numpy's fp16
conversion, float64 matmul on exactly representable cases), closed forms and
invariants, and fp64 brute force within the recursive-summation error bound.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(_HERE, "liboracle.so")

F16, BF16 = 0, 1
B_KN, B_NK = 0, 1
BIAS_COL, BIAS_ROW = 0, 1


def build_cmd() -> list[str]:
    return ["gcc", "-O3", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread",
            "-o", LIB, os.path.join(_HERE, "oracle.c"), "-lm"]


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(src):
        subprocess.check_call(build_cmd())
    return LIB


_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.oracle_half_to_f32.restype = ctypes.c_float
        L.oracle_half_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_f32.restype = ctypes.c_float
        L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_f32_to_half.restype = ctypes.c_uint16
        L.oracle_f32_to_half.argtypes = [ctypes.c_float]
        L.oracle_f32_to_bf16.restype = ctypes.c_uint16
        L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        L.oracle_decode.argtypes = [_P, _I64, ctypes.c_int, _P]
        L.oracle_round.argtypes = [_P, _I64, ctypes.c_int, _P]
        L.oracle_gemm_f32.argtypes = [_P, _I64, _I64, _P, _I64, ctypes.c_int, _P, ctypes.c_int]
        L.oracle_gemm_f64.argtypes = [_P, _I64, _I64, _P, _I64, ctypes.c_int, _P, ctypes.c_int]
        L.oracle_add_bias.argtypes = [_P, _I64, _I64, _P, ctypes.c_int, _P]
        L.oracle_relu.argtypes = [_P, _I64, _P]
        L.oracle_relu_bits.argtypes = [_P, _I64, _P]
        L.oracle_pack_mask.argtypes = [_P, _I64, _I64, _P]
        L.oracle_mask_bit.restype = ctypes.c_int
        L.oracle_mask_bit.argtypes = [_P, _I64, _I64, _I64]
        L.oracle_drelu.argtypes = [_P, _I64, _I64, _P, _P, _P]
        L.oracle_colsum.argtypes = [_P, _I64, _I64, _P]
        L.oracle_gelu_tanh.restype = ctypes.c_double
        L.oracle_gelu_tanh.argtypes = [ctypes.c_double]
        L.oracle_dgelu_tanh.restype = ctypes.c_double
        L.oracle_dgelu_tanh.argtypes = [ctypes.c_double]
        L.oracle_gelu.argtypes = [_P, _I64, _P]
        L.oracle_dgelu.argtypes = [_P, _P, _I64, _P]
        L.oracle_gelu.restype = None
        L.oracle_dgelu.restype = None
        L.oracle_sigmoid.restype = ctypes.c_double
        L.oracle_sigmoid.argtypes = [ctypes.c_double]
        L.oracle_silu.restype = ctypes.c_double
        L.oracle_silu.argtypes = [ctypes.c_double]
        L.oracle_swiglu.argtypes = [_P, _P, _I64, _P]
        L.oracle_swiglu.restype = None
        L.oracle_dswiglu.argtypes = [_P, _P, _P, _I64, _P, _P]
        L.oracle_dswiglu.restype = None
        for name in ("oracle_decode", "oracle_round", "oracle_gemm_f32", "oracle_gemm_f64",
                     "oracle_add_bias", "oracle_relu", "oracle_relu_bits", "oracle_pack_mask",
                     "oracle_drelu", "oracle_colsum"):
            getattr(L, name).restype = None
        _lib = L
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _bits(a: np.ndarray) -> np.ndarray:
    """fp16 arrays or uint16 bit arrays -> contiguous uint16 bits."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ------------------------------------------------------------------ formats
def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    """fp16/bf16 bits -> exact fp32 values."""
    b = _bits(bits)
    out = np.empty(b.shape, dtype=np.float32)
    lib().oracle_decode(b.ctypes.data, b.size, dtype, out.ctypes.data)
    return out


def round_to(x: np.ndarray, dtype: int) -> np.ndarray:
    """fp32 -> fp16/bf16 bits (uint16), round to nearest even."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_round(x.ctypes.data, x.size, dtype, out.ctypes.data)
    return out


# --------------------------------------------------------------------- GEMM
def gemm(A: np.ndarray, B: np.ndarray, dtype: int, b_layout: int = B_KN,
         nthreads: int | None = None) -> np.ndarray:
    """acc[r][n] = sum_p A[r][p] B[p][n] in fp32, ascending p ([P2] step 2).

    A: [R, K] fp16/bf16 bits; B: [K, N] (B_KN) or [N, K] (B_NK) bits.
    """
    Af = decode(A, dtype)
    Bf = decode(B, dtype)
    R, K = Af.shape
    N = Bf.shape[1] if b_layout == B_KN else Bf.shape[0]
    assert (Bf.shape[0] if b_layout == B_KN else Bf.shape[1]) == K
    acc = np.empty((R, N), dtype=np.float32)
    lib().oracle_gemm_f32(Af.ctypes.data, R, K, Bf.ctypes.data, N, b_layout, acc.ctypes.data,
                          nthreads or default_threads())
    return acc


def gemm64(A: np.ndarray, B: np.ndarray, dtype: int, b_layout: int = B_KN,
           nthreads: int | None = None) -> np.ndarray:
    """Brute-force reference: exact products summed in double."""
    Af = decode(A, dtype)
    Bf = decode(B, dtype)
    R, K = Af.shape
    N = Bf.shape[1] if b_layout == B_KN else Bf.shape[0]
    acc = np.empty((R, N), dtype=np.float64)
    lib().oracle_gemm_f64(Af.ctypes.data, R, K, Bf.ctypes.data, N, b_layout, acc.ctypes.data,
                          nthreads or default_threads())
    return acc


# ---------------------------------------------------------------- epilogue steps
def add_bias(acc: np.ndarray, bias: np.ndarray, dtype: int, axis: int,
             row_ids: np.ndarray | None = None) -> np.ndarray:
    """z = acc + bias in fp32; COL: bias[n] per column, ROW: bias[m] per row."""
    z = _c(acc, np.float32).copy()
    bf = decode(np.ravel(bias), dtype)
    R, N = z.shape
    rid = None if row_ids is None else _c(row_ids, np.int64)
    if axis == BIAS_COL:
        assert bf.size == N
    else:
        assert bf.size >= (int(rid.max()) + 1 if rid is not None and rid.size else R)
    lib().oracle_add_bias(z.ctypes.data, R, N, bf.ctypes.data, axis,
                          rid.ctypes.data if rid is not None else None)
    return z


def relu(z: np.ndarray) -> np.ndarray:
    z = _c(z, np.float32)
    y = np.empty_like(z)
    lib().oracle_relu(z.ctypes.data, z.size, y.ctypes.data)
    return y


def relu_bits(z: np.ndarray) -> np.ndarray:
    z = _c(z, np.float32)
    b = np.empty(z.shape, dtype=np.uint8)
    lib().oracle_relu_bits(z.ctypes.data, z.size, b.ctypes.data)
    return b


def pack_mask(bits: np.ndarray) -> np.ndarray:
    """bits [M, N] -> column words uint32 [ceil(M/32), N]."""
    b = _c(bits, np.uint8)
    M, N = b.shape
    w = np.empty(((M + 31) // 32, N), dtype=np.uint32)
    lib().oracle_pack_mask(b.ctypes.data, M, N, w.ctypes.data)
    return w


def mask_bit(words: np.ndarray, i: int, j: int) -> int:
    w = _c(words, np.uint32)
    return int(lib().oracle_mask_bit(w.ctypes.data, w.shape[1], i, j))


def drelu(g: np.ndarray, words: np.ndarray, row_ids: np.ndarray | None = None) -> np.ndarray:
    """dz = g where the forward ReLU mask bit is set, else 0 (fp32)."""
    g = _c(g, np.float32)
    w = _c(words, np.uint32)
    R, N = g.shape
    assert w.shape[1] == N
    rid = None if row_ids is None else _c(row_ids, np.int64)
    dz = np.empty_like(g)
    lib().oracle_drelu(g.ctypes.data, R, N, rid.ctypes.data if rid is not None else None,
                       w.ctypes.data, dz.ctypes.data)
    return dz


def colsum(dz: np.ndarray) -> np.ndarray:
    """Column sums over the batch (rows), in double, ascending rows."""
    dz = _c(dz, np.float32)
    M, N = dz.shape
    out = np.empty(N, dtype=np.float64)
    lib().oracle_colsum(dz.ctypes.data, M, N, out.ctypes.data)
    return out


# ---------------------------------------------------------------- epilogs
def epilog_none(A, B, dtype, b_layout=B_KN, nthreads=None):
    """out = round(A B)."""
    return round_to(gemm(A, B, dtype, b_layout, nthreads), dtype)


def relu_bias(A, B, bias, dtype, b_layout=B_KN, axis=BIAS_COL, row_ids=None, nthreads=None):
    """RELU_BIAS ([P1] "The problem addressed by fused epilogs"):
    Y = round(ReLU(A B + bias)). Returns (Y bits, z fp32).

    A holds rows ``row_ids`` of the full left operand when given (ROW bias
    and mask rows follow the global row index)."""
    acc = gemm(A, B, dtype, b_layout, nthreads)
    z = add_bias(acc, bias, dtype, axis, row_ids)
    y = round_to(relu(z), dtype)
    return y, z


def relu_aux_bias(A, B, bias, dtype, b_layout=B_KN, axis=BIAS_COL, nthreads=None):
    """RELU_AUX_BIAS ([P1] "Forward-pass capabilities in the source"):
    RELU_BIAS plus relu_aux, the packed mask of z > 0. Full M only.
    Returns (Y bits, aux words, z fp32)."""
    y, z = relu_bias(A, B, bias, dtype, b_layout, axis, None, nthreads)
    return y, pack_mask(relu_bits(z)), z


def drelu_bgrad(G_A, G_B, words, dtype, b_layout=B_NK, row_ids=None, nthreads=None):
    """DRELU_BGRAD ([P1] "Backward-pass path shown in the example"):
    g = G_A G_B (e.g. dY W^T); dz = g masked by relu_aux; out = round(dz);
    bgrad = column sums of dz over the batch (only when all rows are given).
    Returns (dz bits, bgrad fp32 or None, g fp32)."""
    g = gemm(G_A, G_B, dtype, b_layout, nthreads)
    dz = drelu(g, words, row_ids)
    out = round_to(dz, dtype)
    bgrad = colsum(dz).astype(np.float32) if row_ids is None else None
    return out, bgrad, g


# ------------------------------------------------------------------ GELU
def gelu_scalar(z: float) -> float:
    return float(lib().oracle_gelu_tanh(z))


def dgelu_scalar(z: float) -> float:
    return float(lib().oracle_dgelu_tanh(z))


def gelu(z: np.ndarray) -> np.ndarray:
    """tanh-form GELU (Hendrycks & Gimpel 2016), in double, stored as fp32."""
    z = _c(z, np.float32)
    y = np.empty_like(z)
    lib().oracle_gelu(z.ctypes.data, z.size, y.ctypes.data)
    return y


def dgelu(g: np.ndarray, z: np.ndarray) -> np.ndarray:
    """dz = g * gelu'(z) (double, stored as fp32)."""
    g = _c(g, np.float32)
    z = _c(z, np.float32)
    assert g.shape == z.shape
    dz = np.empty_like(g)
    lib().oracle_dgelu(g.ctypes.data, z.ctypes.data, g.size, dz.ctypes.data)
    return dz


def gelu_bias(A, B, bias, dtype, b_layout=B_KN, axis=BIAS_COL, row_ids=None, nthreads=None):
    """GELU_BIAS (nvmath-python / cuBLASLt page, "other epilogs"):
    Y = round(GELU(A B + bias)). Returns (Y bits, z fp32)."""
    acc = gemm(A, B, dtype, b_layout, nthreads)
    z = add_bias(acc, bias, dtype, axis, row_ids)
    return round_to(gelu(z), dtype), z


def gelu_aux_bias(A, B, bias, dtype, b_layout=B_KN, axis=BIAS_COL, row_ids=None, nthreads=None):
    """GELU_AUX_BIAS: GELU_BIAS plus the pre-activation z saved in the
    operand dtype for the backward. Returns (Y bits, aux bits, z fp32)."""
    y, z = gelu_bias(A, B, bias, dtype, b_layout, axis, row_ids, nthreads)
    return y, round_to(z, dtype), z


def dgelu_bgrad(G_A, G_B, aux, dtype, b_layout=B_NK, full_rows=True, nthreads=None):
    """DGELU_BGRAD: g = G_A G_B; dz = g * gelu'(z) with z the saved
    pre-activation (aux bits of dtype, same rows as G_A); out = round(dz);
    bgrad = column sums of dz over the batch (when all rows are given)."""
    g = gemm(G_A, G_B, dtype, b_layout, nthreads)
    z = decode(aux, dtype)
    dz = dgelu(g, z)
    out = round_to(dz, dtype)
    bgrad = colsum(dz).astype(np.float32) if full_rows else None
    return out, bgrad, g


# ---------------------------------------------------------------- SwiGLU
def sigmoid_scalar(g: float) -> float:
    return float(lib().oracle_sigmoid(g))


def silu_scalar(g: float) -> float:
    return float(lib().oracle_silu(g))


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """h = silu(g) * u (double, stored as fp32)."""
    g = _c(g, np.float32)
    u = _c(u, np.float32)
    assert g.shape == u.shape
    h = np.empty_like(g)
    lib().oracle_swiglu(g.ctypes.data, u.ctypes.data, g.size, h.ctypes.data)
    return h


def dswiglu(dh: np.ndarray, g: np.ndarray, u: np.ndarray):
    """(d_gate, d_up) of h = silu(g) * u applied to dh (double, stored fp32)."""
    dh = _c(dh, np.float32)
    g = _c(g, np.float32)
    u = _c(u, np.float32)
    assert dh.shape == g.shape == u.shape
    dg = np.empty_like(dh)
    du = np.empty_like(dh)
    lib().oracle_dswiglu(dh.ctypes.data, g.ctypes.data, u.ctypes.data, dh.size, dg.ctypes.data,
                         du.ctypes.data)
    return dg, du


def swiglu_forward(x, Wg, Wu, dtype, nthreads=None):
    """The fused gate+up forward of gemm_swiglu_mlp_fusion.py (docstring):
    g = x Wg^T, u = x Wu^T (Wg, Wu stored [I, H]: B_NK), h = silu(g) * u.
    Returns (h bits, g bits, u bits, g fp32, u fp32); g and u rounded are
    what the forward saves for the backward."""
    g = gemm(x, Wg, dtype, B_NK, nthreads)
    u = gemm(x, Wu, dtype, B_NK, nthreads)
    h = round_to(swiglu(g, u), dtype)
    return h, round_to(g, dtype), round_to(u, dtype), g, u


def dswiglu_backward(dout, Wd, g_bits, u_bits, dtype, nthreads=None):
    """dh = dout Wd (Wd stored [H, I]: B_KN), then the dSwiGLU of the saved
    g, u as its epilogue (gemm_swiglu_mlp_fusion.py, docstring).
    Returns (d_gate bits, d_up bits, dh fp32)."""
    dh = gemm(dout, Wd, dtype, B_KN, nthreads)
    dg, du = dswiglu(dh, decode(g_bits, dtype), decode(u_bits, dtype))
    return round_to(dg, dtype), round_to(du, dtype), dh
