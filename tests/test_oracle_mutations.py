"""The oracle's pins are discriminating: each test plants one plausible
mistake in a step of the CPU oracle (a dropped term, a wrong sign, axis or
bit index, a transposed operand, another rounding or summation order) by
replacing that step in the ``oracle`` module for the duration of the test, and
checks that every pin listed for it fails. The pins are first run on the
unmodified oracle, where they must pass. Nothing here touches a GPU."""
import math

import numpy as np
import pytest

import oracle
import test_oracle_gelu_pins as G
import test_oracle_pins as P

torch = pytest.importorskip("torch")
import test_oracle_swiglu_pins as S  # noqa: E402  (needs torch)

_orig = {name: getattr(oracle, name) for name in (
    "gemm", "gemm64", "decode", "round_to", "add_bias", "relu", "relu_bits", "pack_mask", "drelu",
    "colsum", "gelu", "dgelu", "gelu_scalar", "dgelu_scalar", "silu_scalar", "swiglu",
    "dswiglu")}


# ------------------------------------------------------------------ mutants
def _gemm_layout_flipped(A, B, dtype, b_layout=oracle.B_KN, nthreads=None):
    return _orig["gemm"](A, B, dtype, 1 - b_layout, nthreads)


def _gemm_in_double(A, B, dtype, b_layout=oracle.B_KN, nthreads=None):
    return _orig["gemm64"](A, B, dtype, b_layout, nthreads).astype(np.float32)


def _gemm_descending_k(A, B, dtype, b_layout=oracle.B_KN, nthreads=None):
    Af = _orig["decode"](A, dtype)
    Bf = _orig["decode"](B, dtype)
    if b_layout == oracle.B_NK:
        Bf = Bf.T
    acc = np.zeros((Af.shape[0], Bf.shape[1]), dtype=np.float32)
    for p in reversed(range(Af.shape[1])):
        acc += np.outer(Af[:, p], Bf[p])  # products of 16-bit values are exact in fp32
    return acc


def _gemm_tail_dropped(A, B, dtype, b_layout=oracle.B_KN, nthreads=None):
    K = np.asarray(A).shape[1]
    K16 = K // 16 * 16
    if K16 == 0:
        R = np.asarray(A).shape[0]
        N = np.asarray(B).shape[1] if b_layout == oracle.B_KN else np.asarray(B).shape[0]
        return np.zeros((R, N), dtype=np.float32)
    A = np.ascontiguousarray(np.asarray(A)[:, :K16])
    B = np.ascontiguousarray(np.asarray(B)[:K16] if b_layout == oracle.B_KN
                             else np.asarray(B)[:, :K16])
    return _orig["gemm"](A, B, dtype, b_layout, nthreads)


def _decode_ignores_dtype(bits, dtype):
    return _orig["decode"](bits, oracle.F16)


def _round_toward_zero(x, dtype):
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == oracle.BF16:
        return (x.view(np.uint32) >> 16).astype(np.uint16)
    with np.errstate(over="ignore"):
        h = x.astype(np.float16)
    bits = h.view(np.uint16).copy()
    over = np.isfinite(x) & (np.abs(h.astype(np.float32)) > np.abs(x))
    bits[over] -= 1  # one step toward zero in sign-magnitude
    return bits


def _bias_dropped(acc, bias, dtype, axis, row_ids=None):
    return np.ascontiguousarray(acc, dtype=np.float32).copy()


def _bias_subtracted(acc, bias, dtype, axis, row_ids=None):
    neg = _orig["round_to"](-_orig["decode"](np.ravel(bias), dtype), dtype).reshape(np.shape(bias))
    return _orig["add_bias"](acc, neg, dtype, axis, row_ids)


def _bias_other_axis(acc, bias, dtype, axis, row_ids=None):
    return _orig["add_bias"](acc, bias, dtype, 1 - axis, row_ids)


def _relu_dropped(z):
    return np.ascontiguousarray(z, dtype=np.float32).copy()


def _relu_bits_ge(z):
    return (np.asarray(z) >= 0).astype(np.uint8)


def _relu_bits_sign(z):
    return (~np.signbit(np.asarray(z, dtype=np.float32))).astype(np.uint8)


def _pack_mask_msb_first(bits):
    b = np.asarray(bits, dtype=np.uint8)
    M, N = b.shape
    w = np.zeros(((M + 31) // 32, N), dtype=np.uint32)
    for i in range(M):
        w[i // 32] |= b[i].astype(np.uint32) << np.uint32(31 - i % 32)
    return w


def _pack_mask_row_words(bits):
    # words run along a row ([M][ceil(N/32)]) instead of down a column
    b = np.asarray(bits, dtype=np.uint8)
    M, N = b.shape
    w = np.zeros((M, (N + 31) // 32), dtype=np.uint32)
    for j in range(N):
        w[:, j // 32] |= b[:, j].astype(np.uint32) << np.uint32(j % 32)
    return w


def _drelu_unmasked(g, words, row_ids=None):
    return np.ascontiguousarray(g, dtype=np.float32).copy()


def _drelu_inverted(g, words, row_ids=None):
    return _orig["drelu"](g, ~np.ascontiguousarray(words, dtype=np.uint32), row_ids)


def _drelu_local_rows(g, words, row_ids=None):
    return _orig["drelu"](g, words, None)


def _colsum_rows(dz):
    return np.ascontiguousarray(dz, dtype=np.float32).astype(np.float64).sum(axis=1)


def _gelu_no_cubic(z):
    return 0.5 * z * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * z))


def _gelu_erf(z):
    return 0.5 * z * (1.0 + math.erf(z / math.sqrt(2.0)))


def _dgelu_no_product_rule(z):
    return 0.5 * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (z + 0.044715 * z ** 3)))


def _dgelu_sech_sign(z):
    u = math.sqrt(2.0 / math.pi) * (z + 0.044715 * z ** 3)
    du = math.sqrt(2.0 / math.pi) * (1.0 + 3 * 0.044715 * z * z)
    t = math.tanh(u)
    return 0.5 * (1.0 + t) - 0.5 * z * (1.0 - t * t) * du


def _dgelu_vector_uses_gelu(g, z):
    return (np.asarray(g, np.float64) * _orig["gelu"](z).astype(np.float64)).astype(np.float32)


def _silu_is_sigmoid(g):
    return 1.0 / (1.0 + math.exp(-g))


def _swiglu_gate_up_swapped(g, u):
    return _orig["swiglu"](u, g)


def _dswiglu_outputs_swapped(dh, g, u):
    dg, du = _orig["dswiglu"](dh, g, u)
    return du, dg


def _dswiglu_gate_no_sigmoid_slope(dh, g, u):
    # d_gate = dh * u * sigmoid(g): drops the g * s * (1 - s) term of silu'
    dh, g, u = (np.asarray(a, np.float64) for a in (dh, g, u))
    s = 1.0 / (1.0 + np.exp(-g))
    dg = (dh * u * s).astype(np.float32)
    du = (dh * g * s).astype(np.float32)
    return dg, du


# ------------------------------------------------------------------ table
def _hand_col(dtype=oracle.F16, layout=oracle.B_KN):
    return lambda: P.test_hand_col_bias(dtype, layout)


MUTANTS = {
    # GEMM
    "B read in the other layout": (
        {"gemm": _gemm_layout_flipped}, [_hand_col(), _hand_col(oracle.F16, oracle.B_NK)]),
    "fp32 accumulation replaced by double": (
        {"gemm": _gemm_in_double}, [P.test_gemm_order_is_ascending_k]),
    "k summed in descending order": (
        {"gemm": _gemm_descending_k}, [P.test_gemm_order_is_ascending_k]),
    "ragged k tail dropped": (
        {"gemm": _gemm_tail_dropped},
        [_hand_col(), lambda: P.test_gemm_exact_on_small_integers(oracle.B_KN, oracle.F16)]),
    # number formats
    "bf16 decoded as fp16": (
        {"decode": _decode_ignores_dtype},
        [P.test_bf16_against_torch, _hand_col(oracle.BF16, oracle.B_KN)]),
    "rounding toward zero instead of to nearest even": (
        {"round_to": _round_toward_zero},
        [P.test_half_rounding_matches_numpy, P.test_bf16_against_torch]),
    # forward epilogue
    "bias dropped": ({"add_bias": _bias_dropped}, [_hand_col(), P.test_hand_row_bias]),
    "bias subtracted": ({"add_bias": _bias_subtracted}, [_hand_col(), P.test_hand_row_bias]),
    "bias broadcast along the other axis": (
        {"add_bias": _bias_other_axis}, [_hand_col(), P.test_hand_row_bias]),
    "ReLU dropped": ({"relu": _relu_dropped}, [_hand_col(), P.test_hand_row_bias]),
    "mask bit set for z >= 0": ({"relu_bits": _relu_bits_ge}, [_hand_col()]),
    "mask bit from the sign bit": ({"relu_bits": _relu_bits_sign}, [_hand_col()]),
    "mask bits packed most significant first": (
        {"pack_mask": _pack_mask_msb_first},
        [_hand_col(), P.test_pack_mask_brute_force, P.test_nonnegative_inputs_closed_form]),
    "mask words along rows": ({"pack_mask": _pack_mask_row_words}, [_hand_col()]),
    # backward epilogue
    "dReLU mask ignored": (
        {"drelu": _drelu_unmasked},
        [P.test_hand_drelu_bgrad, P.test_drelu_identity_and_colsum_invariant]),
    "dReLU mask inverted": (
        {"drelu": _drelu_inverted},
        [P.test_hand_drelu_bgrad, P.test_drelu_bgrad_closed_forms]),
    "dReLU mask taken at the local row": ({"drelu": _drelu_local_rows}, [P.test_hand_drelu_row_ids]),
    "bias gradient summed along rows": ({"colsum": _colsum_rows}, [P.test_hand_drelu_bgrad]),
    # GELU
    "GELU without the cubic term": (
        {"gelu_scalar": _gelu_no_cubic},
        [G.test_gelu_closed_forms, G.test_gelu_matches_torch_float64]),
    "erf GELU in place of the tanh form": (
        {"gelu_scalar": _gelu_erf}, [G.test_gelu_closed_forms, G.test_gelu_matches_torch_float64]),
    "dGELU without the product-rule term": (
        {"dgelu_scalar": _dgelu_no_product_rule}, [G.test_dgelu_is_the_derivative]),
    "dGELU with the sech^2 term's sign flipped": (
        {"dgelu_scalar": _dgelu_sech_sign}, [G.test_dgelu_is_the_derivative]),
    "DGELU_BGRAD multiplying by gelu instead of gelu'": (
        {"dgelu": _dgelu_vector_uses_gelu}, [G.test_vector_steps_round_once]),
    # SwiGLU
    "sigmoid in place of silu": (
        {"silu_scalar": _silu_is_sigmoid}, [S.test_closed_forms, S.test_silu_matches_torch]),
    "gate and up swapped": (
        {"swiglu": _swiglu_gate_up_swapped},
        [S.test_dswiglu_matches_autograd, S.test_forward_is_the_samples_composite]),
    "d_gate and d_up swapped": (
        {"dswiglu": _dswiglu_outputs_swapped},
        [S.test_closed_forms, S.test_dswiglu_matches_autograd,
         S.test_backward_is_autograd_of_the_composite]),
    "d_gate without silu's slope term": (
        {"dswiglu": _dswiglu_gate_no_sigmoid_slope},
        [S.test_dswiglu_matches_autograd, S.test_backward_is_autograd_of_the_composite]),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    patches, pins = MUTANTS[name]
    for pin in pins:
        pin()  # the unmodified oracle passes every pin
    for attr, fn in patches.items():
        monkeypatch.setattr(oracle, attr, fn)
    missed = []
    for pin in pins:
        try:
            pin()
        except AssertionError:
            continue
        missed.append(getattr(pin, "__name__", repr(pin)))
    assert not missed, f"planted mistake '{name}' passed {missed}"
