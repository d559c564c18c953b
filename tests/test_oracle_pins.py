"""Pins of the CPU oracle against things other than itself.

Each test fixes part of the oracle by something the pages or mathematics
decide: hand-worked examples (tests/golden/hand_4x4.json), library routines
(numpy's IEEE fp16 conversion, torch's bf16 conversion, float64 matmul on
exactly representable cases), closed forms, invariants and fp64 brute force
within the recursive-summation error bound (Higham, "Accuracy and Stability of
Numerical Algorithms", 2nd ed., eq. 3.4 / Lemma 3.1: |fl(sum) - sum| <=
gamma_n * sum |terms|, gamma_n = n u / (1 - n u)).

Definitions pinned (web pages on fused matmul epilogs):
 "Fusing Matmul Epilogs with nvmath-python": "The problem addressed by fused
 epilogs", "Forward-pass capabilities in the source", "Backward-pass path shown
 in the example"; the nvmath-python/cuBLASLt page, steps 1-2.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden", "hand_4x4.json")


def gold():
    with open(GOLD) as f:
        g = json.load(f)
    return g


def f16(a):
    """Literal list (with "-0" strings) -> fp16 array."""
    a = np.array([[-0.0 if v == "-0" else v for v in r] if isinstance(r, list) else
                  (-0.0 if r == "-0" else r) for r in a], dtype=np.float64)
    return a.astype(np.float16)


def vals(bits, dtype=oracle.F16):
    return oracle.decode(bits, dtype)


# ----------------------------------------------------------- hand-worked 4x4
@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
@pytest.mark.parametrize("layout", [oracle.B_KN, oracle.B_NK])
def test_hand_col_bias(dtype, layout):
    g = gold()
    A, B, bias = f16(g["A"]), f16(g["B_kn"]), f16(g["bias_col"])
    if dtype == oracle.BF16:
        A, B, bias = (oracle.round_to(x.astype(np.float32), oracle.BF16) for x in (A, B, bias))
    Bl = B if layout == oracle.B_KN else np.ascontiguousarray(B.T)
    acc = oracle.gemm(A, Bl, dtype, layout)
    assert np.array_equal(acc, np.array(g["acc"], dtype=np.float32))
    y, words, z = oracle.relu_aux_bias(A, Bl, bias, dtype, layout, oracle.BIAS_COL)
    assert np.array_equal(z, np.array(g["z_col"], dtype=np.float32))
    assert np.array_equal(vals(y, dtype), np.array(g["y_col"], dtype=np.float32))
    assert np.array_equal(oracle.relu_bits(z), np.array(g["bits_col"], dtype=np.uint8))
    assert np.array_equal(words, np.array(g["words_col"], dtype=np.uint32))
    # the z == 0 entries, including 0 + (-0), give ReLU 0 and mask bit 0
    assert z[2, 3] == 0 and not np.signbit(z[2, 3])


def test_hand_row_bias():
    g = gold()
    A, B, bias = f16(g["A"]), f16(g["B_kn"]), f16(g["bias_row"])
    y, z = oracle.relu_bias(A, B, bias.reshape(4, 1), oracle.F16, oracle.B_KN, oracle.BIAS_ROW)
    assert np.array_equal(z, np.array(g["z_row"], dtype=np.float32))
    assert np.array_equal(vals(y), np.array(g["y_row"], dtype=np.float32))
    assert np.array_equal(oracle.pack_mask(oracle.relu_bits(z)),
                          np.array(g["words_row"], dtype=np.uint32))
    # a subset of rows with their global index picks the right bias rows
    y2, z2 = oracle.relu_bias(A[[3, 1]], B, bias, oracle.F16, oracle.B_KN, oracle.BIAS_ROW,
                              row_ids=np.array([3, 1]))
    assert np.array_equal(z2, z[[3, 1]])


def test_hand_drelu_bgrad():
    g = gold()
    A, B = f16(g["A"]), f16(g["B_kn"])
    words = np.array(g["drelu_words"], dtype=np.uint32)
    out, bgrad, gm = oracle.drelu_bgrad(A, np.ascontiguousarray(B.T), words, oracle.F16,
                                        oracle.B_NK)
    assert np.array_equal(vals(out), np.array(g["drelu_dz"], dtype=np.float32))
    assert np.array_equal(bgrad, np.array(g["drelu_bgrad"], dtype=np.float32))


def test_hand_drelu_row_ids():
    # rows 3 and 1 alone, with their global row indices, take the mask bits
    # of rows 3 and 1 (word bits 3 and 1), not of rows 0 and 1
    g = gold()
    A, B = f16(g["A"]), f16(g["B_kn"])
    words = np.array(g["drelu_words"], dtype=np.uint32)
    out, bgrad, _ = oracle.drelu_bgrad(A[[3, 1]], np.ascontiguousarray(B.T), words, oracle.F16,
                                       oracle.B_NK, row_ids=np.array([3, 1]))
    assert bgrad is None
    assert np.array_equal(vals(out), np.array(g["drelu_dz"], dtype=np.float32)[[3, 1]])


# -------------------------------------------------------------- number formats
def _special_f32():
    r = np.random.default_rng(0)
    xs = [r.standard_normal(20000).astype(np.float32) * s for s in (1e-6, 1e-3, 1, 300, 7e4)]
    ties = np.array([1 + 2.0**-11, 1 + 3 * 2.0**-11, 2.0**-24 * 1.5, 2.0**-24 * 2.5, 2.0**-25,
                     2.0**-26, 65504, 65519.99, 65520, 65536, 1e10, 2.0**-14, 2.0**-14 * 0.99,
                     0.0, -0.0, np.inf, -np.inf], dtype=np.float64)
    return np.concatenate(xs + [ties.astype(np.float32), -ties.astype(np.float32)])


def test_half_rounding_matches_numpy():
    x = _special_f32()
    mine = oracle.round_to(x, oracle.F16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(mine, ref)
    nan = oracle.round_to(np.array([np.nan], np.float32), oracle.F16)
    assert np.isnan(nan.view(np.float16)[0])


def test_half_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.decode(bits, oracle.F16)
    ref = bits.view(np.float16).astype(np.float32)
    same = (mine == ref) | (np.isnan(mine) & np.isnan(ref))
    assert same.all()
    assert np.array_equal(np.signbit(mine[~np.isnan(mine)]), np.signbit(ref[~np.isnan(ref)]))


def test_bf16_against_torch():
    torch = pytest.importorskip("torch")
    x = _special_f32()
    mine = oracle.round_to(x, oracle.BF16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    dec = oracle.decode(bits, oracle.BF16)
    tref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    same = (dec == tref) | (np.isnan(dec) & np.isnan(tref))
    assert same.all()


# ----------------------------------------------------------------------- GEMM
@pytest.mark.parametrize("layout", [oracle.B_KN, oracle.B_NK])
@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
def test_gemm_exact_on_small_integers(layout, dtype):
    # integers in [-8, 8] with K = 203: every partial sum is an integer below
    # 2^24, so fp32 accumulation is exact and must equal float64 matmul
    r = np.random.default_rng(1)
    A = r.integers(-8, 9, (37, 203)).astype(np.float32)
    B = r.integers(-8, 9, (203, 29)).astype(np.float32)
    Ab, Bb = oracle.round_to(A, dtype), oracle.round_to(B, dtype)
    Bl = Bb if layout == oracle.B_KN else np.ascontiguousarray(Bb.T)
    acc = oracle.gemm(Ab, Bl, dtype, layout, nthreads=3)
    assert np.array_equal(acc.astype(np.float64), A.astype(np.float64) @ B.astype(np.float64))


@pytest.mark.parametrize("layout", [oracle.B_KN, oracle.B_NK])
def test_gemm_within_summation_bound(layout):
    r = np.random.default_rng(2)
    K = 777
    A = r.standard_normal((19, K)).astype(np.float16)
    B = r.standard_normal((K, 23)).astype(np.float16)
    Bl = B if layout == oracle.B_KN else np.ascontiguousarray(B.T)
    acc = oracle.gemm(A, Bl, oracle.F16, layout).astype(np.float64)
    exact = A.astype(np.float64) @ B.astype(np.float64)
    u = 2.0**-24
    gamma = K * u / (1 - K * u)
    bound = gamma * (np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64)))
    assert np.all(np.abs(acc - exact) <= bound)
    # not trivially exact: fp32 accumulation does differ from the exact sum
    assert np.any(acc != exact)
    g64 = oracle.gemm64(A, Bl, oracle.F16, layout)
    assert np.allclose(g64, exact, rtol=1e-13, atol=1e-11)


def test_gemm_order_is_ascending_k():
    # 1 + 2^-24 + 2^-24 ... : ascending-order fp32 summation loses each tiny
    # term against 1 (ties to even), so the sum stays 1 exactly
    K = 64
    A = np.ones((1, K), dtype=np.float32)
    B = np.full((K, 1), 2.0**-24, dtype=np.float32)
    B[0, 0] = 1.0
    acc = oracle.gemm(oracle.round_to(A, oracle.BF16), oracle.round_to(B, oracle.BF16),
                      oracle.BF16)
    assert acc[0, 0] == 1.0


# ---------------------------------------------------------------- epilogue steps
def test_pack_mask_brute_force():
    r = np.random.default_rng(3)
    M, N = 70, 5
    bits = (r.random((M, N)) < 0.5).astype(np.uint8)
    w = oracle.pack_mask(bits)
    assert w.shape == (3, N)
    for i in range(M):
        for j in range(N):
            assert (int(w[i // 32, j]) >> (i % 32)) & 1 == bits[i, j]
            assert oracle.mask_bit(w, i, j) == bits[i, j]
    assert np.all(w[2] >> (M - 64) == 0)
    # the same words by numpy's little-endian packbits along rows
    padded = np.zeros((96, N), dtype=np.uint8)
    padded[:M] = bits
    lib = np.packbits(padded.reshape(3, 32, N).transpose(0, 2, 1), axis=2, bitorder="little")
    assert np.array_equal(w, lib.view("<u4").reshape(3, N))


def test_drelu_identity_and_colsum_invariant():
    r = np.random.default_rng(4)
    M, N = 100, 48
    z = r.standard_normal((M, N)).astype(np.float32)
    z[3, 4] = 0.0
    g = r.standard_normal((M, N)).astype(np.float32)
    words = oracle.pack_mask(oracle.relu_bits(z))
    dz = oracle.drelu(g, words)
    assert np.array_equal(dz, np.where(z > 0, g, np.float32(0)))  # G * 1[Z > 0]
    cs = oracle.colsum(dz)
    assert np.allclose(cs, dz.astype(np.float64).sum(axis=0), rtol=1e-14, atol=1e-12)


def test_drelu_bgrad_closed_forms():
    r = np.random.default_rng(5)
    M, N, K = 96, 40, 24
    dY = r.standard_normal((M, K)).astype(np.float16)
    W = (r.standard_normal((N, K)) * 0.2).astype(np.float16)  # W stored [N, K]
    ones = np.full(((M + 31) // 32, N), 0xFFFFFFFF, dtype=np.uint32)
    out, bgrad, gm = oracle.drelu_bgrad(dY, W, ones, oracle.F16, oracle.B_NK)
    # all-ones mask: bgrad = (1^T dY) W^T up to the fp32 accumulation of g
    closed = dY.astype(np.float64).sum(axis=0) @ W.astype(np.float64).T
    u = 2.0**-24
    bound = (K * u / (1 - K * u)) * (np.abs(dY.astype(np.float64)).sum(0)
                                     @ np.abs(W.astype(np.float64)).T) + 1e-6 * np.abs(closed)
    assert np.all(np.abs(bgrad.astype(np.float64) - closed) <= bound + 1e-6)
    assert np.array_equal(vals(out), np.array(oracle.decode(oracle.round_to(gm, 0), 0)))
    zeros = np.zeros_like(ones)
    out0, bgrad0, _ = oracle.drelu_bgrad(dY, W, zeros, oracle.F16, oracle.B_NK)
    assert not np.any(vals(out0)) and not np.any(bgrad0)


def test_nonnegative_inputs_closed_form():
    r = np.random.default_rng(6)
    A = np.abs(r.standard_normal((33, 64))).astype(np.float16)
    B = np.abs(r.standard_normal((64, 40))).astype(np.float16)
    bias = np.abs(r.standard_normal(40)).astype(np.float16)
    y, words, z = oracle.relu_aux_bias(A, B, bias, oracle.F16)
    assert np.all(z > 0)
    full = np.full((2, 40), 0xFFFFFFFF, dtype=np.uint32)
    full[1] = 1  # row 32 only; rows 33..63 are padding
    assert np.array_equal(words, full)
    # Y = AB + bias exactly as fp16 of the fp32 sum
    acc = oracle.gemm(A, B, oracle.F16)
    assert np.array_equal(y, (acc + bias.astype(np.float32)).astype(np.float16).view(np.uint16))


def test_epilog_none_is_rounded_gemm():
    r = np.random.default_rng(7)
    A = r.standard_normal((17, 48)).astype(np.float16)
    B = r.standard_normal((48, 24)).astype(np.float16)
    out = oracle.epilog_none(A, B, oracle.F16)
    assert np.array_equal(out, oracle.gemm(A, B, oracle.F16).astype(np.float16).view(np.uint16))


def test_sampled_rows_equal_full_rows():
    w = synth.LINEAR_PAIR_LARGE  # shape recipe only; a small stand-in here
    M, K, N = 200, 64, 48
    X = synth.normal((M, K), synth.F16, 0, synth.TID_A, 1.0)
    W = synth.normal((K, N), synth.F16, 0, synth.TID_B, 1 / 8)
    b = synth.normal((N,), synth.F16, 0, synth.TID_BIAS, 0.1)
    rows = synth.sample_rows(M, 16, 0)
    y_full, z_full = oracle.relu_bias(X, W, b, oracle.F16)
    Xs = synth.normal((M, K), synth.F16, 0, synth.TID_A, 1.0, rows=rows)
    y_s, z_s = oracle.relu_bias(Xs, W, b, oracle.F16, row_ids=rows)
    assert np.array_equal(y_s, y_full[rows]) and np.array_equal(z_s, z_full[rows])
    assert w.tensors["X"].shape == (65536, 16384)
