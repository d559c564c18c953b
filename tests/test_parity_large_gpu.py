"""Parity at the full sizes of the pages' large workloads, in the launch
configuration the benchmark times (the plan's own kernel choice).

Linear-layer pair, fp16 (the (65536,16384) x (16384,8192) workload of
"Fusing Matmul Epilogs with nvmath-python", section "Suitable evaluation
scenarios"): 64 seeded sampled rows of the forward (Y and the relu_aux bits)
and of the backward (dZ) against the oracle; every bias-gradient column
against (a) the fp64 column sum of the device's own dZ and (b) the closed form
(1^T dY) W^T of an all-ones mask, computed on the host from the generator.

GELU at 8192 x 16384 x 4096, bf16: sampled rows of the forward (out and the
saved pre-activation) and backward, and every bias-gradient column against the
closed form 0.5 (1^T dY) W^T of a zero pre-activation (gelu'(0) = 1/2).
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import (BGRAD_NMAX, BGRAD_REL, assert_close, mask_mismatch, to_host_f32,
                     to_host_words, unpack_words)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import gemm_epilogue_tmem_gb300 as gf  # noqa: E402

SEED = 0


def _dev(shape, dtype, tid, sigma):
    tdt = torch.float16 if dtype == synth.F16 else torch.bfloat16
    t = torch.empty(shape, dtype=tdt, device="cuda")
    synth.dev_normal(t, dtype, SEED, tid, sigma)
    return t


def _host_colsum(shape, dtype, tid, sigma, chunk=4096):
    """1^T X in float64 for a generated [R, C] matrix, regenerated on the host."""
    R, C = shape
    s = np.zeros(C, dtype=np.float64)
    for r0 in range(0, R, chunk):
        rows = np.arange(r0, min(R, r0 + chunk))
        x = synth.normal(shape, dtype, SEED, tid, sigma, rows=rows)
        xf = oracle.decode(x, dtype) if dtype == synth.BF16 else x.astype(np.float32)
        s += xf.astype(np.float64).sum(axis=0)
    return s


@pytest.fixture(scope="module")
def linear_pair():
    w = synth.LINEAR_PAIR_LARGE
    M, K = w.tensors["X"].shape
    N = w.tensors["W"].shape[1]
    W_host = synth.normal((K, N), synth.F16, SEED, synth.TID_B, 1 / 128)
    return M, K, N, W_host


def test_large_forward_sampled_rows(linear_pair):
    M, K, N, W_host = linear_pair
    X = _dev((M, K), synth.F16, synth.TID_A, 1.0)
    W = _dev((K, N), synth.F16, synth.TID_B, 1 / 128)
    bias = _dev((N,), synth.F16, synth.TID_BIAS, 0.1)
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    aux = torch.empty((M // 32, N), dtype=torch.int32, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, N, K, gf.GF_F16, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL,
                                gf.GF_B_KN)
    gf.gf_matmul_execute(plan, X, W, bias=bias, out=Y, aux_out=aux)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    rows = synth.sample_rows(M, 64, SEED)
    ridx = torch.from_numpy(rows).cuda()
    y_dev = to_host_f32(Y.index_select(0, ridx))
    words_dev = to_host_words(aux.index_select(0, torch.from_numpy(rows // 32).cuda()))
    bits_dev = ((words_dev >> (rows % 32)[:, None].astype(np.uint32)) & 1).astype(np.uint8)
    del X, W, Y, aux
    torch.cuda.empty_cache()
    Xs = synth.normal((M, K), synth.F16, SEED, synth.TID_A, 1.0, rows=rows)
    b_host = synth.normal((N,), synth.F16, SEED, synth.TID_BIAS, 0.1)
    y_o, z_o = oracle.relu_bias(Xs, W_host, b_host, oracle.F16, row_ids=rows)
    assert_close(y_dev, oracle.decode(y_o, oracle.F16), what="Y sampled rows")
    outside, inside = mask_mismatch(bits_dev, z_o)
    assert outside == 0, f"{outside} relu_aux bits differ outside the band ({inside} inside)"


def test_large_backward_sampled_rows_and_bgrad(linear_pair):
    M, K, N, W_host = linear_pair
    dY = _dev((M, N), synth.F16, synth.TID_DY, 1.0)
    W = _dev((K, N), synth.F16, synth.TID_B, 1 / 128)
    mask = torch.empty((M // 32, K), dtype=torch.int32, device="cuda")
    synth.dev_mask_words(mask, M, K, SEED)
    dZ = torch.empty((M, K), dtype=torch.float16, device="cuda")
    bgrad = torch.empty((K,), dtype=torch.float32, device="cuda")
    # backward of the pair: dY [M, N] . W^T, W [K, N] being the [n, k] storage of B = W^T
    plan = gf.gf_matmul_plan_ex(M, K, N, gf.GF_F16, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL,
                                gf.GF_B_NK)
    gf.gf_matmul_execute(plan, dY, W, out=dZ, aux_in=mask, bgrad=bgrad)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    rows = synth.sample_rows(M, 64, SEED)
    dz_dev = to_host_f32(dZ.index_select(0, torch.from_numpy(rows).cuda()))
    bgrad_dev = bgrad.cpu().numpy()
    colsum_dev = dZ.double().sum(0).cpu().numpy()
    # the all-ones mask: dz = g everywhere
    mask.fill_(-1)
    gf.gf_matmul_execute(plan, dY, W, out=dZ, aux_in=mask, bgrad=bgrad)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    bgrad_ones = bgrad.cpu().numpy()
    plan.free()
    del dY, W, mask, dZ
    torch.cuda.empty_cache()

    assert_close(bgrad_dev, colsum_dev, BGRAD_NMAX, BGRAD_REL, what="bgrad vs 1^T dZ (device)")
    s = _host_colsum((M, N), synth.F16, synth.TID_DY, 1.0)
    closed = W_host.astype(np.float64) @ s  # [K]: sum_i sum_n dY[i, n] W[k, n]
    assert_close(bgrad_ones, closed, BGRAD_NMAX, BGRAD_REL, what="bgrad, all-ones mask")
    dYs = synth.normal((M, N), synth.F16, SEED, synth.TID_DY, 1.0, rows=rows)
    words = synth.mask_words(M, K, SEED)
    dz_o, _, _ = oracle.drelu_bgrad(dYs, W_host, words, oracle.F16, oracle.B_NK, row_ids=rows)
    assert_close(dz_dev, oracle.decode(dz_o, oracle.F16), what="dZ sampled rows")


@pytest.fixture(scope="module")
def gelu_shapes():
    w = synth.GELU_BIAS
    M, K = w.tensors["X"].shape
    N = w.tensors["W"].shape[1]
    W_host = synth.normal((K, N), synth.BF16, SEED, synth.TID_B, 1 / 64)
    return M, K, N, W_host


def test_large_gelu_forward_sampled_rows(gelu_shapes):
    M, K, N, W_host = gelu_shapes
    X = _dev((M, K), synth.BF16, synth.TID_A, 1.0)
    W = _dev((K, N), synth.BF16, synth.TID_B, 1 / 64)
    bias = _dev((N,), synth.BF16, synth.TID_BIAS, 0.1)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    aux = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, N, K, gf.GF_BF16, gf.GF_EPILOG_GELU_AUX_BIAS, gf.GF_BIAS_COL,
                                gf.GF_B_KN)
    gf.gf_matmul_execute(plan, X, W, bias=bias, out=Y, aux_out=aux)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    rows = synth.sample_rows(M, 64, SEED)
    ridx = torch.from_numpy(rows).cuda()
    y_dev = to_host_f32(Y.index_select(0, ridx))
    aux_dev = to_host_f32(aux.index_select(0, ridx))
    Xs = synth.normal((M, K), synth.BF16, SEED, synth.TID_A, 1.0, rows=rows)
    b_host = synth.normal((N,), synth.BF16, SEED, synth.TID_BIAS, 0.1)
    y_o, aux_o, _ = oracle.gelu_aux_bias(Xs, W_host, b_host, oracle.BF16, row_ids=rows)
    assert_close(y_dev, oracle.decode(y_o, oracle.BF16), what="GELU out sampled rows")
    assert_close(aux_dev, oracle.decode(aux_o, oracle.BF16), what="pre-activation sampled rows")


def test_large_dgelu_sampled_rows_and_bgrad(gelu_shapes):
    M, K, N, W_host = gelu_shapes
    # backward: dY [M, N] . W^T -> [M, K]; W [K, N] is the [n, k] storage of W^T
    dY = _dev((M, N), synth.BF16, synth.TID_DY, 1.0)
    W = _dev((K, N), synth.BF16, synth.TID_B, 1 / 64)
    pre = _dev((M, K), synth.BF16, synth.TID_PREACT, 1.0)
    out = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    bgrad = torch.empty((K,), dtype=torch.float32, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, K, N, gf.GF_BF16, gf.GF_EPILOG_DGELU_BGRAD, gf.GF_BIAS_COL,
                                gf.GF_B_NK)
    gf.gf_matmul_execute(plan, dY, W, out=out, aux_in=pre, bgrad=bgrad)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    rows = synth.sample_rows(M, 64, SEED)
    out_dev = to_host_f32(out.index_select(0, torch.from_numpy(rows).cuda()))
    bgrad_dev = bgrad.cpu().numpy()
    colsum_dev = out.double().sum(0).cpu().numpy()
    pre.zero_()  # gelu'(0) = 1/2: bgrad = (1/2) (1^T dY) W^T
    gf.gf_matmul_execute(plan, dY, W, out=out, aux_in=pre, bgrad=bgrad)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    bgrad_half = bgrad.cpu().numpy()
    plan.free()
    del dY, W, pre, out
    torch.cuda.empty_cache()
    assert_close(bgrad_dev, colsum_dev, BGRAD_NMAX, 2e-2, what="dgelu bgrad vs 1^T out (device)")
    s = _host_colsum((M, N), synth.BF16, synth.TID_DY, 1.0)
    closed = 0.5 * (oracle.decode(W_host, oracle.BF16).astype(np.float64) @ s)
    assert_close(bgrad_half, closed, BGRAD_NMAX, BGRAD_REL, what="dgelu bgrad, zero pre-act")
    dYs = synth.normal((M, N), synth.BF16, SEED, synth.TID_DY, 1.0, rows=rows)
    pres = synth.normal((M, K), synth.BF16, SEED, synth.TID_PREACT, 1.0, rows=rows)
    dz_o, _, _ = oracle.dgelu_bgrad(dYs, W_host, pres, oracle.BF16, oracle.B_NK, full_rows=False)
    assert_close(out_dev, oracle.decode(dz_o, oracle.BF16), what="dgelu out sampled rows")
