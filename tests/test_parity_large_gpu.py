"""Parity at the full sizes of the pages' large workloads, in the launch
configuration the benchmark times (the plan's own kernel choice).

Linear-layer pair, fp16 (the (65536,16384) x (16384,8192) workload of
"Fusing Matmul Epilogs with nvmath-python", section "Suitable evaluation
scenarios"): 64 seeded sampled rows of the forward (Y and the relu_aux bits)
and of the backward (dZ) against the oracle; every bias-gradient column
against (a) the fp64 column sum of the device's own dZ and (b) the closed form
(1^T dY) W^T of an all-ones mask, computed on the host from the generator.

The backward's bias gradient under the seeded Bernoulli mask is also checked
against the oracle itself on 64 seeded sampled columns: for those columns the
oracle forms dZ over all 65536 rows (the columns of a product are independent)
and sums it, so the masked path is pinned, not only the device's own 1^T dZ.

GELU at 8192 x 16384 x 4096, bf16: sampled rows of the forward (out and the
saved pre-activation) and backward, every bias-gradient column against the
closed form 0.5 (1^T dY) W^T of a zero pre-activation (gelu'(0) = 1/2), and 64
sampled columns of the dGELU output and its bias gradient against the oracle.

SwiGLU MLP at H = 5120, I = 17408 with 0.02-scaled weights, bf16
(gemm_swiglu_mlp_fusion.py, module docstring), M = 2048 and 16384: 64 sampled
rows of h, the saved g and u and the down projection from the fused gate+up
forward, and of d_gate and d_up from dh = dout Wd with the dSwiGLU epilogue.
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
    cols = synth.sample_cols(K, 64, SEED)
    dz_dev = to_host_f32(dZ.index_select(0, torch.from_numpy(rows).cuda()))
    dz_cols_dev = to_host_f32(dZ.index_select(1, torch.from_numpy(cols).cuda()))
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
    dY_all = synth.normal((M, N), synth.F16, SEED, synth.TID_DY, 1.0)
    s = np.zeros(N, dtype=np.float64)
    for r0 in range(0, M, 4096):
        s += dY_all[r0:r0 + 4096].astype(np.float64).sum(axis=0)
    closed = W_host.astype(np.float64) @ s  # [K]: sum_i sum_n dY[i, n] W[k, n]
    assert_close(bgrad_ones, closed, BGRAD_NMAX, BGRAD_REL, what="bgrad, all-ones mask")
    words = synth.mask_words(M, K, SEED)
    dz_o, _, _ = oracle.drelu_bgrad(dY_all[rows], W_host, words, oracle.F16, oracle.B_NK,
                                    row_ids=rows)
    assert_close(dz_dev, oracle.decode(dz_o, oracle.F16), what="dZ sampled rows")
    # sampled columns over every row, under the Bernoulli mask: the oracle's
    # dZ columns and their column sums (its bias gradient for those columns)
    dzc_o, bgrad_o, _ = oracle.drelu_bgrad(dY_all, W_host[cols], words[:, cols], oracle.F16,
                                           oracle.B_NK)
    assert_close(dz_cols_dev, oracle.decode(dzc_o, oracle.F16), what="dZ sampled columns")
    assert_close(bgrad_dev[cols], bgrad_o, BGRAD_NMAX, BGRAD_REL,
                 what="bgrad sampled columns vs oracle")


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
    cols = synth.sample_cols(K, 64, SEED)
    out_dev = to_host_f32(out.index_select(0, torch.from_numpy(rows).cuda()))
    out_cols_dev = to_host_f32(out.index_select(1, torch.from_numpy(cols).cuda()))
    bgrad_dev = bgrad.cpu().numpy()
    colsum_dev = out.double().sum(0).cpu().numpy()
    pre.zero_()  # gelu'(0) = 1/2: bgrad = (1/2) (1^T dY) W^T
    gf.gf_matmul_execute(plan, dY, W, out=out, aux_in=pre, bgrad=bgrad)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    bgrad_half = bgrad.cpu().numpy()
    plan.free()
    del dY, W, pre, out
    torch.cuda.empty_cache()
    assert_close(bgrad_dev, colsum_dev, BGRAD_NMAX, BGRAD_REL,
                 what="dgelu bgrad vs 1^T out (device)")
    s = _host_colsum((M, N), synth.BF16, synth.TID_DY, 1.0)
    closed = 0.5 * (oracle.decode(W_host, oracle.BF16).astype(np.float64) @ s)
    assert_close(bgrad_half, closed, BGRAD_NMAX, BGRAD_REL, what="dgelu bgrad, zero pre-act")
    dYs = synth.normal((M, N), synth.BF16, SEED, synth.TID_DY, 1.0, rows=rows)
    pres = synth.normal((M, K), synth.BF16, SEED, synth.TID_PREACT, 1.0, rows=rows)
    dz_o, _, _ = oracle.dgelu_bgrad(dYs, W_host, pres, oracle.BF16, oracle.B_NK, full_rows=False)
    assert_close(out_dev, oracle.decode(dz_o, oracle.BF16), what="dgelu out sampled rows")
    # sampled columns over every row: the oracle's dGELU output and bias gradient
    dY_all = synth.normal((M, N), synth.BF16, SEED, synth.TID_DY, 1.0)
    pre_all = synth.normal((M, K), synth.BF16, SEED, synth.TID_PREACT, 1.0)
    dzc_o, bgrad_o, _ = oracle.dgelu_bgrad(dY_all, W_host[cols], pre_all[:, cols], oracle.BF16,
                                           oracle.B_NK)
    assert_close(out_cols_dev, oracle.decode(dzc_o, oracle.BF16), what="dgelu out sampled columns")
    assert_close(bgrad_dev[cols], bgrad_o, BGRAD_NMAX, BGRAD_REL,
                 what="dgelu bgrad sampled columns vs oracle")


@pytest.fixture(scope="module")
def swiglu_weights():
    w = synth.swiglu(2048)
    H = w.tensors["x"].shape[1]
    I = w.tensors["Wg"].shape[0]
    sg = {n: w.tensors[n].sigma for n in ("Wg", "Wu", "Wd")}
    host = {n: synth.normal(w.tensors[n].shape, synth.BF16, SEED, w.tensors[n].tensor_id, sg[n])
            for n in ("Wg", "Wu", "Wd")}
    return w, H, I, host


@pytest.mark.parametrize("M", [2048, 16384])
def test_large_swiglu_forward_sampled_rows(swiglu_weights, M):
    w, H, I, host = swiglu_weights
    tw = w.tensors
    x = _dev((M, H), synth.BF16, tw["x"].tensor_id, tw["x"].sigma)
    Wg = _dev((I, H), synth.BF16, tw["Wg"].tensor_id, tw["Wg"].sigma)
    Wu = _dev((I, H), synth.BF16, tw["Wu"].tensor_id, tw["Wu"].sigma)
    Wd = _dev((H, I), synth.BF16, tw["Wd"].tensor_id, tw["Wd"].sigma)
    h, g, u = (torch.empty((M, I), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    out = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    fwd = gf.gf_swiglu_plan(M, I, H, gf.GF_BF16, save_gu=True)
    down = gf.gf_matmul_plan_ex(M, H, I, gf.GF_BF16, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL,
                                gf.GF_B_NK)
    gf.gf_swiglu_execute(fwd, x, Wg, Wu, h, g, u)
    gf.gf_matmul_execute(down, h, Wd, out=out)
    for p in (fwd, down):
        assert gf.gf_plan_status(p) == gf.GF_OK
        p.free()
    rows = synth.sample_rows(M, 64, SEED)
    ridx = torch.from_numpy(rows).cuda()
    h_dev, g_dev, u_dev, out_dev = (to_host_f32(t.index_select(0, ridx)) for t in (h, g, u, out))
    del x, Wg, Wu, Wd, h, g, u, out
    torch.cuda.empty_cache()
    xs = synth.normal((M, H), synth.BF16, SEED, tw["x"].tensor_id, tw["x"].sigma, rows=rows)
    h_o, g_o, u_o, _, _ = oracle.swiglu_forward(xs, host["Wg"], host["Wu"], oracle.BF16)
    assert_close(h_dev, oracle.decode(h_o, oracle.BF16), what="h sampled rows")
    assert_close(g_dev, oracle.decode(g_o, oracle.BF16), what="saved g sampled rows")
    assert_close(u_dev, oracle.decode(u_o, oracle.BF16), what="saved u sampled rows")
    # the down projection h Wd^T of the oracle's own h (Wd [H, I] is B given [n, k])
    out_o = oracle.epilog_none(h_o, host["Wd"], oracle.BF16, oracle.B_NK)
    assert_close(out_dev, oracle.decode(out_o, oracle.BF16), what="down projection sampled rows")


@pytest.mark.parametrize("M", [2048, 16384])
def test_large_dswiglu_sampled_rows(swiglu_weights, M):
    w, H, I, host = swiglu_weights
    tw = w.tensors
    # saved g and u with the spread the forward gives them: x Wg^T with x ~ N(0, 1)
    # and 0.02-scaled weights over H = 5120 terms
    s_gu = tw["Wg"].sigma * float(np.sqrt(H))
    dout = _dev((M, H), synth.BF16, tw["dout"].tensor_id, tw["dout"].sigma)
    Wd = _dev((H, I), synth.BF16, tw["Wd"].tensor_id, tw["Wd"].sigma)
    g = _dev((M, I), synth.BF16, synth.TID_G_SAVED, s_gu)
    u = _dev((M, I), synth.BF16, synth.TID_U_SAVED, s_gu)
    d_gate = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
    d_up = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
    plan = gf.gf_dswiglu_plan(M, I, H, gf.GF_BF16)
    gf.gf_dswiglu_execute(plan, dout, Wd, g, u, d_gate, d_up)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    rows = synth.sample_rows(M, 64, SEED)
    ridx = torch.from_numpy(rows).cuda()
    dg_dev, du_dev = (to_host_f32(t.index_select(0, ridx)) for t in (d_gate, d_up))
    del dout, Wd, g, u, d_gate, d_up
    torch.cuda.empty_cache()
    ds = synth.normal((M, H), synth.BF16, SEED, tw["dout"].tensor_id, tw["dout"].sigma, rows=rows)
    gs = synth.normal((M, I), synth.BF16, SEED, synth.TID_G_SAVED, s_gu, rows=rows)
    us = synth.normal((M, I), synth.BF16, SEED, synth.TID_U_SAVED, s_gu, rows=rows)
    dg_o, du_o, _ = oracle.dswiglu_backward(ds, host["Wd"], gs, us, oracle.BF16)
    assert_close(dg_dev, oracle.decode(dg_o, oracle.BF16), what="d_gate sampled rows")
    assert_close(du_dev, oracle.decode(du_o, oracle.BF16), what="d_up sampled rows")
