"""Both kernels with several output tiles per persistent CTA (or CTA pair),
so that the two tensor-memory accumulator buffers are each reused and the
shared-memory ring wraps many times: checked against the oracle."""
import numpy as np
import pytest

import oracle
import synth
from helpers import (BGRAD_NMAX, BGRAD_REL, assert_close, mask_mismatch, to_dev, to_host_f32,
                     to_host_words, unpack_words)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import gemm_epilogue_tmem_gb300 as gf  # noqa: E402

M, N, K = 4096, 4096, 320


@pytest.fixture(scope="module")
def data():
    X = synth.normal((M, K), synth.F16, 21, synth.TID_A, 1.0)
    W = synth.normal((K, N), synth.F16, 21, synth.TID_B, 1 / np.sqrt(K))
    Wt = synth.normal((N, K), synth.F16, 21, synth.TID_W2, 1 / np.sqrt(K))
    b = synth.normal((N,), synth.F16, 21, synth.TID_BIAS, 0.1)
    words = synth.mask_words(M, N, 21)
    y_o, z_o = oracle.relu_bias(X, W, b, oracle.F16)
    dz_o, bgrad_o, _ = oracle.drelu_bgrad(X, Wt, words, oracle.F16, oracle.B_NK)
    return X, W, Wt, b, words, y_o, z_o, dz_o, bgrad_o


@pytest.mark.parametrize("kernel,tile_n", [(1, 256), (1, 128), (2, 0)])
def test_forward_many_tiles(data, kernel, tile_n):
    X, W, Wt, b, words, y_o, z_o, dz_o, bgrad_o = data
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    aux = torch.empty((M // 32, N), dtype=torch.int32, device="cuda")
    plan = gf.gf_matmul_plan(M, N, K, gf.GF_F16, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL)
    gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, kernel)
    if tile_n:
        gf.gf_plan_set_option(plan, gf.GF_OPT_TILE_N, tile_n)
    d = gf.gf_plan_describe(plan)
    tiles = (M // d["tile_m"]) * (N // d["tile_n"])
    per = d["grid"] if d["tile_m"] == 128 else d["grid"] // 2
    assert tiles >= 3 * per, (tiles, d)
    gf.gf_matmul_execute(plan, to_dev(X, 0), to_dev(W, 0), bias=to_dev(b, 0), out=out,
                         aux_out=aux)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    assert_close(to_host_f32(out), oracle.decode(y_o, 0), what="Y")
    outside, _ = mask_mismatch(unpack_words(to_host_words(aux), M), z_o)
    assert outside == 0


@pytest.mark.parametrize("kernel,tile_n", [(1, 256), (1, 128), (2, 0)])
def test_backward_many_tiles(data, kernel, tile_n):
    X, W, Wt, b, words, y_o, z_o, dz_o, bgrad_o = data
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    bgrad = torch.empty((N,), dtype=torch.float32, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, N, K, gf.GF_F16, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL,
                                gf.GF_B_NK)
    gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, kernel)
    if tile_n:
        gf.gf_plan_set_option(plan, gf.GF_OPT_TILE_N, tile_n)
    gf.gf_matmul_execute(plan, to_dev(X, 0), to_dev(Wt, 0), out=out, aux_in=to_dev(words, 0),
                         bgrad=bgrad)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    assert_close(to_host_f32(out), oracle.decode(dz_o, 0), what="dZ")
    assert_close(bgrad.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL, what="bgrad")
