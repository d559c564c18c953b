"""GPU parity of the GELU epilogs (GELU_BIAS named on the nvmath-python /
cuBLASLt page, "other epilogs"; tanh-form GELU) against the CPU oracle:
GELU_BIAS, GELU_AUX_BIAS (saves the pre-activation) and DGELU_BGRAD (the
backward from that pre-activation, with the column-sum bias gradient)."""
import numpy as np
import pytest

import oracle
import synth
from helpers import BGRAD_NMAX, BGRAD_REL, assert_close, to_dev, to_host_f32, torch_dtype

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import gemm_epilogue_tmem_gb300 as gf  # noqa: E402

SHAPES = [(256, 256, 128), (300, 200, 72), (1000, 520, 1000), (2048, 1024, 512)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("dtype", [synth.BF16, synth.F16])
@pytest.mark.parametrize("kernel", [1, 2])
def test_gelu_aux_bias(M, N, K, dtype, kernel):
    X = synth.normal((M, K), dtype, 7, synth.TID_A, 1.0)
    W = synth.normal((K, N), dtype, 7, synth.TID_B, 1 / np.sqrt(K))
    bias = synth.normal((N,), dtype, 7, synth.TID_BIAS, 0.1)
    tdt = torch_dtype(dtype)
    out = torch.empty((M, N), dtype=tdt, device="cuda")
    aux = torch.empty((M, N), dtype=tdt, device="cuda")
    out2 = torch.empty((M, N), dtype=tdt, device="cuda")
    for epi, o, a in ((gf.GF_EPILOG_GELU_AUX_BIAS, out, aux), (gf.GF_EPILOG_GELU_BIAS, out2, None)):
        plan = gf.gf_matmul_plan_ex(M, N, K, dtype, epi, gf.GF_BIAS_COL, gf.GF_B_KN)
        gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, kernel)
        gf.gf_matmul_execute(plan, to_dev(X, dtype), to_dev(W, dtype), bias=to_dev(bias, dtype),
                             out=o, aux_out=a)
        assert gf.gf_plan_status(plan) == gf.GF_OK
        plan.free()
    y_o, aux_o, z = oracle.gelu_aux_bias(X, W, bias, dtype)
    assert_close(to_host_f32(out), oracle.decode(y_o, dtype), what="gelu out")
    assert_close(to_host_f32(out2), oracle.decode(y_o, dtype), what="gelu out (no aux)")
    assert_close(to_host_f32(aux), oracle.decode(aux_o, dtype), what="pre-activation aux")


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("dtype", [synth.BF16, synth.F16])
@pytest.mark.parametrize("kernel,mode", [(1, 0), (2, 0), (1, 1)])
def test_dgelu_bgrad(M, N, K, dtype, kernel, mode):
    dY = synth.normal((M, K), dtype, 8, synth.TID_DY, 1.0)
    W = synth.normal((N, K), dtype, 8, synth.TID_B, 1 / np.sqrt(K))
    pre = synth.normal((M, N), dtype, 8, synth.TID_PREACT, 1.0)
    tdt = torch_dtype(dtype)
    out = torch.empty((M, N), dtype=tdt, device="cuda")
    bgrad = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, N, K, dtype, gf.GF_EPILOG_DGELU_BGRAD, gf.GF_BIAS_COL,
                                gf.GF_B_NK)
    gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, kernel)
    gf.gf_plan_set_option(plan, gf.GF_OPT_BGRAD_MODE, mode)
    gf.gf_matmul_execute(plan, to_dev(dY, dtype), to_dev(W, dtype), out=out,
                         aux_in=to_dev(pre, dtype), bgrad=bgrad)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    dz_o, bgrad_o, _ = oracle.dgelu_bgrad(dY, W, pre, dtype, oracle.B_NK)
    assert_close(to_host_f32(out), oracle.decode(dz_o, dtype), what="dgelu out")
    assert_close(bgrad.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL, what="dgelu bgrad")


def test_gelu_forward_backward_pair():
    """GELU_AUX_BIAS forward, then DGELU_BGRAD on the saved pre-activation
    (the oracle's own aux feeds the device backward; the device's aux is
    compared separately above)."""
    M, K, N = 512, 256, 384
    d = synth.BF16
    X = synth.normal((M, K), d, 9, synth.TID_A, 1.0)
    W = synth.normal((K, N), d, 9, synth.TID_B, 1 / 16)
    b = synth.normal((N,), d, 9, synth.TID_BIAS, 0.1)
    dY = synth.normal((M, 128), d, 9, synth.TID_DY, 1.0)
    W2 = synth.normal((N, 128), d, 9, synth.TID_W2, 1 / np.sqrt(N))
    _, aux_o, _ = oracle.gelu_aux_bias(X, W, b, d)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    bgrad = torch.empty(N, dtype=torch.float32, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, N, 128, d, gf.GF_EPILOG_DGELU_BGRAD, gf.GF_BIAS_COL, gf.GF_B_NK)
    gf.gf_matmul_execute(plan, to_dev(dY, d), to_dev(W2, d), out=out, aux_in=to_dev(aux_o, d),
                         bgrad=bgrad)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    dz_o, bgrad_o, _ = oracle.dgelu_bgrad(dY, W2, aux_o, d, oracle.B_NK)
    assert_close(to_host_f32(out), oracle.decode(dz_o, d))
    assert_close(bgrad.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL)
