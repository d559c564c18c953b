"""GPU parity of the SwiGLU MLP path (gemm_swiglu_mlp_fusion.py, module
docstring): the gate+up forward as one kernel (two accumulators per tile,
SiLU * mul epilogue, optionally saving g and u), the down projection as a
plain GEMM, and the dSwiGLU fused as the epilogue of dh = dout Wd."""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_close, to_dev, to_host_f32, torch_dtype

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import gemm_epilogue_tmem_gb300 as gf  # noqa: E402

SHAPES = [(256, 128, 128), (300, 200, 72), (1000, 520, 1000), (2048, 2048, 512), (4096, 4096, 256)]


def _weights(M, H, I, d, seed):
    x = synth.normal((M, H), d, seed, synth.TID_A, 1.0)
    Wg = synth.normal((I, H), d, seed, synth.TID_WG, 0.02 * 8)
    Wu = synth.normal((I, H), d, seed, synth.TID_WU, 0.02 * 8)
    return x, Wg, Wu


@pytest.mark.parametrize("M,I,H", SHAPES)
@pytest.mark.parametrize("dtype", [synth.BF16, synth.F16])
@pytest.mark.parametrize("kernel", [1, 2, 3])
def test_swiglu_forward(M, I, H, dtype, kernel):
    x, Wg, Wu = _weights(M, H, I, dtype, 3)
    tdt = torch_dtype(dtype)
    h = torch.empty((M, I), dtype=tdt, device="cuda")
    g = torch.empty((M, I), dtype=tdt, device="cuda")
    u = torch.empty((M, I), dtype=tdt, device="cuda")
    h2 = torch.empty((M, I), dtype=tdt, device="cuda")
    xd, Wgd, Wud = to_dev(x, dtype), to_dev(Wg, dtype), to_dev(Wu, dtype)
    for save, hh in ((True, h), (False, h2)):
        plan = gf.gf_swiglu_plan(M, I, H, dtype, save_gu=save)
        gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, kernel)
        gf.gf_swiglu_execute(plan, xd, Wgd, Wud, hh, g if save else None, u if save else None)
        assert gf.gf_plan_status(plan) == gf.GF_OK
        plan.free()
    h_o, g_o, u_o, _, _ = oracle.swiglu_forward(x, Wg, Wu, dtype)
    assert_close(to_host_f32(h), oracle.decode(h_o, dtype), what="h")
    assert_close(to_host_f32(h2), oracle.decode(h_o, dtype), what="h (no save)")
    assert_close(to_host_f32(g), oracle.decode(g_o, dtype), what="saved g")
    assert_close(to_host_f32(u), oracle.decode(u_o, dtype), what="saved u")


@pytest.mark.parametrize("M,I,H", SHAPES)
@pytest.mark.parametrize("dtype", [synth.BF16, synth.F16])
@pytest.mark.parametrize("kernel", [1, 2, 3])
def test_dswiglu(M, I, H, dtype, kernel):
    dout = synth.normal((M, H), dtype, 4, synth.TID_DOUT, 1.0)
    Wd = synth.normal((H, I), dtype, 4, synth.TID_WD, 1 / np.sqrt(H))
    g = synth.normal((M, I), dtype, 4, synth.TID_G_SAVED, 2.0)
    u = synth.normal((M, I), dtype, 4, synth.TID_U_SAVED, 1.0)
    tdt = torch_dtype(dtype)
    d_gate = torch.empty((M, I), dtype=tdt, device="cuda")
    d_up = torch.empty((M, I), dtype=tdt, device="cuda")
    plan = gf.gf_dswiglu_plan(M, I, H, dtype)
    gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, kernel)
    gf.gf_dswiglu_execute(plan, to_dev(dout, dtype), to_dev(Wd, dtype), to_dev(g, dtype),
                          to_dev(u, dtype), d_gate, d_up)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    dg_o, du_o, _ = oracle.dswiglu_backward(dout, Wd, g, u, dtype)
    assert_close(to_host_f32(d_gate), oracle.decode(dg_o, dtype), what="d_gate")
    assert_close(to_host_f32(d_up), oracle.decode(du_o, dtype), what="d_up")


def test_mlp_forward_backward_chain():
    """x -> (gate+up, saved g, u) -> h -> down GEMM; dout -> dh -> (d_gate,
    d_up), on the device, with the oracle's own saved g and u feeding the
    oracle's backward (the device's saved g and u feed the device's)."""
    M, H, I = 512, 256, 384
    d = synth.BF16
    x, Wg, Wu = _weights(M, H, I, d, 5)
    Wd = synth.normal((H, I), d, 5, synth.TID_WD, 1 / np.sqrt(I))
    dout = synth.normal((M, H), d, 5, synth.TID_DOUT, 1.0)
    t = torch.bfloat16
    h = torch.empty((M, I), dtype=t, device="cuda")
    g = torch.empty((M, I), dtype=t, device="cuda")
    u = torch.empty((M, I), dtype=t, device="cuda")
    out = torch.empty((M, H), dtype=t, device="cuda")
    dgt = torch.empty((M, I), dtype=t, device="cuda")
    dup = torch.empty((M, I), dtype=t, device="cuda")
    fwd = gf.gf_swiglu_plan(M, I, H, d, save_gu=True)
    down = gf.gf_matmul_plan_ex(M, H, I, d, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL, gf.GF_B_NK)
    bwd = gf.gf_dswiglu_plan(M, I, H, d)
    Wdd = to_dev(Wd, d)
    gf.gf_swiglu_execute(fwd, to_dev(x, d), to_dev(Wg, d), to_dev(Wu, d), h, g, u)
    gf.gf_matmul_execute(down, h, Wdd, out=out)
    gf.gf_dswiglu_execute(bwd, to_dev(dout, d), Wdd, g, u, dgt, dup)
    for p in (fwd, down, bwd):
        assert gf.gf_plan_status(p) == gf.GF_OK
        p.free()
    h_o, g_o, u_o, _, _ = oracle.swiglu_forward(x, Wg, Wu, d)
    out_o = oracle.epilog_none(h_o, Wd, d, oracle.B_NK)
    dg_o, du_o, _ = oracle.dswiglu_backward(dout, Wd, g_o, u_o, d)
    assert_close(to_host_f32(out), oracle.decode(out_o, d), what="MLP out")
    assert_close(to_host_f32(dgt), oracle.decode(dg_o, d), what="d_gate")
    assert_close(to_host_f32(dup), oracle.decode(du_o, d), what="d_up")
