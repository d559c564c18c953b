"""A seeded sweep of random problems against the oracle: shapes (M any size,
N and K multiples of 8, from tiny to several tiles with ragged tails), every
gf_matmul epilog, fp16 and bf16, both B layouts, both bias axes, every kernel
form (the plan's choice, single CTA at both tile widths, CTA pair, wide pair),
k split or not, bias-gradient mode, and dependent launch on or off; and the
SwiGLU entry points the same way. The cases are drawn once from a fixed seed,
so every run checks the same ones."""
import numpy as np
import pytest

import oracle
import synth
from helpers import (BGRAD_NMAX, BGRAD_REL, assert_close, mask_mismatch, to_dev, to_host_f32,
                     to_host_words, torch_dtype, unpack_words)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import gemm_epilogue_tmem_gb300 as gf  # noqa: E402

FWD = [gf.GF_EPILOG_NONE, gf.GF_EPILOG_BIAS, gf.GF_EPILOG_RELU_BIAS, gf.GF_EPILOG_RELU_AUX_BIAS,
       gf.GF_EPILOG_GELU_BIAS, gf.GF_EPILOG_GELU_AUX_BIAS]
BWD = [gf.GF_EPILOG_DRELU_BGRAD, gf.GF_EPILOG_DGELU_BGRAD]


def _cases(n=120, seed=2024):
    r = np.random.default_rng(seed)
    out = []
    for i in range(n):
        M = int(r.choice([1, 31, 33, 127, 129, 255, 257]) if r.random() < 0.3
                else r.integers(1, 1500))
        N = 8 * int(r.integers(1, 150))
        K = 8 * int(r.integers(1, 160))
        epi = int(r.choice(FWD + BWD))
        axis = int(r.integers(0, 2)) if epi in (gf.GF_EPILOG_BIAS, gf.GF_EPILOG_RELU_BIAS,
                                                 gf.GF_EPILOG_RELU_AUX_BIAS,
                                                 gf.GF_EPILOG_GELU_BIAS) else gf.GF_BIAS_COL
        out.append(dict(i=i, M=M, N=N, K=K, epi=epi, axis=axis, dtype=int(r.integers(0, 2)),
                        layout=int(r.integers(0, 2)), kernel=int(r.choice([0, 1, 1, 2, 3])),
                        tile_n=int(r.choice([0, 128, 256])), split=int(r.choice([0, 1, 2, 3])),
                        mode=int(r.integers(0, 2)), pdl=int(r.integers(0, 2))))
    return out


CASES = _cases()


def _id(c):
    return (f"{c['i']}-{c['M']}x{c['N']}x{c['K']}-e{c['epi']}-d{c['dtype']}-l{c['layout']}"
            f"-k{c['kernel']}-s{c['split']}")


@pytest.fixture(scope="module", autouse=True)
def _built():
    gf.build()
    synth.build_host()
    oracle.build()


@pytest.mark.parametrize("c", CASES, ids=_id)
def test_random_problem(c):
    M, N, K, epi, axis, d, layout = c["M"], c["N"], c["K"], c["epi"], c["axis"], c["dtype"], \
        c["layout"]
    seed = 100 + c["i"]
    bwd = epi in BWD
    A = synth.normal((M, K), d, seed, synth.TID_DY if bwd else synth.TID_A, 1.0)
    B = synth.normal((K, N) if layout == gf.GF_B_KN else (N, K), d, seed, synth.TID_B,
                     1 / np.sqrt(K))
    plan = gf.gf_matmul_plan_ex(M, N, K, d, epi, axis, layout)
    if c["kernel"]:
        gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, c["kernel"])
    if c["kernel"] == 1 and c["tile_n"]:
        gf.gf_plan_set_option(plan, gf.GF_OPT_TILE_N, c["tile_n"])
    if c["split"]:
        gf.gf_plan_set_option(plan, gf.GF_OPT_SPLIT_K, c["split"])
    gf.gf_plan_set_option(plan, gf.GF_OPT_PDL, c["pdl"])
    tdt = torch_dtype(d)
    out = torch.empty((M, N), dtype=tdt, device="cuda")
    if not bwd:
        bias = synth.normal((M if axis == gf.GF_BIAS_ROW else N,), d, seed, synth.TID_BIAS, 0.1)
        words = torch.zeros(((M + 31) // 32, N), dtype=torch.int32, device="cuda")
        pre = torch.empty((M, N), dtype=tdt, device="cuda")
        aux = (words if epi == gf.GF_EPILOG_RELU_AUX_BIAS else
               pre if epi == gf.GF_EPILOG_GELU_AUX_BIAS else None)
        gf.gf_matmul_execute(plan, to_dev(A, d), to_dev(B, d), bias=to_dev(bias, d), out=out,
                             aux_out=aux)
        assert gf.gf_plan_status(plan) == gf.GF_OK
        plan.free()
        acc = oracle.gemm(A, B, d, layout)
        if epi == gf.GF_EPILOG_NONE:
            assert_close(to_host_f32(out), oracle.decode(oracle.round_to(acc, d), d), what="out")
            return
        z = oracle.add_bias(acc, bias, d, axis)
        if epi == gf.GF_EPILOG_BIAS:
            y = oracle.round_to(z, d)
        elif epi in (gf.GF_EPILOG_RELU_BIAS, gf.GF_EPILOG_RELU_AUX_BIAS):
            y = oracle.round_to(oracle.relu(z), d)
        else:
            y = oracle.round_to(oracle.gelu(z), d)
        assert_close(to_host_f32(out), oracle.decode(y, d), what="out")
        if epi == gf.GF_EPILOG_RELU_AUX_BIAS:
            outside, _ = mask_mismatch(unpack_words(to_host_words(words), M), z)
            assert outside == 0
        if epi == gf.GF_EPILOG_GELU_AUX_BIAS:
            assert_close(to_host_f32(pre), oracle.decode(oracle.round_to(z, d), d),
                         what="pre-activation")
        return
    bgrad = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    gf.gf_plan_set_option(plan, gf.GF_OPT_BGRAD_MODE, c["mode"])
    if epi == gf.GF_EPILOG_DRELU_BGRAD:
        aux_h = synth.mask_words(M, N, seed)
    else:
        aux_h = synth.normal((M, N), d, seed, synth.TID_PREACT, 1.0)
    gf.gf_matmul_execute(plan, to_dev(A, d), to_dev(B, d), out=out, aux_in=to_dev(aux_h, d),
                         bgrad=bgrad)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    if epi == gf.GF_EPILOG_DRELU_BGRAD:
        dz_o, bgrad_o, _ = oracle.drelu_bgrad(A, B, aux_h, d, layout)
    else:
        dz_o, bgrad_o, _ = oracle.dgelu_bgrad(A, B, aux_h, d, layout)
    assert_close(to_host_f32(out), oracle.decode(dz_o, d), what="dZ")
    assert_close(bgrad.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL, what="bgrad")


def _swiglu_cases(n=40, seed=2025):
    r = np.random.default_rng(seed)
    out = []
    for i in range(n):
        M = int(r.choice([1, 33, 129, 257]) if r.random() < 0.3 else r.integers(1, 900))
        out.append(dict(i=i, M=M, I=8 * int(r.integers(1, 100)), H=8 * int(r.integers(1, 100)),
                        dtype=int(r.integers(0, 2)), backward=bool(r.integers(0, 2)),
                        save=bool(r.integers(0, 2)), kernel=int(r.choice([0, 1, 2, 3])),
                        pdl=int(r.integers(0, 2))))
    return out


@pytest.mark.parametrize("c", _swiglu_cases(),
                         ids=lambda c: (f"{c['i']}-{c['M']}x{c['I']}x{c['H']}-d{c['dtype']}"
                                        f"-{'bwd' if c['backward'] else 'fwd'}-k{c['kernel']}"))
def test_random_swiglu(c):
    """The gate+up forward (saving g and u or not) and the dSwiGLU backward
    on random shapes, kernel forms (the wide pair only for the backward,
    which has one B operand) and launch modes."""
    M, I, H, d = c["M"], c["I"], c["H"], c["dtype"]
    seed = 300 + c["i"]
    tdt = torch_dtype(d)
    if not c["backward"]:
        x = synth.normal((M, H), d, seed, synth.TID_A, 1.0)
        Wg = synth.normal((I, H), d, seed, synth.TID_WG, 1 / np.sqrt(H))
        Wu = synth.normal((I, H), d, seed, synth.TID_WU, 1 / np.sqrt(H))
        plan = gf.gf_swiglu_plan(M, I, H, d, save_gu=c["save"])
        if c["kernel"] in (1, 2):
            gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, c["kernel"])
        gf.gf_plan_set_option(plan, gf.GF_OPT_PDL, c["pdl"])
        h, g, u = (torch.empty((M, I), dtype=tdt, device="cuda") for _ in range(3))
        gf.gf_swiglu_execute(plan, to_dev(x, d), to_dev(Wg, d), to_dev(Wu, d), h,
                             g if c["save"] else None, u if c["save"] else None)
        assert gf.gf_plan_status(plan) == gf.GF_OK
        plan.free()
        h_o, g_o, u_o, _, _ = oracle.swiglu_forward(x, Wg, Wu, d)
        assert_close(to_host_f32(h), oracle.decode(h_o, d), what="h")
        if c["save"]:
            assert_close(to_host_f32(g), oracle.decode(g_o, d), what="saved g")
            assert_close(to_host_f32(u), oracle.decode(u_o, d), what="saved u")
        return
    dout = synth.normal((M, H), d, seed, synth.TID_DOUT, 1.0)
    Wd = synth.normal((H, I), d, seed, synth.TID_WD, 1 / np.sqrt(H))
    g = synth.normal((M, I), d, seed, synth.TID_G_SAVED, 2.0)
    u = synth.normal((M, I), d, seed, synth.TID_U_SAVED, 1.0)
    plan = gf.gf_dswiglu_plan(M, I, H, d)
    if c["kernel"]:
        gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, c["kernel"])
    gf.gf_plan_set_option(plan, gf.GF_OPT_PDL, c["pdl"])
    dg, du = (torch.empty((M, I), dtype=tdt, device="cuda") for _ in range(2))
    gf.gf_dswiglu_execute(plan, to_dev(dout, d), to_dev(Wd, d), to_dev(g, d), to_dev(u, d), dg, du)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    dg_o, du_o, _ = oracle.dswiglu_backward(dout, Wd, g, u, d)
    assert_close(to_host_f32(dg), oracle.decode(dg_o, d), what="d_gate")
    assert_close(to_host_f32(du), oracle.decode(du_o, d), what="d_up")
