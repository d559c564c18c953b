"""No kernel stores outside its outputs: every output (16-bit result, the
relu_aux words, a saved activation, the bias gradient) is placed between two
8 KB guard zones filled with a canary pattern; after a call on ragged shapes
(M, N not multiples of any tile width; N a multiple of 64 or not, which
selects the 3-D or the 2-D B loads) the guards must be untouched and the
outputs must match the oracle. Covers the single-CTA kernel (128- and
256-wide tiles), the CTA pair (256 x 256) and the wide pair (256 x 512), with
direct and staged (shared-memory transposed) stores, and each form's split-k
hand-over."""
import numpy as np
import pytest

import oracle
import synth
from helpers import (BGRAD_NMAX, BGRAD_REL, assert_close, mask_mismatch, to_dev, to_host_f32,
                     unpack_words)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import gemm_epilogue_tmem_gb300 as gf  # noqa: E402

GUARD = 4096  # elements on each side
CANARY16 = 0x5A5A
CANARY32 = 0x5A5A5A5A
KERNELS = [(1, 128), (1, 256), (2, 0), (3, 0)]


class Guarded:
    """A flat buffer [guard | n | guard] of 16- or 32-bit words; `view` is the
    middle n elements as `dtype`."""

    def __init__(self, n, dtype):
        self.bits32 = dtype in (torch.float32, torch.int32)
        raw = torch.int32 if self.bits32 else torch.int16
        self.canary = CANARY32 if self.bits32 else CANARY16
        self.flat = torch.full((2 * GUARD + n,), self.canary, dtype=raw, device="cuda")
        self.view = self.flat[GUARD:GUARD + n].view(dtype)

    def intact(self) -> bool:
        head, tail = self.flat[:GUARD], self.flat[-GUARD:]
        return bool(torch.all(head == self.canary)) and bool(torch.all(tail == self.canary))


def _set(plan, kernel, tile_n):
    gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, kernel)
    if tile_n:
        gf.gf_plan_set_option(plan, gf.GF_OPT_TILE_N, tile_n)


@pytest.mark.parametrize("kernel,tile_n", KERNELS)
@pytest.mark.parametrize("N", [776, 832])
def test_guards_relu_aux_bias(kernel, tile_n, N):
    M, K = 1000, 200
    X = synth.normal((M, K), synth.F16, 61, synth.TID_A, 1.0)
    W = synth.normal((K, N), synth.F16, 61, synth.TID_B, 1 / np.sqrt(K))
    b = synth.normal((N,), synth.F16, 61, synth.TID_BIAS, 0.1)
    out = Guarded(M * N, torch.float16)
    aux = Guarded(((M + 31) // 32) * N, torch.int32)
    plan = gf.gf_matmul_plan(M, N, K, gf.GF_F16, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL)
    _set(plan, kernel, tile_n)
    gf.gf_matmul_execute(plan, to_dev(X, 0), to_dev(W, 0), bias=to_dev(b, 0), out=out.view,
                         aux_out=aux.view)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    assert out.intact() and aux.intact()
    y_o, z_o = oracle.relu_bias(X, W, b, oracle.F16)
    assert_close(to_host_f32(out.view.view(M, N)), oracle.decode(y_o, 0), what="Y")
    words = aux.view.view((M + 31) // 32, N).cpu().numpy().view(np.uint32)
    outside, _ = mask_mismatch(unpack_words(words, M), z_o)
    assert outside == 0


@pytest.mark.parametrize("kernel,tile_n", KERNELS)
@pytest.mark.parametrize("mode", [gf.GF_BGRAD_TWO_PASS, gf.GF_BGRAD_ATOMIC])
def test_guards_drelu_bgrad(kernel, tile_n, mode):
    M, N, K = 1000, 776, 200
    G_A = synth.normal((M, K), synth.F16, 62, synth.TID_DY, 1.0)
    Wt = synth.normal((N, K), synth.F16, 62, synth.TID_W2, 1 / np.sqrt(K))
    words = synth.mask_words(M, N, 62)
    out = Guarded(M * N, torch.float16)
    bgrad = Guarded(N, torch.float32)
    plan = gf.gf_matmul_plan_ex(M, N, K, gf.GF_F16, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL,
                                gf.GF_B_NK)
    _set(plan, kernel, tile_n)
    gf.gf_plan_set_option(plan, gf.GF_OPT_BGRAD_MODE, mode)
    gf.gf_matmul_execute(plan, to_dev(G_A, 0), to_dev(Wt, 0), out=out.view,
                         aux_in=to_dev(words, 0), bgrad=bgrad.view)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    assert out.intact() and bgrad.intact()
    dz_o, bgrad_o, _ = oracle.drelu_bgrad(G_A, Wt, words, oracle.F16, oracle.B_NK)
    assert_close(to_host_f32(out.view.view(M, N)), oracle.decode(dz_o, 0), what="dZ")
    assert_close(bgrad.view.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL, what="bgrad")


@pytest.mark.parametrize("kernel,tile_n", KERNELS)
def test_guards_gelu_aux_bias(kernel, tile_n):
    M, N, K = 1000, 832, 200
    d = synth.BF16
    X = synth.normal((M, K), d, 63, synth.TID_A, 1.0)
    W = synth.normal((K, N), d, 63, synth.TID_B, 1 / np.sqrt(K))
    b = synth.normal((N,), d, 63, synth.TID_BIAS, 0.1)
    out = Guarded(M * N, torch.bfloat16)
    aux = Guarded(M * N, torch.bfloat16)
    plan = gf.gf_matmul_plan(M, N, K, d, gf.GF_EPILOG_GELU_AUX_BIAS, gf.GF_BIAS_COL)
    _set(plan, kernel, tile_n)
    gf.gf_matmul_execute(plan, to_dev(X, d), to_dev(W, d), bias=to_dev(b, d), out=out.view,
                         aux_out=aux.view)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    assert out.intact() and aux.intact()
    y_o, aux_o, _ = oracle.gelu_aux_bias(X, W, b, d)
    assert_close(to_host_f32(out.view.view(M, N)), oracle.decode(y_o, d), what="gelu out")
    assert_close(to_host_f32(aux.view.view(M, N)), oracle.decode(aux_o, d), what="pre-activation")


@pytest.mark.parametrize("kernel", [1, 2, 3])
def test_guards_swiglu_save(kernel):
    M, I, H = 1000, 776, 200
    d = synth.BF16
    x = synth.normal((M, H), d, 64, synth.TID_A, 1.0)
    Wg = synth.normal((I, H), d, 64, synth.TID_WG, 0.1)
    Wu = synth.normal((I, H), d, 64, synth.TID_WU, 0.1)
    h, g, u = (Guarded(M * I, torch.bfloat16) for _ in range(3))
    plan = gf.gf_swiglu_plan(M, I, H, d, save_gu=True)
    gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, kernel)
    gf.gf_swiglu_execute(plan, to_dev(x, d), to_dev(Wg, d), to_dev(Wu, d), h.view, g.view, u.view)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    assert h.intact() and g.intact() and u.intact()
    h_o, g_o, u_o, _, _ = oracle.swiglu_forward(x, Wg, Wu, d)
    assert_close(to_host_f32(h.view.view(M, I)), oracle.decode(h_o, d), what="h")
    assert_close(to_host_f32(g.view.view(M, I)), oracle.decode(g_o, d), what="g")
    assert_close(to_host_f32(u.view.view(M, I)), oracle.decode(u_o, d), what="u")


@pytest.mark.parametrize("kernel", [1, 2, 3])
def test_guards_dswiglu(kernel):
    M, I, H = 1000, 776, 200
    d = synth.BF16
    dout = synth.normal((M, H), d, 65, synth.TID_DOUT, 1.0)
    Wd = synth.normal((H, I), d, 65, synth.TID_WD, 1 / np.sqrt(H))
    g = synth.normal((M, I), d, 65, synth.TID_G_SAVED, 1.0)
    u = synth.normal((M, I), d, 65, synth.TID_U_SAVED, 1.0)
    dg, du = Guarded(M * I, torch.bfloat16), Guarded(M * I, torch.bfloat16)
    plan = gf.gf_dswiglu_plan(M, I, H, d)
    gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, kernel)
    gf.gf_dswiglu_execute(plan, to_dev(dout, d), to_dev(Wd, d), to_dev(g, d), to_dev(u, d),
                          dg.view, du.view)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    assert dg.intact() and du.intact()
    dg_o, du_o, _ = oracle.dswiglu_backward(dout, Wd, g, u, d)
    assert_close(to_host_f32(dg.view.view(M, I)), oracle.decode(dg_o, d), what="d_gate")
    assert_close(to_host_f32(du.view.view(M, I)), oracle.decode(du_o, d), what="d_up")


@pytest.mark.parametrize("kernel,tile_n", KERNELS)
@pytest.mark.parametrize("N", [776, 832])
def test_guards_split_k(kernel, tile_n, N):
    """Every tile's k split 3 ways (a ragged last split): the partial sums go
    through the plan's workspace and only the output's own elements are
    written."""
    M, K = 1000, 1000
    d = synth.BF16
    A = synth.normal((M, K), d, 65, synth.TID_A, 1.0)
    B = synth.normal((K, N), d, 65, synth.TID_B, 1 / np.sqrt(K))
    out = Guarded(M * N, torch.bfloat16)
    plan = gf.gf_matmul_plan_ex(M, N, K, d, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL, gf.GF_B_KN)
    _set(plan, kernel, tile_n)
    gf.gf_plan_set_option(plan, gf.GF_OPT_SPLIT_K, 3)
    assert gf.gf_plan_describe(plan)["k_splits"] == 3
    gf.gf_matmul_execute(plan, to_dev(A, d), to_dev(B, d), out=out.view)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    assert out.intact()
    assert_close(to_host_f32(out.view.view(M, N)), oracle.decode(oracle.epilog_none(A, B, d), d),
                 what="NONE, split k")
