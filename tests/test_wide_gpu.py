"""The CTA-pair kernel with 256 x 512 tiles (GF_OPT_KERNEL = 3): one
512-column accumulator per pair, drained in two halves while the next tile
starts on the first half and the last k-slices of a tile finish the first
half early (with the two SwiGLU operands: 256 x 256 tiles). Checked against
the oracle on
ragged shapes (N not a multiple of 512 or of 64, K not a multiple of 64, fewer
k-slices than ring stages, K = 0), on every epilog family it serves, with many
tiles per CTA pair, under both schedules, and through a bounded wait that runs
out."""
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

WIDE = 3
SHAPES = [(3000, 2568, 264), (1000, 2560, 64), (700, 1088, 520), (520, 1032, 0),
          # longer k loops: head, middle and tail of the half schedule all present
          (1000, 1088, 1344), (600, 2568, 2056)]


def _wide(plan):
    gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, WIDE)
    d = gf.gf_plan_describe(plan)
    assert (d["tile_m"], d["tile_n"]) == (256, 512), d
    return d


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("b_layout", [gf.GF_B_KN, gf.GF_B_NK])
def test_wide_relu_aux_bias(M, N, K, b_layout):
    seed = 41
    X = synth.normal((M, K), synth.F16, seed, synth.TID_A, 1.0)
    shape_b = (K, N) if b_layout == gf.GF_B_KN else (N, K)
    W = synth.normal(shape_b, synth.F16, seed, synth.TID_B, 1 / np.sqrt(max(K, 1)))
    b = synth.normal((N,), synth.F16, seed, synth.TID_BIAS, 0.1)
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    aux = torch.empty(((M + 31) // 32, N), dtype=torch.int32, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, N, K, gf.GF_F16, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL,
                                b_layout)
    _wide(plan)
    gf.gf_matmul_execute(plan, to_dev(X, 0) if K else None, to_dev(W, 0) if K else None,
                         bias=to_dev(b, 0), out=out, aux_out=aux)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    ob = oracle.B_KN if b_layout == gf.GF_B_KN else oracle.B_NK
    y_o, z_o = oracle.relu_bias(X, W, b, oracle.F16, ob)
    assert_close(to_host_f32(out), oracle.decode(y_o, 0), what="Y")
    outside, _ = mask_mismatch(unpack_words(to_host_words(aux), M), z_o)
    assert outside == 0


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("mode", [gf.GF_BGRAD_TWO_PASS, gf.GF_BGRAD_ATOMIC])
def test_wide_drelu_bgrad(M, N, K, mode):
    seed = 42
    G_A = synth.normal((M, K), synth.F16, seed, synth.TID_DY, 1.0)
    Wt = synth.normal((N, K), synth.F16, seed, synth.TID_W2, 1 / np.sqrt(max(K, 1)))
    words = synth.mask_words(M, N, seed)
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    bgrad = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, N, K, gf.GF_F16, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL,
                                gf.GF_B_NK)
    _wide(plan)
    gf.gf_plan_set_option(plan, gf.GF_OPT_BGRAD_MODE, mode)
    gf.gf_matmul_execute(plan, to_dev(G_A, 0) if K else None, to_dev(Wt, 0) if K else None,
                         out=out, aux_in=to_dev(words, 0), bgrad=bgrad)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    dz_o, bgrad_o, _ = oracle.drelu_bgrad(G_A, Wt, words, oracle.F16, oracle.B_NK)
    assert_close(to_host_f32(out), oracle.decode(dz_o, 0), what="dZ")
    assert_close(bgrad.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL, what="bgrad")


@pytest.mark.parametrize("M,N,K", SHAPES[:3] + SHAPES[4:])
def test_wide_none_and_bias(M, N, K):
    d = synth.BF16
    A = synth.normal((M, K), d, 43, synth.TID_A, 1.0)
    B = synth.normal((K, N), d, 43, synth.TID_B, 1 / np.sqrt(K))
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, N, K, d, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL, gf.GF_B_KN)
    _wide(plan)
    gf.gf_matmul_execute(plan, to_dev(A, d), to_dev(B, d), out=out)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    assert_close(to_host_f32(out), oracle.decode(oracle.epilog_none(A, B, d), d), what="NONE")


@pytest.mark.parametrize("M,N,K", SHAPES[:3] + SHAPES[4:])
def test_wide_gelu_forward_backward(M, N, K):
    d = synth.BF16
    X = synth.normal((M, K), d, 44, synth.TID_A, 1.0)
    W = synth.normal((K, N), d, 44, synth.TID_B, 1 / np.sqrt(K))
    b = synth.normal((N,), d, 44, synth.TID_BIAS, 0.1)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    aux = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, N, K, d, gf.GF_EPILOG_GELU_AUX_BIAS, gf.GF_BIAS_COL, gf.GF_B_KN)
    _wide(plan)
    gf.gf_matmul_execute(plan, to_dev(X, d), to_dev(W, d), bias=to_dev(b, d), out=out, aux_out=aux)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    y_o, aux_o, _ = oracle.gelu_aux_bias(X, W, b, d)
    assert_close(to_host_f32(out), oracle.decode(y_o, d), what="gelu out")
    assert_close(to_host_f32(aux), oracle.decode(aux_o, d), what="pre-activation")

    dY = synth.normal((M, K), d, 45, synth.TID_DY, 1.0)
    Wb = synth.normal((N, K), d, 45, synth.TID_W2, 1 / np.sqrt(K))
    pre = synth.normal((M, N), d, 45, synth.TID_PREACT, 1.0)
    dz = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    bgrad = torch.empty((N,), dtype=torch.float32, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, N, K, d, gf.GF_EPILOG_DGELU_BGRAD, gf.GF_BIAS_COL, gf.GF_B_NK)
    _wide(plan)
    gf.gf_matmul_execute(plan, to_dev(dY, d), to_dev(Wb, d), out=dz, aux_in=to_dev(pre, d),
                         bgrad=bgrad)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    dz_o, bgrad_o, _ = oracle.dgelu_bgrad(dY, Wb, pre, d, oracle.B_NK)
    assert_close(to_host_f32(dz), oracle.decode(dz_o, d), what="dgelu out")
    assert_close(bgrad.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL, what="dgelu bgrad")


def test_wide_dswiglu():
    M, I, H = 1000, 1536, 320
    d = synth.BF16
    dout = synth.normal((M, H), d, 46, synth.TID_DOUT, 1.0)
    Wd = synth.normal((H, I), d, 46, synth.TID_WD, 1 / np.sqrt(H))
    g = synth.normal((M, I), d, 46, synth.TID_G_SAVED, 1.0)
    u = synth.normal((M, I), d, 46, synth.TID_U_SAVED, 1.0)
    dg = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
    du = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
    plan = gf.gf_dswiglu_plan(M, I, H, d)
    _wide(plan)
    gf.gf_dswiglu_execute(plan, to_dev(dout, d), to_dev(Wd, d), to_dev(g, d), to_dev(u, d), dg, du)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    dg_o, du_o, _ = oracle.dswiglu_backward(dout, Wd, g, u, d)
    assert_close(to_host_f32(dg), oracle.decode(dg_o, d), what="d_gate")
    assert_close(to_host_f32(du), oracle.decode(du_o, d), what="d_up")


@pytest.mark.parametrize("save", [True, False])
def test_wide_two_operands_same_bits(save):
    """Gate+up SwiGLU on 256 x 256 wide tiles (each CTA loads two 128-row
    parts of its weight) gives the same bits as on the 256 x 128 two-operand
    tiles: every output sums its k-slices in the same order. Several tiles
    per CTA pair, a ragged last column block."""
    M, I, H = 4096, 8200, 2048
    d = synth.BF16
    x = to_dev(synth.normal((M, H), d, 49, synth.TID_A, 1.0), d)
    Wg = to_dev(synth.normal((I, H), d, 49, synth.TID_WG, 0.02), d)
    Wu = to_dev(synth.normal((I, H), d, 49, synth.TID_WU, 0.02), d)
    outs = []
    for kern in (2, WIDE):
        h, g, u = (torch.full((M, I), float("nan"), dtype=torch.bfloat16, device="cuda")
                   for _ in range(3))
        plan = gf.gf_swiglu_plan(M, I, H, d, save_gu=save)
        gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, kern)
        dsc = gf.gf_plan_describe(plan)
        assert (dsc["tile_m"], dsc["tile_n"]) == ((256, 256) if kern == WIDE else (256, 128)), dsc
        gf.gf_swiglu_execute(plan, x, Wg, Wu, h, g if save else None, u if save else None)
        assert gf.gf_plan_status(plan) == gf.GF_OK
        plan.free()
        outs.append((h, g, u) if save else (h,))
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


MT, NT, KT = 8192, 8192, 128  # 512 wide tiles: several per CTA pair


@pytest.fixture(scope="module")
def many():
    X = synth.normal((MT, KT), synth.F16, 47, synth.TID_A, 1.0)
    W = synth.normal((KT, NT), synth.F16, 47, synth.TID_B, 1 / np.sqrt(KT))
    Wt = synth.normal((NT, KT), synth.F16, 47, synth.TID_W2, 1 / np.sqrt(KT))
    b = synth.normal((NT,), synth.F16, 47, synth.TID_BIAS, 0.1)
    words = synth.mask_words(MT, NT, 47)
    y_o, z_o = oracle.relu_bias(X, W, b, oracle.F16)
    dz_o, bgrad_o, _ = oracle.drelu_bgrad(X, Wt, words, oracle.F16, oracle.B_NK)
    return X, W, Wt, b, words, y_o, z_o, dz_o, bgrad_o


@pytest.mark.parametrize("schedule,group_m", [(0, 0), (3, 0), (2, 16), (1, 0)])
def test_wide_many_tiles(many, schedule, group_m):
    X, W, Wt, b, words, y_o, z_o, dz_o, bgrad_o = many
    out = torch.empty((MT, NT), dtype=torch.float16, device="cuda")
    aux = torch.empty((MT // 32, NT), dtype=torch.int32, device="cuda")
    fwd = gf.gf_matmul_plan(MT, NT, KT, gf.GF_F16, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL)
    d = _wide(fwd)
    assert (MT // 256) * (NT // 512) >= 3 * (d["grid"] // 2) or schedule == 1
    gf.gf_plan_set_option(fwd, gf.GF_OPT_SCHEDULE, schedule)
    if group_m:
        gf.gf_plan_set_option(fwd, gf.GF_OPT_GROUP_M, group_m)
    for _ in range(2):
        out.zero_()
        gf.gf_matmul_execute(fwd, to_dev(X, 0), to_dev(W, 0), bias=to_dev(b, 0), out=out,
                             aux_out=aux)
        assert gf.gf_plan_status(fwd) == gf.GF_OK
        assert_close(to_host_f32(out), oracle.decode(y_o, 0), what="Y")
        outside, _ = mask_mismatch(unpack_words(to_host_words(aux), MT), z_o)
        assert outside == 0
    fwd.free()

    bgrad = torch.empty((NT,), dtype=torch.float32, device="cuda")
    bwd = gf.gf_matmul_plan_ex(MT, NT, KT, gf.GF_F16, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL,
                               gf.GF_B_NK)
    _wide(bwd)
    gf.gf_plan_set_option(bwd, gf.GF_OPT_SCHEDULE, schedule)
    gf.gf_matmul_execute(bwd, to_dev(X, 0), to_dev(Wt, 0), out=out, aux_in=to_dev(words, 0),
                         bgrad=bgrad)
    assert gf.gf_plan_status(bwd) == gf.GF_OK
    bwd.free()
    assert_close(to_host_f32(out), oracle.decode(dz_o, 0), what="dZ")
    assert_close(bgrad.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL, what="bgrad")


def test_wide_wait_limit():
    """A skipped stage load: the bounded wait gives up, the status says so,
    and the next call on the same plan is correct."""
    Mw, Nw, Kw = 1024, 2048, 512
    X = synth.normal((Mw, Kw), synth.F16, 34, synth.TID_A, 1.0)
    W = synth.normal((Kw, Nw), synth.F16, 34, synth.TID_B, 1 / np.sqrt(Kw))
    b = synth.normal((Nw,), synth.F16, 34, synth.TID_BIAS, 0.1)
    Xd, Wd, bd = to_dev(X, 0), to_dev(W, 0), to_dev(b, 0)
    out = torch.empty((Mw, Nw), dtype=torch.float16, device="cuda")
    plan = gf.gf_matmul_plan(Mw, Nw, Kw, gf.GF_F16, gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_COL)
    _wide(plan)
    gf.gf_plan_set_option(plan, gf.GF_OPT_WAIT_LIMIT_US, 20000)
    gf.gf_plan_set_option(plan, gf.GF_OPT_FAULT_DROP_LOAD, 3)
    gf.gf_matmul_execute(plan, Xd, Wd, bias=bd, out=out)
    assert gf.gf_plan_status(plan) == gf.GF_ERR_DEVICE_TIMEOUT
    gf.gf_plan_set_option(plan, gf.GF_OPT_FAULT_DROP_LOAD, 0)
    out.fill_(float("nan"))
    gf.gf_matmul_execute(plan, Xd, Wd, bias=bd, out=out)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    y_o, _ = oracle.relu_bias(X, W, b, oracle.F16)
    assert_close(to_host_f32(out), oracle.decode(y_o, oracle.F16), what="Y after the time-out")


def test_wide_many_tiles_long_k():
    """Several wide tiles per CTA pair with 21 k-slices each: the head and
    tail half-passes of consecutive tiles interleave with their drains."""
    M, N, K = 4096, 8192, 1344
    X = synth.normal((M, K), synth.F16, 48, synth.TID_A, 1.0)
    W = synth.normal((K, N), synth.F16, 48, synth.TID_B, 1 / np.sqrt(K))
    b = synth.normal((N,), synth.F16, 48, synth.TID_BIAS, 0.1)
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    aux = torch.empty((M // 32, N), dtype=torch.int32, device="cuda")
    fwd = gf.gf_matmul_plan(M, N, K, gf.GF_F16, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL)
    d = _wide(fwd)
    assert (M // 256) * (N // 512) >= 3 * (d["grid"] // 2)
    gf.gf_matmul_execute(fwd, to_dev(X, 0), to_dev(W, 0), bias=to_dev(b, 0), out=out, aux_out=aux)
    assert gf.gf_plan_status(fwd) == gf.GF_OK
    fwd.free()
    y_o, z_o = oracle.relu_bias(X, W, b, oracle.F16)
    assert_close(to_host_f32(out), oracle.decode(y_o, 0), what="Y")
    outside, _ = mask_mismatch(unpack_words(to_host_words(aux), M), z_o)
    assert outside == 0

    Wt = synth.normal((N, K), synth.F16, 48, synth.TID_W2, 1 / np.sqrt(K))
    words = synth.mask_words(M, N, 48)
    bgrad = torch.empty((N,), dtype=torch.float32, device="cuda")
    bwd = gf.gf_matmul_plan_ex(M, N, K, gf.GF_F16, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL,
                               gf.GF_B_NK)
    _wide(bwd)
    gf.gf_matmul_execute(bwd, to_dev(X, 0), to_dev(Wt, 0), out=out, aux_in=to_dev(words, 0),
                         bgrad=bgrad)
    assert gf.gf_plan_status(bwd) == gf.GF_OK
    bwd.free()
    dz_o, bgrad_o, _ = oracle.drelu_bgrad(X, Wt, words, oracle.F16, oracle.B_NK)
    assert_close(to_host_f32(out), oracle.decode(dz_o, 0), what="dZ")
    assert_close(bgrad.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL, what="bgrad")


def test_wide_row_bias():
    """A per-row bias (bias[m]) through the wide tiles, whose column-bias
    prefetch into shared memory must then stay unused."""
    M, N, K = 1000, 1088, 1344
    X = synth.normal((M, K), synth.F16, 49, synth.TID_A, 1.0)
    W = synth.normal((K, N), synth.F16, 49, synth.TID_B, 1 / np.sqrt(K))
    b = synth.normal((M,), synth.F16, 49, synth.TID_BIAS, 0.5)
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    plan = gf.gf_matmul_plan(M, N, K, gf.GF_F16, gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_ROW)
    _wide(plan)
    gf.gf_matmul_execute(plan, to_dev(X, 0), to_dev(W, 0), bias=to_dev(b, 0), out=out)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    y_o, _ = oracle.relu_bias(X, W, b, oracle.F16, oracle.B_KN, oracle.BIAS_ROW)
    assert_close(to_host_f32(out), oracle.decode(y_o, 0), what="Y (row bias)")
