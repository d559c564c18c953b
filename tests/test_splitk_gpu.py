"""Split k in the single-CTA kernel: the k-blocks of each output tile shared
by several CTAs whose fp32 partial sums meet in the plan's workspace, the
last CTA of a tile running the epilogue. Every epilog against the oracle on
ragged shapes (a k tail in the last split, rows and columns past M and N),
both B layouts and tile widths, more work units than SMs, bit-for-bit
repeatability across launches, guard zones around every output, the
time-out path and the plan's own choice on the (1024, 512, 2048) row-bias
GEMM. The CTA-pair kernel's split (256 x 256 and 256 x 512 tiles,
EPILOG_NONE): every tile split, and the plan's split of a mostly empty last
wave, against the oracle."""
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

GUARD = 4096


@pytest.fixture(scope="module", autouse=True)
def _built():
    gf.build()
    synth.build_host()
    oracle.build()


def _plan(M, N, K, dtype, epilog, axis, layout, split, tile_n=128):
    plan = gf.gf_matmul_plan_ex(M, N, K, dtype, epilog, axis, layout)
    gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, 1)
    gf.gf_plan_set_option(plan, gf.GF_OPT_TILE_N, tile_n)
    gf.gf_plan_set_option(plan, gf.GF_OPT_SPLIT_K, split)
    return plan


def _expected_splits(K, split):
    kb = (K + 63) // 64
    kps = (kb + split - 1) // split
    return (kb + kps - 1) // kps


def _fwd_inputs(M, N, K, dtype, layout, seed, axis):
    A = synth.normal((M, K), dtype, seed, synth.TID_A, 1.0)
    sb = 1 / np.sqrt(K)
    B = (synth.normal((K, N), dtype, seed, synth.TID_B, sb) if layout == gf.GF_B_KN
         else synth.normal((N, K), dtype, seed, synth.TID_B, sb))
    bias = synth.normal((M if axis == gf.GF_BIAS_ROW else N,), dtype, seed, synth.TID_BIAS, 0.1)
    return A, B, bias


def _oracle_fwd(epilog, A, B, bias, dtype, layout, axis):
    """(out bits, aux, z) of a forward epilog."""
    acc = oracle.gemm(A, B, dtype, layout)
    if epilog == gf.GF_EPILOG_NONE:
        return oracle.round_to(acc, dtype), None, acc
    z = oracle.add_bias(acc, bias, dtype, axis)
    if epilog == gf.GF_EPILOG_BIAS:
        return oracle.round_to(z, dtype), None, z
    if epilog in (gf.GF_EPILOG_RELU_BIAS, gf.GF_EPILOG_RELU_AUX_BIAS):
        return oracle.round_to(oracle.relu(z), dtype), None, z
    y = oracle.round_to(oracle.gelu(z), dtype)
    return y, oracle.round_to(z, dtype), z


FWD = [gf.GF_EPILOG_NONE, gf.GF_EPILOG_BIAS, gf.GF_EPILOG_RELU_BIAS, gf.GF_EPILOG_RELU_AUX_BIAS,
       gf.GF_EPILOG_GELU_BIAS, gf.GF_EPILOG_GELU_AUX_BIAS]


@pytest.mark.parametrize("epilog", FWD)
@pytest.mark.parametrize("split", [2, 3, 5])
def test_forward_epilogs(epilog, split):
    M, N, K = 300, 200, 1000  # 16 k-blocks, the last one 40 wide
    dtype = 1 if epilog in (gf.GF_EPILOG_GELU_BIAS, gf.GF_EPILOG_GELU_AUX_BIAS) else 0
    axis, layout = gf.GF_BIAS_COL, gf.GF_B_KN
    A, B, bias = _fwd_inputs(M, N, K, dtype, layout, 11, axis)
    tdt = torch_dtype(dtype)
    out = torch.empty((M, N), dtype=tdt, device="cuda")
    aux_words = torch.zeros(((M + 31) // 32, N), dtype=torch.int32, device="cuda")
    aux_pre = torch.empty((M, N), dtype=tdt, device="cuda")
    plan = _plan(M, N, K, dtype, epilog, axis, layout, split)
    assert gf.gf_plan_describe(plan)["k_splits"] == _expected_splits(K, split)
    aux = (aux_words if epilog == gf.GF_EPILOG_RELU_AUX_BIAS else
           aux_pre if epilog == gf.GF_EPILOG_GELU_AUX_BIAS else None)
    gf.gf_matmul_execute(plan, to_dev(A, dtype), to_dev(B, dtype), bias=to_dev(bias, dtype),
                         out=out, aux_out=aux)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    y_o, pre_o, z_o = _oracle_fwd(epilog, A, B, bias, dtype, layout, axis)
    assert_close(to_host_f32(out), oracle.decode(y_o, dtype), what=f"out split {split}")
    if epilog == gf.GF_EPILOG_RELU_AUX_BIAS:
        outside, _ = mask_mismatch(unpack_words(to_host_words(aux_words), M), z_o)
        assert outside == 0
    if epilog == gf.GF_EPILOG_GELU_AUX_BIAS:
        assert_close(to_host_f32(aux_pre), oracle.decode(pre_o, dtype), what="pre-activation")


@pytest.mark.parametrize("layout", [gf.GF_B_KN, gf.GF_B_NK])
@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("axis", [gf.GF_BIAS_COL, gf.GF_BIAS_ROW])
def test_layouts_tiles_axes(layout, tile_n, axis):
    M, N, K = 520, 392, 2056
    A, B, bias = _fwd_inputs(M, N, K, 0, layout, 12, axis)
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    aux = torch.zeros(((M + 31) // 32, N), dtype=torch.int32, device="cuda")
    plan = _plan(M, N, K, 0, gf.GF_EPILOG_RELU_AUX_BIAS, axis, layout, 4, tile_n)
    assert gf.gf_plan_describe(plan)["k_splits"] == 4
    gf.gf_matmul_execute(plan, to_dev(A, 0), to_dev(B, 0), bias=to_dev(bias, 0), out=out,
                         aux_out=aux)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    y_o, _, z_o = _oracle_fwd(gf.GF_EPILOG_RELU_AUX_BIAS, A, B, bias, 0, layout, axis)
    assert_close(to_host_f32(out), oracle.decode(y_o, 0), what="Y")
    outside, _ = mask_mismatch(unpack_words(to_host_words(aux), M), z_o)
    assert outside == 0


@pytest.mark.parametrize("epilog", [gf.GF_EPILOG_DRELU_BGRAD, gf.GF_EPILOG_DGELU_BGRAD])
@pytest.mark.parametrize("mode", [gf.GF_BGRAD_TWO_PASS, gf.GF_BGRAD_ATOMIC])
@pytest.mark.parametrize("split", [2, 6])
def test_backward_epilogs(epilog, mode, split):
    M, N, K = 777, 456, 1280
    dtype = 0 if epilog == gf.GF_EPILOG_DRELU_BGRAD else 1
    dY = synth.normal((M, K), dtype, 13, synth.TID_DY, 1.0)
    W = synth.normal((N, K), dtype, 13, synth.TID_B, 1 / np.sqrt(K))
    if epilog == gf.GF_EPILOG_DRELU_BGRAD:
        aux_h = synth.mask_words(M, N, 13)
    else:
        aux_h = synth.normal((M, N), dtype, 13, synth.TID_PREACT, 1.0)
    tdt = torch_dtype(dtype)
    out = torch.empty((M, N), dtype=tdt, device="cuda")
    bgrad = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    plan = _plan(M, N, K, dtype, epilog, gf.GF_BIAS_COL, gf.GF_B_NK, split)
    gf.gf_plan_set_option(plan, gf.GF_OPT_BGRAD_MODE, mode)
    assert gf.gf_plan_describe(plan)["k_splits"] == _expected_splits(K, split)
    gf.gf_matmul_execute(plan, to_dev(dY, dtype), to_dev(W, dtype), out=out,
                         aux_in=to_dev(aux_h, dtype), bgrad=bgrad)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    if epilog == gf.GF_EPILOG_DRELU_BGRAD:
        dz_o, bgrad_o, _ = oracle.drelu_bgrad(dY, W, aux_h, dtype, oracle.B_NK)
    else:
        dz_o, bgrad_o, _ = oracle.dgelu_bgrad(dY, W, aux_h, dtype, oracle.B_NK)
    assert_close(to_host_f32(out), oracle.decode(dz_o, dtype), what="dZ")
    assert_close(bgrad.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL, what="bgrad")


def test_more_units_than_sms_and_repeatable():
    """512 work units on at most 152 CTAs: both accumulator buffers and the
    counters are reused within a launch and across launches; the sum runs in
    split order, so every launch gives the same bits."""
    M, N, K = 2048, 2048, 512
    A, B, bias = _fwd_inputs(M, N, K, 0, gf.GF_B_KN, 14, gf.GF_BIAS_COL)
    Ad, Bd, bd = to_dev(A, 0), to_dev(B, 0), to_dev(bias, 0)
    plan = _plan(M, N, K, 0, gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_COL, gf.GF_B_KN, 2)
    assert gf.gf_plan_describe(plan)["k_splits"] == 2
    outs = []
    for _ in range(3):
        out = torch.empty((M, N), dtype=torch.float16, device="cuda")
        gf.gf_matmul_execute(plan, Ad, Bd, bias=bd, out=out)
        outs.append(out)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    rows = synth.sample_rows(M, 64, 14)
    y_o, _ = oracle.relu_bias(np.ascontiguousarray(A[rows]), B, bias, 0)
    assert_close(to_host_f32(outs[0])[rows], oracle.decode(y_o, 0), what="sampled rows")


def test_guard_zones():
    M, N, K = 1000, 776, 2000
    A, B, bias = _fwd_inputs(M, N, K, 0, gf.GF_B_KN, 15, gf.GF_BIAS_COL)
    flat = torch.full((2 * GUARD + M * N,), 0x5A5A, dtype=torch.int16, device="cuda")
    wflat = torch.full((2 * GUARD + ((M + 31) // 32) * N,), 0x5A5A5A5A, dtype=torch.int32,
                       device="cuda")
    out = flat[GUARD:GUARD + M * N].view(torch.float16)
    aux = wflat[GUARD:GUARD + ((M + 31) // 32) * N]
    plan = _plan(M, N, K, 0, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL, gf.GF_B_KN, 3)
    gf.gf_matmul_execute(plan, to_dev(A, 0), to_dev(B, 0), bias=to_dev(bias, 0), out=out,
                         aux_out=aux)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    for f, c in ((flat, 0x5A5A), (wflat, 0x5A5A5A5A)):
        assert bool(torch.all(f[:GUARD] == c)) and bool(torch.all(f[-GUARD:] == c))
    y_o, _, z_o = _oracle_fwd(gf.GF_EPILOG_RELU_AUX_BIAS, A, B, bias, 0, gf.GF_B_KN,
                              gf.GF_BIAS_COL)
    assert_close(to_host_f32(out.view(M, N)), oracle.decode(y_o, 0), what="Y")
    outside, _ = mask_mismatch(unpack_words(to_host_words(aux.view((M + 31) // 32, N)), M), z_o)
    assert outside == 0


def test_timeout_then_reuse():
    """Every CTA skips a stage load: the bounded waits run out, the host reads
    GF_ERR_DEVICE_TIMEOUT, the tile counters left part-way are reset, and the
    next launch of the same plan is correct."""
    M, N, K = 256, 256, 2048
    A, B, bias = _fwd_inputs(M, N, K, 0, gf.GF_B_KN, 16, gf.GF_BIAS_COL)
    Ad, Bd, bd = to_dev(A, 0), to_dev(B, 0), to_dev(bias, 0)
    plan = _plan(M, N, K, 0, gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_COL, gf.GF_B_KN, 4)
    gf.gf_plan_set_option(plan, gf.GF_OPT_WAIT_LIMIT_US, 20000)
    gf.gf_plan_set_option(plan, gf.GF_OPT_FAULT_DROP_LOAD, 3)
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    gf.gf_matmul_execute(plan, Ad, Bd, bias=bd, out=out)
    assert gf.gf_plan_status(plan) == gf.GF_ERR_DEVICE_TIMEOUT
    gf.gf_plan_set_option(plan, gf.GF_OPT_FAULT_DROP_LOAD, 0)
    gf.gf_matmul_execute(plan, Ad, Bd, bias=bd, out=out)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    y_o, _ = oracle.relu_bias(A, B, bias, 0)
    assert_close(to_host_f32(out), oracle.decode(y_o, 0), what="Y after the time-out")


def test_plan_choice():
    """The plan splits the (1024, 512, 2048) row-bias GEMM (32 tiles of
    128 x 128, 32 k-blocks) four ways; not the tiny MLP layer (8 k-blocks),
    not a CTA-pair plan, not the two-operand SwiGLU."""
    p = gf.gf_matmul_plan(1024, 512, 2048, 0, gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_ROW)
    d = gf.gf_plan_describe(p)
    assert (d["tile_m"], d["tile_n"], d["k_splits"], d["grid"]) == (128, 128, 4, 128)
    assert d["workspace_bytes"] >= 32 * 4 * 128 * 128 * 4
    gf.gf_plan_set_option(p, gf.GF_OPT_SPLIT_K, 1)
    assert gf.gf_plan_describe(p)["k_splits"] == 1
    p.free()
    p = gf.gf_matmul_plan(256, 384, 512, 0, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL)
    assert gf.gf_plan_describe(p)["k_splits"] == 1
    p.free()
    p = gf.gf_matmul_plan(8192, 8192, 4096, 0, gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_COL)
    gf.gf_plan_set_option(p, gf.GF_OPT_SPLIT_K, 4)
    d = gf.gf_plan_describe(p)
    assert d["tile_m"] == 256 and d["k_splits"] == 1
    p.free()
    p = gf.gf_swiglu_plan(256, 512, 4096, 1)
    gf.gf_plan_set_option(p, gf.GF_OPT_KERNEL, 1)
    gf.gf_plan_set_option(p, gf.GF_OPT_SPLIT_K, 4)
    assert gf.gf_plan_describe(p)["k_splits"] == 1
    p.free()
    with pytest.raises(gf.GfError):
        p = gf.gf_matmul_plan(128, 128, 128, 0, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL)
        try:
            gf.gf_plan_set_option(p, gf.GF_OPT_SPLIT_K, 65)
        finally:
            p.free()


def test_autotune_keeps_a_correct_split():
    M, N, K = 1024, 512, 2048
    A, B, bias = _fwd_inputs(M, N, K, 0, gf.GF_B_KN, 17, gf.GF_BIAS_ROW)
    Ad, Bd, bd = to_dev(A, 0), to_dev(B, 0), to_dev(bias, 0)
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    plan = gf.gf_matmul_plan(M, N, K, 0, gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_ROW)
    gf.gf_matmul_autotune(plan, Ad, Bd, bias=bd, out=out, reps=3)
    out.fill_(float("nan"))
    gf.gf_matmul_execute(plan, Ad, Bd, bias=bd, out=out)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    y_o, _ = oracle.relu_bias(A, B, bias, 0, axis=oracle.BIAS_ROW)
    assert_close(to_host_f32(out), oracle.decode(y_o, 0), what="Y after autotune")


# ----------------------------------------------------------- CTA-pair kernel
def _pair_plan(M, N, K, dtype, layout, split, kernel=2):
    plan = gf.gf_matmul_plan_ex(M, N, K, dtype, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL, layout)
    gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, kernel)
    gf.gf_plan_set_option(plan, gf.GF_OPT_SPLIT_K, split)
    d = gf.gf_plan_describe(plan)
    assert (d["tile_m"], d["tile_n"]) == (256, 256 if kernel == 2 else 512), d
    return plan


@pytest.mark.parametrize("M,N,K", [(1000, 1032, 1000), (512, 2568, 4104), (300, 264, 520)])
@pytest.mark.parametrize("layout", [gf.GF_B_KN, gf.GF_B_NK])
@pytest.mark.parametrize("split", [2, 3, 8])
@pytest.mark.parametrize("kernel", [2, 3])
def test_pair_split_every_tile(M, N, K, layout, split, kernel):
    """CTA-pair tiles (256 x 256, or 256 x 512 with the accumulator drained
    in halves) with every tile split k ways (a ragged last split, rows and
    columns past M and N): against the oracle, twice in a row (the per-tile
    counters are back at zero after each launch), the same bits both
    times."""
    d = synth.BF16
    A, B, _ = _fwd_inputs(M, N, K, d, layout, 71, gf.GF_BIAS_COL)
    plan = _pair_plan(M, N, K, d, layout, split, kernel)
    assert gf.gf_plan_describe(plan)["k_splits"] == _expected_splits(K, split)
    Ad, Bd = to_dev(A, d), to_dev(B, d)
    outs = []
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        gf.gf_matmul_execute(plan, Ad, Bd, out=out)
        assert gf.gf_plan_status(plan) == gf.GF_OK
        outs.append(out)
    plan.free()
    ob = oracle.B_KN if layout == gf.GF_B_KN else oracle.B_NK
    assert_close(to_host_f32(outs[0]), oracle.decode(oracle.epilog_none(A, B, d, ob), d),
                 what="NONE, pair split")
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


@pytest.mark.parametrize("kernel", [2, 3])
def test_pair_split_timeout_then_reuse(kernel):
    """The CTA-pair kernel with every tile split: each CTA skips a stage load,
    the bounded waits run out (the epilogue warps agree on it before any
    barrier of the hand-over), the host reads GF_ERR_DEVICE_TIMEOUT and resets
    the per-tile counters left part-way, and the next launch of the same plan
    matches the oracle."""
    d = synth.BF16
    M, N, K = 512, 1024, 2048
    A, B, _ = _fwd_inputs(M, N, K, d, gf.GF_B_NK, 74, gf.GF_BIAS_COL)
    Ad, Bd = to_dev(A, d), to_dev(B, d)
    plan = _pair_plan(M, N, K, d, gf.GF_B_NK, 2, kernel)
    assert gf.gf_plan_describe(plan)["k_splits"] == 2
    gf.gf_plan_set_option(plan, gf.GF_OPT_WAIT_LIMIT_US, 20000)
    gf.gf_plan_set_option(plan, gf.GF_OPT_FAULT_DROP_LOAD, 3)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    gf.gf_matmul_execute(plan, Ad, Bd, out=out)
    assert gf.gf_plan_status(plan) == gf.GF_ERR_DEVICE_TIMEOUT
    gf.gf_plan_set_option(plan, gf.GF_OPT_FAULT_DROP_LOAD, 0)
    out.fill_(float("nan"))
    gf.gf_matmul_execute(plan, Ad, Bd, out=out)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    assert_close(to_host_f32(out), oracle.decode(oracle.epilog_none(A, B, d, oracle.B_NK), d),
                 what="NONE after the time-out")


def test_pair_split_last_wave_plan_choice():
    """The plan's own choice on a product whose 256 x 256 tiles fill two waves
    of the resident CTA pairs and leave 3 tiles for a third: those are split
    (the tiles before run whole), and the result matches the oracle on
    sampled rows."""
    d = synth.BF16
    big = gf.gf_matmul_plan_ex(4096, 8192, 128, d, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL, gf.GF_B_NK)
    gf.gf_plan_set_option(big, gf.GF_OPT_KERNEL, 2)
    pairs = gf.gf_plan_describe(big)["grid"] // 2  # 512 tiles: every resident pair
    big.free()
    M, K = 256, 2048
    N = 256 * (2 * pairs + 3)
    A = synth.normal((M, K), d, 72, synth.TID_A, 1.0)
    B = synth.normal((N, K), d, 72, synth.TID_B, 1 / np.sqrt(K))
    plan = gf.gf_matmul_plan_ex(M, N, K, d, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL, gf.GF_B_NK)
    gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, 2)
    ks = gf.gf_plan_describe(plan)["k_splits"]
    assert 2 <= ks <= 8, ks
    outs = []
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        gf.gf_matmul_execute(plan, to_dev(A, d), to_dev(B, d), out=out)
        assert gf.gf_plan_status(plan) == gf.GF_OK
        outs.append(out)
    plan.free()
    rows = synth.sample_rows(M, 32, 72)
    o_rows = oracle.decode(oracle.epilog_none(A[rows], B, d, oracle.B_NK), d)
    assert_close(to_host_f32(outs[0])[rows], o_rows, what="NONE, plan's split")
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


@pytest.mark.parametrize("M", [2048, 8192])
def test_pair_split_swiglu_down_shape(M):
    """The SwiGLU MLP's down projection (h[M, 17408] · Wdᵀ, Wd stored
    [5120, 17408]): at M = 2048 80 tiles of 256 x 512 fill one wave of the
    resident CTA pairs and leave a few tiles over, at M = 8192 320 fill four
    and leave a few; the plan splits those; 32 sampled rows against the
    oracle."""
    d = synth.BF16
    N, K = 5120, 17408
    h = synth.normal((M, K), d, 73, synth.TID_A, 1.0)
    Wd = synth.normal((N, K), d, 73, synth.TID_WD, 0.02)
    plan = gf.gf_matmul_plan_ex(M, N, K, d, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL, gf.GF_B_NK)
    desc = gf.gf_plan_describe(plan)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    gf.gf_matmul_execute(plan, to_dev(h, d), to_dev(Wd, d), out=out)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    # the documented rule: a last wave at most half full, k >= 128 blocks
    # beyond three waves (here 272 blocks)
    pairs = desc["grid"] // 2
    tiles = (M // 256) * -(-N // desc["tile_n"])
    rem = tiles % pairs
    assert desc["tile_m"] == 256, desc
    if rem and 2 * rem <= pairs:
        assert desc["k_splits"] >= 2, desc
    rows = synth.sample_rows(M, 32, 73)
    o_rows = oracle.decode(oracle.epilog_none(h[rows], Wd, d, oracle.B_NK), d)
    assert_close(to_host_f32(out)[rows], o_rows, what="down projection")
