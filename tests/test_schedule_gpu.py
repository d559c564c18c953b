"""Tile schedules of the persistent kernels (static, one tile per CTA pair,
dynamic counter) and raster groups give the oracle's results; the dynamic
schedule also keeps its bounded waits (a skipped load is reported, and the
next call is correct), and plans running at once on several streams do not
disturb each other."""
import numpy as np
import pytest

import oracle
import synth
from helpers import BGRAD_NMAX, BGRAD_REL, assert_close, mask_mismatch, to_dev, to_host_f32, \
    to_host_words, unpack_words

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import gemm_epilogue_tmem_gb300 as gf  # noqa: E402

M, N, K = 3000, 2568, 264


@pytest.fixture(scope="module")
def data():
    X = synth.normal((M, K), synth.F16, 31, synth.TID_A, 1.0)
    W = synth.normal((K, N), synth.F16, 31, synth.TID_B, 1 / np.sqrt(K))
    Wt = synth.normal((N, K), synth.F16, 31, synth.TID_W2, 1 / np.sqrt(K))
    b = synth.normal((N,), synth.F16, 31, synth.TID_BIAS, 0.1)
    words = synth.mask_words(M, N, 31)
    y_o, z_o = oracle.relu_bias(X, W, b, oracle.F16)
    dz_o, bgrad_o, _ = oracle.drelu_bgrad(X, Wt, words, oracle.F16, oracle.B_NK)
    return X, W, Wt, b, words, y_o, z_o, dz_o, bgrad_o


@pytest.mark.parametrize("schedule", [0, 1, 2, 3])
@pytest.mark.parametrize("group_m", [1, 4, 8])
def test_forward_schedules(data, schedule, group_m):
    X, W, Wt, b, words, y_o, z_o, dz_o, bgrad_o = data
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    aux = torch.empty(((M + 31) // 32, N), dtype=torch.int32, device="cuda")
    plan = gf.gf_matmul_plan(M, N, K, gf.GF_F16, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL)
    gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, 2)
    gf.gf_plan_set_option(plan, gf.GF_OPT_SCHEDULE, schedule)
    gf.gf_plan_set_option(plan, gf.GF_OPT_GROUP_M, group_m)
    for _ in range(2):  # the dynamic counter is reset for every call
        gf.gf_matmul_execute(plan, to_dev(X, 0), to_dev(W, 0), bias=to_dev(b, 0), out=out,
                             aux_out=aux)
        assert gf.gf_plan_status(plan) == gf.GF_OK
        assert_close(to_host_f32(out), oracle.decode(y_o, 0), what="Y")
        outside, _ = mask_mismatch(unpack_words(to_host_words(aux), M), z_o)
        assert outside == 0
        out.zero_()
    plan.free()


@pytest.mark.parametrize("schedule", [0, 3])
@pytest.mark.parametrize("mode", [gf.GF_BGRAD_TWO_PASS, gf.GF_BGRAD_ATOMIC])
def test_backward_schedules(data, schedule, mode):
    X, W, Wt, b, words, y_o, z_o, dz_o, bgrad_o = data
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    bgrad = torch.empty((N,), dtype=torch.float32, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, N, K, gf.GF_F16, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL,
                                gf.GF_B_NK)
    gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, 2)
    gf.gf_plan_set_option(plan, gf.GF_OPT_SCHEDULE, schedule)
    gf.gf_plan_set_option(plan, gf.GF_OPT_BGRAD_MODE, mode)
    gf.gf_matmul_execute(plan, to_dev(X, 0), to_dev(Wt, 0), out=out, aux_in=to_dev(words, 0),
                         bgrad=bgrad)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    assert_close(to_host_f32(out), oracle.decode(dz_o, 0), what="dZ")
    assert_close(bgrad.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL, what="bgrad")


def test_dynamic_schedule_swiglu_and_gelu():
    Mh, I, H = 1536, 1032, 256
    d = synth.BF16
    x = synth.normal((Mh, H), d, 32, synth.TID_A, 1.0)
    Wg = synth.normal((I, H), d, 32, synth.TID_WG, 0.1)
    Wu = synth.normal((I, H), d, 32, synth.TID_WU, 0.1)
    h = torch.empty((Mh, I), dtype=torch.bfloat16, device="cuda")
    plan = gf.gf_swiglu_plan(Mh, I, H, d)
    gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, 2)
    gf.gf_plan_set_option(plan, gf.GF_OPT_SCHEDULE, 2)
    gf.gf_swiglu_execute(plan, to_dev(x, d), to_dev(Wg, d), to_dev(Wu, d), h)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    h_o = oracle.swiglu_forward(x, Wg, Wu, d)[0]
    assert_close(to_host_f32(h), oracle.decode(h_o, d), what="h")


def test_dynamic_schedule_wait_limit():
    Mw, Nw, Kw = 1024, 1024, 512
    X = synth.normal((Mw, Kw), synth.F16, 33, synth.TID_A, 1.0)
    W = synth.normal((Kw, Nw), synth.F16, 33, synth.TID_B, 1 / np.sqrt(Kw))
    b = synth.normal((Nw,), synth.F16, 33, synth.TID_BIAS, 0.1)
    Xd, Wd, bd = to_dev(X, 0), to_dev(W, 0), to_dev(b, 0)
    out = torch.empty((Mw, Nw), dtype=torch.float16, device="cuda")
    plan = gf.gf_matmul_plan(Mw, Nw, Kw, gf.GF_F16, gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_COL)
    gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, 2)
    gf.gf_plan_set_option(plan, gf.GF_OPT_SCHEDULE, 2)
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


@pytest.mark.parametrize("epilog", ["fwd", "bwd"])
def test_autotune_keeps_a_correct_choice(data, epilog):
    """The autotuned plan still gives the oracle's results, and its
    description is one of the candidate configurations."""
    X, W, Wt, b, words, y_o, z_o, dz_o, bgrad_o = data
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    if epilog == "fwd":
        aux = torch.empty(((M + 31) // 32, N), dtype=torch.int32, device="cuda")
        plan = gf.gf_matmul_plan(M, N, K, gf.GF_F16, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL)
        args = dict(A=to_dev(X, 0), B=to_dev(W, 0), bias=to_dev(b, 0), out=out, aux_out=aux)
    else:
        bgrad = torch.empty((N,), dtype=torch.float32, device="cuda")
        plan = gf.gf_matmul_plan_ex(M, N, K, gf.GF_F16, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL,
                                    gf.GF_B_NK)
        args = dict(A=to_dev(X, 0), B=to_dev(Wt, 0), out=out, aux_in=to_dev(words, 0),
                    bgrad=bgrad)
    desc = gf.gf_matmul_autotune(plan, reps=2, **args)
    assert (desc["tile_m"], desc["tile_n"]) in ((256, 512), (256, 256), (128, 256), (128, 128))
    out.zero_()
    gf.gf_matmul_execute(plan, **args)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    assert gf.gf_plan_describe(plan) == desc
    plan.free()
    if epilog == "fwd":
        assert_close(to_host_f32(out), oracle.decode(y_o, 0), what="Y")
        outside, _ = mask_mismatch(unpack_words(to_host_words(aux), M), z_o)
        assert outside == 0
    else:
        assert_close(to_host_f32(out), oracle.decode(dz_o, 0), what="dZ")
        assert_close(bgrad.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL, what="bgrad")


def test_autotune_rejects_bad_reps():
    plan = gf.gf_matmul_plan(256, 256, 64, gf.GF_F16, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL)
    a = torch.zeros((256, 64), dtype=torch.float16, device="cuda")
    w = torch.zeros((64, 256), dtype=torch.float16, device="cuda")
    o = torch.empty((256, 256), dtype=torch.float16, device="cuda")
    for reps in (0, 101):
        with pytest.raises(gf.GfError):
            gf.gf_matmul_autotune(plan, a, w, out=o, reps=reps)
    plan.free()


@pytest.mark.parametrize("kernel", [1, 2, 3])
def test_raster_orders_give_the_same_bits(data, kernel):
    """Groups of row blocks or of column blocks (GF_OPT_RASTER 1 / 2), of
    several sizes, visit the same tiles in another order: the forward output,
    its mask and the backward's dZ and two-pass bias gradient are identical
    bit for bit, and match the oracle."""
    X, W, Wt, b, words, y_o, z_o, dz_o, bgrad_o = data
    Xd, Wd, Wtd, bd, wd = to_dev(X, 0), to_dev(W, 0), to_dev(Wt, 0), to_dev(b, 0), to_dev(words, 0)
    results = []
    for raster, group in ((0, 0), (1, 8), (2, 4), (2, 1), (2, 3)):
        fwd = gf.gf_matmul_plan(M, N, K, gf.GF_F16, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL)
        bwd = gf.gf_matmul_plan_ex(M, N, K, gf.GF_F16, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL,
                                   gf.GF_B_NK)
        for p in (fwd, bwd):
            gf.gf_plan_set_option(p, gf.GF_OPT_KERNEL, kernel)
            gf.gf_plan_set_option(p, gf.GF_OPT_RASTER, raster)
            gf.gf_plan_set_option(p, gf.GF_OPT_GROUP_M, group)
        y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        aux = torch.empty(((M + 31) // 32, N), dtype=torch.int32, device="cuda")
        dz = torch.empty((M, N), dtype=torch.float16, device="cuda")
        bg = torch.empty((N,), dtype=torch.float32, device="cuda")
        gf.gf_matmul_execute(fwd, Xd, Wd, bias=bd, out=y, aux_out=aux)
        gf.gf_matmul_execute(bwd, Xd, Wtd, out=dz, aux_in=wd, bgrad=bg)
        assert gf.gf_plan_status(fwd) == gf.GF_OK and gf.gf_plan_status(bwd) == gf.GF_OK
        fwd.free()
        bwd.free()
        results.append((y, aux, dz, bg))
    for r in results[1:]:
        for a, c in zip(results[0], r):
            assert torch.equal(a, c)
    y, aux, dz, bg = results[0]
    assert_close(to_host_f32(y), oracle.decode(y_o, 0), what="Y")
    assert mask_mismatch(unpack_words(to_host_words(aux), M), z_o)[0] == 0
    assert_close(to_host_f32(dz), oracle.decode(dz_o, 0), what="dZ")
    assert_close(bg.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL, what="bgrad")


def test_plans_on_two_streams_at_once():
    """A forward plan and a backward plan (and a wide-tile forward) enqueued on
    three streams so that their persistent kernels overlap, several times in
    a row: each plan's tile counter and status word are its own, so every
    output is the same bits as when the plans run one after the other."""
    Mc, Nc, Kc = 4096, 4096, 2048
    X = to_dev(synth.normal((Mc, Kc), synth.F16, 50, synth.TID_A, 1.0), 0)
    W = to_dev(synth.normal((Kc, Nc), synth.F16, 50, synth.TID_B, 1 / np.sqrt(Kc)), 0)
    Wt = to_dev(synth.normal((Nc, Kc), synth.F16, 50, synth.TID_W2, 1 / np.sqrt(Kc)), 0)
    b = to_dev(synth.normal((Nc,), synth.F16, 50, synth.TID_BIAS, 0.1), 0)
    words = to_dev(synth.mask_words(Mc, Nc, 50), 0)
    fwd = gf.gf_matmul_plan(Mc, Nc, Kc, gf.GF_F16, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL)
    gf.gf_plan_set_option(fwd, gf.GF_OPT_KERNEL, 2)
    wide = gf.gf_matmul_plan(Mc, Nc, Kc, gf.GF_F16, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL)
    gf.gf_plan_set_option(wide, gf.GF_OPT_KERNEL, 3)
    bwd = gf.gf_matmul_plan_ex(Mc, Nc, Kc, gf.GF_F16, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL,
                               gf.GF_B_NK)

    def outs():
        return (torch.empty((Mc, Nc), dtype=torch.float16, device="cuda"),
                torch.empty((Mc // 32, Nc), dtype=torch.int32, device="cuda"),
                torch.empty((Mc, Nc), dtype=torch.float16, device="cuda"),
                torch.empty((Mc // 32, Nc), dtype=torch.int32, device="cuda"),
                torch.empty((Mc, Nc), dtype=torch.float16, device="cuda"),
                torch.empty((Nc,), dtype=torch.float32, device="cuda"))

    def launch(o, streams):
        s1, s2, s3 = (s.cuda_stream for s in streams)
        gf.gf_matmul_execute(fwd, X, W, bias=b, out=o[0], aux_out=o[1], stream=s1)
        gf.gf_matmul_execute(wide, X, W, bias=b, out=o[2], aux_out=o[3], stream=s2)
        gf.gf_matmul_execute(bwd, X, Wt, out=o[4], aux_in=words, bgrad=o[5], stream=s3)

    cur = torch.cuda.current_stream()
    ref = outs()
    launch(ref, (cur, cur, cur))  # one after the other
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(3)]
    for _ in range(3):
        o = outs()
        launch(o, streams)
        torch.cuda.synchronize()
        for a, r in zip(o, ref):
            assert torch.equal(a.view(torch.uint8), r.view(torch.uint8))
    for p in (fwd, wide, bwd):
        assert gf.gf_plan_status(p) == gf.GF_OK
        p.free()
