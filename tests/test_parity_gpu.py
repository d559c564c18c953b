"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs, element by element.

Workloads follow the pages' examples (see synth): the tiny 2-layer ReLU MLP
step, the (1024,512,2048) RELU_BIAS GEMM with a (m,1) bias, plus ragged and
degenerate shapes that span several tiles and a tail in every dimension.
"""
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    gf.build()
    synth.build_host()
    oracle.build()


def _inputs(M, N, K, dtype, layout, seed, sigma_b=None, bias_len=None):
    A = synth.normal((M, K), dtype, seed, synth.TID_A, 1.0)
    sb = sigma_b if sigma_b is not None else 1 / np.sqrt(max(K, 1))
    B = (synth.normal((K, N), dtype, seed, synth.TID_B, sb) if layout == oracle.B_KN
         else synth.normal((N, K), dtype, seed, synth.TID_B, sb))
    bias = synth.normal((bias_len or N,), dtype, seed, synth.TID_BIAS, 0.1)
    return A, B, bias


def _run_fwd(M, N, K, dtype, epilog, axis, layout, A, B, bias, tile_n=0):
    tdt = torch_dtype(dtype)
    Ad, Bd, bd = to_dev(A, dtype), to_dev(B, dtype), to_dev(bias, dtype)
    out = torch.empty((M, N), dtype=tdt, device="cuda")
    aux = torch.zeros((max((M + 31) // 32, 1), max(N, 1)), dtype=torch.int32, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, N, K, dtype, epilog, axis, layout)
    if tile_n:
        gf.gf_plan_set_option(plan, gf.GF_OPT_TILE_N, tile_n)
    gf.gf_matmul_execute(plan, Ad, Bd, bias=bd, out=out,
                         aux_out=aux if epilog == gf.GF_EPILOG_RELU_AUX_BIAS else None)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    return plan, out, aux


def _check_fwd(M, N, K, dtype, epilog, axis, layout, seed=0, tile_n=0, sigma_b=None):
    A, B, bias = _inputs(M, N, K, dtype, layout, seed, sigma_b,
                         bias_len=M if axis == gf.GF_BIAS_ROW else N)
    plan, out, aux = _run_fwd(M, N, K, dtype, epilog, axis, layout, A, B, bias, tile_n)
    acc = oracle.gemm(A, B, dtype, layout)
    if epilog == gf.GF_EPILOG_NONE:
        ref, z = oracle.round_to(acc, dtype), acc
    else:
        z = oracle.add_bias(acc, bias, dtype, axis)
        ref = oracle.round_to(z if epilog == gf.GF_EPILOG_BIAS else oracle.relu(z), dtype)
    errs = assert_close(to_host_f32(out), oracle.decode(ref, dtype), what=f"out {M}x{N}x{K}")
    if epilog == gf.GF_EPILOG_RELU_AUX_BIAS:
        words = to_host_words(aux)
        bits = unpack_words(words, M)
        outside, inside = mask_mismatch(bits, z)
        assert outside == 0, f"{outside} mask bits differ outside the band"
        if M % 32:
            assert np.all(words[-1] >> (M % 32) == 0), "padding bits must be 0"
    plan.free()
    return errs


# ---------------------------------------------------------------- workloads
def test_mlp_tiny_step():
    """2-layer ReLU MLP step: layer-1 RELU_AUX_BIAS forward, then DRELU_BGRAD
    of G = dY W2^T with the relu_aux mask (all fp16, seed 0)."""
    w = synth.MLP_TINY
    s = 0
    T = {k: synth.normal(v.shape, w.dtype, s, v.tensor_id, v.sigma) for k, v in w.tensors.items()}
    X, W1, b1, W2, dY = T["X"], T["W1"], T["b1"], T["W2"], T["dY"]
    M, K = X.shape
    N = W1.shape[1]
    plan, Y, aux = _run_fwd(M, N, K, 0, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL, gf.GF_B_KN,
                            X, W1, b1)
    y_o, words_o, z_o = oracle.relu_aux_bias(X, W1, b1, oracle.F16)
    assert_close(to_host_f32(Y), oracle.decode(y_o, 0), what="Y1")
    outside, inside = mask_mismatch(unpack_words(to_host_words(aux), M), z_o)
    assert outside == 0
    # backward: W2 is [384, 128] = [N, K2]: G = dY . W2^T is B_NK with W2
    K2 = dY.shape[1]
    dZ = torch.empty((M, N), dtype=torch.float16, device="cuda")
    bgrad = torch.empty(N, dtype=torch.float32, device="cuda")
    bwd = gf.gf_matmul_plan_ex(M, N, K2, 0, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL, gf.GF_B_NK)
    gf.gf_matmul_execute(bwd, to_dev(dY, 0), to_dev(W2, 0), out=dZ, aux_in=to_dev(words_o, 0),
                         bgrad=bgrad)
    assert gf.gf_plan_status(bwd) == gf.GF_OK
    dz_o, bgrad_o, _ = oracle.drelu_bgrad(dY, W2, words_o, oracle.F16, oracle.B_NK)
    assert_close(to_host_f32(dZ), oracle.decode(dz_o, 0), what="dZ")
    assert_close(bgrad.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL, what="bgrad1")
    # the paired flow on the GPU alone: the device's own mask gives the same
    # result wherever the two masks agree
    dZ2 = torch.empty_like(dZ)
    gf.gf_matmul_execute(bwd, to_dev(dY, 0), to_dev(W2, 0), out=dZ2, aux_in=aux, bgrad=bgrad)
    same = unpack_words(to_host_words(aux), M) == oracle.relu_bits(z_o)
    assert np.array_equal(to_host_f32(dZ2)[same], to_host_f32(dZ)[same])
    plan.free()
    bwd.free()


@pytest.mark.parametrize("seed", [0, 1, 2, 3, 4])
def test_relu_bias_row_bias(seed):
    """m=1024, k=2048, n=512 RELU_BIAS with a (1024,1) bias, A, B, bias ~ N(0,1)."""
    _check_fwd(1024, 512, 2048, 0, gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_ROW, gf.GF_B_KN, seed=seed,
               sigma_b=1.0)


# ------------------------------------------------------- shapes and variants
SHAPES = [
    (128, 128, 64),     # exactly one tile
    (300, 200, 72),     # ragged M, N and K
    (1000, 520, 1000),  # several tiles, ragged
    (33, 8, 8),         # tiny
    (129, 264, 136),
    (4096, 1024, 512),  # more tiles than SMs
    (4096, 4096, 256),  # 3 to 4 tiles per CTA: both accumulator buffers reused
]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("layout", [gf.GF_B_KN, gf.GF_B_NK])
@pytest.mark.parametrize("epilog", [gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_EPILOG_NONE])
def test_forward_shapes(M, N, K, layout, epilog):
    _check_fwd(M, N, K, 0, epilog, gf.GF_BIAS_COL, layout)


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("epilog,axis", [
    (gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_COL), (gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_ROW),
    (gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_ROW), (gf.GF_EPILOG_BIAS, gf.GF_BIAS_COL),
])
def test_forward_variants(tile_n, dtype, epilog, axis):
    for layout in (gf.GF_B_KN, gf.GF_B_NK):
        _check_fwd(700, 392, 328, dtype, epilog, axis, layout, seed=3, tile_n=tile_n)


def _check_drelu(M, N, K, dtype, layout, seed=0, mode=gf.GF_BGRAD_TWO_PASS, tile_n=0):
    dY = synth.normal((M, K), dtype, seed, synth.TID_DY, 1.0)
    W = (synth.normal((N, K), dtype, seed, synth.TID_B, 1 / np.sqrt(max(K, 1)))
         if layout == gf.GF_B_NK else
         synth.normal((K, N), dtype, seed, synth.TID_B, 1 / np.sqrt(max(K, 1))))
    words = synth.mask_words(M, N, seed)
    tdt = torch_dtype(dtype)
    out = torch.empty((M, N), dtype=tdt, device="cuda")
    bgrad = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, N, K, dtype, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL, layout)
    gf.gf_plan_set_option(plan, gf.GF_OPT_BGRAD_MODE, mode)
    if tile_n:
        gf.gf_plan_set_option(plan, gf.GF_OPT_TILE_N, tile_n)
    gf.gf_matmul_execute(plan, to_dev(dY, dtype), to_dev(W, dtype), out=out,
                         aux_in=to_dev(words, dtype), bgrad=bgrad)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    dz_o, bgrad_o, _ = oracle.drelu_bgrad(dY, W, words, dtype, layout)
    assert_close(to_host_f32(out), oracle.decode(dz_o, dtype), what=f"dZ {M}x{N}x{K}")
    assert_close(bgrad.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL, what="bgrad")
    # invariant: bgrad = 1^T dz (the device's own output, summed in fp64)
    colsum = out.double().sum(0).cpu().numpy()
    assert_close(bgrad.cpu().numpy(), colsum, BGRAD_NMAX, BGRAD_REL, what="bgrad vs 1^T dZ")
    plan.free()
    return out, bgrad


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("layout", [gf.GF_B_NK, gf.GF_B_KN])
def test_drelu_bgrad_shapes(M, N, K, layout):
    _check_drelu(M, N, K, 0, layout)


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("mode", [gf.GF_BGRAD_TWO_PASS, gf.GF_BGRAD_ATOMIC])
@pytest.mark.parametrize("tile_n", [128, 256])
def test_drelu_bgrad_variants(dtype, mode, tile_n):
    _check_drelu(777, 456, 264, dtype, gf.GF_B_NK, seed=2, mode=mode, tile_n=tile_n)


def test_drelu_two_pass_is_deterministic():
    a_out, a_b = _check_drelu(1500, 520, 256, 0, gf.GF_B_NK, seed=5)
    b_out, b_b = _check_drelu(1500, 520, 256, 0, gf.GF_B_NK, seed=5)
    assert torch.equal(a_b, b_b) and torch.equal(a_out, b_out)


# ------------------------------------------------------------ degenerate cases
def test_k_zero():
    M, N = 200, 136
    bias = synth.normal((N,), 0, 0, synth.TID_BIAS, 0.1)
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    aux = torch.empty(((M + 31) // 32, N), dtype=torch.int32, device="cuda")
    plan = gf.gf_matmul_plan(M, N, 0, 0, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL)
    gf.gf_matmul_execute(plan, None, None, bias=to_dev(bias, 0), out=out, aux_out=aux)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    z = np.broadcast_to(bias.astype(np.float32), (M, N))
    assert np.array_equal(to_host_f32(out), np.maximum(z, 0).astype(np.float16).astype(np.float32))
    assert np.array_equal(unpack_words(to_host_words(aux), M), (z > 0).astype(np.uint8))


@pytest.mark.parametrize("M,N", [(0, 64), (64, 0), (0, 0)])
def test_empty(M, N):
    bgrad = torch.full((max(N, 1),), 7.0, dtype=torch.float32, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, N, 64, 0, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL, gf.GF_B_NK)
    gf.gf_matmul_execute(plan, None, None, out=None, aux_in=None, bgrad=bgrad if N else None)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    if N:
        assert torch.all(bgrad[:N] == 0)


def test_execute_rejects_bad_pointers():
    M, N, K = 128, 128, 64
    A = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    B = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    plan = gf.gf_matmul_plan(M, N, K, 0, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL)
    with pytest.raises(gf.GfError) as e:  # aux_out missing
        gf.gf_matmul_execute(plan, A, B, bias=torch.zeros(N, dtype=torch.float16, device="cuda"),
                             out=out)
    assert e.value.status == gf.GF_ERR_INVALID_VALUE
    with pytest.raises(gf.GfError):  # misaligned A
        gf.gf_matmul_execute(plan, A.data_ptr() + 2, B, bias=out, out=out, aux_out=out)
    plan.free()


def test_wait_limit_reports_timeout():
    """A skipped stage load makes the MMA warp's bounded wait run out: the
    kernel returns, the host reads GF_ERR_DEVICE_TIMEOUT and the context stays
    usable for the next call."""
    M, N, K = 256, 256, 256
    A, B, bias = _inputs(M, N, K, 0, gf.GF_B_KN, 0)
    plan = gf.gf_matmul_plan(M, N, K, 0, gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_COL)
    gf.gf_plan_set_option(plan, gf.GF_OPT_WAIT_LIMIT_US, 20000)
    gf.gf_plan_set_option(plan, gf.GF_OPT_FAULT_DROP_LOAD, 2)
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    gf.gf_matmul_execute(plan, to_dev(A, 0), to_dev(B, 0), bias=to_dev(bias, 0), out=out)
    assert gf.gf_plan_status(plan) == gf.GF_ERR_DEVICE_TIMEOUT
    gf.gf_plan_set_option(plan, gf.GF_OPT_FAULT_DROP_LOAD, 0)
    gf.gf_matmul_execute(plan, to_dev(A, 0), to_dev(B, 0), bias=to_dev(bias, 0), out=out)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    plan.free()
    _check_fwd(256, 256, 256, 0, gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_COL, gf.GF_B_KN)


def _kernel_nodes(graph_handle: int) -> int:
    """Kernel nodes of a captured CUDA graph, through the CUDA runtime that
    this process already loaded (the graph is a driver object)."""
    import ctypes
    path = None
    with open("/proc/self/maps") as f:
        for line in f:
            if "libcudart.so" in line:
                path = line.split()[-1]
                break
    assert path, "no CUDA runtime loaded"
    rt = ctypes.CDLL(path)
    n = ctypes.c_size_t(0)
    assert rt.cudaGraphGetNodes(ctypes.c_void_p(graph_handle), None, ctypes.byref(n)) == 0
    nodes = (ctypes.c_void_p * max(n.value, 1))()
    assert rt.cudaGraphGetNodes(ctypes.c_void_p(graph_handle), nodes, ctypes.byref(n)) == 0
    kernels = 0
    for i in range(n.value):
        t = ctypes.c_int(-1)
        assert rt.cudaGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) == 0
        kernels += t.value == 0  # cudaGraphNodeTypeKernel
    return kernels


def test_one_fused_launch():
    """One execute = one kernel launch, plus the bgrad finalize for the
    two-pass backward (single-CTA and CTA-pair kernels). Counted from a CUDA
    graph capture of execute, and equal to what gf_plan_launches reports
    (the SwiGLU sample counts launches too, so that "1 kernel" is shown:
    gemm_swiglu_mlp_fusion.py, ``_demo``)."""
    M, N, K = 512, 512, 256
    A = torch.randn((M, K), device="cuda").half()
    B = torch.randn((K, N), device="cuda").half()
    bias = torch.randn(N, device="cuda").half()
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    aux = torch.empty((M // 32, N), dtype=torch.int32, device="cuda")
    mask = torch.randint(-2**31, 2**31 - 1, (M // 32, N), dtype=torch.int32, device="cuda")
    bgrad = torch.empty(N, dtype=torch.float32, device="cuda")
    fwd = gf.gf_matmul_plan(M, N, K, 0, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL)
    bwd = gf.gf_matmul_plan_ex(M, N, K, 0, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL, gf.GF_B_NK)
    bwd_pair = gf.gf_matmul_plan_ex(M, N, K, 0, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL,
                                    gf.GF_B_NK)
    gf.gf_plan_set_option(bwd_pair, gf.GF_OPT_KERNEL, 2)
    counts, declared = [], []
    for plan, kw in ((fwd, dict(bias=bias, out=out, aux_out=aux)),
                     (bwd, dict(out=out, aux_in=mask, bgrad=bgrad)),
                     (bwd_pair, dict(out=out, aux_in=mask, bgrad=bgrad))):
        declared.append(gf.gf_plan_describe(plan)["launches"])
        gf.gf_matmul_execute(plan, A, B, **kw)
        torch.cuda.synchronize()
        ref = out.clone()
        g = torch.cuda.CUDAGraph(keep_graph=True)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                gf.gf_matmul_execute(plan, A, B, **kw, stream=s)
        counts.append(_kernel_nodes(g.raw_cuda_graph()))
        out.zero_()
        g.replay()  # the captured launch replays to the same result
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert counts == [1, 2, 2] and declared == counts, (counts, declared)
    fwd.free()
    bwd.free()
    bwd_pair.free()


def test_dependent_launch_changes_nothing():
    """Programmatic dependent launch (GF_OPT_PDL, the default) against plain
    stream order: the tiny MLP step (forward GEMM, backward GEMM, bias-gradient
    finalize back to back, every kernel reading what the one before wrote),
    directly and captured in a CUDA graph, gives the same bits."""
    w = synth.MLP_TINY
    T = {k: to_dev(synth.normal(v.shape, w.dtype, 3, v.tensor_id, v.sigma), 0)
         for k, v in w.tensors.items()}
    M, K = w.tensors["X"].shape
    N = w.tensors["W1"].shape[1]
    K2 = w.tensors["dY"].shape[1]
    results = {}
    for pdl in (0, 1):
        fwd = gf.gf_matmul_plan(M, N, K, 0, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL)
        bwd = gf.gf_matmul_plan_ex(M, N, K2, 0, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL,
                                   gf.GF_B_NK)
        for p in (fwd, bwd):
            gf.gf_plan_set_option(p, gf.GF_OPT_PDL, pdl)
        Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        aux = torch.empty(((M + 31) // 32, N), dtype=torch.int32, device="cuda")
        G = torch.empty((M, N), dtype=torch.float16, device="cuda")
        bg = torch.empty(N, dtype=torch.float32, device="cuda")

        def step(s=None):
            for _ in range(5):
                gf.gf_matmul_execute(fwd, T["X"], T["W1"], bias=T["b1"], out=Y, aux_out=aux,
                                     stream=s)
                gf.gf_matmul_execute(bwd, T["dY"], T["W2"], out=G, aux_in=aux, bgrad=bg,
                                     stream=s)

        step()
        torch.cuda.synchronize()
        direct = [t.clone() for t in (Y, aux, G, bg)]
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                step(s)
        for t in (Y, aux, G, bg):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert gf.gf_plan_status(fwd) == gf.GF_OK and gf.gf_plan_status(bwd) == gf.GF_OK
        results[pdl] = direct + [t.clone() for t in (Y, aux, G, bg)]
        fwd.free()
        bwd.free()
    for a, b in zip(results[0], results[1]):
        assert torch.equal(a, b)
    for a, b in zip(results[1][:4], results[1][4:]):
        assert torch.equal(a, b)


# ------------------------------------------------------------- CTA-pair kernel
PAIR_SHAPES = [
    (256, 256, 64),     # one pair tile
    (300, 520, 200),    # the second CTA's rows partly past M; ragged N and K
    (129, 264, 136),    # the peer CTA entirely past M
    (2048, 2048, 512),  # nearly one pair tile per resident pair
    (4096, 4096, 256),  # 3 to 4 pair tiles per pair: both accumulator buffers reused
    (6000, 2056, 328),  # several tiles per pair, ragged everywhere
]


def _force_pair(plan):
    gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, 2)
    assert gf.gf_plan_describe(plan)["tile_m"] == 256


@pytest.mark.parametrize("M,N,K", PAIR_SHAPES)
@pytest.mark.parametrize("layout", [gf.GF_B_KN, gf.GF_B_NK])
@pytest.mark.parametrize("epilog,axis", [
    (gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL), (gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_ROW),
    (gf.GF_EPILOG_NONE, gf.GF_BIAS_COL),
])
def test_pair_forward(M, N, K, layout, epilog, axis):
    dtype = 0 if K != 200 else 1
    A, B, bias = _inputs(M, N, K, dtype, layout, 1, bias_len=M if axis == gf.GF_BIAS_ROW else N)
    tdt = torch_dtype(dtype)
    out = torch.empty((M, N), dtype=tdt, device="cuda")
    aux = torch.zeros(((M + 31) // 32, N), dtype=torch.int32, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, N, K, dtype, epilog, axis, layout)
    _force_pair(plan)
    gf.gf_matmul_execute(plan, to_dev(A, dtype), to_dev(B, dtype), bias=to_dev(bias, dtype),
                         out=out, aux_out=aux if epilog == gf.GF_EPILOG_RELU_AUX_BIAS else None)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    acc = oracle.gemm(A, B, dtype, layout)
    if epilog == gf.GF_EPILOG_NONE:
        ref, z = oracle.round_to(acc, dtype), acc
    else:
        z = oracle.add_bias(acc, bias, dtype, axis)
        ref = oracle.round_to(oracle.relu(z), dtype)
    assert_close(to_host_f32(out), oracle.decode(ref, dtype), what=f"pair out {M}x{N}x{K}")
    if epilog == gf.GF_EPILOG_RELU_AUX_BIAS:
        outside, _ = mask_mismatch(unpack_words(to_host_words(aux), M), z)
        assert outside == 0
    plan.free()


@pytest.mark.parametrize("M,N,K", PAIR_SHAPES)
@pytest.mark.parametrize("mode", [gf.GF_BGRAD_TWO_PASS, gf.GF_BGRAD_ATOMIC])
def test_pair_drelu_bgrad(M, N, K, mode):
    dtype = 0
    dY = synth.normal((M, K), dtype, 4, synth.TID_DY, 1.0)
    W = synth.normal((N, K), dtype, 4, synth.TID_B, 1 / np.sqrt(K))
    words = synth.mask_words(M, N, 4)
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    bgrad = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    plan = gf.gf_matmul_plan_ex(M, N, K, dtype, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL,
                                gf.GF_B_NK)
    _force_pair(plan)
    gf.gf_plan_set_option(plan, gf.GF_OPT_BGRAD_MODE, mode)
    gf.gf_matmul_execute(plan, to_dev(dY, 0), to_dev(W, 0), out=out, aux_in=to_dev(words, 0),
                         bgrad=bgrad)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    dz_o, bgrad_o, _ = oracle.drelu_bgrad(dY, W, words, dtype, gf.GF_B_NK)
    assert_close(to_host_f32(out), oracle.decode(dz_o, 0), what="pair dZ")
    assert_close(bgrad.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL, what="pair bgrad")
    plan.free()


def test_pair_wait_limit_reports_timeout():
    M, N, K = 512, 512, 256
    A, B, bias = _inputs(M, N, K, 0, gf.GF_B_KN, 0)
    plan = gf.gf_matmul_plan(M, N, K, 0, gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_COL)
    _force_pair(plan)
    gf.gf_plan_set_option(plan, gf.GF_OPT_WAIT_LIMIT_US, 20000)
    gf.gf_plan_set_option(plan, gf.GF_OPT_FAULT_DROP_LOAD, 2)
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    gf.gf_matmul_execute(plan, to_dev(A, 0), to_dev(B, 0), bias=to_dev(bias, 0), out=out)
    assert gf.gf_plan_status(plan) == gf.GF_ERR_DEVICE_TIMEOUT
    gf.gf_plan_set_option(plan, gf.GF_OPT_FAULT_DROP_LOAD, 0)
    gf.gf_matmul_execute(plan, to_dev(A, 0), to_dev(B, 0), bias=to_dev(bias, 0), out=out)
    assert gf.gf_plan_status(plan) == gf.GF_OK
    z = oracle.add_bias(oracle.gemm(A, B, 0), bias, 0, 0)
    assert_close(to_host_f32(out), oracle.decode(oracle.round_to(oracle.relu(z), 0), 0))
    plan.free()
