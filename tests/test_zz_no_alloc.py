"""The allocation-free DRELU_BGRAD entry point (gf_drelu_bgrad_noalloc).

It serves callers that cannot call cudaMalloc: it keeps its scratch (the
per-block partial column sums of the bias gradient and a status word) in a
fixed array inside the library instead of a plan's workspace. Here it is
called through the C ABI and must give what the plan-based entry point
(gf_matmul_execute on a DRELU_BGRAD plan) gives and what the CPU oracle
gives, on two calls in a row (the second reuses the scratch the first one
left behind), with the scratch's status word clear after every call
(gf_noalloc_status).

This file is named so that pytest collects it last.
"""
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


def _case(M, N, K, seed, layout, dtype):
    dY = synth.normal((M, K), dtype, seed, synth.TID_DY, 1.0)
    shape = (N, K) if layout == gf.GF_B_NK else (K, N)
    W = synth.normal(shape, dtype, seed, synth.TID_B, 1 / np.sqrt(max(K, 1)))
    words = synth.mask_words(M, N, seed)
    return dY, W, words


@pytest.mark.parametrize("M,N,K,layout,dtype", [(1000, 520, 264, gf.GF_B_NK, gf.GF_F16),
                                                (4096, 2048, 512, gf.GF_B_NK, gf.GF_F16),
                                                (300, 136, 72, gf.GF_B_KN, gf.GF_F16),
                                                (1000, 520, 264, gf.GF_B_NK, gf.GF_BF16),
                                                (520, 264, 136, gf.GF_B_KN, gf.GF_BF16)])
def test_noalloc_matches_plan_and_oracle_twice(M, N, K, layout, dtype):
    gf.build()
    tdt = torch_dtype(dtype)
    plan = gf.gf_matmul_plan_ex(M, N, K, dtype, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL, layout)
    for call, seed in enumerate((11, 12)):  # two calls in a row, different data
        dY_h, W_h, words_h = _case(M, N, K, seed, layout, dtype)
        dY, W, mask = to_dev(dY_h, dtype), to_dev(W_h, dtype), to_dev(words_h, dtype)
        ref_out = torch.empty((M, N), dtype=tdt, device="cuda")
        ref_bgrad = torch.empty(N, dtype=torch.float32, device="cuda")
        gf.gf_matmul_execute(plan, dY, W, out=ref_out, aux_in=mask, bgrad=ref_bgrad)
        assert gf.gf_plan_status(plan) == gf.GF_OK
        out = torch.full((M, N), float("nan"), dtype=tdt, device="cuda")
        bgrad = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
        gf.gf_drelu_bgrad_noalloc(M, N, K, dtype, layout, dY, W, out, mask, bgrad)
        assert gf.gf_noalloc_status() == gf.GF_OK  # the status word stayed clear
        assert_close(to_host_f32(out), to_host_f32(ref_out), what=f"dZ vs plan, call {call}")
        assert_close(bgrad.cpu().numpy(), ref_bgrad.cpu().numpy(), BGRAD_NMAX, BGRAD_REL,
                     what=f"bgrad vs plan, call {call}")
        dz_o, bgrad_o, _ = oracle.drelu_bgrad(dY_h, W_h, words_h, dtype, layout)
        assert_close(to_host_f32(out), oracle.decode(dz_o, dtype), what=f"dZ vs oracle, call {call}")
        assert_close(bgrad.cpu().numpy(), bgrad_o, BGRAD_NMAX, BGRAD_REL,
                     what=f"bgrad vs oracle, call {call}")
    plan.free()


@pytest.mark.parametrize("dtype", [gf.GF_F16, gf.GF_BF16])
def test_noalloc_empty_k_gives_zeros(dtype):
    """k = 0: the product is zero, so dZ = 0 and the bias gradient is 0, even
    over a scratch array that the previous call left full of partial sums."""
    gf.build()
    M, N = 300, 136
    words = to_dev(synth.mask_words(M, N, 5), dtype)
    out = torch.full((M, N), float("nan"), dtype=torch_dtype(dtype), device="cuda")
    bgrad = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    gf.gf_drelu_bgrad_noalloc(M, N, 0, dtype, gf.GF_B_NK, None, None, out, words, bgrad)
    assert gf.gf_noalloc_status() == gf.GF_OK
    assert torch.count_nonzero(out.float()).item() == 0
    assert torch.count_nonzero(bgrad).item() == 0


def test_noalloc_rejects_beyond_scratch():
    gf.build()
    N = 4096
    M = 128 * (gf.GF_NOALLOC_MAX_PARTIALS // N) + 1  # one 128-row block too many
    t = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(gf.GfError) as e:
        gf.gf_drelu_bgrad_noalloc(M, N, 64, gf.GF_F16, gf.GF_B_NK, t, t, t, t, t)
    assert e.value.status == gf.GF_ERR_UNSUPPORTED
    assert gf.gf_last_error() == gf.GF_ERR_UNSUPPORTED
