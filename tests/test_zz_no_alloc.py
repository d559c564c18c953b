"""The allocation-free DRELU_BGRAD entry point (gf_drelu_bgrad_noalloc).

It serves callers that cannot call cudaMalloc: it keeps its scratch (the
per-block partial column sums of the bias gradient and a status word) in a
fixed array inside the library instead of a plan's workspace. Here it is
called through the C ABI and must give what the plan-based entry point
(gf_matmul_execute on a DRELU_BGRAD plan) gives, on two calls in a row
(the second reuses the scratch the first one left behind).

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest

import synth
from helpers import BGRAD_NMAX, BGRAD_REL, assert_close, to_dev, to_host_f32

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import gemm_epilogue_tmem_gb300 as gf  # noqa: E402


def _case(M, N, K, seed, layout):
    dY = synth.normal((M, K), synth.F16, seed, synth.TID_DY, 1.0)
    shape = (N, K) if layout == gf.GF_B_NK else (K, N)
    W = synth.normal(shape, synth.F16, seed, synth.TID_B, 1 / np.sqrt(K))
    words = synth.mask_words(M, N, seed)
    return to_dev(dY, 0), to_dev(W, 0), to_dev(words, 0)


@pytest.mark.parametrize("M,N,K,layout", [(1000, 520, 264, gf.GF_B_NK),
                                          (4096, 2048, 512, gf.GF_B_NK),
                                          (300, 136, 72, gf.GF_B_KN)])
def test_noalloc_matches_plan_twice(M, N, K, layout):
    gf.build()
    plan = gf.gf_matmul_plan_ex(M, N, K, gf.GF_F16, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL,
                                layout)
    for call, seed in enumerate((11, 12)):  # two calls in a row, different data
        dY, W, mask = _case(M, N, K, seed, layout)
        ref_out = torch.empty((M, N), dtype=torch.float16, device="cuda")
        ref_bgrad = torch.empty(N, dtype=torch.float32, device="cuda")
        gf.gf_matmul_execute(plan, dY, W, out=ref_out, aux_in=mask, bgrad=ref_bgrad)
        assert gf.gf_plan_status(plan) == gf.GF_OK
        out = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        bgrad = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
        gf.gf_drelu_bgrad_noalloc(M, N, K, gf.GF_F16, layout, dY, W, out, mask, bgrad)
        torch.cuda.synchronize()
        assert_close(to_host_f32(out), to_host_f32(ref_out), what=f"dZ call {call}")
        assert_close(bgrad.cpu().numpy(), ref_bgrad.cpu().numpy(), BGRAD_NMAX, BGRAD_REL,
                     what=f"bgrad call {call}")
    plan.free()


def test_noalloc_rejects_beyond_scratch():
    gf.build()
    N = 4096
    M = 128 * (gf.GF_NOALLOC_MAX_PARTIALS // N) + 1  # one 128-row block too many
    t = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(gf.GfError) as e:
        gf.gf_drelu_bgrad_noalloc(M, N, 64, gf.GF_F16, gf.GF_B_NK, t, t, t, t, t)
    assert e.value.status == gf.GF_ERR_UNSUPPORTED
