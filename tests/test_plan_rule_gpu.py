"""The plan's tile and split choice for CTA-pair products follows the rule its
documentation states (include/gf.h, GF_OPT_KERNEL and GF_OPT_SPLIT_K):
256 x 512 tiles (256 x 256 with two B operands) when k >= 2048 and their
schedule, counted in waves of the resident pairs with the last-wave split of
EPILOG_NONE plans, is no longer than the 256 x 256 (256 x 128) tiles'
weighed by the wide tile's gain (12 %, 4 % with two operands); the split of
a last wave at most half full, when k has at least 32 blocks within three
waves and 128 beyond. Restated here in Python and compared with the plans
the library makes on this device, over the workloads' shapes and a grid
around them (no kernel runs)."""
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import gemm_epilogue_tmem_gb300 as gf  # noqa: E402


def _cdiv(a, b):
    return -(-a // b)


@pytest.fixture(scope="module")
def pairs():
    big = gf.gf_matmul_plan_ex(8192, 8192, 2048, gf.GF_BF16, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL,
                               gf.GF_B_NK)
    gf.gf_plan_set_option(big, gf.GF_OPT_KERNEL, 2)
    n = gf.gf_plan_describe(big)["grid"] // 2  # 1024 tiles: every resident pair
    big.free()
    return n


def _expected(M, N, K, dual, none, cl):
    m2 = _cdiv(M, 256)
    nn, nw = (128, 256) if dual else (256, 512)
    t_narrow, t_wide = m2 * _cdiv(N, nn), m2 * _cdiv(N, nw)
    nkb = _cdiv(K, 64)

    def split(tiles):
        if dual or not none:
            return 0
        rem = tiles % cl
        if rem == 0 or 2 * rem > cl or nkb < (32 if tiles <= 3 * cl else 128):
            return 0
        w = min(8, cl // rem, nkb // 8)
        return w if w >= 2 else 0

    def eighths(tiles):
        w, full = split(tiles), tiles // cl
        return 8 * full + (0 if tiles == full * cl else (_cdiv(8, w) if w else 8))

    gain = 104 if dual else 112
    wide = K >= 2048 and 100 * 2 * eighths(t_wide) <= gain * eighths(t_narrow)
    tiles = t_wide if wide else t_narrow
    want = split(tiles)
    ks = 1
    if want >= 2:
        kps = _cdiv(nkb, want)
        ks = _cdiv(nkb, kps)
        tn = nw if wide else nn
        if (tiles - tiles // cl * cl) * 2 * ks * 128 * tn * 4 > (256 << 20) or ks < 2:
            ks = 1
    return (nw if wide else nn), ks


SHAPES = [(M, N, K) for M in (2048, 4096, 8192, 16384) for N in (5120, 8192, 16384, 17408)
          for K in (1024, 4096, 8192, 17408)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_matmul_none_plan_rule(M, N, K, pairs):
    p = gf.gf_matmul_plan_ex(M, N, K, gf.GF_BF16, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL, gf.GF_B_NK)
    d = gf.gf_plan_describe(p)
    p.free()
    assert d["tile_m"] == 256, d
    assert (d["tile_n"], d["k_splits"]) == _expected(M, N, K, False, True, pairs), d


@pytest.mark.parametrize("M,N,K", SHAPES[::3])
def test_matmul_fused_plan_rule(M, N, K, pairs):
    p = gf.gf_matmul_plan_ex(M, N, K, gf.GF_BF16, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL,
                             gf.GF_B_KN)
    d = gf.gf_plan_describe(p)
    p.free()
    assert d["tile_m"] == 256, d
    assert (d["tile_n"], d["k_splits"]) == _expected(M, N, K, False, False, pairs), d


@pytest.mark.parametrize("M", [2048, 4096, 8192, 16384])
def test_swiglu_gate_up_plan_rule(M, pairs):
    I, H = 17408, 5120
    p = gf.gf_swiglu_plan(M, I, H, gf.GF_BF16, save_gu=True)
    d = gf.gf_plan_describe(p)
    p.free()
    assert d["tile_m"] == 256, d
    assert (d["tile_n"], d["k_splits"]) == _expected(M, I, H, True, False, pairs), d
