"""Pins of the oracle's SwiGLU steps (gemm_swiglu_mlp_fusion.py, module
docstring: silu(x Wg^T) * (x Wu^T), and the dSwiGLU backward): closed forms,
torch's SiLU and autograd in float64, and the sample's own composite formula
``F.silu(x @ Wg.t()) * (x @ Wu.t())`` on small inputs."""
import math

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
F = torch.nn.functional


def test_closed_forms():
    assert oracle.sigmoid_scalar(0.0) == 0.5
    assert oracle.silu_scalar(0.0) == 0.0
    assert oracle.silu_scalar(40.0) == 40.0
    assert abs(oracle.silu_scalar(-40.0)) < 1e-15
    assert abs(oracle.silu_scalar(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    # d/dg silu at 0 is 1/2: d_gate = dh * u * 0.5 * (1 + 0)
    dg, du = oracle.dswiglu(np.array([2.0], np.float32), np.array([0.0], np.float32),
                            np.array([3.0], np.float32))
    assert dg[0] == 3.0 and du[0] == 0.0


def test_silu_matches_torch():
    g = np.linspace(-20, 20, 4001)
    ref = F.silu(torch.from_numpy(g)).numpy()
    mine = np.array([oracle.silu_scalar(v) for v in g])
    assert np.max(np.abs(mine - ref)) < 1e-13


def test_dswiglu_matches_autograd():
    r = np.random.default_rng(0)
    g = (r.standard_normal(5000) * 3).astype(np.float32)
    u = r.standard_normal(5000).astype(np.float32)
    dh = r.standard_normal(5000).astype(np.float32)
    gt = torch.from_numpy(g.astype(np.float64)).requires_grad_(True)
    ut = torch.from_numpy(u.astype(np.float64)).requires_grad_(True)
    (F.silu(gt) * ut).backward(torch.from_numpy(dh.astype(np.float64)))
    dg, du = oracle.dswiglu(dh, g, u)
    assert np.allclose(dg, gt.grad.numpy(), rtol=1e-6, atol=1e-6)
    assert np.allclose(du, ut.grad.numpy(), rtol=1e-6, atol=1e-6)
    h = oracle.swiglu(g, u)
    assert np.allclose(h, (F.silu(gt) * ut).detach().numpy(), rtol=1e-6, atol=1e-6)


def test_forward_is_the_samples_composite():
    r = np.random.default_rng(1)
    M, H, I = 37, 64, 48
    x = r.standard_normal((M, H)).astype(np.float32)
    Wg = (r.standard_normal((I, H)) * 0.1).astype(np.float32)
    Wu = (r.standard_normal((I, H)) * 0.1).astype(np.float32)
    xb, Wgb, Wub = (oracle.round_to(a, oracle.BF16) for a in (x, Wg, Wu))
    h, gb, ub, g, u = oracle.swiglu_forward(xb, Wgb, Wub, oracle.BF16)
    xt, Wgt, Wut = (torch.from_numpy(oracle.decode(a, oracle.BF16).astype(np.float64))
                    for a in (xb, Wgb, Wub))
    ref = (F.silu(xt @ Wgt.t()) * (xt @ Wut.t())).numpy()
    hv = oracle.decode(h, oracle.BF16)
    # one bf16 rounding (2^-9 relative) on top of fp32 accumulation
    assert np.all(np.abs(hv - ref) <= 2.0**-8 * np.abs(ref) + 1e-6)
    assert np.allclose(oracle.decode(gb, oracle.BF16), (xt @ Wgt.t()).numpy(), rtol=2**-8, atol=1e-6)


def test_backward_is_autograd_of_the_composite():
    r = np.random.default_rng(2)
    M, H, I = 29, 40, 56
    dout = oracle.round_to(r.standard_normal((M, H)).astype(np.float32), oracle.BF16)
    Wd = oracle.round_to((r.standard_normal((H, I)) * 0.1).astype(np.float32), oracle.BF16)
    g = oracle.round_to((r.standard_normal((M, I)) * 2).astype(np.float32), oracle.BF16)
    u = oracle.round_to(r.standard_normal((M, I)).astype(np.float32), oracle.BF16)
    dg, du, dh = oracle.dswiglu_backward(dout, Wd, g, u, oracle.BF16)
    gt = torch.from_numpy(oracle.decode(g, oracle.BF16).astype(np.float64)).requires_grad_(True)
    ut = torch.from_numpy(oracle.decode(u, oracle.BF16).astype(np.float64)).requires_grad_(True)
    dht = torch.from_numpy(oracle.decode(dout, oracle.BF16).astype(np.float64)) @ \
        torch.from_numpy(oracle.decode(Wd, oracle.BF16).astype(np.float64))
    (F.silu(gt) * ut).backward(dht)
    for mine, ref in ((dg, gt.grad.numpy()), (du, ut.grad.numpy())):
        v = oracle.decode(mine, oracle.BF16)
        assert np.all(np.abs(v - ref) <= 2.0**-8 * np.abs(ref) + 1e-4 * np.abs(ref).max())
