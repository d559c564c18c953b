"""Pins of the oracle's GELU steps (the GELU_BIAS epilog named on the
nvmath-python / cuBLASLt page, "other epilogs"; tanh form of Hendrycks &
Gimpel 2016): closed forms, an exact symmetry, the library routine, and the
derivative against a finite difference."""
import math

import numpy as np
import pytest

import oracle


def test_gelu_closed_forms():
    assert oracle.gelu_scalar(0.0) == 0.0
    assert oracle.dgelu_scalar(0.0) == 0.5
    assert oracle.gelu_scalar(30.0) == 30.0          # tanh saturates to 1
    assert oracle.gelu_scalar(-30.0) == 0.0          # ... and to -1 (0.5 z (1 - 1))
    assert abs(oracle.dgelu_scalar(30.0) - 1.0) < 1e-15
    assert abs(oracle.dgelu_scalar(-30.0)) < 1e-15
    # by hand at z = 1: u = sqrt(2/pi) * 1.044715
    u = math.sqrt(2 / math.pi) * 1.044715
    assert abs(oracle.gelu_scalar(1.0) - 0.5 * (1 + math.tanh(u))) < 1e-15


@pytest.mark.parametrize("z", [0.1, 0.7, 1.3, 2.9, 5.0])
def test_gelu_odd_part_is_identity(z):
    # the tanh form satisfies gelu(z) - gelu(-z) = z exactly (tanh is odd)
    assert abs((oracle.gelu_scalar(z) - oracle.gelu_scalar(-z)) - z) < 1e-14 * max(1, z)


def test_gelu_matches_torch_float64():
    torch = pytest.importorskip("torch")
    z = np.linspace(-8, 8, 4001)
    ref = torch.nn.functional.gelu(torch.from_numpy(z), approximate="tanh").numpy()
    mine = np.array([oracle.gelu_scalar(v) for v in z])
    assert np.max(np.abs(mine - ref)) < 1e-14


def test_dgelu_is_the_derivative():
    z = np.linspace(-6, 6, 1201)
    h = 1e-6
    fd = np.array([(oracle.gelu_scalar(v + h) - oracle.gelu_scalar(v - h)) / (2 * h) for v in z])
    d = np.array([oracle.dgelu_scalar(v) for v in z])
    assert np.max(np.abs(fd - d)) < 1e-8


def test_vector_steps_round_once():
    z = np.array([-3.0, -0.5, 0.0, 0.25, 4.0], dtype=np.float32)
    y = oracle.gelu(z)
    assert np.array_equal(y, np.array([np.float32(oracle.gelu_scalar(float(v))) for v in z]))
    g = np.array([1.0, -2.0, 3.0, 0.5, -1.0], dtype=np.float32)
    dz = oracle.dgelu(g, z)
    ref = np.array([np.float32(float(a) * oracle.dgelu_scalar(float(b))) for a, b in zip(g, z)])
    assert np.array_equal(dz, ref)
    assert dz[2] == 1.5  # g * gelu'(0) = 3 * 0.5


def test_dgelu_bgrad_invariant():
    r = np.random.default_rng(0)
    M, N, K = 70, 24, 40
    dY = r.standard_normal((M, K)).astype(np.float16)
    W = (r.standard_normal((N, K)) * 0.2).astype(np.float16)
    aux = oracle.round_to(r.standard_normal((M, N)).astype(np.float32), oracle.F16)
    out, bgrad, g = oracle.dgelu_bgrad(dY, W, aux, oracle.F16, oracle.B_NK)
    dz = oracle.dgelu(g, oracle.decode(aux, oracle.F16))
    assert np.allclose(bgrad, dz.astype(np.float64).sum(0), rtol=1e-6, atol=1e-6)
