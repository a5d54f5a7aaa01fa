"""Pins for the oracle's output activations (CPU only).

Each activation is checked against torch's float64 implementation (an
independent library routine), against exact identities of its definition,
and on its special values; LIPSCHITZ is checked against finite differences.
"""
import math

import numpy as np
import pytest
import torch

import oracle

GRID = np.concatenate([np.linspace(-30.0, 30.0, 6001), [0.0, -0.0, 1e-300, -1e-300, 1e-8, -1e-8,
                                                        700.0, -700.0, 1e10, -1e10]])


def torch_ref(x, act):
    t = torch.from_numpy(x.astype(np.float64))
    f = torch.nn.functional
    return {
        oracle.ACT_NONE: lambda: t,
        oracle.ACT_RELU: lambda: f.relu(t),
        oracle.ACT_SILU: lambda: f.silu(t),
        oracle.ACT_GELU_TANH: lambda: f.gelu(t, approximate="tanh"),
        oracle.ACT_GELU_ERF: lambda: f.gelu(t, approximate="none"),
    }[act]().numpy()


@pytest.mark.parametrize("act", [oracle.ACT_NONE, oracle.ACT_RELU, oracle.ACT_SILU,
                                 oracle.ACT_GELU_TANH, oracle.ACT_GELU_ERF])
def test_matches_torch_float64(act):
    got = oracle.activate(GRID, act)
    want = torch_ref(GRID, act)
    # atol: both sides cancel in 1 + tanh(u) or 1 + erf(y/sqrt 2) for y << 0
    assert np.allclose(got, want, rtol=1e-12, atol=1e-14), np.max(np.abs(got - want))


@pytest.mark.parametrize("act", [oracle.ACT_SILU, oracle.ACT_GELU_TANH, oracle.ACT_GELU_ERF])
def test_odd_part_is_the_identity(act):
    """x*g(x) with g(x) + g(-x) = 1 (sigmoid, the tanh form's and the erf
    form's Phi): act(x) - act(-x) = x exactly in the reals."""
    x = np.linspace(-12.0, 12.0, 2401)
    d = oracle.activate(x, act) - oracle.activate(-x, act)
    assert np.allclose(d, x, rtol=0, atol=1e-13)


def test_special_values():
    nan = np.array([np.nan])
    for act in range(5):
        assert np.isnan(oracle.activate(nan, act))[0]
    z = oracle.activate(np.array([-0.0, -1.0, -1e-30]), oracle.ACT_RELU)
    assert np.all(z == 0.0) and not np.any(np.signbit(z))  # +0 for y <= 0
    # sigmoid(0) = Phi(0) = 1/2: every smooth form has slope 1/2 at 0
    h = 1e-6
    for act in (oracle.ACT_SILU, oracle.ACT_GELU_TANH, oracle.ACT_GELU_ERF):
        slope = (oracle.activate(np.array([h]), act) - oracle.activate(np.array([-h]), act))[0] / (2 * h)
        assert abs(slope - 0.5) < 1e-9
    # GELU (erf form) at 1 is Phi(1) = (1 + erf(1/sqrt 2)) / 2
    assert oracle.activate(np.array([1.0]), oracle.ACT_GELU_ERF)[0] == pytest.approx(
        0.5 * (1 + math.erf(1 / math.sqrt(2))), rel=1e-15)
    # large |y|: identity above, zero below
    for act in (oracle.ACT_SILU, oracle.ACT_GELU_TANH, oracle.ACT_GELU_ERF):
        v = oracle.activate(np.array([50.0, -50.0]), act)
        assert v[0] == 50.0 and abs(v[1]) < 1e-20


@pytest.mark.parametrize("act", [oracle.ACT_RELU, oracle.ACT_SILU, oracle.ACT_GELU_TANH,
                                 oracle.ACT_GELU_ERF])
def test_lipschitz_bound(act):
    x = np.linspace(-20.0, 20.0, 400001)
    d = np.abs(np.diff(oracle.activate(x, act)) / np.diff(x))
    assert d.max() <= oracle.LIPSCHITZ[act]
    assert d.max() >= oracle.LIPSCHITZ[act] - 0.02  # and the bound is tight


def test_gemv_ex_applies_activation_last():
    from nvfp4_block_scaled_gemv_gb300 import synthetic
    M, K, L = 40, 256, 2
    p = synthetic.make_problem(M, K, L, seed=3)
    bias = (np.random.default_rng(0).standard_normal((L, M))).astype(np.float16).view(np.uint16)
    c0, y0, t0 = oracle.gemv_ex(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L, alpha=0.25, bias=bias)
    for act in range(5):
        c, y, t = oracle.gemv_ex(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L, alpha=0.25,
                                 bias=bias, activation=act)
        assert np.array_equal(y, oracle.activate(y0, act))
        assert np.array_equal(c, oracle.fp16_rne(oracle.activate(y0, act)))
        assert np.allclose(t, oracle.LIPSCHITZ[act] * t0)
    with pytest.raises(ValueError):
        oracle.activate(np.zeros(1), 9)
