"""Pins of the gated RMSNorm oracle (CPU): a hand-computed example, the
special cases that reduce it to plain RMSNorm and to a pure gate, scale
invariance, and central finite differences of every gradient."""
import numpy as np

from oracle import norm_gate


def test_hand_example():
    # x = (3, 4): mean x^2 = 12.5, r = 1/sqrt(12.5 + 1e-6); g = 0 -> sigmoid = 1/2; w = (2, 1)
    x = np.array([[3.0, 4.0]])
    y = norm_gate.forward(x, np.zeros((1, 2)), np.array([2.0, 1.0]))
    r = 1.0 / np.sqrt(12.5 + 1e-6)
    np.testing.assert_allclose(y, [[3.0 * r * 2.0 * 0.5, 4.0 * r * 1.0 * 0.5]], rtol=1e-15)


def test_open_gate_unit_weight_is_rms_normalisation():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(5, 64))
    y = norm_gate.forward(x, np.full((5, 64), 60.0), np.ones(64), eps=0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-12)


def test_scale_invariance_without_eps():
    rng = np.random.default_rng(2)
    x, g, w = rng.normal(size=(4, 16)), rng.normal(size=(4, 16)), rng.normal(size=16)
    np.testing.assert_allclose(norm_gate.forward(7.5 * x, g, w, eps=0.0), norm_gate.forward(x, g, w, eps=0.0),
                               rtol=1e-12)


def test_finite_differences():
    rng = np.random.default_rng(3)
    x, g, w, dy = rng.normal(size=(3, 8)), rng.normal(size=(3, 8)), rng.normal(size=8), rng.normal(size=(3, 8))
    dx, dg, dw = norm_gate.backward(x, g, w, dy)
    h = 1e-6

    def loss(xx, gg, ww):
        return float((norm_gate.forward(xx, gg, ww) * dy).sum())

    for arr, grad, idx in ((x, dx, (1, 3)), (g, dg, (2, 5)), (w, dw, (4,))):
        p, m = arr.copy(), arr.copy()
        p[idx] += h
        m[idx] -= h
        args_p = [p if a is arr else a for a in (x, g, w)]
        args_m = [m if a is arr else a for a in (x, g, w)]
        fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (idx, fd, grad[idx])
