"""Pins of the short causal convolution oracle (CPU): impulse response,
document reset (a packed row equals separate runs), the identity filter,
causality, and central finite differences of dx and dw."""
import numpy as np

from oracle import short_conv


def test_impulse_response_is_the_filter_through_silu():
    C, K = 3, 4
    w = np.arange(C * K, dtype=float).reshape(C, K) / 10.0 - 0.4
    x = np.zeros((8, C))
    x[2] = 1.0
    y = short_conv.forward(x, w, activation="none")
    for j in range(K):  # y_{2 + K-1-j} = w_j
        np.testing.assert_allclose(y[2 + K - 1 - j], w[:, j], rtol=0, atol=0)
    assert np.all(y[:2] == 0) and np.all(y[6:] == 0)
    ys = short_conv.forward(x, w)
    np.testing.assert_allclose(ys, y / (1.0 + np.exp(-y)), rtol=1e-15)


def test_document_reset_equals_separate_runs():
    rng = np.random.default_rng(4)
    lens = [5, 1, 0, 9, 3]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x, w = rng.normal(size=(cu[-1], 6)), rng.normal(size=(6, 4))
    dy = rng.normal(size=x.shape)
    y = short_conv.forward(x, w, cu)
    dx, dw = short_conv.backward(x, w, dy, cu)
    dw_sum = np.zeros_like(w)
    for a, b in zip(cu[:-1], cu[1:]):
        if b > a:
            np.testing.assert_allclose(y[a:b], short_conv.forward(x[a:b], w), rtol=1e-15)
            dxs, dws = short_conv.backward(x[a:b], w, dy[a:b])
            np.testing.assert_allclose(dx[a:b], dxs, rtol=1e-15)
            dw_sum += dws
    np.testing.assert_allclose(dw, dw_sum, rtol=1e-12)


def test_identity_filter_and_causality():
    rng = np.random.default_rng(5)
    x = rng.normal(size=(10, 4))
    w = np.zeros((4, 4))
    w[:, 3] = 1.0  # tap on x_t only
    np.testing.assert_allclose(short_conv.forward(x, w, activation="none"), x, rtol=0)
    w2 = rng.normal(size=(4, 4))
    y1 = short_conv.forward(x, w2)
    x2 = x.copy()
    x2[6:] += 1.0  # changing the future leaves the past unchanged
    np.testing.assert_array_equal(short_conv.forward(x2, w2)[:6], y1[:6])


def test_finite_differences():
    rng = np.random.default_rng(6)
    cu = np.array([0, 4, 11])
    x, w, dy = rng.normal(size=(11, 3)), rng.normal(size=(3, 4)), rng.normal(size=(11, 3))
    dx, dw = short_conv.backward(x, w, dy, cu)
    h = 1e-6

    def loss(xx, ww):
        return float((short_conv.forward(xx, ww, cu) * dy).sum())

    for idx in [(0, 1), (3, 0), (4, 2), (10, 1)]:
        p, m = x.copy(), x.copy()
        p[idx] += h
        m[idx] -= h
        fd = (loss(p, w) - loss(m, w)) / (2 * h)
        assert abs(fd - dx[idx]) <= 1e-7 * max(1.0, abs(fd)), (idx, fd, dx[idx])
    for idx in [(0, 0), (1, 3), (2, 2)]:
        p, m = w.copy(), w.copy()
        p[idx] += h
        m[idx] -= h
        fd = (loss(x, p) - loss(x, m)) / (2 * h)
        assert abs(fd - dw[idx]) <= 1e-7 * max(1.0, abs(fd)), (idx, fd, dw[idx])
