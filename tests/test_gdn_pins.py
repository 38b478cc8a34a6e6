"""Pins of the scalar-gate reading of the oracle (CPU).

The scalar-gated variant is the per-channel recurrence with equal channel
gates.  These tests pin that reduction against an independent scalar form of
the recurrence, S_t = exp(g_t) (S_{t-1} - beta_t k_t (k_t^T S_{t-1})) + beta_t
k_t v_t^T, written out here directly, and pin the summed gate gradient with
central finite differences in f."""
import numpy as np

from kimi_delta_attention_bwd_gb300.inputs import custom, make_inputs
from _common import run_oracle


def _scalar_recurrence(x, scale):
    Ntok, H, dk = x["q"].shape
    dv = x["v"].shape[-1]
    o = np.zeros((Ntok, H, dv))
    S = np.zeros((H, dk, dv))
    for t in range(Ntok):
        for h in range(H):
            q = x["q"][t, h] / np.sqrt((x["q"][t, h] ** 2).sum() + 1e-6)
            k = x["k"][t, h] / np.sqrt((x["k"][t, h] ** 2).sum() + 1e-6)
            z = x["f"][t, h] + x["dt_bias"][h]
            g = -np.exp(x["A_log"][h]) * np.logaddexp(0.0, z)
            beta = 1.0 / (1.0 + np.exp(-x["b"][t, h]))
            Sh = np.exp(g) * (S[h] - beta * np.outer(k, k @ S[h])) + beta * np.outer(k, x["v"][t, h])
            S[h] = Sh
            o[t, h] = scale * Sh.T @ q
    return o, S


def _inputs(seed):
    inp = make_inputs(custom(1, 9, 2, 4, 3, dtype="f32", gate="scalar"), seed=seed)
    from kimi_delta_attention_bwd_gb300.inputs import numpy_f64
    return inp, numpy_f64(inp)


def test_scalar_gate_oracle_equals_direct_scalar_recurrence():
    inp, x = _inputs(5)
    ref = run_oracle(inp, backward=False)
    o, S = _scalar_recurrence(x, inp["scale"])
    np.testing.assert_allclose(ref["o"], o, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(ref["h_final"][0], S, rtol=1e-10, atol=1e-12)


def test_scalar_gate_gradient_by_finite_differences():
    inp, x = _inputs(6)
    ref = run_oracle(inp, backward=True)
    dO = x["dO"]
    eps = 1e-6
    for (t, h) in [(0, 0), (4, 1), (8, 0)]:
        fp = inp["f"].double()  # perturb in float64: a float32 step would be quantised
        fm = inp["f"].double()
        fp[0, t, h] += eps
        fm[0, t, h] -= eps
        lp = (run_oracle(dict(inp, f=fp), backward=False)["o"] * dO).sum()
        lm = (run_oracle(dict(inp, f=fm), backward=False)["o"] * dO).sum()
        fd = (lp - lm) / (2 * eps)
        assert abs(fd - ref["df"][t, h]) <= 1e-6 * max(1.0, abs(fd)), (t, h, fd, ref["df"][t, h])
