"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test fixes the oracle to something other than itself: closed forms of
the gate pieces, special cases of the recurrence that reduce to textbook
results (pure decay, the ungated delta rule's exact retrieval of orthonormal
keys, the retrieval property of a beta=1 write), linearity, an independent
dense formulation built from explicit matrix products, the chunked WY form
solved with a library inverse, central finite differences for every gradient,
and the packed-versus-separate identity of the torchtitan packing PR.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import oracle

PREC = ["f64", "f32"]
TOL = {"f64": 1e-11, "f32": 2e-5}
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny(lens, H=2, dk=4, dv=3, seed=0, h0=False, gate_scale=1.0):
    rng = np.random.RandomState(seed)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(cu[-1])
    x = {
        "q": rng.randn(N, H, dk), "k": rng.randn(N, H, dk), "v": rng.randn(N, H, dv),
        "f": rng.randn(N, H, dk) * gate_scale, "b": rng.randn(N, H),
        "A_log": np.log(rng.uniform(1, 16, H)),
        "cu_seqlens": cu, "scale": 1.0 / math.sqrt(dk),
    }
    dt = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), (H, dk)))
    x["dt_bias"] = dt + np.log(-np.expm1(-dt))
    x["h0"] = rng.randn(len(lens), H, dk, dv) * 0.5 if h0 else None
    return x


def unit(a, eps=0.0):
    return a / np.sqrt((a * a).sum(-1, keepdims=True) + eps)


def softplus_np(x):
    return np.logaddexp(0.0, x)  # library routine, independent of the oracle's form


# ---------------------------------------------------------------- gate pieces
@pytest.mark.parametrize("p", PREC)
def test_gate_closed_forms(p):
    tol = TOL[p] * 10
    # A_log = 0, x = 0: g = -softplus(0) = -ln 2
    assert abs(oracle.gate(0.0, 0.0, p) + math.log(2.0)) < tol
    # softplus(ln(e - 1)) = 1, so with A_log = ln 2 the gate is -2
    assert abs(oracle.gate(math.log(2.0), math.log(math.e - 1.0), p) + 2.0) < tol
    # far tails: softplus(50) = 50 (to 1e-22), softplus(-50) = e^-50 (relative 1e-22)
    assert abs(oracle.gate(math.log(3.0), 50.0, p) + 150.0) < 150.0 * tol
    assert abs(oracle.gate(0.0, -50.0, p) / -math.exp(-50.0) - 1.0) < tol
    # sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4, sigmoid(-ln 3) = 1/4
    assert abs(oracle.sigmoid(0.0, p) - 0.5) < tol
    assert abs(oracle.sigmoid(math.log(3.0), p) - 0.75) < tol
    assert abs(oracle.sigmoid(-math.log(3.0), p) - 0.25) < tol


def test_f32_variant_is_fp32():
    assert oracle.load("f32").kda_oracle_real_bytes() == 4
    assert oracle.load("f64").kda_oracle_real_bytes() == 8


# ------------------------------------------------------------ special cases
@pytest.mark.parametrize("p", PREC)
def test_one_step_from_zero_state(p):
    """From S = 0 one token gives S_1 = beta k^ v^T and o_1 = scale beta (k^.q^) v,
    whatever the gate (decay of a zero state is zero)."""
    x = tiny([1, 1, 1], H=3, dk=5, dv=4, seed=1, gate_scale=3.0)
    o, hf = oracle.forward(x, precision=p)
    qh, kh = unit(x["q"], 1e-6), unit(x["k"], 1e-6)
    beta = 1.0 / (1.0 + np.exp(-x["b"]))
    for t in range(3):
        for h in range(3):
            S1 = beta[t, h] * np.outer(kh[t, h], x["v"][t, h])
            np.testing.assert_allclose(hf[t, h], S1, rtol=TOL[p], atol=TOL[p])
            o1 = x["scale"] * beta[t, h] * (kh[t, h] @ qh[t, h]) * x["v"][t, h]
            np.testing.assert_allclose(o[t, h], o1, rtol=TOL[p] * 10, atol=TOL[p])


@pytest.mark.parametrize("p", PREC)
def test_beta_zero_is_pure_decay(p):
    """beta = 0 (b = -1000, sigmoid underflows to exactly 0): the state only
    decays, S_t = Diag(exp(sum_{s<=t} g_s)) h0, decaying key channels (rows)."""
    x = tiny([7, 5], H=2, dk=4, dv=3, seed=2, h0=True)
    x["b"][:] = -1000.0
    o, hf = oracle.forward(x, precision=p)
    qh = unit(x["q"], 1e-6)
    for s in range(2):
        t0, t1 = x["cu_seqlens"][s], x["cu_seqlens"][s + 1]
        for h in range(2):
            g = -np.exp(x["A_log"][h]) * softplus_np(x["f"][t0:t1, h] + x["dt_bias"][h])
            G = np.cumsum(g, axis=0)
            for t in range(t1 - t0):
                St = np.exp(G[t])[:, None] * x["h0"][s, h]
                np.testing.assert_allclose(o[t0 + t, h], x["scale"] * St.T @ qh[t0 + t, h],
                                           rtol=TOL[p] * 10, atol=TOL[p])
            np.testing.assert_allclose(hf[s, h], np.exp(G[-1])[:, None] * x["h0"][s, h],
                                       rtol=TOL[p] * 10, atol=TOL[p])


@pytest.mark.parametrize("p", PREC)
def test_ungated_delta_rule_orthonormal_keys(p):
    """A_log = -1000 makes the decay exactly 1 (g = -0); with beta = 1 the
    ungated delta rule stores orthonormal keys exactly: S = sum k_i v_i^T, and
    re-writing a key replaces its value (S = k v_new^T for that key)."""
    dk, dv, H = 6, 5, 1
    rng = np.random.RandomState(3)
    Qm, _ = np.linalg.qr(rng.randn(dk, dk))
    keys = Qm.T  # orthonormal rows
    order = [0, 1, 2, 3, 1, 4]  # key 1 is written twice
    N = len(order)
    x = tiny([N], H=H, dk=dk, dv=dv, seed=4)
    x["eps"] = 0.0
    x["k"][:, 0] = keys[order]
    x["A_log"][:] = -1000.0
    x["b"][:] = 1000.0
    o, hf = oracle.forward(x, precision=p)
    last = {}
    for t, i in enumerate(order):
        last[i] = x["v"][t, 0]
        S = sum(np.outer(keys[j], vj) for j, vj in last.items())
        qh = unit(x["q"][t, 0])
        np.testing.assert_allclose(o[t, 0], x["scale"] * S.T @ qh, rtol=1e-4 if p == "f32" else 1e-10,
                                   atol=1e-5 if p == "f32" else 1e-12)
    S = sum(np.outer(keys[j], vj) for j, vj in last.items())
    np.testing.assert_allclose(hf[0, 0], S, atol=1e-5 if p == "f32" else 1e-12)


@pytest.mark.parametrize("p", PREC)
def test_beta_one_write_is_retrievable(p):
    """With beta = 1 the correction is computed on the decayed state, so the
    new state maps the written key to its value exactly: S_t^T k^_t = v_t,
    for any gate.  Reading with q = k gives o_t = scale v_t."""
    x = tiny([9, 6], H=2, dk=5, dv=4, seed=5, h0=True, gate_scale=2.0)
    x["eps"] = 0.0
    x["b"][:] = 1000.0
    x["q"] = x["k"].copy()
    o, _ = oracle.forward(x, precision=p)
    np.testing.assert_allclose(o, x["scale"] * x["v"], rtol=1e-4 if p == "f32" else 1e-10,
                               atol=1e-5 if p == "f32" else 1e-12)


@pytest.mark.parametrize("p", PREC)
def test_linear_in_v_and_column_independent(p):
    """With h0 = 0 the output is linear in v (scaling v by 2 is exact in
    binary floating point) and the dv columns never mix."""
    x = tiny([8, 3], H=2, dk=4, dv=5, seed=6)
    o1, h1 = oracle.forward(x, precision=p)
    x2 = dict(x, v=2.0 * x["v"])
    o2, h2 = oracle.forward(x2, precision=p)
    assert np.array_equal(o2, 2.0 * o1) and np.array_equal(h2, 2.0 * h1)
    perm = np.array([3, 0, 4, 1, 2])
    x3 = dict(x, v=x["v"][:, :, perm])
    o3, h3 = oracle.forward(x3, precision=p)
    assert np.array_equal(o3, o1[:, :, perm]) and np.array_equal(h3, h1[..., perm])


# ------------------------------------------------ independent formulations
def dense_transfer(x, s, h):
    """States S_r of one document built by brute force from explicit matrix
    products of the per-token transfer M_t = (I - beta_t k_t k_t^T) Diag(exp g_t)
    and the write W_t = beta_t k_t v_t^T:
        S_r = M_r ... M_0 h0 + sum_{t<=r} M_r ... M_{t+1} W_t."""
    t0, t1 = x["cu_seqlens"][s], x["cu_seqlens"][s + 1]
    dk, dv = x["q"].shape[2], x["v"].shape[2]
    eps = x.get("eps", 1e-6)
    qh, kh = unit(x["q"], eps), unit(x["k"], eps)
    beta = 1.0 / (1.0 + np.exp(-x["b"]))
    g = -np.exp(x["A_log"][h]) * softplus_np(x["f"][:, h] + x["dt_bias"][h])
    Ms, Ws = [], []
    for t in range(t0, t1):
        k_ = kh[t, h][:, None]
        Ms.append((np.eye(dk) - beta[t, h] * k_ @ k_.T) @ np.diag(np.exp(g[t])))
        Ws.append(beta[t, h] * k_ @ x["v"][t, h][None, :])

    def chain(a, b):  # M_b M_{b-1} ... M_a, identity when a > b
        P = np.eye(dk)
        for t in range(a, b + 1):
            P = Ms[t] @ P
        return P
    h0 = np.zeros((dk, dv)) if x.get("h0") is None else x["h0"][s, h]
    outs = []
    for r in range(len(Ms)):
        S = chain(0, r) @ h0
        for t in range(r + 1):
            S = S + chain(t + 1, r) @ Ws[t]
        outs.append(S)
    return outs, qh[t0:t1, h]


@pytest.mark.parametrize("p", PREC)
def test_dense_transfer_products(p):
    x = tiny([6, 0, 5], H=2, dk=4, dv=3, seed=7, h0=True, gate_scale=2.0)
    o, hf = oracle.forward(x, precision=p)
    for s in range(3):
        t0 = x["cu_seqlens"][s]
        for h in range(2):
            Sr, qh = dense_transfer(x, s, h)
            for r, S in enumerate(Sr):
                np.testing.assert_allclose(o[t0 + r, h], x["scale"] * S.T @ qh[r],
                                           rtol=TOL[p] * 100, atol=TOL[p] * 10)
            final = Sr[-1] if Sr else x["h0"][s, h]
            np.testing.assert_allclose(hf[s, h], final, rtol=TOL[p] * 100, atol=TOL[p] * 10)


def chunked_wy(x, s, h, C):
    """The chunk form the CUDA kernels implement, solved with numpy's inverse:
    per chunk with entry state S and in-chunk cumulative log-decay G,
      A = strict_lower(diag(beta) (K^ K^T with ratios exp(G_r - G_s)))
      E = (I + A)^-1 diag(beta) (V - (K^ * exp(G)) S)
      O = scale [ (Q^ * exp(G)) S + inclusive_lower(Q^ K^T with ratios) E ]
      S <- Diag(exp(G_last)) S + (K^ * exp(G_last - G))^T E."""
    t0, t1 = x["cu_seqlens"][s], x["cu_seqlens"][s + 1]
    eps = x.get("eps", 1e-6)
    qh, kh = unit(x["q"][t0:t1, h], eps), unit(x["k"][t0:t1, h], eps)
    V = x["v"][t0:t1, h]
    beta = 1.0 / (1.0 + np.exp(-x["b"][t0:t1, h]))
    g = -np.exp(x["A_log"][h]) * softplus_np(x["f"][t0:t1, h] + x["dt_bias"][h])
    S = np.zeros((qh.shape[1], V.shape[1])) if x.get("h0") is None else x["h0"][s, h].copy()
    O = np.zeros_like(V)
    for c0 in range(0, t1 - t0, C):
        sl = slice(c0, min(c0 + C, t1 - t0))
        L = sl.stop - sl.start
        G = np.cumsum(g[sl], axis=0)
        R = np.exp(G[:, None, :] - G[None, :, :])  # [r, s, i] ratio exp(G_r - G_s)
        KK = np.einsum("ri,si,rsi->rs", kh[sl], kh[sl], R)
        QK = np.einsum("ri,si,rsi->rs", qh[sl], kh[sl], R)
        A = np.tril(beta[sl][:, None] * KK, -1)
        E = np.linalg.inv(np.eye(L) + A) @ (beta[sl][:, None] * (V[sl] - (kh[sl] * np.exp(G)) @ S))
        O[sl] = x["scale"] * ((qh[sl] * np.exp(G)) @ S + np.tril(QK) @ E)
        S = np.exp(G[-1])[:, None] * S + (kh[sl] * np.exp(G[-1] - G)).T @ E
    return O, S


@pytest.mark.parametrize("C", [4, 5, 64])
def test_chunked_wy_form_matches(C):
    x = tiny([13, 1, 9], H=2, dk=4, dv=3, seed=8, h0=True)
    o, hf = oracle.forward(x)
    for s in range(3):
        t0, t1 = x["cu_seqlens"][s], x["cu_seqlens"][s + 1]
        for h in range(2):
            O, S = chunked_wy(x, s, h, C)
            np.testing.assert_allclose(o[t0:t1, h], O, rtol=1e-9, atol=1e-11)
            np.testing.assert_allclose(hf[s, h], S, rtol=1e-9, atol=1e-11)


# ------------------------------------------------------- finite differences
def loss(x, dO, dhf):
    o, hf = oracle.forward(x, threads=1)
    return float((o * dO).sum() + (hf * dhf).sum())


def test_finite_differences_every_gradient():
    """Central differences (h = 1e-6, float64) of L = sum(o dO) + sum(h_final
    dh_final) against every analytic gradient, on two documents and a
    zero-length one, with an initial state."""
    x = tiny([5, 0, 4], H=2, dk=3, dv=2, seed=9, h0=True, gate_scale=1.5)
    rng = np.random.RandomState(10)
    dO = rng.randn(*x["v"].shape)
    dhf = rng.randn(*x["h0"].shape)
    g = oracle.backward(x, dO, dhf, threads=1)
    hstep = 1e-6
    names = [("q", "dq"), ("k", "dk"), ("v", "dv"), ("f", "df"), ("b", "db"),
             ("A_log", "dA_log"), ("dt_bias", "ddt_bias"), ("h0", "dh0")]
    for inp, grad in names:
        base = x[inp]
        num = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = base.copy(), base.copy()
            xp[idx] += hstep
            xm[idx] -= hstep
            num[idx] = (loss(dict(x, **{inp: xp}), dO, dhf) - loss(dict(x, **{inp: xm}), dO, dhf)) / (2 * hstep)
        ana = g[grad]
        err = np.abs(num - ana).max() / max(1e-12, np.abs(num).max())
        assert err < 1e-6, (grad, err)


def test_finite_differences_across_checkpoint_segments():
    """The backward rebuilds S_{t-1} from states checkpointed every 64 tokens.
    On documents of 70 and 140 tokens (two and three checkpoint segments),
    with an initial state and a final-state gradient, central differences at
    entries sampled in every segment (both sides of each segment boundary)
    match every analytic gradient.  A checkpoint restored one segment off, or
    taken after its segment instead of before, gives the tokens of that
    segment the wrong previous states and fails here."""
    x = tiny([70, 140], H=2, dk=3, dv=2, seed=18, h0=True)
    rng = np.random.RandomState(19)
    dO = rng.randn(*x["v"].shape)
    dhf = rng.randn(*x["h0"].shape)
    g = oracle.backward(x, dO, dhf, threads=1)
    hstep = 1e-6
    # document 0: tokens 0..69 (segments [0, 64), [64, 70)); document 1: 70..209
    # (segments [70, 134), [134, 198), [198, 210))
    toks = [0, 31, 63, 64, 69, 70, 100, 133, 134, 170, 197, 198, 209]

    def fd(inp, idx):
        base = x[inp]
        xp, xm = base.copy(), base.copy()
        xp[idx] += hstep
        xm[idx] -= hstep
        return (loss(dict(x, **{inp: xp}), dO, dhf) - loss(dict(x, **{inp: xm}), dO, dhf)) / (2 * hstep)

    cases = []
    for inp, grad in [("q", "dq"), ("k", "dk"), ("v", "dv"), ("f", "df"), ("b", "db")]:
        shape = x[inp].shape
        for t in toks:
            rest = tuple(rng.randint(0, n) for n in shape[1:])
            cases.append((inp, grad, (t,) + rest))
    for inp, grad in [("A_log", "dA_log"), ("dt_bias", "ddt_bias"), ("h0", "dh0")]:
        for idx in np.ndindex(x[inp].shape):
            cases.append((inp, grad, idx))
    by_grad = {}
    for inp, grad, idx in cases:
        by_grad.setdefault(grad, []).append((fd(inp, idx), g[grad][idx]))
    for grad, pairs in by_grad.items():
        num = np.array([p[0] for p in pairs])
        ana = np.array([p[1] for p in pairs])
        err = np.abs(num - ana).max() / max(1e-12, np.abs(num).max())
        assert err < 1e-6, (grad, err)


def test_gradients_with_large_gates_and_no_h0():
    x = tiny([7, 3], H=1, dk=3, dv=2, seed=11, gate_scale=4.0)
    rng = np.random.RandomState(12)
    dO = rng.randn(*x["v"].shape)
    g = oracle.backward(x, dO, None, threads=1)
    hstep = 1e-6
    for inp, grad in [("f", "df"), ("k", "dk"), ("b", "db"), ("dt_bias", "ddt_bias")]:
        base = x[inp]
        num = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            xp, xm = base.copy(), base.copy()
            xp[idx] += hstep
            xm[idx] -= hstep
            num[idx] = (loss(dict(x, **{inp: xp}), dO, 0.0) - loss(dict(x, **{inp: xm}), dO, 0.0)) / (2 * hstep)
        err = np.abs(num - g[grad]).max() / max(1e-12, np.abs(num).max())
        assert err < 1e-6, (grad, err)


# ------------------------------------------------------------- segmentation
def test_packed_equals_separate_torchtitan_fixture():
    """torchtitan PR "[kimi k3] Support sample packing in KDA", Verification:
    two documents of 96 and 160 tokens, packed with cu_seqlens (0, 96, 256),
    reproduce the separate runs bitwise; without the offsets the second
    document is contaminated."""
    with open(os.path.join(GOLDEN, "torchtitan_packing.json")) as fh:
        fx = json.load(fh)
    lens = fx["lengths"]
    x = tiny(lens, H=2, dk=4, dv=3, seed=13)
    assert list(x["cu_seqlens"]) == fx["cu_seqlens"]
    rng = np.random.RandomState(14)
    dO = rng.randn(*x["v"].shape)
    o, hf = oracle.forward(x)
    gp = oracle.backward(x, dO)
    for s, (t0, t1) in enumerate(zip(fx["cu_seqlens"][:-1], fx["cu_seqlens"][1:])):
        xs = {kk: (vv[t0:t1] if kk in ("q", "k", "v", "f", "b") else vv) for kk, vv in x.items()}
        xs["cu_seqlens"] = np.array([0, t1 - t0], np.int32)
        os_, hs = oracle.forward(xs)
        assert np.array_equal(os_, o[t0:t1]) and np.array_equal(hs[0], hf[s])
        gs = oracle.backward(xs, dO[t0:t1])
        for n in ("dq", "dk", "dv", "df", "db"):
            assert np.array_equal(gs[n], gp[n][t0:t1])
    xj = dict(x, cu_seqlens=np.array([0, sum(lens)], np.int32))
    oj, _ = oracle.forward(xj)
    assert np.array_equal(oj[:96], o[:96])
    assert not np.allclose(oj[96:], o[96:])


def test_zero_length_document_passes_state_through():
    x = tiny([3, 0, 2], H=2, dk=3, dv=2, seed=15, h0=True)
    rng = np.random.RandomState(16)
    dO = rng.randn(*x["v"].shape)
    dhf = rng.randn(*x["h0"].shape)
    _, hf = oracle.forward(x)
    np.testing.assert_array_equal(hf[1], x["h0"][1])
    g = oracle.backward(x, dO, dhf)
    np.testing.assert_array_equal(g["dh0"][1], dhf[1])


def test_f32_oracle_tracks_f64():
    x = tiny([40, 25], H=2, dk=8, dv=6, seed=17, h0=True)
    o64, h64 = oracle.forward(x, precision="f64")
    o32, h32 = oracle.forward(x, precision="f32")
    assert np.abs(o32 - o64).max() / np.sqrt((o64 ** 2).mean()) < 1e-5
    assert np.linalg.norm(h32 - h64) / np.linalg.norm(h64) < 1e-5
