"""Pins for the fp64 oracle: each test ties it to something other than itself.

- hand-worked tiny cases (tests/golden/*.txt): scalar recurrence, state orientation,
  grouped heads, scalar gradient;
- closed form for beta = 0 (pure decay);
- the delta-rule projection for g = 0, beta = 1, unit k;
- the chunk (WY/UT) form against the token recurrence, at several chunk sizes;
- grouped heads against explicitly repeated heads;
- joint linearity in (v, state_in);
- central finite differences for the backward;
- zero-length sequences.
The operator is the gated delta rule named in the IsoExec page's section
"Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet".
"""
import os

import numpy as np
import pytest

import oracle
from gated_deltanet_cpr_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(":")
            vals[key.strip()] = np.array([float(x) for x in rest.split()], dtype=np.float64)
    return vals


def rnd_inputs(rng, lengths, hqk, hv, dk, dv, unit=True, g_scale=1.0):
    T = int(sum(lengths))
    q = rng.standard_normal((T, hqk, dk))
    k = rng.standard_normal((T, hqk, dk))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, hv, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, hv))))
    g = -np.log1p(np.exp(rng.standard_normal((T, hv)))) * g_scale
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return q, k, v, g, beta, cu


# ---------------------------------------------------------------- golden cases ----

def test_golden_scalar_three_tokens():
    G = read_golden("scalar_three_tokens.txt")
    T = len(G["a"])
    sh = lambda x: x.reshape(T, 1, 1)
    o, st, _ = oracle.fwd(sh(G["q"]), sh(G["k"]), sh(G["v"]), np.log(G["a"]).reshape(T, 1),
                          G["beta"].reshape(T, 1), [0, T], G["state_in"].reshape(1, 1, 1, 1))
    np.testing.assert_allclose(o.ravel(), G["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(st.ravel(), G["state_out"], rtol=0, atol=1e-14)


def test_golden_orientation():
    G = read_golden("orientation_dk2_dv3.txt")
    dk, dv = int(G["dk"][0]), int(G["dv"][0])
    T = len(G["a"])
    o, st, _ = oracle.fwd(G["q"].reshape(T, 1, dk), G["k"].reshape(T, 1, dk),
                          G["v"].reshape(T, 1, dv), np.log(G["a"]).reshape(T, 1),
                          G["beta"].reshape(T, 1), [0, T], G["state_in"].reshape(1, 1, dv, dk))
    np.testing.assert_allclose(o.ravel(), G["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(st.ravel(), G["state_out"], rtol=0, atol=1e-14)


def test_golden_grouped_heads():
    G = read_golden("grouped_heads.txt")
    dk, dv, hqk, hv = (int(G[x][0]) for x in ("dk", "dv", "hqk", "hv"))
    o, st, _ = oracle.fwd(G["q"].reshape(1, hqk, dk), G["k"].reshape(1, hqk, dk),
                          G["v"].reshape(1, hv, dv), np.log(G["a"]).reshape(1, hv),
                          G["beta"].reshape(1, hv), [0, 1])
    np.testing.assert_allclose(o.ravel(), G["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(st.ravel(), G["state_out"], rtol=0, atol=1e-14)


def test_golden_scalar_backward():
    G = read_golden("scalar_backward.txt")
    sh3 = lambda x: x.reshape(1, 1, 1)
    sh2 = lambda x: x.reshape(1, 1)
    args = (sh3(G["q"]), sh3(G["k"]), sh3(G["v"]), sh2(G["g"]), sh2(G["beta"]), [0, 1])
    s0 = G["s0"].reshape(1, 1, 1, 1)
    o, st, _ = oracle.fwd(*args, state_in=s0)
    assert o.ravel()[0] == pytest.approx(G["o"][0], abs=1e-14)
    assert st.ravel()[0] == pytest.approx(G["state_out"][0], abs=1e-14)
    gr = oracle.bwd(*args, dout=np.ones((1, 1, 1)), state_in=s0)
    for key in ("dq", "dk", "dv", "dg", "dbeta", "dstate_in"):
        assert gr[key].ravel()[0] == pytest.approx(G[key][0], abs=1e-13), key


# ---------------------------------------------------------------- closed forms ----

def test_beta_zero_is_pure_decay():
    """beta = 0: S_t = exp(G_t) S_0 with G_t = g_1 + ... + g_t, and o_t = S_t q_t."""
    rng = np.random.default_rng(1)
    lengths = [7, 1, 12]
    q, k, v, g, beta, cu = rnd_inputs(rng, lengths, 2, 4, 5, 3)
    beta[:] = 0.0
    s0 = rng.standard_normal((3, 4, 3, 5))
    o, st, _ = oracle.fwd(q, k, v, g, beta, cu, state_in=s0)
    for s in range(3):
        G = np.cumsum(g[cu[s]:cu[s + 1]], axis=0)  # [L, Hv]
        for h in range(4):
            hq = h // 2
            for t in range(cu[s], cu[s + 1]):
                dec = np.exp(G[t - cu[s], h])
                np.testing.assert_allclose(o[t, h], dec * s0[s, h] @ q[t, hq], rtol=1e-12, atol=1e-14)
            final = np.exp(G[-1, h]) * s0[s, h]
            np.testing.assert_allclose(st[s, h], final, rtol=1e-12, atol=1e-14)


def test_unit_key_write_projects_out_k():
    """g = 0, beta = 1, |k| = 1: after token t, S_t k_t = v_t exactly and S_t x = S_{t-1} x
    for every x orthogonal to k_t (the delta rule replaces the value stored at key k_t)."""
    rng = np.random.default_rng(2)
    T, dk, dv = 9, 6, 4
    q, k, v, g, beta, cu = rnd_inputs(rng, [T], 1, 1, dk, dv)
    g[:] = 0.0
    beta[:] = 1.0
    s0 = rng.standard_normal((1, 1, dv, dk))
    _, st, bnd = oracle.fwd(q, k, v, g, beta, cu, state_in=s0, chunk=1)
    states = list(bnd[:, 0]) + [st[0, 0]]  # states[t] = state before token t
    for t in range(T):
        kt = k[t, 0]
        S_prev, S_t = states[t], states[t + 1]
        np.testing.assert_allclose(S_t @ kt, v[t, 0], rtol=0, atol=1e-12)
        x = rng.standard_normal(dk)
        x -= (x @ kt) * kt
        np.testing.assert_allclose(S_t @ x, S_prev @ x, rtol=0, atol=1e-12)


def test_single_token_closed_form():
    """T = 1: S_1 = e^g S_0 (I - beta k k^T) + beta v k^T (matrix form), o = S_1 q."""
    rng = np.random.default_rng(3)
    dk, dv = 5, 3
    q, k, v, g, beta, cu = rnd_inputs(rng, [1], 1, 1, dk, dv, unit=False)
    s0 = rng.standard_normal((1, 1, dv, dk))
    o, st, _ = oracle.fwd(q, k, v, g, beta, cu, state_in=s0)
    kk = k[0, 0]
    S1 = np.exp(g[0, 0]) * s0[0, 0] @ (np.eye(dk) - beta[0, 0] * np.outer(kk, kk)) \
        + beta[0, 0] * np.outer(v[0, 0], kk)
    np.testing.assert_allclose(st[0, 0], S1, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(o[0, 0], S1 @ q[0, 0], rtol=1e-13, atol=1e-14)


# ------------------------------------------------------------- chunk form pins ----

@pytest.mark.parametrize("chunk", [1, 3, 16, 64])
def test_chunk_form_equals_token_recurrence(chunk):
    """The WY/UT chunk form (what the CPR boundary pass evaluates) reproduces the token
    recurrence's state at every chunk boundary and at the end of every sequence."""
    rng = np.random.default_rng(10 + chunk)
    lengths = [0, 1, 17, 64, 130, 5]
    q, k, v, g, beta, cu = rnd_inputs(rng, lengths, 2, 4, 8, 6, g_scale=0.2)
    s0 = rng.standard_normal((len(lengths), 4, 6, 8))
    _, st_r, bnd_r = oracle.fwd(q, k, v, g, beta, cu, state_in=s0, chunk=chunk)
    bnd_c, st_c = oracle.chunk_states(k, v, g, beta, cu, chunk, state_in=s0)
    np.testing.assert_allclose(bnd_c, bnd_r, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(st_c, st_r, rtol=1e-10, atol=1e-11)


def test_chunk_count():
    assert oracle.num_chunks([0, 0, 1, 65, 129], 64) == 0 + 1 + 1 + 1
    assert oracle.num_chunks([0, 128, 128], 64) == 2


# ------------------------------------------------------------------ invariants ----

def test_grouped_heads_equal_repeated_heads():
    rng = np.random.default_rng(4)
    lengths = [11, 6]
    q, k, v, g, beta, cu = rnd_inputs(rng, lengths, 2, 6, 4, 4)
    o, st, _ = oracle.fwd(q, k, v, g, beta, cu)
    rep = np.repeat(np.arange(2), 3)  # value head h -> key head h // 3
    o2, st2, _ = oracle.fwd(q[:, rep], k[:, rep], v, g, beta, cu)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(st, st2)


def test_linear_in_values_and_state():
    """For fixed q, k, g, beta the map (v, S_0) -> (o, S_T) is linear."""
    rng = np.random.default_rng(5)
    lengths = [13, 4]
    q, k, v1, g, beta, cu = rnd_inputs(rng, lengths, 1, 2, 5, 3)
    v2 = rng.standard_normal(v1.shape)
    s1 = rng.standard_normal((2, 2, 3, 5))
    s2 = rng.standard_normal((2, 2, 3, 5))
    alpha = -1.7
    oa, sa, _ = oracle.fwd(q, k, v1, g, beta, cu, state_in=s1)
    ob, sb, _ = oracle.fwd(q, k, v2, g, beta, cu, state_in=s2)
    oc, sc, _ = oracle.fwd(q, k, alpha * v1 + v2, g, beta, cu, state_in=alpha * s1 + s2)
    np.testing.assert_allclose(oc, alpha * oa + ob, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sc, alpha * sa + sb, rtol=1e-12, atol=1e-12)


def test_zero_length_sequences_pass_state_through():
    rng = np.random.default_rng(6)
    lengths = [0, 3, 0]
    q, k, v, g, beta, cu = rnd_inputs(rng, lengths, 1, 1, 4, 4)
    s0 = rng.standard_normal((3, 1, 4, 4))
    o, st, _ = oracle.fwd(q, k, v, g, beta, cu, state_in=s0)
    np.testing.assert_array_equal(st[0], s0[0])
    np.testing.assert_array_equal(st[2], s0[2])
    assert o.shape == (3, 1, 4)


def test_synthetic_generator_shapes_and_rounding():
    x = synth.make_inputs([5, 3], 2, 4, 8, dtype=synth.BF16, seed=0, state_in=True, dout=True)
    assert x["q"].shape == (8, 2, 8) and x["v"].shape == (8, 4, 8)
    assert x["cu_seqlens"].tolist() == [0, 5, 8]
    assert float(x["g"].max()) < 0 and 0 < float(x["beta"].min()) and float(x["beta"].max()) < 1
    # seeded: same seed, same bits
    y = synth.make_inputs([5, 3], 2, 4, 8, dtype=synth.BF16, seed=0, state_in=True, dout=True)
    assert all(bool((x[n] == y[n]).all()) for n in ("q", "k", "v", "g", "beta", "state_in"))


# ---------------------------------------------------------- backward vs FD -------

def _loss(params, cu, dout, dstate_out):
    q, k, v, g, beta, s0 = params
    o, st, _ = oracle.fwd(q, k, v, g, beta, cu, state_in=s0, n_threads=1)
    return float((o * dout).sum() + (st * dstate_out).sum())


@pytest.mark.parametrize("lengths,hqk,hv,dk,dv", [([5, 3], 1, 2, 3, 2), ([4], 2, 2, 2, 3)])
def test_backward_matches_central_differences(lengths, hqk, hv, dk, dv):
    rng = np.random.default_rng(7)
    q, k, v, g, beta, cu = rnd_inputs(rng, lengths, hqk, hv, dk, dv, unit=False)
    s0 = rng.standard_normal((len(lengths), hv, dv, dk))
    dout = rng.standard_normal(v.shape)
    dso = rng.standard_normal(s0.shape)
    gr = oracle.bwd(q, k, v, g, beta, cu, dout, state_in=s0, dstate_out=dso, n_threads=1)
    params = [q, k, v, g, beta, s0]
    names = ["dq", "dk", "dv", "dg", "dbeta", "dstate_in"]
    h = 1e-6
    for p, name in zip(params, names):
        fd = np.zeros_like(p)
        flat = p.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + h
            lp = _loss(params, cu, dout, dso)
            flat[i] = old - h
            lm = _loss(params, cu, dout, dso)
            flat[i] = old
            fd.reshape(-1)[i] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(gr[name], fd, rtol=1e-6, atol=1e-7, err_msg=name)


def test_backward_across_checkpoint_segments():
    """A sequence longer than the oracle's 64-token checkpoint spacing, checked by central
    differences on a seeded sample of coordinates of every input."""
    rng = np.random.default_rng(8)
    lengths = [150]
    q, k, v, g, beta, cu = rnd_inputs(rng, lengths, 1, 1, 2, 2, g_scale=0.05)
    s0 = rng.standard_normal((1, 1, 2, 2))
    dout = rng.standard_normal(v.shape)
    dso = rng.standard_normal(s0.shape)
    gr = oracle.bwd(q, k, v, g, beta, cu, dout, state_in=s0, dstate_out=dso, n_threads=1)
    params = [q, k, v, g, beta, s0]
    names = ["dq", "dk", "dv", "dg", "dbeta", "dstate_in"]
    h = 1e-6
    for p, name in zip(params, names):
        flat = p.reshape(-1)
        idx = rng.choice(flat.size, size=min(12, flat.size), replace=False)
        for i in idx:
            old = flat[i]
            flat[i] = old + h
            lp = _loss(params, cu, dout, dso)
            flat[i] = old - h
            lm = _loss(params, cu, dout, dso)
            flat[i] = old
            fd = (lp - lm) / (2 * h)
            assert gr[name].reshape(-1)[i] == pytest.approx(fd, rel=1e-5, abs=1e-6), (name, i)
