"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test names what it pins.  Sources: the recurrence and gate of the model card
"Qwen3.5 Gated Delta Net NKI Kernel for AWS Neuron" ("How It Works", "Correctness Contract"),
the direct-solve chunked form of PR #164 "Fused DeltaNet Direct-Solve Follow-Up", and plain
mathematics (closed forms, invariants, library routines, exact rational brute force).
"""
import math

import numpy as np
import pytest
import scipy.special as sps

import oracle


def _unit_rows(rng, n, d):
    x = rng.standard_normal((n, d))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


def _rand_case(rng, T, dk, dv, g_scale=1.0):
    q = _unit_rows(rng, T, dk)
    k = _unit_rows(rng, T, dk)
    v = rng.standard_normal((T, dv))
    g = -g_scale * rng.uniform(0.0, 3.0, T)
    beta = sps.expit(rng.standard_normal(T))
    S0 = 0.3 * rng.standard_normal((dv, dk))
    return q, k, v, g, beta, S0


# ------------------------------------------------------------------ elementwise prologue

def test_sigmoid_softplus_match_scipy():
    """P12: sigmoid == scipy.special.expit; softplus(x) == -log_expit(-x) (library routines)."""
    for x in np.linspace(-40, 40, 161):
        assert oracle.sigmoid(x) == pytest.approx(sps.expit(x), rel=1e-15, abs=1e-300)
        assert oracle.softplus(x) == pytest.approx(-sps.log_expit(-x), rel=1e-14, abs=1e-300)
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-16)
    # softplus(x) - softplus(-x) = x
    for x in (-3.0, -0.5, 0.25, 7.0):
        assert oracle.softplus(x) - oracle.softplus(-x) == pytest.approx(x, rel=1e-14)


def test_gate_is_never_positive_and_matches_contract():
    """The gate of the model card's correctness contract: g = -exp(A_log) softplus(a+dt_bias),
    so exp(g) lies in (0, 1].  Closed values: A_log=0, a=0 -> -ln 2; A_log=ln 16 -> 16x."""
    assert oracle.gate(0.0, 0.0) == pytest.approx(-math.log(2.0), rel=1e-15)
    assert oracle.gate(0.0, math.log(16.0)) == pytest.approx(-16 * math.log(2.0), rel=1e-14)
    assert oracle.gate(1.0, 0.0, -1.0) == pytest.approx(-math.log(2.0), rel=1e-15)
    rng = np.random.default_rng(0)
    for a in rng.standard_normal(200) * 5:
        g = oracle.gate(a, rng.uniform(0, math.log(16)))
        assert g <= 0.0 and 0.0 < math.exp(g) <= 1.0


def test_l2norm_against_numpy_linalg():
    """P12: l2norm output has unit norm (eps=0) and the direction of the input (numpy.linalg)."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal(128)
    y = oracle.l2norm(x, eps=0.0)
    assert np.linalg.norm(y) == pytest.approx(1.0, rel=1e-15)
    np.testing.assert_allclose(y * np.linalg.norm(x), x, rtol=1e-14)
    y2 = oracle.l2norm(x, eps=1e-6, scale=0.5)
    np.testing.assert_allclose(y2, 0.5 * x / math.sqrt(x @ x + 1e-6), rtol=1e-15)


# ------------------------------------------------------------------ recurrence

def test_worked_example_exact_rationals():
    """Brute force in exact rational arithmetic (sympy) of the matrix form
    S_t = e^{g_t} S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T, o_t = S_t q_t,
    on a 2x3 (dv x dk) non-square, non-symmetric case with e^{g} in {1/2, 1, 1/4}: a
    transposed state, a swapped read/decay order or a dropped term all change the result."""
    sp = pytest.importorskip("sympy")
    R = sp.Rational
    dv, dk = 2, 3
    S = sp.Matrix([[R(1, 3), R(-1, 2), R(2)], [R(0), R(1, 5), R(-1)]])
    ks = [sp.Matrix([R(1), R(2), R(-1)]), sp.Matrix([R(0), R(1, 2), R(3)]),
          sp.Matrix([R(-2), R(1), R(1, 3)])]
    qs = [sp.Matrix([R(1, 2), R(0), R(1)]), sp.Matrix([R(-1), R(1), R(2)]),
          sp.Matrix([R(3), R(-1, 3), R(0)])]
    vs = [sp.Matrix([R(1), R(-1)]), sp.Matrix([R(2), R(1, 2)]), sp.Matrix([R(-1, 4), R(3)])]
    decays = [R(1, 2), R(1), R(1, 4)]
    betas = [R(1, 2), R(3, 4), R(1, 3)]
    S0 = np.array(S.tolist(), dtype=float)
    outs = []
    for t in range(3):
        S = decays[t] * S * (sp.eye(dk) - betas[t] * ks[t] * ks[t].T) + betas[t] * vs[t] * ks[t].T
        outs.append(S * qs[t])
    o_ref = np.array([[float(e) for e in o] for o in outs])
    S_ref = np.array(S.tolist(), dtype=float)
    q = np.array([[float(e) for e in x] for x in qs])
    k = np.array([[float(e) for e in x] for x in ks])
    v = np.array([[float(e) for e in x] for x in vs])
    g = np.log(np.array([float(d) for d in decays]))
    beta = np.array([float(b) for b in betas])
    o, S_T = oracle.recurrence(q, k, v, g, beta, S0)
    np.testing.assert_allclose(o, o_ref, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(S_T, S_ref, rtol=1e-14, atol=1e-14)
    o2, S2 = oracle.chunked(q, k, v, g, beta, S0, chunk=2)
    np.testing.assert_allclose(o2, o_ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(S2, S_ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("T", [1, 2, 3, 15, 16, 17, 63, 64, 65, 129, 200])
@pytest.mark.parametrize("C", [4, 8, 16, 64])
def test_chunked_equals_sequential(T, C):
    """P1: the chunked WY/UT form (direct solve) equals the token-by-token recurrence in fp64,
    including a last chunk shorter than C."""
    rng = np.random.default_rng(100 * T + C)
    q, k, v, g, beta, S0 = _rand_case(rng, T, 16, 12)
    o1, S1 = oracle.recurrence(q, k, v, g, beta, S0)
    o2, S2 = oracle.chunked(q, k, v, g, beta, S0, chunk=C)
    scale = max(1.0, np.abs(o1).max())
    assert np.abs(o1 - o2).max() / scale < 1e-10
    assert np.abs(S1 - S2).max() / max(1.0, np.abs(S1).max()) < 1e-10


def test_chunked_equals_sequential_full_head():
    """P1 at the real head size d = 128 and chunk 64, T = 129 (ragged)."""
    rng = np.random.default_rng(7)
    q, k, v, g, beta, S0 = _rand_case(rng, 129, 128, 128)
    o1, S1 = oracle.recurrence(q, k, v, g, beta, S0)
    o2, S2 = oracle.chunked(q, k, v, g, beta, S0, chunk=64)
    assert np.abs(o1 - o2).max() / np.abs(o1).max() < 1e-10
    assert np.abs(S1 - S2).max() / np.abs(S1).max() < 1e-10


@pytest.mark.parametrize("g", [0.0, -0.7, -5.0])
def test_single_write_stores_value(g):
    """P2: beta = 1 and ||k|| = 1 => after the write S_t k_t = v_t exactly, for any decay and
    any earlier state (e^g S (k - k (k.k)) + v (k.k) = v)."""
    rng = np.random.default_rng(3)
    dk, dv = 16, 10
    S0 = rng.standard_normal((dv, dk))
    k = _unit_rows(rng, 1, dk)
    q = _unit_rows(rng, 1, dk)
    v = rng.standard_normal((1, dv))
    _, S1 = oracle.recurrence(q, k, v, np.array([g]), np.array([1.0]), S0)
    np.testing.assert_allclose(S1 @ k[0], v[0], rtol=1e-13, atol=1e-13)


def test_orthonormal_keys_form_exact_memory():
    """P3: g = 0, beta = 1, orthonormal k_1..k_n => S_n k_j = v_j for every j (S0 = 0)."""
    rng = np.random.default_rng(4)
    dk, dv, n = 32, 8, 20
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm[:, :n].T.copy()
    v = rng.standard_normal((n, dv))
    q = _unit_rows(rng, n, dk)
    _, S = oracle.recurrence(q, k, v, np.zeros(n), np.ones(n), np.zeros((dv, dk)))
    np.testing.assert_allclose(k @ S.T, v, rtol=1e-12, atol=1e-12)
    _, S2 = oracle.chunked(q, k, v, np.zeros(n), np.ones(n), np.zeros((dv, dk)), chunk=8)
    np.testing.assert_allclose(k @ S2.T, v, rtol=1e-12, atol=1e-12)


def test_beta_zero_only_decays():
    """P4: beta = 0 => S_T = e^{sum g} S0 and o_t = e^{G_t} S0 q_t (G_t = cumulative g)."""
    rng = np.random.default_rng(5)
    T, dk, dv = 37, 16, 12
    q, k, v, g, _, S0 = _rand_case(rng, T, dk, dv)
    beta = np.zeros(T)
    for fn in (oracle.recurrence, lambda *a: oracle.chunked(*a, chunk=16)):
        o, S = fn(q, k, v, g, beta, S0)
        G = np.cumsum(g)
        np.testing.assert_allclose(S, np.exp(G[-1]) * S0, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(o, np.exp(G)[:, None] * (q @ S0.T), rtol=1e-12, atol=1e-15)


def test_erase_off_is_gated_linear_attention():
    """P5: with the erase term off, the chunked form (T = I) and the sequential one both equal
    the direct gated-linear-attention sum
    o_t = e^{G_t} S0 q_t + sum_{s<=t} e^{G_t - G_s} beta_s (k_s . q_t) v_s."""
    rng = np.random.default_rng(6)
    T, dk, dv = 45, 16, 12
    q, k, v, g, beta, S0 = _rand_case(rng, T, dk, dv)
    G = np.cumsum(g)
    o_ref = np.zeros((T, dv))
    for t in range(T):
        o_ref[t] = np.exp(G[t]) * (S0 @ q[t])
        for s in range(t + 1):
            o_ref[t] += np.exp(G[t] - G[s]) * beta[s] * (k[s] @ q[t]) * v[s]
    S_ref = np.exp(G[-1]) * S0 + sum(np.exp(G[-1] - G[s]) * beta[s] * np.outer(v[s], k[s])
                                     for s in range(T))
    o1, S1 = oracle.recurrence(q, k, v, g, beta, S0, erase=False)
    o2, S2 = oracle.chunked(q, k, v, g, beta, S0, chunk=16, erase=False)
    for o, S in ((o1, S1), (o2, S2)):
        np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(S, S_ref, rtol=1e-11, atol=1e-12)


def test_first_token_output_order():
    """P6: T = 1, S0 = 0 => o = beta (k . q) v: the output is read after the write."""
    rng = np.random.default_rng(8)
    dk, dv = 16, 9
    q, k = _unit_rows(rng, 1, dk), _unit_rows(rng, 1, dk)
    v = rng.standard_normal((1, dv))
    beta = np.array([0.37])
    o, _ = oracle.recurrence(q, k, v, np.array([-0.4]), beta, np.zeros((dv, dk)))
    np.testing.assert_allclose(o[0], beta[0] * (k[0] @ q[0]) * v[0], rtol=1e-14)


def test_value_row_permutation():
    """P11: rows of S are independent: permuting the d_v index of v and S0 permutes o and S."""
    rng = np.random.default_rng(9)
    T, dk, dv = 21, 16, 12
    q, k, v, g, beta, S0 = _rand_case(rng, T, dk, dv)
    perm = rng.permutation(dv)
    o, S = oracle.recurrence(q, k, v, g, beta, S0)
    op, Sp = oracle.recurrence(q, k, v[:, perm], g, beta, S0[perm])
    np.testing.assert_allclose(op, o[:, perm], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(Sp, S[perm], rtol=1e-14, atol=1e-15)


def test_strong_decay_is_stable():
    """P13: per-token log-decay down to -50 (cumulative far below fp32 range): finite, and
    chunked == sequential.  The direct solve never forms exp of a positive number."""
    rng = np.random.default_rng(10)
    T, dk, dv = 200, 16, 8
    q, k, v, _, beta, S0 = _rand_case(rng, T, dk, dv)
    g = -rng.uniform(0.0, 50.0, T)
    o1, S1 = oracle.recurrence(q, k, v, g, beta, S0)
    o2, S2 = oracle.chunked(q, k, v, g, beta, S0, chunk=64)
    assert np.isfinite(o2).all() and np.isfinite(S2).all()
    assert np.abs(o1 - o2).max() / np.abs(o1).max() < 1e-10
    assert np.abs(S1 - S2).max() / np.abs(S1).max() < 1e-10


# ------------------------------------------------------------------ direct solve

@pytest.mark.parametrize("n", [1, 4, 16, 64])
def test_unit_lower_inverse_matches_numpy(n):
    """P8: the forward-substitution inverse of I + A (A strictly lower) matches
    numpy.linalg.inv and satisfies (I + A) T = I."""
    rng = np.random.default_rng(n)
    A = np.tril(rng.standard_normal((n, n)) * 0.3, -1)
    T = oracle.unit_lower_inverse(A)
    M = np.eye(n) + A
    np.testing.assert_allclose(T, np.linalg.inv(M), rtol=1e-10, atol=1e-12)
    assert np.abs(M @ T - np.eye(n)).max() < 1e-12
    assert np.allclose(np.triu(T, 1), 0.0)


# ------------------------------------------------------------------ conv

def test_conv_matches_numpy_convolve():
    """P9: the depthwise causal conv equals numpy.convolve per channel (taps reversed: the
    last tap multiplies the current token), with the state as left context."""
    rng = np.random.default_rng(11)
    B, T, C, W = 2, 9, 5, 4
    x = rng.standard_normal((B, T, C))
    w = rng.standard_normal((C, W))
    st = rng.standard_normal((B, W - 1, C))
    y, st_out = oracle.conv1d(x, w, state=st)
    for b in range(B):
        for c in range(C):
            full = np.concatenate([st[b, :, c], x[b, :, c]])
            ref = np.convolve(full, w[c, ::-1], mode="valid")
            np.testing.assert_allclose(y[b, :, c], ref, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(st_out[b], x[b, -(W - 1):], rtol=0, atol=0)
    ys, _ = oracle.conv1d(x, w, state=st, silu=True)
    np.testing.assert_allclose(ys, y * sps.expit(y), rtol=1e-14)


@pytest.mark.parametrize("T1", [1, 2, 3, 7])
def test_conv_split_equals_whole(T1):
    """P9: conv over [x1; x2] == conv(x1), then conv(x2 | state after x1), including a first
    piece shorter than W - 1 (the state then mixes old state and new inputs)."""
    rng = np.random.default_rng(12 + T1)
    B, T, C, W = 1, 10, 6, 4
    x = rng.standard_normal((B, T, C))
    w = rng.standard_normal((C, W))
    st = rng.standard_normal((B, W - 1, C))
    y, s_end = oracle.conv1d(x, w, state=st)
    y1, s1 = oracle.conv1d(x[:, :T1], w, state=st)
    y2, s2 = oracle.conv1d(x[:, T1:], w, state=s1)
    np.testing.assert_array_equal(np.concatenate([y1, y2], 1), y)
    np.testing.assert_array_equal(s2, s_end)


# ------------------------------------------------------------------ the whole layer

def _layer_case(seed, B, T, Hk, Hv, d, W):
    rng = np.random.default_rng(seed)
    C = (2 * Hk + Hv) * d
    kw = dict(num_k_heads=Hk, num_v_heads=Hv, head_dim=d,
              a=rng.standard_normal((B, T, Hv)), b=rng.standard_normal((B, T, Hv)),
              A_log=rng.uniform(0, math.log(16), Hv), dt_bias=0.1 * rng.standard_normal(Hv),
              state=0.02 * rng.standard_normal((B, Hv, d, d)))
    if W:
        kw.update(x=rng.standard_normal((B, T, C)),
                  conv_weight=rng.standard_normal((C, W)) / 2,
                  conv_state=rng.standard_normal((B, W - 1, C)))
    else:
        kw.update(q=rng.standard_normal((B, T, Hk, d)), k=rng.standard_normal((B, T, Hk, d)),
                  v=rng.standard_normal((B, T, Hv, d)))
    return kw


def _manual_layer(kw, scale=1.0, eps=1e-6):
    """Composition of the separately pinned pieces: conv -> split q|k|v -> l2norm -> gates ->
    recurrence, value head h reading key head h // (Hv/Hk)."""
    Hk, Hv, d = kw["num_k_heads"], kw["num_v_heads"], kw["head_dim"]
    a, b = kw["a"], kw["b"]
    B, T, _ = a.shape
    if "x" in kw:
        y, cs = oracle.conv1d(kw["x"], kw["conv_weight"], state=kw["conv_state"], silu=True)
        q = y[:, :, : Hk * d].reshape(B, T, Hk, d)
        k = y[:, :, Hk * d: 2 * Hk * d].reshape(B, T, Hk, d)
        v = y[:, :, 2 * Hk * d:].reshape(B, T, Hv, d)
    else:
        q, k, v, cs = kw["q"], kw["k"], kw["v"], None
    out = np.zeros((B, T, Hv, d))
    S = kw["state"].copy()
    r = Hv // Hk
    for bi in range(B):
        for h in range(Hv):
            kh = h // r
            qn = np.stack([oracle.l2norm(q[bi, t, kh], eps, scale) for t in range(T)])
            kn = np.stack([oracle.l2norm(k[bi, t, kh], eps) for t in range(T)])
            g = np.array([oracle.gate(a[bi, t, h], kw["A_log"][h], kw["dt_bias"][h])
                          for t in range(T)])
            beta = sps.expit(b[bi, :, h])
            o, S[bi, h] = oracle.recurrence(qn, kn, v[bi, :, h], g, beta, S[bi, h])
            out[bi, :, h] = o
    return out, S, cs


@pytest.mark.parametrize("W", [0, 4])
def test_layer_equals_composition_with_gqa(W):
    """The layer entry point (per-token conv, norm, gates, recurrence, threads over units)
    equals the composition of the separately pinned pieces; Hv/Hk = 3 exercises the GQA
    head map, W = 4 the q|k|v channel split and the conv state."""
    kw = _layer_case(20 + W, 2, 11, 2, 6, 8, W)
    res = oracle.layer(**kw, scale=0.5, nthreads=3)
    out, S, cs = _manual_layer(kw, scale=0.5)
    np.testing.assert_allclose(res.out, out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(res.state, S, rtol=1e-12, atol=1e-13)
    if W:
        np.testing.assert_array_equal(res.conv_state, cs)


@pytest.mark.parametrize("split", [1, 2, 5, 8])
def test_checkpoint_resume_equals_uninterrupted(split):
    """P7: run a prefix, keep (recurrent state, conv state), continue on the rest == one
    uninterrupted run, exactly (hybrid prefix-reuse semantics)."""
    kw = _layer_case(30, 1, 13, 1, 2, 8, 4)
    full = oracle.layer(**kw)
    first = {**kw, "a": kw["a"][:, :split], "b": kw["b"][:, :split], "x": kw["x"][:, :split]}
    r1 = oracle.layer(**first)
    second = {**kw, "a": kw["a"][:, split:], "b": kw["b"][:, split:], "x": kw["x"][:, split:],
              "state": r1.state, "conv_state": r1.conv_state}
    r2 = oracle.layer(**second)
    np.testing.assert_array_equal(np.concatenate([r1.out, r2.out], 1), full.out)
    np.testing.assert_array_equal(r2.state, full.state)
    np.testing.assert_array_equal(r2.conv_state, full.conv_state)


def test_prefill_equals_repeated_decode():
    """P10: a T-token layer call == T single-token calls carrying both states (exact)."""
    kw = _layer_case(40, 2, 6, 2, 4, 8, 4)
    full = oracle.layer(**kw)
    S, cs = kw["state"], kw["conv_state"]
    outs = []
    for t in range(6):
        step = {**kw, "a": kw["a"][:, t:t + 1], "b": kw["b"][:, t:t + 1],
                "x": kw["x"][:, t:t + 1], "state": S, "conv_state": cs}
        r = oracle.layer(**step)
        S, cs = r.state, r.conv_state
        outs.append(r.out)
    np.testing.assert_array_equal(np.concatenate(outs, 1), full.out)
    np.testing.assert_array_equal(S, full.state)


def test_layer_rejects_bad_geometry():
    kw = _layer_case(50, 1, 3, 2, 3, 8, 0)   # Hv % Hk != 0
    with pytest.raises(ValueError):
        oracle.layer(**kw)


# ------------------------------------------------------------------ gated output norm

def test_gated_rmsnorm_worked_example():
    """o = (3, 4), w = 1, z = ln 3 in both channels: mean square 12.5 and
    silu(ln 3) = ln 3 * sigmoid(ln 3) = (3/4) ln 3, so y = o / sqrt(12.5) * (3/4) ln 3."""
    y = oracle.gated_rmsnorm(np.array([[3.0, 4.0]]), np.full((1, 2), math.log(3.0)),
                             np.ones(2), eps=0.0)
    g = 0.75 * math.log(3.0)
    np.testing.assert_allclose(y[0], [3.0 / math.sqrt(12.5) * g, 4.0 / math.sqrt(12.5) * g],
                               rtol=1e-15)


def test_gated_rmsnorm_closed_forms():
    """A constant vector c has RMS |c|: y = sign(c) * w * silu(z).  z = 0 closes the gate
    (silu(0) = 0); a large z opens it to z itself; a very negative z closes it."""
    rng = np.random.default_rng(11)
    n = 128
    w = rng.uniform(0.5, 2.0, n)
    z = rng.standard_normal((2, n))
    o = np.stack([np.full(n, 0.37), np.full(n, -5.0)])
    y = oracle.gated_rmsnorm(o, z, w, eps=0.0)
    silu = z * sps.expit(z)
    np.testing.assert_allclose(y[0], w * silu[0], rtol=1e-14)
    np.testing.assert_allclose(y[1], -w * silu[1], rtol=1e-14)
    o = rng.standard_normal((3, n))
    assert np.all(oracle.gated_rmsnorm(o, np.zeros((3, n)), w, eps=0.0) == 0.0)
    big = oracle.gated_rmsnorm(o, np.full((3, n), 60.0), np.ones(n), eps=0.0)
    rms = np.sqrt(np.mean(o * o, axis=1, keepdims=True))
    np.testing.assert_allclose(big, o / rms * 60.0, rtol=1e-13)
    assert np.all(np.abs(oracle.gated_rmsnorm(o, np.full((3, n), -60.0), np.ones(n))) < 1e-20)


def test_gated_rmsnorm_invariants():
    """Without eps: invariant to positive scaling of o, odd in o, and the normalised vector
    y / (w silu(z)) has mean square exactly 1 (mean over n channels, not a sum).  With eps,
    o = 0 gives 0 (no division by zero) and a tiny o is damped, not blown up."""
    rng = np.random.default_rng(12)
    n = 128
    o = rng.standard_normal((5, n))
    z = rng.standard_normal((5, n))
    w = rng.uniform(0.5, 2.0, n)
    y = oracle.gated_rmsnorm(o, z, w, eps=0.0)
    np.testing.assert_allclose(oracle.gated_rmsnorm(7.5 * o, z, w, eps=0.0), y, rtol=1e-13)
    np.testing.assert_allclose(oracle.gated_rmsnorm(-o, z, w, eps=0.0), -y, rtol=1e-15)
    unit = y / (w * z * sps.expit(z))
    np.testing.assert_allclose(np.mean(unit * unit, axis=1), 1.0, rtol=1e-13)
    assert np.all(oracle.gated_rmsnorm(np.zeros((1, n)), z[:1], w, eps=1e-6) == 0.0)
    tiny = oracle.gated_rmsnorm(1e-6 * o, z, w, eps=1e-6)
    assert np.max(np.abs(tiny)) < np.max(np.abs(y)) * 2e-3
