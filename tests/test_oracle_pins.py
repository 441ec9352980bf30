"""Pins for the fp64 oracle against what the pages and mathematics fix.

Source of the definitions: gist.science technical summary of "Higher-order Linear
Attention", section 1 (prefix summaries S^K, C^QV, m^Q; cross summaries G, h;
masked output; ratio normalisation), section 4 (segment concatenation with cross
term S_B C_A; exclusive scan equals the serial recurrence), "Resultaten en claims"
(exactness, strict causality).

Every check here compares the oracle with something computed another way: a
brute-force sum over index triples, the dense masked-matrix form, integer
fixtures derived by hand, closed forms, or a structural property.
"""
import glob
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_inputs(rng, B, H, n, d, dv, positive=False):
    q = rng.standard_normal((B, H, n, d))
    k = rng.standard_normal((B, H, n, d))
    v = rng.standard_normal((B, H, n, dv))
    if positive:
        q, k = np.abs(q) + 0.1, np.abs(k) + 0.1
    return q, k, v


def brute_force(q, k, v, g=1.0, normalize=False, eps=0.0):
    """o_t = sum_{a<=b<=t} g^{(t-a)+(t-b)} (q_t.k_a)(k_a.q_b) v_b, straight triple loop."""
    n, dv = q.shape[0], v.shape[1]
    o = np.zeros((n, dv))
    for t in range(n):
        num = np.zeros(dv)
        den = 0.0
        for b in range(t + 1):
            for a in range(b + 1):
                w = (g ** ((t - a) + (t - b))) * (q[t] @ k[a]) * (k[a] @ q[b])
                num += w * v[b]
                den += w
        o[t] = num / (den + eps) if normalize else num
    return o


def brute_state(q, k, v, g=1.0):
    """The five summaries after the last token, each from its own definition."""
    n, d = q.shape
    dv = v.shape[1]
    T = n - 1
    S = sum(g ** (T - a) * np.outer(k[a], k[a]) for a in range(n))
    C = sum(g ** (T - b) * np.outer(q[b], v[b]) for b in range(n))
    m = sum(g ** (T - b) * q[b] for b in range(n))
    G = np.zeros((d, dv))
    h = np.zeros(d)
    for a in range(n):
        for b in range(a):  # strictly earlier query/value index: the "future" pairs
            w = g ** ((T - a) + (T - b)) * (k[a] @ q[b])
            G += w * np.outer(k[a], v[b])
            h += w * k[a]
    return S, C, m, G, h


def rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# --------------------------------------------------------------------------- T1
@pytest.mark.parametrize("decay", [False, True])
@pytest.mark.parametrize("normalize", [False, True])
@pytest.mark.parametrize("n,d,dv", [(1, 1, 1), (7, 3, 2), (19, 4, 3), (24, 2, 4)])
def test_brute_force_outputs(decay, normalize, n, d, dv):
    rng = np.random.default_rng(100 + n * 7 + d)
    B, H = 2, 2
    q, k, v = rand_inputs(rng, B, H, n, d, dv, positive=normalize)
    gamma = np.array([0.9, 0.6]) if decay else None
    eps = 1e-3 if normalize else 0.0
    o, st = oracle.forward(q, k, v, gamma=gamma, normalize=normalize, eps=eps)
    for b in range(B):
        for h in range(H):
            g = gamma[h] if decay else 1.0
            ref = brute_force(q[b, h], k[b, h], v[b, h], g, normalize, eps)
            assert rel(o[b, h], ref) < 1e-12
            S, C, m, G, hh = brute_state(q[b, h], k[b, h], v[b, h], g)
            u = b * H + h
            for got, want in zip((st.S[u], st.C[u], st.m[u], st.G[u], st.h[u]), (S, C, m, G, hh)):
                assert rel(got, want) < 1e-12


# --------------------------------------------------------------------------- T2
def test_dense_matrix_form():
    """No decay: O = [L o ((L o QK^T)(L o QK^T)^T)] V with L the lower-triangular ones."""
    rng = np.random.default_rng(7)
    n, d, dv = 40, 5, 3
    q, k, v = rand_inputs(rng, 1, 1, n, d, dv)
    L = np.tril(np.ones((n, n)))
    A = L * (q[0, 0] @ k[0, 0].T)
    ref = (L * (A @ A.T)) @ v[0, 0]
    o, _ = oracle.forward(q, k, v)
    assert rel(o[0, 0], ref) < 1e-12
    # normalised: the denominator is the row sum of the same masked weights
    qp, kp = np.abs(q) + 0.1, np.abs(k) + 0.1
    A = L * (qp[0, 0] @ kp[0, 0].T)
    W = L * (A @ A.T)
    ref = (W @ v[0, 0]) / (W.sum(axis=1, keepdims=True) + 1e-6)
    o, _ = oracle.forward(qp, kp, v, normalize=True, eps=1e-6)
    assert rel(o[0, 0], ref) < 1e-12


# ---------------------------------------------------------------------- golden
@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(GOLDEN, "*.json"))))
def test_hand_fixtures(path):
    fx = json.load(open(path))
    q = np.array(fx["q"], dtype=np.float64)[None, None]
    k = np.array(fx["k"], dtype=np.float64)[None, None]
    v = np.array(fx["v"], dtype=np.float64)[None, None]
    gamma = None if fx["gamma"] is None else np.array([fx["gamma"]])
    o, _ = oracle.forward(q, k, v, gamma=gamma, normalize=fx["normalize"], eps=fx["eps"])
    np.testing.assert_allclose(o[0, 0], np.array(fx["o"], dtype=np.float64), rtol=1e-14, atol=1e-14)


# ------------------------------------------------------------------ closed forms
def test_constant_inputs_closed_form():
    """Constant q,k,v: every triple contributes (q.k)^2 v and there are t(t+1)/2 pairs."""
    rng = np.random.default_rng(3)
    n, d, dv = 50, 6, 4
    q1, k1, v1 = rng.standard_normal(d), rng.standard_normal(d), rng.standard_normal(dv)
    q = np.broadcast_to(q1, (1, 1, n, d)).copy()
    k = np.broadcast_to(k1, (1, 1, n, d)).copy()
    v = np.broadcast_to(v1, (1, 1, n, dv)).copy()
    o, _ = oracle.forward(q, k, v)
    t = np.arange(1, n + 1)[:, None]
    ref = (q1 @ k1) ** 2 * t * (t + 1) / 2 * v1[None, :]
    assert rel(o[0, 0], ref) < 1e-13


def test_single_token():
    rng = np.random.default_rng(4)
    q, k, v = rand_inputs(rng, 3, 2, 1, 5, 3)
    o, _ = oracle.forward(q, k, v)
    ref = np.einsum("bhnd,bhnd->bhn", q, k)[..., None] ** 2 * v
    assert rel(o, ref) < 1e-14
    o, _ = oracle.forward(q, k, v, normalize=True, eps=0.5)
    s = np.einsum("bhnd,bhnd->bhn", q, k)[..., None] ** 2
    assert rel(o, s * v / (s + 0.5)) < 1e-14


def test_scalar_d1_cumulative_form():
    """d = 1: o_t = q_t * cumsum_b( cumsum_a(k_a^2)_b * q_b * v_b )_t."""
    rng = np.random.default_rng(5)
    n, dv = 64, 3
    q, k, v = rand_inputs(rng, 1, 1, n, 1, dv)
    K2 = np.cumsum(k[0, 0, :, 0] ** 2)
    inner = np.cumsum((K2 * q[0, 0, :, 0])[:, None] * v[0, 0], axis=0)
    ref = q[0, 0, :, 0][:, None] * inner
    o, _ = oracle.forward(q, k, v)
    assert rel(o[0, 0], ref) < 1e-12


def test_decay_zero_and_one():
    rng = np.random.default_rng(6)
    q, k, v = rand_inputs(rng, 1, 2, 30, 4, 3)
    # gamma = 1 is the undecayed operator
    o1, s1 = oracle.forward(q, k, v, gamma=np.array([1.0, 1.0]))
    o0, s0 = oracle.forward(q, k, v)
    assert rel(o1, o0) < 1e-14 and rel(s1.G, s0.G) < 1e-14
    # gamma = 0 keeps only a = b = t: o_t = (q_t.k_t)^2 v_t
    oz, _ = oracle.forward(q, k, v, gamma=np.array([0.0, 0.0]))
    ref = np.einsum("bhnd,bhnd->bhn", q, k)[..., None] ** 2 * v
    assert rel(oz, ref) < 1e-14


# --------------------------------------------------------------------------- T3
@pytest.mark.parametrize("decay", [False, True])
@pytest.mark.parametrize("normalize", [False, True])
def test_chunked_scan_equals_serial_every_chunk(decay, normalize):
    """Exactness claim: the chunk-parallel scan reproduces the serial activations,
    for every chunk size including ones that do not divide n."""
    rng = np.random.default_rng(11)
    B, H, n, d, dv = 1, 2, 23, 3, 2
    q, k, v = rand_inputs(rng, B, H, n, d, dv, positive=normalize)
    gamma = np.array([0.95, 0.7]) if decay else None
    # a non-zero incoming state, itself from a real prefix
    qp, kp, vp = rand_inputs(rng, B, H, 9, d, dv, positive=normalize)
    _, st0 = oracle.forward(qp, kp, vp, gamma=gamma)
    o_ser, s_ser = oracle.forward(q, k, v, gamma=gamma, normalize=normalize, eps=1e-3, state_in=st0)
    for c in range(1, n + 2):
        o_c, s_c = oracle.forward(q, k, v, gamma=gamma, normalize=normalize, eps=1e-3, state_in=st0, chunk=c)
        assert rel(o_c, o_ser) < 1e-12, c
        for a, b in zip(s_c.astuple(), s_ser.astuple()):
            assert rel(a, b) < 1e-12, c


# --------------------------------------------------------------------------- T4
def _rand_state(rng, units, d, dv):
    return oracle.State(rng.standard_normal((units, d, d)), rng.standard_normal((units, d, dv)),
                        rng.standard_normal((units, d)), rng.standard_normal((units, d, dv)),
                        rng.standard_normal((units, d)))


def test_combine_associative_identity_noncommutative():
    rng = np.random.default_rng(12)
    u, d, dv = 5, 4, 3
    A, Bs, Cs = (_rand_state(rng, u, d, dv) for _ in range(3))
    fB, fC = rng.uniform(0.2, 1.0, u), rng.uniform(0.2, 1.0, u)
    left = oracle.combine(oracle.combine(A, Bs, fB), Cs, fC)
    right = oracle.combine(A, oracle.combine(Bs, Cs, fC), fB * fC)
    for a, b in zip(left.astuple(), right.astuple()):
        assert rel(a, b) < 1e-13
    Z = oracle.State.zeros(u, d, dv)
    for a, b in zip(oracle.combine(A, Z).astuple(), A.astuple()):
        assert rel(a, b) < 1e-15
    for a, b in zip(oracle.combine(Z, A).astuple(), A.astuple()):
        assert rel(a, b) < 1e-15
    AB, BA = oracle.combine(A, Bs), oracle.combine(Bs, A)
    assert rel(AB.G, BA.G) > 1e-3


def test_combine_equals_concatenated_sequence():
    """State of seq_A ++ seq_B equals state(A) (+) state(B) with f = gamma^len(B)."""
    rng = np.random.default_rng(13)
    d, dv, na, nb = 4, 3, 11, 6
    gamma = np.array([0.8, 1.0])
    qa, ka, va = rand_inputs(rng, 1, 2, na, d, dv)
    qb, kb, vb = rand_inputs(rng, 1, 2, nb, d, dv)
    _, sa = oracle.forward(qa, ka, va, gamma=gamma)
    _, sb = oracle.forward(qb, kb, vb, gamma=gamma)
    _, sab = oracle.forward(np.concatenate([qa, qb], 2), np.concatenate([ka, kb], 2),
                            np.concatenate([va, vb], 2), gamma=gamma)
    comb = oracle.combine(sa, sb, gamma ** nb)
    for a, b in zip(comb.astuple(), sab.astuple()):
        assert rel(a, b) < 1e-12


# --------------------------------------------------------------------------- T5
@pytest.mark.parametrize("normalize", [False, True])
def test_strict_causality(normalize):
    rng = np.random.default_rng(14)
    n, d, dv = 30, 4, 3
    q, k, v = rand_inputs(rng, 1, 2, n, d, dv, positive=normalize)
    gamma = np.array([0.9, 1.0])
    o, _ = oracle.forward(q, k, v, gamma=gamma, normalize=normalize, eps=1e-3)
    for t in (0, 7, 20):
        q2, k2, v2 = q.copy(), k.copy(), v.copy()
        q2[:, :, t + 1:] += 1.0
        k2[:, :, t + 1:] -= 2.0
        v2[:, :, t + 1:] *= 3.0
        o2, _ = oracle.forward(q2, k2, v2, gamma=gamma, normalize=normalize, eps=1e-3)
        assert np.array_equal(o2[:, :, : t + 1], o[:, :, : t + 1])
        assert not np.allclose(o2[:, :, t + 1:], o[:, :, t + 1:])


# --------------------------------------------------------------------------- T7
def test_unmasked_identity():
    """q_t^T S_t C_t equals the sum over all key/value index pairs, and the masked
    output is that minus q_t^T G_t."""
    rng = np.random.default_rng(15)
    n, d, dv = 12, 3, 2
    q, k, v = rand_inputs(rng, 1, 1, n, d, dv)
    o, _ = oracle.forward(q, k, v)
    for t in (0, 5, 11):
        _, st = oracle.forward(q[:, :, : t + 1], k[:, :, : t + 1], v[:, :, : t + 1])
        qt = q[0, 0, t]
        unmasked = qt @ st.S[0] @ st.C[0]
        allpairs = sum((qt @ k[0, 0, a]) * (k[0, 0, a] @ q[0, 0, b]) * v[0, 0, b]
                       for a in range(t + 1) for b in range(t + 1))
        assert rel(unmasked, allpairs) < 1e-12
        assert rel(unmasked - qt @ st.G[0], o[0, 0, t]) < 1e-12


# --------------------------------------------------------------------------- T8
def test_split_resume_and_decode_continuation():
    rng = np.random.default_rng(16)
    B, H, n, d, dv = 2, 2, 21, 4, 3
    q, k, v = rand_inputs(rng, B, H, n, d, dv, positive=True)
    gamma = np.array([0.9, 0.99])
    for normalize in (False, True):
        o, s = oracle.forward(q, k, v, gamma=gamma, normalize=normalize, eps=1e-3)
        n1 = 13
        o1, s1 = oracle.forward(q[:, :, :n1], k[:, :, :n1], v[:, :, :n1], gamma=gamma,
                                normalize=normalize, eps=1e-3)
        o2, s2 = oracle.forward(q[:, :, n1:], k[:, :, n1:], v[:, :, n1:], gamma=gamma,
                                normalize=normalize, eps=1e-3, state_in=s1)
        assert rel(np.concatenate([o1, o2], 2), o) < 1e-13
        for a, b in zip(s2.astuple(), s.astuple()):
            assert rel(a, b) < 1e-13
        # decode steps from s1 reproduce the remaining outputs
        st = s1.copy()
        for t in range(n1, n):
            od = oracle.decode_step(st, q[:, :, t].reshape(B * H, d), k[:, :, t].reshape(B * H, d),
                                    v[:, :, t].reshape(B * H, dv), H, gamma=gamma,
                                    normalize=normalize, eps=1e-3)
            assert rel(od.reshape(B, H, dv), o[:, :, t]) < 1e-13
        for a, b in zip(st.astuple(), s.astuple()):
            assert rel(a, b) < 1e-13


def test_empty_sequence_keeps_state():
    rng = np.random.default_rng(17)
    q, k, v = rand_inputs(rng, 1, 1, 5, 3, 2)
    _, s = oracle.forward(q, k, v)
    o, s2 = oracle.forward(q[:, :, :0], k[:, :, :0], v[:, :, :0], state_in=s)
    assert o.shape == (1, 1, 0, 2)
    for a, b in zip(s2.astuple(), s.astuple()):
        assert np.array_equal(a, b)


# ------------------------------------------------------------- unmasked variant
# Skill card "Higher-order linear attention", section "Linear-Time Higher-Order
# Interactions", bullet "Streaming Computation": o_t = q_t^T S_t C_t; the ratio form
# divides by q_t^T S_t m_t.  Its operators are the linear part of the concatenation
# rule (gist.science "Belangrijkste bijdragen" item 2).
def brute_force_unmasked(q, k, v, g=1.0, normalize=False, eps=0.0):
    """o_t = sum_{a<=t} sum_{b<=t} g^{(t-a)+(t-b)} (q_t.k_a)(k_a.q_b) v_b: every key
    index and every query/value index up to t, in any order."""
    n, dv = q.shape[0], v.shape[1]
    o = np.zeros((n, dv))
    for t in range(n):
        num = np.zeros(dv)
        den = 0.0
        for a in range(t + 1):
            for b in range(t + 1):
                w = (g ** ((t - a) + (t - b))) * (q[t] @ k[a]) * (k[a] @ q[b])
                num += w * v[b]
                den += w
        o[t] = num / (den + eps) if normalize else num
    return o


@pytest.mark.parametrize("decay", [False, True])
@pytest.mark.parametrize("normalize", [False, True])
@pytest.mark.parametrize("n,d,dv", [(1, 1, 1), (9, 3, 2), (17, 4, 3)])
def test_unmasked_brute_force_and_state(decay, normalize, n, d, dv):
    rng = np.random.default_rng(300 + n + d)
    B, H = 2, 2
    q, k, v = rand_inputs(rng, B, H, n, d, dv, positive=normalize)
    gamma = np.array([0.85, 0.5]) if decay else None
    o, st = oracle.forward(q, k, v, gamma=gamma, normalize=normalize, eps=1e-3, unmasked=True)
    for b in range(B):
        for h in range(H):
            g = gamma[h] if decay else 1.0
            ref = brute_force_unmasked(q[b, h], k[b, h], v[b, h], g, normalize, 1e-3)
            assert rel(o[b, h], ref) < 1e-12
            S, C, m, _, _ = brute_state(q[b, h], k[b, h], v[b, h], g)
            u = b * H + h
            assert rel(st.S[u], S) < 1e-12 and rel(st.C[u], C) < 1e-12 and rel(st.m[u], m) < 1e-12
    assert not st.G.any() and not st.h.any()  # not carried by this variant


def test_unmasked_dense_form_and_masked_relation():
    """O = [L o ((L o QK^T)(QK^T)^T)] V, and the masked output is the unmasked one
    minus q_t^T G_t (G from the masked state after t)."""
    rng = np.random.default_rng(31)
    n, d, dv = 14, 3, 2
    q, k, v = rand_inputs(rng, 1, 1, n, d, dv)
    o, _ = oracle.forward(q, k, v, unmasked=True)
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    L = np.tril(np.ones((n, n)))
    A = Q @ K.T
    assert rel(o[0, 0], (L * ((L * A) @ A.T)) @ V) < 1e-12
    om, _ = oracle.forward(q, k, v)
    for t in (0, 6, 13):
        _, st = oracle.forward(q[:, :, : t + 1], k[:, :, : t + 1], v[:, :, : t + 1])
        assert rel(o[0, 0, t] - Q[t] @ st.G[0], om[0, 0, t]) < 1e-12


@pytest.mark.parametrize("decay", [False, True])
def test_unmasked_chunked_resume_decode(decay):
    rng = np.random.default_rng(32)
    B, H, n, d, dv = 2, 2, 23, 3, 4
    q, k, v = rand_inputs(rng, B, H, n, d, dv, positive=True)
    gamma = np.array([0.9, 0.7]) if decay else None
    kw = dict(gamma=gamma, normalize=True, eps=1e-3, unmasked=True)
    o, s = oracle.forward(q, k, v, **kw)
    for c in (1, 4, 7, 23, 40):
        oc, sc = oracle.forward(q, k, v, chunk=c, **kw)
        assert rel(oc, o) < 1e-12
        for a, b in zip(sc.astuple(), s.astuple()):
            assert np.allclose(a, b, rtol=1e-12, atol=1e-12)
    n1 = 11
    _, s1 = oracle.forward(q[:, :, :n1], k[:, :, :n1], v[:, :, :n1], **kw)
    o2, _ = oracle.forward(q[:, :, n1:], k[:, :, n1:], v[:, :, n1:], state_in=s1, **kw)
    assert rel(o2, o[:, :, n1:]) < 1e-12
    st = s1.copy()
    for t in range(n1, n):
        od = oracle.decode_step(st, q[:, :, t].reshape(B * H, d), k[:, :, t].reshape(B * H, d),
                                v[:, :, t].reshape(B * H, dv), H, **kw)
        assert rel(od.reshape(B, H, dv), o[:, :, t]) < 1e-12
    for a, b in zip(st.astuple(), s.astuple()):
        assert np.allclose(a, b, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- shared key/value heads
# Skill card, section "Architecture Overview", bullet "Multi-Head Support": keys and
# values shared by a group of query heads.  The result must equal ordinary
# multi-head attention with each group's keys and values repeated per query head.
@pytest.mark.parametrize("unmasked", [False, True])
@pytest.mark.parametrize("H,Hkv", [(4, 1), (6, 2), (3, 3)])
def test_shared_kv_heads_equal_repeated_heads(unmasked, H, Hkv):
    rng = np.random.default_rng(40 + H * 3 + Hkv)
    B, n, d, dv = 2, 10, 3, 2
    q = rng.standard_normal((B, H, n, d))
    k = rng.standard_normal((B, Hkv, n, d))
    v = rng.standard_normal((B, Hkv, n, dv))
    gamma = np.linspace(0.6, 0.95, H)
    rep = lambda a: np.repeat(a, H // Hkv, axis=1)
    kw = dict(gamma=gamma, unmasked=unmasked)
    o, s = oracle.forward(q, k, v, **kw)
    o_ref, s_ref = oracle.forward(q, rep(k), rep(v), **kw)
    assert np.array_equal(o, o_ref)
    for a, b in zip(s.astuple(), s_ref.astuple()):
        assert np.array_equal(a, b)
    oc, _ = oracle.forward(q, k, v, chunk=4, **kw)
    assert rel(oc, o) < 1e-12
    # decode: key/value rows per (sequence, key/value head)
    st, st_ref = s.copy(), s.copy()
    qd = rng.standard_normal((B * H, d))
    kd = rng.standard_normal((B * Hkv, d))
    vd = rng.standard_normal((B * Hkv, dv))
    od = oracle.decode_step(st, qd, kd, vd, H, **kw)
    rep2 = lambda a: np.repeat(a.reshape(B, Hkv, -1), H // Hkv, axis=1).reshape(B * H, -1)
    od_ref = oracle.decode_step(st_ref, qd, rep2(kd), rep2(vd), H, **kw)
    assert np.array_equal(od, od_ref)
    for a, b in zip(st.astuple(), st_ref.astuple()):
        assert np.array_equal(a, b)


# ------------------------------------------------------------- asymmetric variant (AHLA)
# gist.science summary, section 2 "Asymmetrische Hogere-orde Lineaire Aandacht": the
# operator Q (K^T Q)(K^T V) = A A V, A = Q K^T, routed through an intermediate key
# index; masked: o_t = sum_{a<=b<=t} (q_t.k_b)(q_b.k_a) v_a; summaries P^KV, m^K, E, n.
def brute_force_asym(q, k, v, g=1.0, normalize=False, eps=0.0):
    n, dv = q.shape[0], v.shape[1]
    o = np.zeros((n, dv))
    for t in range(n):
        num, den = np.zeros(dv), 0.0
        for b in range(t + 1):
            for a in range(b + 1):
                w = (g ** (t - a)) * (q[t] @ k[b]) * (q[b] @ k[a])
                num += w * v[a]
                den += w
        o[t] = num / (den + eps) if normalize else num
    return o


def brute_state_asym(q, k, v, g=1.0):
    """R, P, m^K, E, n after the last token, each from its definition."""
    n = q.shape[0]
    T = n - 1
    R = sum(np.outer(k[b], q[b]) for b in range(n))
    P = sum(g ** (T - a) * np.outer(k[a], v[a]) for a in range(n))
    m = sum(g ** (T - a) * k[a] for a in range(n))
    E = sum(g ** (T - a) * (q[b] @ k[a]) * np.outer(k[b], v[a]) for b in range(n) for a in range(b + 1))
    nn = sum(g ** (T - a) * (q[b] @ k[a]) * k[b] for b in range(n) for a in range(b + 1))
    return R, P, m, E, nn


@pytest.mark.parametrize("decay", [False, True])
@pytest.mark.parametrize("normalize", [False, True])
@pytest.mark.parametrize("n,d,dv", [(1, 1, 1), (8, 3, 2), (15, 4, 3)])
def test_asym_brute_force_and_state(decay, normalize, n, d, dv):
    rng = np.random.default_rng(500 + n + d)
    B, H = 2, 2
    q, k, v = rand_inputs(rng, B, H, n, d, dv, positive=normalize)
    gamma = np.array([0.8, 0.55]) if decay else None
    o, st = oracle.forward(q, k, v, gamma=gamma, normalize=normalize, eps=1e-3, asymmetric=True)
    for b in range(B):
        for h in range(H):
            g = gamma[h] if decay else 1.0
            assert rel(o[b, h], brute_force_asym(q[b, h], k[b, h], v[b, h], g, normalize, 1e-3)) < 1e-12
            u = b * H + h
            for got, ref in zip(st.astuple(), brute_state_asym(q[b, h], k[b, h], v[b, h], g)):
                assert rel(got[u], ref) < 1e-12


def test_asym_dense_form_and_constant_inputs():
    rng = np.random.default_rng(51)
    n, d, dv = 13, 3, 2
    q, k, v = rand_inputs(rng, 1, 1, n, d, dv)
    o, _ = oracle.forward(q, k, v, asymmetric=True)
    L = np.tril(np.ones((n, n)))
    A = q[0, 0] @ k[0, 0].T
    assert rel(o[0, 0], (L * A) @ (L * A) @ v[0, 0]) < 1e-12
    # constant q = k = x, v = y: (x.x)^2 times the number of pairs a <= b <= t
    x, y = np.array([0.5, -1.0, 2.0]), np.array([1.5, -0.25])
    qc = np.tile(x, (1, 1, n, 1)); vc = np.tile(y, (1, 1, n, 1))
    oc, _ = oracle.forward(qc, qc, vc, asymmetric=True)
    for t in range(n):
        assert rel(oc[0, 0, t], (x @ x) ** 2 * (t + 1) * (t + 2) / 2 * y) < 1e-13


@pytest.mark.parametrize("decay", [False, True])
def test_asym_chunked_combine_resume_decode(decay):
    rng = np.random.default_rng(52)
    B, H, n, d, dv = 2, 2, 22, 3, 4
    q, k, v = rand_inputs(rng, B, H, n, d, dv, positive=True)
    gamma = np.array([0.9, 0.7]) if decay else None
    kw = dict(gamma=gamma, normalize=True, eps=1e-3, asymmetric=True)
    o, s = oracle.forward(q, k, v, **kw)
    for c in (1, 3, 8, 22, 30):
        oc, sc = oracle.forward(q, k, v, chunk=c, **kw)
        assert rel(oc, o) < 1e-12
        for a, b in zip(sc.astuple(), s.astuple()):
            assert np.allclose(a, b, rtol=1e-12, atol=1e-12)
    # the concatenation of two halves' states equals the state of the whole sequence
    n1 = 9
    _, s1 = oracle.forward(q[:, :, :n1], k[:, :, :n1], v[:, :, :n1], **kw)
    _, s2 = oracle.forward(q[:, :, n1:], k[:, :, n1:], v[:, :, n1:], **kw)
    f = np.tile(gamma ** (n - n1), B) if decay else None
    sj = oracle.combine(s1, s2, f, asymmetric=True)
    for a, b in zip(sj.astuple(), s.astuple()):
        assert np.allclose(a, b, rtol=1e-11, atol=1e-11)
    # associativity with a third piece
    n2 = 15
    _, sa = oracle.forward(q[:, :, :n1], k[:, :, :n1], v[:, :, :n1], **kw)
    _, sb = oracle.forward(q[:, :, n1:n2], k[:, :, n1:n2], v[:, :, n1:n2], **kw)
    _, sc3 = oracle.forward(q[:, :, n2:], k[:, :, n2:], v[:, :, n2:], **kw)
    fb = np.tile(gamma ** (n2 - n1), B) if decay else None
    fc = np.tile(gamma ** (n - n2), B) if decay else None
    fbc = np.tile(gamma ** (n - n1), B) if decay else None
    left = oracle.combine(oracle.combine(sa, sb, fb, asymmetric=True), sc3, fc, asymmetric=True)
    right = oracle.combine(sa, oracle.combine(sb, sc3, fc, asymmetric=True), fbc, asymmetric=True)
    for a, b in zip(left.astuple(), right.astuple()):
        assert np.allclose(a, b, rtol=1e-11, atol=1e-11)
    # resume and decode continuation
    o2, _ = oracle.forward(q[:, :, n1:], k[:, :, n1:], v[:, :, n1:], state_in=s1, **kw)
    assert rel(o2, o[:, :, n1:]) < 1e-12
    st = s1.copy()
    for t in range(n1, n):
        od = oracle.decode_step(st, q[:, :, t].reshape(B * H, d), k[:, :, t].reshape(B * H, d),
                                v[:, :, t].reshape(B * H, dv), H, **kw)
        assert rel(od.reshape(B, H, dv), o[:, :, t]) < 1e-12


# ------------------------------------------------------------------ backward
# The pages give no gradient formulas.  The oracle's reverse-mode recurrence is
# pinned by central finite differences of the forward oracle and by the gradient
# of the dense masked-matrix form O = [L o (Q U^T)] V, U = (L o QK^T) K.
@pytest.mark.parametrize("decay", [False, True])
def test_backward_finite_differences(decay):
    rng = np.random.default_rng(61)
    B, H, n, d, dv = 1, 2, 6, 3, 2
    q, k, v = rand_inputs(rng, B, H, n, d, dv)
    go = rng.standard_normal((B, H, n, dv))
    gamma = np.array([0.8, 0.6]) if decay else None
    dq, dk, dvv = oracle.backward(q, k, v, go, gamma)
    loss = lambda q_, k_, v_: float(np.sum(go * oracle.forward(q_, k_, v_, gamma=gamma, want_state=False)[0]))
    eps = 1e-6
    for x, grad, which in ((q, dq, 0), (k, dk, 1), (v, dvv, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [q, k, v]; args_m = [q, k, v]
            args_p[which] = xp; args_m[which] = xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        assert rel(grad, num) < 1e-7, which


def test_backward_dense_form():
    rng = np.random.default_rng(62)
    n, d, dv = 11, 4, 3
    q, k, v = rand_inputs(rng, 1, 1, n, d, dv)
    go = rng.standard_normal((1, 1, n, dv))
    dq, dk, dvv = oracle.backward(q, k, v, go)
    Q, K, V, G = q[0, 0], k[0, 0], v[0, 0], go[0, 0]
    L = np.tril(np.ones((n, n)))
    At = L * (Q @ K.T)            # A-tilde
    U = At @ K
    M = L * (Q @ U.T)
    dV = M.T @ G
    dM = L * (G @ V.T)
    dU = dM.T @ Q
    dAt = L * (dU @ K.T)
    dQ = dM @ U + dAt @ K
    dK = At.T @ dU + dAt.T @ Q
    assert rel(dq[0, 0], dQ) < 1e-12 and rel(dk[0, 0], dK) < 1e-12 and rel(dvv[0, 0], dV) < 1e-12


def test_backward_shared_kv_heads_is_group_sum_of_repeated_heads():
    """Keys and values shared by groups of query heads: the gradient equals that of the
    same computation with every key/value head repeated for its query heads, with dk
    and dv summed over each group (chain rule through the repetition)."""
    rng = np.random.default_rng(12)
    B, H, Hkv, n, d, dv = 2, 6, 2, 9, 3, 2
    q = rng.standard_normal((B, H, n, d))
    k = rng.standard_normal((B, Hkv, n, d))
    v = rng.standard_normal((B, Hkv, n, dv))
    go = rng.standard_normal((B, H, n, dv))
    g = rng.uniform(0.8, 1.0, H)
    rep = H // Hkv
    kr, vr = np.repeat(k, rep, axis=1), np.repeat(v, rep, axis=1)
    dq_r, dk_r, dv_r = oracle.backward(q, kr, vr, go, g)
    dq, dk, dvv = oracle.backward(q, k, v, go, g)
    assert rel(dq, dq_r) < 1e-13
    assert rel(dk, dk_r.reshape(B, Hkv, rep, n, d).sum(axis=2)) < 1e-13
    assert rel(dvv, dv_r.reshape(B, Hkv, rep, n, dv).sum(axis=2)) < 1e-13


@pytest.mark.parametrize("decay", [False, True])
def test_backward_normalised_finite_differences(decay):
    """Ratio-normalised output o = num / (den + eps): the reverse mode through the
    denominator against central differences of the normalised forward (positive
    features keep the denominator away from zero)."""
    rng = np.random.default_rng(63)
    B, H, n, d, dv = 1, 2, 6, 3, 2
    q, k, v = rand_inputs(rng, B, H, n, d, dv)
    q, k = np.abs(q) + 0.2, np.abs(k) + 0.2
    go = rng.standard_normal((B, H, n, dv))
    gamma = np.array([0.8, 0.6]) if decay else None
    e0 = 1e-3
    dq, dk, dvv = oracle.backward(q, k, v, go, gamma, normalize=True, eps=e0)
    loss = lambda q_, k_, v_: float(np.sum(go * oracle.forward(q_, k_, v_, gamma=gamma, normalize=True, eps=e0,
                                                                want_state=False)[0]))
    h = 1e-6
    for x, grad, which in ((q, dq, 0), (k, dk, 1), (v, dvv, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [q, k, v]; args_m = [q, k, v]
            args_p[which] = xp; args_m[which] = xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert rel(grad, num) < 1e-6, which


def test_backward_normalised_equals_augmented_value():
    """The normalised gradient is the unnormalised one of the augmented values [V | 1]
    (the denominator is the output with every value one) with upstream
    [go / (den + eps) | -(go . o) / (den + eps)]; dv is its first dv columns."""
    rng = np.random.default_rng(64)
    B, H, n, d, dv = 2, 2, 13, 4, 3
    q, k, v = rand_inputs(rng, B, H, n, d, dv)
    q, k = np.abs(q) + 0.1, np.abs(k) + 0.1
    go = rng.standard_normal((B, H, n, dv))
    gamma = np.array([0.9, 0.7])
    e0 = 1e-4
    dq, dk, dvv = oracle.backward(q, k, v, go, gamma, normalize=True, eps=e0)
    num, _ = oracle.forward(q, k, v, gamma=gamma, want_state=False)
    den, _ = oracle.forward(q, k, np.ones((B, H, n, 1)), gamma=gamma, want_state=False)
    r = 1.0 / (den + e0)
    o = num * r
    ga = np.concatenate([go * r, -np.sum(go * o, axis=-1, keepdims=True) * r], axis=-1)
    va = np.concatenate([v, np.ones((B, H, n, 1))], axis=-1)
    dq_a, dk_a, dv_a = oracle.backward(q, k, va, ga, gamma)
    assert rel(dq, dq_a) < 1e-11 and rel(dk, dk_a) < 1e-11 and rel(dvv, dv_a[..., :dv]) < 1e-11
