"""Pins of the third-order oracle's decay and ratio normalisation (oracle/hla_oracle3.c).

The gist.science summary (section 3 "Derde-orde HLA") names the cross summaries
G^(1..3) and h^(1..3) of the masked third-order state and, for the scans of section 4,
the segment maps M^KQP and M^KQm; it prints no formula and states no decayed third
order.  The readings pinned here carry the second order's over (section 1
"Normalisatie"; "Belangrijkste bijdragen" item 2 for decay):

  decay:      every prefix moment decays by gamma per token, so the triple (a, b, c)
              seen at time t has weight gamma^((t-a)+(t-b)+(t-c));
  normalised: o_t = num_t / (den_t + eps), den_t the masked output of unit values.

Each pin is independent of the recurrence: four-index brute force, a dense
masked-matrix form, closed forms and special cases."""
import os
import subprocess
import ctypes

import numpy as np
import pytest

import oracle
from test_oracle_third import brute3, rand, rel

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "hla_oracle3.c")


def brute3_decay(Q, K, V, g):
    """o_t = sum_{b<=t} sum_{a<=b} sum_{c<=b} g^(3t-a-b-c) (q_t.k_a)(k_a.q_b)(q_b.k_c) v_c."""
    n, dv = Q.shape[0], V.shape[1]
    o = np.zeros((n, dv))
    for t in range(n):
        for b in range(t + 1):
            for a in range(b + 1):
                for c in range(b + 1):
                    o[t] += g ** (3 * t - a - b - c) * (Q[t] @ K[a]) * (K[a] @ Q[b]) * (Q[b] @ K[c]) * V[c]
    return o


def dense3_decay(Q, K, V, g):
    """O = (L o G^3 o (A (G o L o A)^T)) ((G o L o A) V) with A = Q K^T, G[i][j] = g^(i-j):
    the weight g^(3t-a-b-c) split as g^(3(t-b)) g^(b-a) g^(b-c)."""
    n = Q.shape[0]
    idx = np.arange(n)
    diff = idx[:, None] - idx[None, :]
    L = (diff >= 0).astype(np.float64)
    G1 = np.where(diff >= 0, g ** np.maximum(diff, 0).astype(np.float64), 0.0)
    G3 = np.where(diff >= 0, g ** (3 * np.maximum(diff, 0)).astype(np.float64), 0.0)
    A = Q @ K.T
    W = G1 * L * A
    return (L * G3 * (A @ W.T)) @ (W @ V)


@pytest.mark.parametrize("g", [0.9, 0.6])
@pytest.mark.parametrize("n,d,dv", [(1, 2, 2), (7, 3, 2), (9, 2, 1)])
def test_decay_brute_force(g, n, d, dv):
    rng = np.random.default_rng(100 + n)
    q, k, v = rand(rng, 1, 2, n, d, dv)
    gam = np.array([g, 1.0])
    o, _ = oracle.forward3(q, k, v, gamma=gam)
    assert rel(o[0, 0], brute3_decay(q[0, 0], k[0, 0], v[0, 0], g)) < 1e-12
    assert rel(o[0, 1], brute3(q[0, 1], k[0, 1], v[0, 1])) < 1e-12  # per-head rate; gamma 1 = no decay


def test_decay_dense_form_and_chunked():
    rng = np.random.default_rng(101)
    n, d, dv, g = 37, 4, 3, 0.93
    q, k, v = rand(rng, 1, 1, n, d, dv)
    ref = dense3_decay(q[0, 0], k[0, 0], v[0, 0], g)
    for chunk in (None, 1, 5, 16):
        o, _ = oracle.forward3(q, k, v, gamma=[g], chunk=chunk)
        assert rel(o[0, 0], ref) < 1e-11, chunk


def test_decay_zero_keeps_only_the_current_token():
    """gamma = 0: only a = b = c = t has a nonzero weight, o_t = (q_t.k_t)^3 v_t."""
    rng = np.random.default_rng(102)
    q, k, v = rand(rng, 1, 1, 12, 3, 2)
    o, _ = oracle.forward3(q, k, v, gamma=[0.0])
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    ref = (np.einsum("td,td->t", Q, K) ** 3)[:, None] * V
    assert rel(o[0, 0], ref) < 1e-13


def test_decay_constant_inputs_closed_form():
    """Constant q, k, v: o_t = (q.k)^3 v sum_{b<=t} g^(3(t-b)) (sum_{j<=b} g^(b-j))^2."""
    rng = np.random.default_rng(103)
    n, d, dv, g = 25, 3, 2, 0.8
    q1, k1, v1 = rng.standard_normal(d), rng.standard_normal(d), rng.standard_normal(dv)
    q = np.broadcast_to(q1, (1, 1, n, d)).copy()
    k = np.broadcast_to(k1, (1, 1, n, d)).copy()
    v = np.broadcast_to(v1, (1, 1, n, dv)).copy()
    o, _ = oracle.forward3(q, k, v, gamma=[g])
    geo = lambda m: (1 - g ** (m + 1)) / (1 - g)  # sum_{j=0..m} g^j
    w = np.array([sum(g ** (3 * (t - b)) * geo(b) ** 2 for b in range(t + 1)) for t in range(n)])
    ref = (q1 @ k1) ** 3 * w[:, None] * v1[None, :]
    assert rel(o[0, 0], ref) < 1e-13


def test_decay_summaries_brute_force():
    """The decayed state against its definitions: every term weighted by g^(t - index)
    per factor (t = the last token)."""
    rng = np.random.default_rng(104)
    n, d, dv, g = 6, 3, 2, 0.85
    q, k, v = rand(rng, 1, 1, n, d, dv)
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    _, st = oracle.forward3(q, k, v, gamma=[g])
    t = n - 1
    w = lambda *ix: g ** sum(t - i for i in ix)
    kk = lambda a: np.outer(K[a], K[a])
    qq = lambda b: np.outer(Q[b], Q[b])
    kv = lambda c: np.outer(K[c], V[c])
    R = range(n)
    ref = {
        "SK": sum(w(a) * kk(a) for a in R), "SQ": sum(w(b) * qq(b) for b in R), "P": sum(w(c) * kv(c) for c in R),
        "Z1": sum(w(a, b) * kk(a) @ qq(b) for a in R for b in R if a > b),
        "Z2": sum(w(b, c) * qq(b) @ kv(c) for b in R for c in R if c > b),
        "G1": sum(w(a, b, c) * kk(a) @ qq(b) @ kv(c) for a in R for b in R for c in R if a > b),
        "G2": sum(w(a, b, c) * kk(a) @ qq(b) @ kv(c) for a in R for b in R for c in R if c > b),
        "G3": sum(w(a, b, c) * kk(a) @ qq(b) @ kv(c) for a in R for b in R for c in R if a > b and c > b),
        "T": sum(w(a, b, c) * kk(a) @ qq(b) @ kv(c) for a in R for b in R for c in R if a <= b and c <= b),
        # the maps carry g^(2(t-b)) on the query b and the factor's own decay inside
        "MQP": sum(w(b, b) * g ** (b - c) * qq(b) @ kv(c) for b in R for c in R if c <= b),
        "MKQ": sum(w(b, b) * g ** (b - a) * kk(a) @ qq(b) for a in R for b in R if a <= b),
    }
    for name, want in ref.items():
        assert rel(st[name][0], want) < 1e-12, name


def _segment(q, k, v, t0, t1, **kw):
    return oracle.forward3(q[:, :, t0:t1], k[:, :, t0:t1], v[:, :, t0:t1], **kw)[1]


def test_decay_concatenation_equals_joined_sequence():
    rng = np.random.default_rng(105)
    H, g = 3, np.array([0.9, 0.97, 0.75])
    q, k, v = rand(rng, 1, H, 19, 3, 2)
    A, Bs, C = (_segment(q, k, v, a, b, gamma=g) for a, b in ((0, 5), (5, 12), (12, 19)))
    whole = _segment(q, k, v, 0, 19, gamma=g)
    left = oracle.combine3(oracle.combine3(A, Bs, g ** 7), C, g ** 7)
    right = oracle.combine3(A, oracle.combine3(Bs, C, g ** 7), g ** 14)
    for name in ("SK", "SQ", "P", "T", "MQP", "MKQ"):
        assert rel(left[name], whole[name]) < 1e-12, name
        assert rel(right[name], whole[name]) < 1e-12, name


def brute3_den(Q, K, g=1.0):
    n = Q.shape[0]
    return brute3_decay(Q, K, np.ones((n, 1)), g)[:, 0]


@pytest.mark.parametrize("g", [None, 0.9])
def test_normalised_brute_force(g):
    rng = np.random.default_rng(106)
    n, d, dv, eps = 8, 3, 2, 0.25
    q, k, v = rand(rng, 1, 1, n, d, dv)
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    gg = 1.0 if g is None else g
    num = brute3_decay(Q, K, V, gg)
    den = brute3_den(Q, K, gg)
    o, st = oracle.forward3(q, k, v, gamma=None if g is None else [g], normalize=True, eps=eps)
    assert rel(o[0, 0], num / (den[:, None] + eps)) < 1e-12
    # the unit column: P is the key mass m^K, q_t^T T gives the last token's denominator
    mk = sum(gg ** (n - 1 - c) * K[c] for c in range(n))
    assert rel(st["P"][0][:, dv], mk) < 1e-12
    assert abs(Q[-1] @ st["T"][0][:, dv] - den[-1]) < 1e-10 * max(1.0, abs(den[-1]))


def test_normalised_constant_values_closed_form():
    """Every value row equal to w: num_t = den_t w, so with eps = 0 the output is w
    wherever den_t != 0 (elu + 1 features keep den_t > 0)."""
    rng = np.random.default_rng(107)
    n, d, dv = 21, 4, 3
    x = rng.standard_normal((2, 1, 1, n, d))
    q, k = (np.where(z > 0, z + 1.0, np.exp(z)) for z in x)
    w = rng.standard_normal(dv)
    v = np.broadcast_to(w, (1, 1, n, dv)).copy()
    for g in (None, [0.9]):
        o, _ = oracle.forward3(q, k, v, gamma=g, normalize=True, eps=0.0)
        assert rel(o[0, 0], np.broadcast_to(w, (n, dv))) < 1e-12


@pytest.mark.parametrize("chunk", [1, 3, 8])
def test_normalised_chunked_and_resume(chunk):
    rng = np.random.default_rng(108)
    q, k, v = rand(rng, 1, 2, 26, 3, 2)
    g = np.array([0.95, 0.8])
    o, st = oracle.forward3(q, k, v, gamma=g, normalize=True, eps=0.1)
    oc, stc = oracle.forward3(q, k, v, gamma=g, normalize=True, eps=0.1, chunk=chunk)
    assert rel(oc, o) < 1e-12
    for name in ("SK", "SQ", "P", "T", "MQP", "MKQ"):
        assert rel(stc[name], st[name]) < 1e-12, name
    _, s1 = oracle.forward3(q[:, :, :10], k[:, :, :10], v[:, :, :10], gamma=g, normalize=True, eps=0.1)
    o2, s2 = oracle.forward3(q[:, :, 10:], k[:, :, 10:], v[:, :, 10:], gamma=g, normalize=True, eps=0.1,
                             state_in=s1, chunk=chunk)
    assert rel(o2, o[:, :, 10:]) < 1e-12
    assert rel(s2["T"], st["T"]) < 1e-12


def test_decay_strict_causality():
    rng = np.random.default_rng(109)
    q, k, v = rand(rng, 1, 1, 14, 3, 2)
    o, _ = oracle.forward3(q, k, v, gamma=[0.9], normalize=True, eps=0.5)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[:, :, 8:] += 1.0
    k2[:, :, 8:] -= 2.0
    v2[:, :, 8:] *= 3.0
    o2, _ = oracle.forward3(q2, k2, v2, gamma=[0.9], normalize=True, eps=0.5)
    assert np.array_equal(o[:, :, :8], o2[:, :, :8])


# Plausible mistakes in the decayed and normalised recurrence, planted in a copy.
MUTATIONS = {
    "g1_decay_power": ("g2 * z1k[i] * v[j] + g * k[i] * ksqp[j]", "g * z1k[i] * v[j] + g * k[i] * ksqp[j]"),
    "z2_no_decay_on_new_pair": ("g2 * s->Z2[i * dv + j] + g * sqk[i] * v[j]", "g2 * s->Z2[i * dv + j] + sqk[i] * v[j]"),
    "g3_correction_undecayed": ("- g * ksqk * k[i] * v[j]", "- ksqk * k[i] * v[j]"),
    "combine_t_power": ("f3 * A->T[i * dv + j]", "f2 * A->T[i * dv + j]"),
    "combine_mkq_power": ("f2 * A->MKQ[i * d + j]", "f * A->MKQ[i * d + j]"),
    "normalise_drops_eps": ("J->normalize ? r[J->dv] + J->eps : 1.0", "J->normalize ? r[J->dv] : 1.0"),
}


def _mutant(tmp_path, name):
    old, new = MUTATIONS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, name
    src = tmp_path / f"mut3x_{name}.c"
    src.write_text(text.replace(old, new))
    lib = tmp_path / f"libmut3x_{name}.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(lib), str(src), "-lm"])
    L = ctypes.CDLL(str(lib))
    dp, i = ctypes.POINTER(ctypes.c_double), ctypes.c_int
    L.hla_oracle3_forward_ex.argtypes = [i] * 6 + [dp, i, ctypes.c_double] + [dp] * 6 + [i]
    return L


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_planted_mistakes(tmp_path, name):
    L = _mutant(tmp_path, name)
    rng = np.random.default_rng(110)
    n, d, dv, g, eps = 9, 3, 2, 0.85, 0.3
    Q, K, V = rng.standard_normal((n, d)), rng.standard_normal((n, d)), rng.standard_normal((n, dv))
    ref = brute3_decay(Q, K, V, g) / (brute3_den(Q, K, g)[:, None] + eps)
    P = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    qq, kk, vv = (np.ascontiguousarray(x[None, None]) for x in (Q, K, V))
    gam = np.array([g])
    # the segment maps of the whole sequence by their definitions (the exported state of
    # the chunked path carries them; the outputs never read the prefix's own maps)
    t = n - 1
    Ve = np.concatenate([V, np.ones((n, 1))], axis=1)
    mqp = sum(g ** (2 * (t - b) + b - c) * np.outer(Q[b], Q[b]) @ np.outer(K[c], Ve[c])
              for b in range(n) for c in range(b + 1))
    mkq = sum(g ** (2 * (t - b) + b - a) * np.outer(K[a], K[a]) @ np.outer(Q[b], Q[b])
              for b in range(n) for a in range(b + 1))
    # Z2 by its definition (it cancels from the output: G2 and G3 take the same k k^T Z2 term)
    z2 = sum(g ** ((t - b) + (t - c)) * np.outer(Q[b], Q[b]) @ np.outer(K[c], Ve[c])
             for b in range(n) for c in range(n) if c > b)
    caught = False
    for chunk in (0, 4):
        o = np.zeros((1, 1, n, dv))
        st = np.zeros((1, 4 * d * d + 7 * d * (dv + 1)))
        assert L.hla_oracle3_forward_ex(1, 1, n, d, dv, chunk, P(gam), 1, eps, P(qq), P(kk), P(vv), None, P(o),
                                        P(st), 1) == 0
        s3 = oracle.state3_unpack(st, 1, d, dv + 1)
        caught = caught or rel(o[0, 0], ref) > 1e-6 or rel(s3["MQP"][0], mqp) > 1e-6 or rel(s3["MKQ"][0], mkq) > 1e-6
        if chunk == 0:
            caught = caught or rel(s3["Z2"][0], z2) > 1e-6
    assert caught, f"mutation {name} not caught"
