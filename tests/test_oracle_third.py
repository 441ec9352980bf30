"""Pins of the third-order oracle (oracle/hla_oracle3.c) against what the pages and
the mathematics fix: the brute-force masked sum of A A^T A (gist.science summary,
section 3 "Derde-orde HLA"), the dense masked-matrix form, hand-derived fixtures,
brute-force definitions of every summary and segment map, a closed form for
constant inputs, and the scan properties of section 4 ("Derde-orde scans")."""
import glob
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN3 = os.path.join(os.path.dirname(__file__), "golden", "third_order")


def rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def rand(rng, B, H, n, d, dv):
    return (rng.standard_normal((B, H, n, d)), rng.standard_normal((B, H, n, d)),
            rng.standard_normal((B, H, n, dv)))


def brute3(Q, K, V):
    """o_t = sum_{b<=t} sum_{a<=b} sum_{c<=b} (q_t.k_a)(k_a.q_b)(q_b.k_c) v_c, all four
    indices looped explicitly."""
    n, dv = Q.shape[0], V.shape[1]
    o = np.zeros((n, dv))
    for t in range(n):
        for b in range(t + 1):
            for a in range(b + 1):
                for c in range(b + 1):
                    o[t] += (Q[t] @ K[a]) * (K[a] @ Q[b]) * (Q[b] @ K[c]) * V[c]
    return o


@pytest.mark.parametrize("n,d,dv", [(1, 3, 2), (6, 3, 2), (9, 1, 1), (8, 4, 3)])
def test_brute_force(n, d, dv):
    rng = np.random.default_rng(n * 10 + d)
    q, k, v = rand(rng, 1, 2, n, d, dv)
    o, _ = oracle.forward3(q, k, v)
    for h in range(2):
        assert rel(o[0, h], brute3(q[0, h], k[0, h], v[0, h])) < 1e-12


def test_shared_key_value_heads_brute_force():
    """Four query heads on two key/value heads: query head h uses key/value head h // 2
    (not h % 2) in the four-index sum."""
    rng = np.random.default_rng(17)
    q = rng.standard_normal((1, 4, 7, 3))
    k = rng.standard_normal((1, 2, 7, 3))
    v = rng.standard_normal((1, 2, 7, 2))
    o, _ = oracle.forward3(q, k, v)
    for h in range(4):
        assert rel(o[0, h], brute3(q[0, h], k[0, h // 2], v[0, h // 2])) < 1e-12
    oc, _ = oracle.forward3(q, k, v, chunk=2)
    assert rel(oc, o) < 1e-12


def test_dense_form():
    rng = np.random.default_rng(2)
    n, d, dv = 40, 5, 3
    q, k, v = rand(rng, 1, 1, n, d, dv)
    L = np.tril(np.ones((n, n)))
    A = L * (q[0, 0] @ k[0, 0].T)
    ref = ((L * (A @ A.T)) @ A) @ v[0, 0]
    o, _ = oracle.forward3(q, k, v)
    assert rel(o[0, 0], ref) < 1e-11


@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(GOLDEN3, "*.json"))))
def test_hand_fixtures(path):
    fx = json.load(open(path))
    q, k, v = (np.array(fx[x], dtype=np.float64)[None, None] for x in "qkv")
    o, _ = oracle.forward3(q, k, v)
    np.testing.assert_allclose(o[0, 0], np.array(fx["o"], dtype=np.float64), rtol=1e-14, atol=1e-14)


def test_constant_inputs_closed_form():
    """Constant q, k, v: each triple contributes (q.k)^3 v; for query index b there are
    b choices of a and b of c, so o_t = (q.k)^3 v sum_{b<=t} b^2 = (q.k)^3 t(t+1)(2t+1)/6 v."""
    rng = np.random.default_rng(3)
    n, d, dv = 30, 4, 3
    q1, k1, v1 = rng.standard_normal(d), rng.standard_normal(d), rng.standard_normal(dv)
    q = np.broadcast_to(q1, (1, 1, n, d)).copy()
    k = np.broadcast_to(k1, (1, 1, n, d)).copy()
    v = np.broadcast_to(v1, (1, 1, n, dv)).copy()
    o, _ = oracle.forward3(q, k, v)
    t = np.arange(1, n + 1)[:, None]
    ref = (q1 @ k1) ** 3 * t * (t + 1) * (2 * t + 1) / 6 * v1[None, :]
    assert rel(o[0, 0], ref) < 1e-13


def test_summaries_brute_force():
    """Every field of the state against its definition as an index sum."""
    rng = np.random.default_rng(4)
    n, d, dv = 7, 3, 2
    q, k, v = rand(rng, 1, 1, n, d, dv)
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    _, st = oracle.forward3(q, k, v)
    kk = lambda a: np.outer(K[a], K[a])
    qq = lambda b: np.outer(Q[b], Q[b])
    kv = lambda c: np.outer(K[c], V[c])
    R = range(n)
    ref = {
        "SK": sum(kk(a) for a in R), "SQ": sum(qq(b) for b in R), "P": sum(kv(c) for c in R),
        "Z1": sum(kk(a) @ qq(b) for a in R for b in R if a > b),
        "Z2": sum(qq(b) @ kv(c) for b in R for c in R if c > b),
        "G1": sum(kk(a) @ qq(b) @ kv(c) for a in R for b in R for c in R if a > b),
        "G2": sum(kk(a) @ qq(b) @ kv(c) for a in R for b in R for c in R if c > b),
        "G3": sum(kk(a) @ qq(b) @ kv(c) for a in R for b in R for c in R if a > b and c > b),
        "T": sum(kk(a) @ qq(b) @ kv(c) for a in R for b in R for c in R if a <= b and c <= b),
        "MQP": sum(qq(b) @ kv(c) for b in R for c in R if c <= b),
        "MKQ": sum(kk(a) @ qq(b) for a in R for b in R if a <= b),
    }
    for name, want in ref.items():
        assert rel(st[name][0], want) < 1e-12, name


@pytest.mark.parametrize("chunk", [1, 2, 3, 5, 16, 40])
def test_chunked_scan_equals_serial(chunk):
    rng = np.random.default_rng(5)
    q, k, v = rand(rng, 2, 2, 23, 4, 3)
    o, st = oracle.forward3(q, k, v)
    oc, stc = oracle.forward3(q, k, v, chunk=chunk)
    assert rel(oc, o) < 1e-12
    for name in ("SK", "SQ", "P", "T", "MQP", "MKQ"):
        assert rel(stc[name], st[name]) < 1e-12, name


def _segment(q, k, v, t0, t1):
    return oracle.forward3(q[:, :, t0:t1], k[:, :, t0:t1], v[:, :, t0:t1])[1]


def test_concatenation_equals_joined_sequence_and_is_associative():
    rng = np.random.default_rng(6)
    q, k, v = rand(rng, 1, 3, 20, 4, 2)
    A, Bs, C = _segment(q, k, v, 0, 6), _segment(q, k, v, 6, 13), _segment(q, k, v, 13, 20)
    whole = _segment(q, k, v, 0, 20)
    left = oracle.combine3(oracle.combine3(A, Bs), C)
    right = oracle.combine3(A, oracle.combine3(Bs, C))
    for name in ("SK", "SQ", "P", "T", "MQP", "MKQ"):
        assert rel(left[name], whole[name]) < 1e-12, name
        assert rel(right[name], whole[name]) < 1e-12, name
    # the operator is not commutative
    swapped = oracle.combine3(Bs, A)
    assert rel(swapped["T"], oracle.combine3(A, Bs)["T"]) > 1e-3


def test_resume_from_state():
    rng = np.random.default_rng(7)
    q, k, v = rand(rng, 1, 2, 25, 3, 3)
    o, st = oracle.forward3(q, k, v)
    _, st1 = oracle.forward3(q[:, :, :11], k[:, :, :11], v[:, :, :11])
    o2, st2 = oracle.forward3(q[:, :, 11:], k[:, :, 11:], v[:, :, 11:], state_in=st1)
    assert rel(o2, o[:, :, 11:]) < 1e-12
    o3, st3 = oracle.forward3(q[:, :, 11:], k[:, :, 11:], v[:, :, 11:], state_in=st1, chunk=4)
    assert rel(o3, o[:, :, 11:]) < 1e-12
    for name in oracle.STATE3_FIELDS:
        assert rel(st2[name], st[name]) < 1e-12, name
    for name in ("SK", "SQ", "P", "T", "MQP", "MKQ"):
        assert rel(st3[name], st[name]) < 1e-12, name


def test_strict_causality():
    rng = np.random.default_rng(8)
    q, k, v = rand(rng, 1, 1, 15, 3, 2)
    o, _ = oracle.forward3(q, k, v)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[:, :, 9:] += 1.0
    k2[:, :, 9:] -= 2.0
    v2[:, :, 9:] *= 3.0
    o2, _ = oracle.forward3(q2, k2, v2)
    assert np.array_equal(o[:, :, :9], o2[:, :, :9])
    assert not np.allclose(o[:, :, 9:], o2[:, :, 9:])
