"""Plant plausible mistakes in a copy of the third-order oracle source and check that
the brute-force pin rejects each one (serial recurrence and chunked scan).  The copy is
compiled to a temporary library; the real oracle is untouched."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from test_oracle_third import brute3, rel

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "hla_oracle3.c")

MUTATIONS = {
    # Z1 built from the query moment after the token (keeps the pair a = b out of the correction)
    "z1_after_sq": ("b += k[j] * s->SQ[j * d + i];", "b += k[j] * (s->SQ[j * d + i] + q[j] * q[i]);"),
    # wrong sign of the doubly forbidden correction
    "g3_sign": ("- q[i] * (s->G1[i * dv + j] + s->G2[i * dv + j] - s->G3[i * dv + j]);",
                "- q[i] * (s->G1[i * dv + j] + s->G2[i * dv + j] + s->G3[i * dv + j]);"),
    # G2 without the term of the new key c = t against earlier queries
    "g2_drops_term": ("s->G2[i * dv + j] = g3 * s->G2[i * dv + j] + g2 * sksqk[i] * v[j] + k[i] * kz2[j];",
                      "s->G2[i * dv + j] = g3 * s->G2[i * dv + j] + k[i] * kz2[j];"),
    # transposed auxiliary product in G1
    "z1_transposed": ("c += s->Z1[i * d + j] * k[j];", "c += s->Z1[j * d + i] * k[j];"),
    # G3 counts the triple a = c = t twice
    "g3_double_count": ("+ z1tk[i] * v[j] - g * ksqk * k[i] * v[j];", "+ z1tk[i] * v[j];"),
}

MUTATIONS_SCAN = {
    # concatenation drops the S^K_A S^Q_B P_A cross term
    "combine_drops_cross": ("+ f * t1 + f * t2 + f2 * t3;", "+ f * t1 + f * t2;"),
    # the cross term S^K_A M^QP_B taken with the later segment's key moment
    "combine_wrong_segment": ("t1 += A->SK[i * d + l] * B->MQP[l * dv + j];", "t1 += B->SK[i * d + l] * B->MQP[l * dv + j];"),
    # M^QP composed with the wrong operand order (visible in the exported state)
    "mqp_order": ("acc += B->SQ[i * d + l] * A->P[l * dv + j];", "acc += A->SQ[i * d + l] * B->P[l * dv + j];"),
}


def _build(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, name
    src = tmp_path / f"mut3_{name}.c"
    src.write_text(text.replace(old, new))
    lib = tmp_path / f"libmut3_{name}.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(lib), str(src), "-lm"])
    L = ctypes.CDLL(str(lib))
    dp, i = ctypes.POINTER(ctypes.c_double), ctypes.c_int
    L.hla_oracle3_forward.argtypes = [i] * 6 + [dp] * 6 + [i]
    return L


def _run(L, q, k, v, chunk, want_state=False):
    n, d, dv = q.shape[0], q.shape[1], v.shape[1]
    o = np.zeros((1, 1, n, dv))
    st = np.zeros((1, 4 * d * d + 7 * d * dv))
    P = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    qq, kk, vv = (np.ascontiguousarray(x[None, None]) for x in (q, k, v))
    assert L.hla_oracle3_forward(1, 1, n, d, dv, chunk, P(qq), P(kk), P(vv), None, P(o), P(st), 1) == 0
    if want_state:
        import oracle
        return o[0, 0], oracle.state3_unpack(st, 1, d, dv)
    return o[0, 0]


def _inputs():
    rng = np.random.default_rng(1)
    n, d, dv = 8, 3, 2
    return rng.standard_normal((n, d)), rng.standard_normal((n, d)), rng.standard_normal((n, dv))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_brute_force_rejects_recurrence_mistake(tmp_path, name):
    L = _build(tmp_path, name, *MUTATIONS[name])
    q, k, v = _inputs()
    assert rel(_run(L, q, k, v, 0), brute3(q, k, v)) > 1e-6, f"mutation {name} not caught"


@pytest.mark.parametrize("name", sorted(MUTATIONS_SCAN))
def test_brute_force_rejects_scan_mistake(tmp_path, name):
    L = _build(tmp_path, name, *MUTATIONS_SCAN[name])
    q, k, v = _inputs()
    ref = brute3(q, k, v)
    assert rel(_run(L, q, k, v, 0), ref) < 1e-12  # the serial path is untouched
    o, st = _run(L, q, k, v, 3, want_state=True)
    # the segment map M^QP of the whole sequence by its definition sum_{c<=b} q_b q_b^T k_c v_c^T
    mqp = sum(np.outer(q[b], q[b]) @ np.outer(k[c], v[c]) for b in range(len(q)) for c in range(b + 1))
    caught = rel(o, ref) > 1e-6 or rel(st["MQP"][0], mqp) > 1e-6
    assert caught, f"mutation {name} not caught"
