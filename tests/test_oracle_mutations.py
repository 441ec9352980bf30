"""Plant plausible mistakes in a copy of the oracle source and check that the
brute-force pin rejects each one.  The copy is compiled to a temporary library;
the real oracle is untouched."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from test_oracle_pins import brute_force, rand_inputs, rel

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "hla_oracle.c")

MUTATIONS = {
    # cross summary built from the updated C instead of C_{t-1}: flips the mask direction
    "g_after_c": ("    /* S_t = g S_{t-1} + k k^T */",
                  "    for (int j = 0; j < dv; ++j) { double acc = 0.0;"
                  " for (int i = 0; i < d; ++i) acc += k[i] * (C[i * dv + j] + q[i] * v[j]);"
                  " for (int i = 0; i < d; ++i) G[i * dv + j] += g * k[i] * (acc - st->kc[j]); }\n"
                  "    /* S_t = g S_{t-1} + k k^T */"),
    # wrong sign of the cross-summary correction
    "plus_g": ("acc += st->qs[i] * C[i * dv + j] - q[i] * G[i * dv + j];",
               "acc += st->qs[i] * C[i * dv + j] + q[i] * G[i * dv + j];"),
    # decay applied once instead of twice to G
    "g_single_decay": ("G[i * dv + j] = g2 * G[i * dv + j]", "G[i * dv + j] = g * G[i * dv + j]"),
    # transposed operand in q^T S
    "qs_transposed": ("acc += q[i] * S[i * d + j];", "acc += q[j] * S[i * d + i];"),
    # key moment built from q
    "s_from_q": ("S[i * d + j] = g * S[i * d + j] + k[i] * k[j];",
                 "S[i * d + j] = g * S[i * d + j] + q[i] * k[j];"),
}


def _build_mutant(tmp_path, name):
    text = open(SRC).read()
    old, new = MUTATIONS[name]
    assert text.count(old) == 1, name
    src = tmp_path / f"mut_{name}.c"
    src.write_text(text.replace(old, new))
    lib = tmp_path / f"libmut_{name}.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(lib), str(src), "-lm"])
    L = ctypes.CDLL(str(lib))
    dp = ctypes.POINTER(ctypes.c_double)
    i, d = ctypes.c_int, ctypes.c_double
    L.hla_oracle_forward.argtypes = [i] * 7 + [dp, dp, dp, dp, i, d] + [dp] * 5 + [dp] + [dp] * 5 + [i]
    return L


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pin_rejects_planted_mistake(tmp_path, name):
    L = _build_mutant(tmp_path, name)
    rng = np.random.default_rng(1)
    n, d, dv = 9, 3, 2
    q, k, v = rand_inputs(rng, 1, 1, n, d, dv)
    g = np.array([0.8])
    o = np.zeros((1, 1, n, dv))
    P = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    none = [None] * 5
    assert L.hla_oracle_forward(1, 1, 1, n, d, dv, 0, P(q), P(k), P(v), P(g), 0, 0.0, *none, P(o), *none, 1) == 0
    ref = brute_force(q[0, 0], k[0, 0], v[0, 0], 0.8)
    assert rel(o[0, 0], ref) > 1e-6, f"mutation {name} not caught by the brute-force pin"


# mistakes in the unmasked variant and in the key/value head mapping, each caught by
# its own pin (all-pairs brute force; repeated-head equivalence)
MUTATIONS_VARIANTS = {
    # the unmasked variant still subtracts the cross summary
    "unmasked_keeps_cross": ("    if (st->variant == 0) {\n        /* k^T C_{t-1} and k^T m_{t-1} */",
                             "    if (st->variant != 2) {\n        /* k^T C_{t-1} and k^T m_{t-1} */"),
    # asymmetric variant: z from P before the current token (drops the pairs a = b)
    "asym_stale_p": ("            for (int i = 0; i < d; ++i) acc += q[i] * C[i * dv + j];\n            st->kc[j] = acc;\n        }\n        for (int i = 0; i < d; ++i) zeta",
                     "            for (int i = 0; i < d; ++i) acc += q[i] * (C[i * dv + j] - k[i] * v[j]);\n            st->kc[j] = acc;\n        }\n        for (int i = 0; i < d; ++i) zeta"),
    # query heads mapped to key/value heads round-robin instead of in groups
    "kv_round_robin": ("return (size_t)b * J->Hkv + hh / (J->H / J->Hkv);",
                       "return (size_t)b * J->Hkv + hh % J->Hkv;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS_VARIANTS))
def test_variant_pins_reject_planted_mistake(tmp_path, name):
    from test_oracle_pins import brute_force_unmasked
    text = open(SRC).read()
    old, new = MUTATIONS_VARIANTS[name]
    assert text.count(old) == 1, name
    src = tmp_path / f"mut_{name}.c"
    src.write_text(text.replace(old, new))
    lib = tmp_path / f"libmut_{name}.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(lib), str(src), "-lm"])
    L = ctypes.CDLL(str(lib))
    dp = ctypes.POINTER(ctypes.c_double)
    i, d = ctypes.c_int, ctypes.c_double
    L.hla_oracle_forward.argtypes = [i] * 7 + [dp, dp, dp, dp, i, d] + [dp] * 5 + [dp] + [dp] * 5 + [i]
    P = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    none = [None] * 5
    rng = np.random.default_rng(2)
    n, dd, dv = 8, 3, 2
    if name == "asym_stale_p":
        from test_oracle_pins import brute_force_asym
        q, k, v = rand_inputs(rng, 1, 1, n, dd, dv)
        o = np.zeros((1, 1, n, dv))
        assert L.hla_oracle_forward(1, 1, 1, n, dd, dv, 2, P(q), P(k), P(v), None, 0, 0.0, *none, P(o), *none,
                                    1) == 0
        assert rel(o[0, 0], brute_force_asym(q[0, 0], k[0, 0], v[0, 0])) > 1e-6, f"mutation {name} not caught"
    elif name == "unmasked_keeps_cross":
        q, k, v = rand_inputs(rng, 1, 1, n, dd, dv)
        o = np.zeros((1, 1, n, dv))
        assert L.hla_oracle_forward(1, 1, 1, n, dd, dv, 1, P(q), P(k), P(v), None, 0, 0.0, *none, P(o), *none,
                                    1) == 0
        ref = brute_force_unmasked(q[0, 0], k[0, 0], v[0, 0])
        assert rel(o[0, 0], ref) > 1e-6, f"mutation {name} not caught"
    else:
        H, Hkv = 4, 2
        q = rng.standard_normal((1, H, n, dd))
        k = rng.standard_normal((1, Hkv, n, dd))
        v = rng.standard_normal((1, Hkv, n, dv))
        o = np.zeros((1, H, n, dv))
        assert L.hla_oracle_forward(1, H, Hkv, n, dd, dv, 0, P(q), P(k), P(v), None, 0, 0.0, *none, P(o), *none,
                                    1) == 0
        kr, vr = np.repeat(k, H // Hkv, axis=1), np.repeat(v, H // Hkv, axis=1)
        ref = np.stack([brute_force(q[0, h], kr[0, h], vr[0, h]) for h in range(H)])
        assert rel(o[0], ref) > 1e-6, f"mutation {name} not caught"


def test_backward_pin_rejects_planted_mistake(tmp_path):
    # dk from Om + Om (dropping the transpose) must fail the finite-difference pin
    text = open(SRC).read()
    old = "acc += (Om[i * d + j] + Om[j * d + i]) * kt[j];"
    assert text.count(old) == 1
    src = tmp_path / "mut_bwd.c"
    src.write_text(text.replace(old, "acc += (Om[i * d + j] + Om[i * d + j]) * kt[j];"))
    lib = tmp_path / "libmut_bwd.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(lib), str(src), "-lm"])
    L = ctypes.CDLL(str(lib))
    dp = ctypes.POINTER(ctypes.c_double)
    L.hla_oracle_backward.argtypes = [ctypes.c_int] * 7 + [ctypes.c_double] + [dp] * 8 + [ctypes.c_int]
    L.hla_oracle_forward.argtypes = [ctypes.c_int] * 7 + [dp, dp, dp, dp, ctypes.c_int, ctypes.c_double] + \
        [dp] * 5 + [dp] + [dp] * 5 + [ctypes.c_int]
    P = lambda a: a.ctypes.data_as(dp)
    rng = np.random.default_rng(3)
    n, d, dv = 5, 3, 2
    q, k, v = rand_inputs(rng, 1, 1, n, d, dv)
    go = rng.standard_normal((1, 1, n, dv))
    dq, dk, dvv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    assert L.hla_oracle_backward(1, 1, 1, n, d, dv, 0, 0.0, P(q), P(k), P(v), None, P(go), P(dq), P(dk), P(dvv),
                                 1) == 0
    none = [None] * 5

    def loss(kk):
        o = np.zeros((1, 1, n, dv))
        assert L.hla_oracle_forward(1, 1, 1, n, d, dv, 0, P(q), P(kk), P(v), None, 0, 0.0, *none, P(o), *none,
                                    1) == 0
        return float(np.sum(go * o))

    num = np.zeros_like(k)
    for idx in np.ndindex(*k.shape):
        kp, km = k.copy(), k.copy()
        kp[idx] += 1e-6
        km[idx] -= 1e-6
        num[idx] = (loss(kp) - loss(km)) / 2e-6
    assert rel(dk, num) > 1e-4, "mutation in the backward not caught by the finite-difference pin"
