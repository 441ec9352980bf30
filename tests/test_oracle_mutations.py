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
    L.hla_oracle_forward.argtypes = [i, i, i, i, i, dp, dp, dp, dp, i, d] + [dp] * 5 + [dp] + [dp] * 5 + [i]
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
    assert L.hla_oracle_forward(1, 1, n, d, dv, P(q), P(k), P(v), P(g), 0, 0.0, *none, P(o), *none, 1) == 0
    ref = brute_force(q[0, 0], k[0, 0], v[0, 0], 0.8)
    assert rel(o[0, 0], ref) > 1e-6, f"mutation {name} not caught by the brute-force pin"
