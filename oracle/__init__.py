"""fp64 CPU oracle for second-order Higher-order Linear Attention (masked and unmasked).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never loads it, and it shares no code with the CUDA path.

The arithmetic lives in ``hla_oracle.c`` (plain loops in the order of the formulas
on the gist.science technical summary of "Higher-order Linear Attention",
section 1 "Tweede-orde HLA" and section 4 "Parallelle training via associatieve
scans").  This module compiles it with gcc and marshals numpy arrays to it.

Pins (what the oracle is checked against, all in ``tests/test_oracle_pins.py``):
brute-force triple sum over key <= query/value index <= t, the dense masked-matrix
form, hand-derived integer fixtures in ``tests/golden/``, closed forms for constant
inputs, n = 1 / d = 1 / decay 0 / decay 1 special cases, chunk-size invariance of
the chunked scan, associativity and identity of segment concatenation, strict
causality, split resume, and the unmasked identity.  The decay variant's formula is
not printed on the pages; its pins are internal consistency only (see the decay
reading in hla_oracle.c).  The unmasked variant (o_t = q_t^T S_t C_t, skill card
"Higher-order linear attention", bullet "Streaming Computation") is pinned by an
all-pairs brute force, the dense form [L o ((L o QK^T)(QK^T)^T)]V, its relation to the
masked output through G, chunk invariance, resume and decode continuation; shared
key/value heads (bullet "Multi-Head Support") by equality with repeated heads.  The
asymmetric variant AHLA (section 2, o_t = sum_{a<=b<=t} (q_t.k_b)(q_b.k_a) v_a) is pinned
by its brute-force triple sum, the dense form (L o A)(L o A)V, brute-force definitions of
its five summaries, a closed form for constant inputs, chunk invariance, associativity
of its concatenation rule, concatenation equal to the joined sequence, resume and
decode continuation.  The backward pass (reverse mode of the masked recurrence; the
pages give no gradient formulas) is pinned by central finite differences of the
forward and by the gradient of the dense masked-matrix form.  The masked third-order
output (``forward3``, section 3 "Derde-orde HLA"; the pages print no formula) is
pinned by its brute-force quadruple-index sum, the dense form
[(L o ((L o A)(L o A)^T))(L o A)]V, brute-force definitions of its cross summaries
and segment maps, a closed form for constant inputs, chunk invariance of the
segment-map scan, associativity of its concatenation and resume.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hla_oracle.c")
_SRC3 = os.path.join(_HERE, "hla_oracle3.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libhla_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile hla_oracle.c and hla_oracle3.c into one shared library (gcc, -O2, no
    fast-math)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_SRC3))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, _SRC3, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        d = ctypes.c_double
        _lib.hla_oracle_forward.argtypes = [i] * 7 + [dp, dp, dp, dp, i, d] + [dp] * 5 + [dp] + [dp] * 5 + [i]
        _lib.hla_oracle_forward_chunked.argtypes = [i] * 8 + [dp, dp, dp, dp, i, d] + [dp] * 5 + [dp] + [dp] * 5 + [i]
        _lib.hla_oracle_decode_step.argtypes = [i] * 6 + [dp, i, d] + [dp] * 5 + [dp, dp, dp, dp, i]
        _lib.hla_oracle_combine.argtypes = [i, i, i, i] + [dp] * 10 + [dp] + [dp] * 5
        _lib.hla_oracle_backward.argtypes = [i] * 7 + [d] + [dp] * 8 + [i]
        _lib.hla_oracle_backward_state.argtypes = [i] * 7 + [d] + [dp] * 5 + [dp] * 5 + [dp] * 3 + [dp] * 5 + [i]
        _lib.hla_oracle3_forward.argtypes = [i] * 6 + [dp] * 6 + [i]
        _lib.hla_oracle3_combine.argtypes = [i, i, i, dp, dp, dp]
        _lib.hla_oracle3_forward_ex.argtypes = [i] * 6 + [dp, i, d] + [dp] * 6 + [i]
        _lib.hla_oracle3_combine_ex.argtypes = [i, i, i, dp, dp, dp, dp]
        for f in (_lib.hla_oracle_forward, _lib.hla_oracle_forward_chunked,
                  _lib.hla_oracle_decode_step, _lib.hla_oracle_combine, _lib.hla_oracle_backward,
                  _lib.hla_oracle_backward_state,
                  _lib.hla_oracle3_forward, _lib.hla_oracle3_combine, _lib.hla_oracle3_forward_ex,
                  _lib.hla_oracle3_combine_ex):
            f.restype = ctypes.c_int
    return _lib


def _p(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


@dataclass
class State:
    """The five summaries of every (b,h): S [BH,d,d], C [BH,d,dv], m [BH,d],
    G [BH,d,dv], h [BH,d], fp64."""
    S: np.ndarray
    C: np.ndarray
    m: np.ndarray
    G: np.ndarray
    h: np.ndarray

    @staticmethod
    def zeros(units: int, d: int, dv: int) -> "State":
        return State(np.zeros((units, d, d)), np.zeros((units, d, dv)), np.zeros((units, d)),
                     np.zeros((units, d, dv)), np.zeros((units, d)))

    def copy(self) -> "State":
        return State(*(np.array(x, dtype=np.float64, copy=True) for x in self.astuple()))

    def astuple(self):
        return (self.S, self.C, self.m, self.G, self.h)


def _state_ptrs(st):
    if st is None:
        return [None] * 5
    return [_p(x) for x in st.astuple()]


def _as_state(st, units, d, dv):
    if st is None:
        return None
    s = State(*(_f64(x) for x in st.astuple()))
    assert s.S.size == units * d * d and s.C.size == units * d * dv and s.m.size == units * d
    return s


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


VARIANTS = {"masked": 0, "unmasked": 1, "asymmetric": 2}


def _variant(unmasked=False, asymmetric=False) -> int:
    assert not (unmasked and asymmetric)
    return 1 if unmasked else (2 if asymmetric else 0)


def forward(q, k, v, gamma=None, normalize=False, eps=0.0, state_in=None,
            want_state=True, chunk=None, nthreads=None, unmasked=False, asymmetric=False):
    """2nd-order HLA forward in fp64: masked (default), unmasked, or the asymmetric
    variant AHLA (its state R, P, m^K, E, n in the S, C, m, G, h arrays).

    q: [B,H,n,d]; k: [B,Hkv,n,d]; v: [B,Hkv,n,dv] with H a multiple of Hkv (query
    head h reads key/value head h // (H // Hkv)); gamma: [H] or None.  chunk=None
    runs the serial recurrence; chunk=c runs the chunked scan (per-chunk summaries
    folded with the segment-concatenation rule).  The unmasked variant carries S, C,
    m only and returns G, h as zeros.  Returns (o [B,H,n,dv], State or None).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, n, d = q.shape
    Hkv = k.shape[1]
    dv = v.shape[-1]
    assert k.shape == (B, Hkv, n, d) and v.shape[:3] == (B, Hkv, n) and H % Hkv == 0
    g = _f64(gamma)
    if g is not None:
        assert g.shape == (H,)
    sin = _as_state(state_in, B * H, d, dv)
    o = np.zeros((B, H, n, dv))
    sout = State.zeros(B * H, d, dv) if want_state else None
    lib = _load()
    nt = nthreads or default_threads()
    args_tail = [_p(q), _p(k), _p(v), _p(g), int(bool(normalize)), float(eps)] + _state_ptrs(sin) + \
        [_p(o)] + _state_ptrs(sout) + [nt]
    um = _variant(unmasked, asymmetric)
    if chunk is None:
        rc = lib.hla_oracle_forward(B, H, Hkv, n, d, dv, um, *args_tail)
    else:
        rc = lib.hla_oracle_forward_chunked(B, H, Hkv, n, d, dv, um, int(chunk), *args_tail)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return o, sout


def decode_step(state: State, q, k, v, H, gamma=None, normalize=False, eps=0.0, nthreads=None,
                unmasked=False, asymmetric=False):
    """One decode step for N (sequence, head) pairs, in place on ``state``.
    q: [N,d]; k: [N/H*Hkv,d]; v: [N/H*Hkv,dv]; pair u uses gamma[u % H] and key/value
    row (u // H) * Hkv + (u % H) // (H // Hkv).  Returns o [N,dv]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    N, d = q.shape
    dv = v.shape[-1]
    Hkv = k.shape[0] * H // max(N, 1) if N else H
    g = _f64(gamma)
    for x in state.astuple():
        assert x.dtype == np.float64 and x.flags.c_contiguous
    o = np.zeros((N, dv))
    rc = _load().hla_oracle_decode_step(N, H, Hkv, d, dv, _variant(unmasked, asymmetric), _p(g), int(bool(normalize)),
                                        float(eps),
                                        *_state_ptrs(state), _p(q), _p(k), _p(v), _p(o),
                                        nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return o


def combine(A: State, Bst: State, decay_pow=None, asymmetric=False) -> State:
    """Segment concatenation out = A (+) B for every item (A earlier than B), by the
    masked rule or the asymmetric variant's rule."""
    A = State(*(_f64(x) for x in A.astuple()))
    Bst = State(*(_f64(x) for x in Bst.astuple()))
    count, d, dv = A.C.shape
    out = State.zeros(count, d, dv)
    f = _f64(decay_pow)
    rc = _load().hla_oracle_combine(count, d, dv, 2 if asymmetric else 0, *_state_ptrs(A), *_state_ptrs(Bst), _p(f),
                                    *_state_ptrs(out))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out


def backward(q, k, v, go, gamma=None, nthreads=None, normalize=False, eps=0.0, state_in=None, want_dstate=False):
    """Gradients (dq, dk, dv) of sum_t go_t . o_t for the masked forward (reverse mode
    of the recurrence in hla_oracle.c), through the ratio normalisation
    o = num / (den + eps) when `normalize`.
    q, go: [B,H,n,d|dv]; k, v: [B,Hkv,n,d|dv] with H a multiple of Hkv (query head h
    reads key/value head h // (H // Hkv); dk, dv sum over the heads of a group);
    gamma: [H] or None.  state_in: the State before the first token (None: zeros).
    want_dstate: also return the gradient with respect to that state (a State)."""
    q, k, v, go = _f64(q), _f64(k), _f64(v), _f64(go)
    B, H, n, d = q.shape
    Hkv = k.shape[1]
    dv = v.shape[-1]
    assert k.shape == (B, Hkv, n, d) and v.shape == (B, Hkv, n, dv) and go.shape == (B, H, n, dv) and H % Hkv == 0
    g = _f64(gamma)
    dq, dk, dvv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    sin = _as_state(state_in, B * H, d, dv)
    dst = State.zeros(B * H, d, dv) if want_dstate else None
    rc = _load().hla_oracle_backward_state(B, H, Hkv, n, d, dv, int(bool(normalize)), float(eps), _p(q), _p(k),
                                           _p(v), _p(g), _p(go), *_state_ptrs(sin), _p(dq), _p(dk), _p(dvv),
                                           *_state_ptrs(dst), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return (dq, dk, dvv, dst) if want_dstate else (dq, dk, dvv)


# ------------------------------------------------------------------ third order
STATE3_FIELDS = ("SK", "SQ", "Z1", "MKQ", "P", "Z2", "G1", "G2", "G3", "T", "MQP")


def _state3_shapes(units, d, dv):
    return {n: (units, d, d) if n in ("SK", "SQ", "Z1", "MKQ") else (units, d, dv) for n in STATE3_FIELDS}


def state3_pack(st: dict, units, d, dv) -> np.ndarray:
    """dict of the eleven third-order arrays -> [units][4d^2 + 7 d dv] in the C layout."""
    shp = _state3_shapes(units, d, dv)
    parts = [np.asarray(st[n], np.float64).reshape(shp[n]).reshape(units, -1) for n in STATE3_FIELDS]
    return np.ascontiguousarray(np.concatenate(parts, axis=1))


def state3_unpack(buf: np.ndarray, units, d, dv) -> dict:
    shp = _state3_shapes(units, d, dv)
    out, off = {}, 0
    for n in STATE3_FIELDS:
        w = int(np.prod(shp[n][1:]))
        out[n] = buf[:, off:off + w].reshape(shp[n]).copy()
        off += w
    return out


def forward3(q, k, v, state_in=None, chunk=None, want_state=True, nthreads=None, gamma=None, normalize=False,
             eps=1e-6):
    """Masked third-order HLA forward in fp64 (hla_oracle3.c): o_t = q_t^T T_t with
    T_t = S^K S^Q P - G1 - G2 + G3.  q, k: [B,H,n,d]; v: [B,H,n,dv].  chunk=None runs
    the serial recurrence in the moments and cross summaries; chunk=c the chunked scan
    over segment summaries (S^K, S^Q, P, T, M^QP, M^KQ; the other fields come back NaN).
    gamma: [H] decay per head (every prefix moment decays by gamma per token; the
    triple a, b, c <= t has weight gamma^(3t-a-b-c)) or None.  normalize: o = num /
    (den + eps), den the output of unit values; the state then has dv + 1 value
    columns, the unit column last (its P is the key mass m^K, its G1..G3 are h^(1..3)).
    state_in / the returned state: dict with the fields of STATE3_FIELDS, each
    [B*H, d, d] or [B*H, d, dve] (T is derived and ignored on input).
    Key/value heads may be shared: k [B,Hkv,n,d], v [B,Hkv,n,dv] with H a multiple of
    Hkv, query head h reading key/value head h // (H // Hkv) (each group's keys and
    values are given to every query head of the group before the recurrence runs).
    Returns (o [B,H,n,dv], state or None)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, n, d = q.shape
    dv = v.shape[-1]
    Hkv = k.shape[1]
    assert k.shape == (B, Hkv, n, d) and v.shape == (B, Hkv, n, dv) and H % Hkv == 0
    if Hkv != H:
        k = np.ascontiguousarray(np.repeat(k, H // Hkv, axis=1))
        v = np.ascontiguousarray(np.repeat(v, H // Hkv, axis=1))
    dve = dv + (1 if normalize else 0)
    units = B * H
    g = None if gamma is None else np.ascontiguousarray(np.asarray(gamma, np.float64).reshape(H))
    sin = state3_pack(state_in, units, d, dve) if state_in is not None else None
    sout = np.zeros((units, 4 * d * d + 7 * d * dve)) if want_state else None
    o = np.zeros((B, H, n, dv))
    rc = _load().hla_oracle3_forward_ex(B, H, n, d, dv, int(chunk or 0), _p(g), int(bool(normalize)), float(eps),
                                        _p(q), _p(k), _p(v), _p(sin), _p(o), _p(sout), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return o, (state3_unpack(sout, units, d, dve) if want_state else None)


def combine3(A: dict, Bst: dict, decay_pow=None) -> dict:
    """Concatenation of third-order segment summaries (A before B) for every item;
    decay_pow: per item gamma^len(B), or None (no decay)."""
    units, d, dv = np.asarray(A["P"]).shape
    a, b = state3_pack(A, units, d, dv), state3_pack(Bst, units, d, dv)
    out = np.zeros_like(a)
    f = None if decay_pow is None else np.ascontiguousarray(np.asarray(decay_pow, np.float64).reshape(units))
    rc = _load().hla_oracle3_combine_ex(units, d, dv, _p(f), _p(a), _p(b), _p(out))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return state3_unpack(out, units, d, dv)
