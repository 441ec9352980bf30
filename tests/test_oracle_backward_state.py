"""Pins of the oracle's backward pass from a given initial state (oracle/hla_oracle.c,
hla_oracle_backward_state): the gradient of sum_t go_t . o_t with respect to q, k, v
and to every entry of the state (S, C, m, G, h) before the first token, against
central differences of the oracle's forward, and the equality with the gradient of
the joined sequence."""
import numpy as np
import pytest

import oracle


def rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def rand_state(rng, units, d, dv, scale=0.5):
    S = rng.standard_normal((units, d, d)) * scale
    S = S + S.transpose(0, 2, 1)  # a key moment is symmetric; the gradient is per array entry all the same
    return oracle.State(S, rng.standard_normal((units, d, dv)) * scale, rng.standard_normal((units, d)) * scale,
                        rng.standard_normal((units, d, dv)) * scale, rng.standard_normal((units, d)) * scale)


def loss(q, k, v, go, st, **kw):
    o, _ = oracle.forward(q, k, v, state_in=st, **kw)
    return float((o * go).sum())


def central(f, x, idx, h):
    x0 = x[idx]
    x[idx] = x0 + h
    a = f()
    x[idx] = x0 - h
    b = f()
    x[idx] = x0
    return (a - b) / (2 * h)


@pytest.mark.parametrize("normalize,decay", [(False, False), (False, True), (True, False), (True, True)])
def test_gradients_against_central_differences(normalize, decay):
    rng = np.random.default_rng(11 + 2 * normalize + decay)
    B, H, n, d, dv = 1, 2, 6, 3, 2
    if normalize:  # positive features keep the denominator away from zero
        q = np.abs(rng.standard_normal((B, H, n, d))) + 0.5
        k = np.abs(rng.standard_normal((B, H, n, d))) + 0.5
    else:
        q, k = rng.standard_normal((B, H, n, d)), rng.standard_normal((B, H, n, d))
    v, go = rng.standard_normal((B, H, n, dv)), rng.standard_normal((B, H, n, dv))
    st = rand_state(rng, B * H, d, dv)
    if normalize:  # a positive initial denominator: S_in m_in - h_in with q > 0
        st.m[:] = np.abs(st.m) + 1.0
        st.S[:] = np.abs(st.S) + np.eye(d)
        st.h[:] = -np.abs(st.h)
    kw = dict(gamma=np.array([0.9, 0.75]) if decay else None, normalize=normalize, eps=0.3)
    dq, dk, dv_, ds = oracle.backward(q, k, v, go, state_in=st, want_dstate=True, **kw)
    h = 1e-5
    tol = 1e-7 if normalize else 1e-9
    f = lambda: loss(q, k, v, go, st, **kw)
    for arr, grad in ((q, dq), (k, dk), (v, dv_)):
        for idx in [(0, 0, 0, 0), (0, 1, 3, 1), (0, 1, n - 1, dv - 1)]:
            assert abs(central(f, arr, idx, h) - grad[idx]) < tol * max(1.0, abs(grad[idx])), idx
    for name in ("S", "C", "m", "G", "h"):
        arr, grad = getattr(st, name), getattr(ds, name)
        for idx in np.ndindex(arr.shape):
            fd = central(f, arr, idx, h)
            assert abs(fd - grad[idx]) < tol * max(1.0, abs(grad[idx])), (name, idx, fd, grad[idx])
    if not normalize:  # m and h enter only the denominator
        assert not np.any(ds.m) and not np.any(ds.h)


@pytest.mark.parametrize("normalize", [False, True])
def test_equals_the_gradient_of_the_joined_sequence(normalize):
    """With the upstream gradient zero on the first part, the gradients of the second
    part's tokens are those of the second part alone from the first part's state."""
    rng = np.random.default_rng(21)
    B, H, n, d, dv, cut = 1, 2, 20, 3, 4, 8
    q = np.abs(rng.standard_normal((B, H, n, d))) + 0.3
    k = np.abs(rng.standard_normal((B, H, n, d))) + 0.3
    v, go = rng.standard_normal((B, H, n, dv)), rng.standard_normal((B, H, n, dv))
    go[:, :, :cut] = 0.0
    kw = dict(gamma=np.array([0.95, 0.85]), normalize=normalize, eps=0.1)
    dq, dk, dv_ = oracle.backward(q, k, v, go, **kw)
    _, st1 = oracle.forward(q[:, :, :cut], k[:, :, :cut], v[:, :, :cut], **kw)
    dq2, dk2, dv2 = oracle.backward(q[:, :, cut:], k[:, :, cut:], v[:, :, cut:], go[:, :, cut:], state_in=st1, **kw)
    for a, b in ((dq2, dq[:, :, cut:]), (dk2, dk[:, :, cut:]), (dv2, dv_[:, :, cut:])):
        assert rel(a, b) < 1e-12


def test_no_tokens_gives_a_zero_state_gradient():
    rng = np.random.default_rng(31)
    st = rand_state(rng, 2, 3, 2)
    z = np.zeros((1, 2, 0, 3))
    dq, dk, dv_, ds = oracle.backward(z, z, np.zeros((1, 2, 0, 2)), np.zeros((1, 2, 0, 2)), state_in=st,
                                      want_dstate=True)
    for x in ds.astuple():
        assert not np.any(x)


def test_zero_state_matches_the_plain_backward():
    rng = np.random.default_rng(41)
    q, k = rng.standard_normal((2, 1, 2, 9, 3))
    v, go = rng.standard_normal((2, 1, 2, 9, 2))
    ref = oracle.backward(q, k, v, go, gamma=np.array([0.9, 1.0]))
    got = oracle.backward(q, k, v, go, gamma=np.array([0.9, 1.0]), state_in=oracle.State.zeros(2, 3, 2))
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)
