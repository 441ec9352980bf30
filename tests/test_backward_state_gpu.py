"""GPU parity of the backward pass from a given initial state, with the gradient of
that state (hla_backward_chunked_state, through the C ABI), against the fp64 oracle's
reverse-mode gradient on the same seeded inputs.  Tolerance per (b,h) relative L2:
1e-4 for fp32 inputs, 2e-2 for bf16 inputs and outputs (fp32 state)."""
import numpy as np
import pytest
import torch

import causal_prefix_scan_gb300 as hla
import oracle
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import TOL_BF16, TOL_F32, per_pair_errors, to_dev

pytestmark = pytest.mark.gpu


def small(**kw):
    base = dict(B=1, H=2, n=150, d=32, dv=32, chunk=32, dtype="f32", qk="l2", seed=61, gamma_lo=0.85,
                gamma_hi=0.999)
    base.update(kw)
    return W.Workload("bwdst", **base)


def rand_state(units, d, dv, seed, scale=0.3):
    """A state as a forward would leave it: symmetric positive S, the rest of the same scale."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((units, d, d)) * scale
    S = a @ a.transpose(0, 2, 1) / d + np.eye(d)
    return oracle.State(S, rng.standard_normal((units, d, dv)) * scale, rng.standard_normal((units, d)) * scale,
                        rng.standard_normal((units, d, dv)) * scale, rng.standard_normal((units, d)) * scale)


def state_dev(st):
    f = lambda a: torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.float32))).cuda()
    return hla.State(*(f(x) for x in st.astuple()))


def run(w, x, g, st, want=True):
    q, k, v = (to_dev(x[n], w.dtype) for n in ("q", "k", "v"))
    dout = to_dev(g, w.dtype)
    gam = None if x.get("gamma") is None else torch.from_numpy(np.asarray(x["gamma"], np.float32)).cuda()
    res = hla.backward(q, k, v, dout, chunk=w.chunk, gamma=gam, state_in=None if st is None else state_dev(st),
                       want_dstate=want)
    hla.hla_sync_status()
    grads = tuple(t.float().cpu().numpy() for t in res[:3])
    dst = res[3] if want else None
    return grads, dst


def check(w, x, g, st, tol, what):
    gam = None if x.get("gamma") is None else np.asarray(x["gamma"], np.float64)
    dq, dk, dv, ds = oracle.backward(x["q"], x["k"], x["v"], g, gam, state_in=st, want_dstate=True)
    (gq, gk, gv), gs = run(w, x, g, st)
    for name, a, b in (("dq", gq, dq), ("dk", gk, dk), ("dv", gv, dv)):
        assert np.all(np.isfinite(a)), f"{what}: non-finite {name}"
        e = per_pair_errors(a, b).max()
        assert e <= tol, f"{what}: {name} max per-(b,h) rel L2 {e:.3e} > {tol}"
    units = w.B * w.H
    for name in ("S", "C", "G"):
        a = getattr(gs, name).double().cpu().numpy().reshape(units, 1, -1)
        b = getattr(ds, name).reshape(units, 1, -1)
        e = per_pair_errors(a, b).max()
        assert e <= tol, f"{what}: d{name} max per-(b,h) rel L2 {e:.3e} > {tol}"
    for name in ("m", "h"):
        assert not torch.any(getattr(gs, name)), f"{what}: d{name} must be zero without normalisation"


@pytest.mark.parametrize("d,dv,chunk,n", [(16, 32, 16, 100), (32, 32, 32, 33), (64, 64, 64, 130), (64, 16, 16, 7),
                                          (32, 16, 32, 1)])
@pytest.mark.parametrize("decay", [False, True])
def test_backward_from_state_f32(d, dv, chunk, n, decay):
    w = small(d=d, dv=dv, chunk=chunk, n=n, decay=decay)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    st = rand_state(w.B * w.H, d, dv, seed=n + d)
    check(w, x, g, st, TOL_F32, f"f32 d{d} dv{dv} c{chunk} n{n} decay={decay}")


@pytest.mark.parametrize("decay", [False, True])
def test_backward_from_state_tensor_core_shape(decay):
    """bf16 at d = dv = chunk = 64: tensor-core local sums and gradients around the
    CUDA-core scan that starts from the given state."""
    w = small(B=2, H=2, n=300, d=64, dv=64, chunk=64, dtype="bf16", decay=decay, seed=62)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    st = rand_state(w.B * w.H, 64, 64, seed=7)
    check(w, x, g, st, TOL_BF16, f"bf16 64/64/64 decay={decay}")


def test_backward_from_state_shared_heads():
    w = small(B=1, H=4, Hkv=2, n=90, d=32, dv=16, chunk=16, decay=True, seed=63)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    st = rand_state(w.B * w.H, 32, 16, seed=8)
    check(w, x, g, st, TOL_F32, "shared key/value heads")


def test_state_gradient_from_a_zero_state():
    """No given state: the gradients of q, k, v are those of hla_backward_chunked and the
    state gradient still comes out (dC = 0, dS = g Om, dG = -g^2 Lam)."""
    w = small(n=77, decay=True, seed=64)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    check(w, x, g, None, TOL_F32, "zero state")
    (a, b, c), _ = run(w, x, g, None, want=False)
    q, k, v = (to_dev(x[n], w.dtype) for n in ("q", "k", "v"))
    gam = torch.from_numpy(np.asarray(x["gamma"], np.float32)).cuda()
    ref = hla.backward(q, k, v, to_dev(g, w.dtype), chunk=w.chunk, gamma=gam)
    hla.hla_sync_status()
    for mine, theirs in zip((a, b, c), ref):
        assert np.array_equal(mine, theirs.float().cpu().numpy())


def test_state_gradient_of_an_empty_sequence_is_zero():
    units, d, dv = 2, 16, 16
    st = state_dev(rand_state(units, d, dv, seed=9))
    z = torch.empty((1, 2, 0, d), device="cuda")
    zv = torch.empty((1, 2, 0, dv), device="cuda")
    dq, dk, dv_, ds = hla.backward(z, z, zv, zv, chunk=16, state_in=st, want_dstate=True)
    hla.hla_sync_status()
    for t in ds.astuple():
        assert not torch.any(t)


@pytest.mark.parametrize("dtype,d,dv,chunk", [("f32", 32, 16, 16), ("f32", 16, 32, 32), ("bf16", 64, 64, 64)])
@pytest.mark.parametrize("decay", [False, True])
def test_normalised_backward_from_state(dtype, d, dv, chunk, decay):
    """Ratio-normalised: the state a forward over a first part leaves (positive
    denominators with elu+1 features), then the gradient of the second part and of that
    state, all five arrays (m and h now carry the denominator's gradient)."""
    cut, eps = 70, 1e-3
    w = small(n=cut + 129, d=d, dv=dv, chunk=chunk, dtype=dtype, decay=decay, qk="elu1", seed=65)
    x = W.make_inputs(w)
    gam = None if x.get("gamma") is None else np.asarray(x["gamma"], np.float64)
    _, st = oracle.forward(x["q"][:, :, :cut], x["k"][:, :, :cut], x["v"][:, :, :cut], gamma=gam, normalize=True,
                           eps=eps)
    second = {n: np.ascontiguousarray(x[n][:, :, cut:]) for n in ("q", "k", "v")}
    second["gamma"] = x["gamma"]
    w2 = small(n=129, d=d, dv=dv, chunk=chunk, dtype=dtype, decay=decay, qk="elu1", seed=66)
    g = W.make_dout(w2)
    dq, dk, dv_, ds = oracle.backward(second["q"], second["k"], second["v"], g, gam, normalize=True, eps=eps,
                                      state_in=st, want_dstate=True)
    q, k, v = (to_dev(second[n], dtype) for n in ("q", "k", "v"))
    gd = None if gam is None else torch.from_numpy(np.asarray(gam, np.float32)).cuda()
    gq, gk, gv, gs = hla.backward(q, k, v, to_dev(g, dtype), chunk=chunk, gamma=gd, normalize=True, eps=eps,
                                  state_in=state_dev(st), want_dstate=True)
    hla.hla_sync_status()
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    for name, a, b in (("dq", gq, dq), ("dk", gk, dk), ("dv", gv, dv_)):
        e = per_pair_errors(a.float().cpu().numpy(), b).max()
        assert e <= tol, f"{name}: {e:.3e}"
    units = w.B * w.H
    for name in ("S", "C", "m", "G", "h"):
        a = getattr(gs, name).double().cpu().numpy().reshape(units, 1, -1)
        b = getattr(ds, name).reshape(units, 1, -1)
        e = per_pair_errors(a, b).max()
        assert e <= tol, f"d{name}: {e:.3e}"

