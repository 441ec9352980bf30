"""GPU parity of third-order HLA with exponential decay and ratio normalisation: the
CUDA forward and decode step (through the C ABI) against the fp64 oracle
(hla_oracle3.c) on the same seeded inputs.  Tolerance per (b,h) relative L2: 1e-4 for
fp32 inputs, 2e-2 for bf16 inputs (fp32 state and arithmetic)."""
import numpy as np
import pytest
import torch

import causal_prefix_scan_gb300 as hla
import oracle
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import TOL_BF16, TOL_F32, per_pair_errors, to_dev

pytestmark = pytest.mark.gpu


def small(**kw):
    base = dict(B=1, H=3, n=200, d=32, dv=32, chunk=32, dtype="f32", qk="l2", seed=51, decay=True,
                gamma_lo=0.75, gamma_hi=0.99)
    base.update(kw)
    return W.Workload("fwd3x", **base)


def gamma_dev(x):
    return None if x["gamma"] is None else torch.from_numpy(np.asarray(x["gamma"], np.float32)).cuda()


def state_dev(st, units, d, dv, normalize):
    """The oracle's state (value columns, then the unit column when normalising) as a State3."""
    f = lambda a: torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.float32))).cuda()
    P, T = np.asarray(st["P"]).reshape(units, d, -1), np.asarray(st["T"]).reshape(units, d, -1)
    s = hla.State3(f(np.asarray(st["SK"]).reshape(units, d, d)), f(P[:, :, :dv]), f(T[:, :, :dv]))
    if normalize:
        s.m, s.h = f(P[:, :, dv]), f(T[:, :, dv])
    return s


def run(x, w, normalize=False, eps=1e-6, state_in=None, chunk=None):
    q, k, v = (to_dev(x[n], w.dtype) for n in ("q", "k", "v"))
    o, st = hla.forward3(q, k, v, chunk=chunk or w.chunk, gamma=gamma_dev(x), normalize=normalize, eps=eps,
                         state_in=state_in, return_state=True)
    hla.hla_sync_status()
    return o.float().cpu().numpy(), st


def check(o, st, o_ref, st_ref, w, tol, what, normalize):
    assert np.all(np.isfinite(o)), f"{what}: non-finite outputs"
    e = per_pair_errors(o, o_ref).max()
    assert e <= tol, f"{what}: output max per-(b,h) rel L2 {e:.3e} > {tol}"
    units, d, dv = w.B * w.H, w.d, w.dv
    P, T = np.asarray(st_ref["P"]).reshape(units, d, -1), np.asarray(st_ref["T"]).reshape(units, d, -1)
    pairs = [("S", st.S, np.asarray(st_ref["SK"]).reshape(units, d, d)), ("P", st.P, P[:, :, :dv]),
             ("T", st.T, T[:, :, :dv])]
    if normalize:
        pairs += [("m", st.m, P[:, :, dv]), ("h", st.h, T[:, :, dv])]
    for name, got, ref in pairs:
        g = got.double().cpu().numpy().reshape(units, 1, -1)
        es = per_pair_errors(g, ref.reshape(units, 1, -1)).max()
        assert es <= tol, f"{what}: state {name} max per-(b,h) rel L2 {es:.3e} > {tol}"
    return float(e)


@pytest.mark.parametrize("d,dv,chunk,n", [(16, 32, 16, 100), (32, 32, 32, 33), (64, 64, 64, 130), (64, 16, 16, 7),
                                          (32, 64, 64, 1)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_forward3_decay(d, dv, chunk, n, dtype):
    w = small(d=d, dv=dv, chunk=chunk, n=n, dtype=dtype)
    x = W.make_inputs(w)
    o, st = run(x, w)
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"], gamma=x["gamma"])
    check(o, st, o_ref, st_ref, w, TOL_F32 if dtype == "f32" else TOL_BF16, f"fwd3 decay {dtype} d{d} dv{dv}", False)


@pytest.mark.parametrize("decay", [False, True])
@pytest.mark.parametrize("dtype,d,dv,chunk", [("f32", 32, 16, 16), ("bf16", 64, 64, 64), ("bf16", 16, 32, 32)])
def test_forward3_normalised(decay, dtype, d, dv, chunk):
    w = small(d=d, dv=dv, chunk=chunk, n=157, dtype=dtype, qk="elu1", decay=decay, seed=52)
    x = W.make_inputs(w)
    o, st = run(x, w, normalize=True, eps=1e-6)
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"], gamma=x["gamma"], normalize=True, eps=1e-6)
    check(o, st, o_ref, st_ref, w, TOL_F32 if dtype == "f32" else TOL_BF16, f"fwd3 norm {dtype} decay={decay}", True)


@pytest.mark.parametrize("normalize", [False, True])
def test_forward3_decay_resume(normalize):
    """state_out of the first part (a split inside a chunk) fed back as state_in, and the
    second part from the oracle's own state."""
    w = small(n=230, d=32, dv=16, chunk=32, qk="elu1" if normalize else "l2", seed=53)
    x = W.make_inputs(w)
    cut = 101
    first = {n: x[n][:, :, :cut] for n in ("q", "k", "v")}
    second = {n: x[n][:, :, cut:] for n in ("q", "k", "v")}
    first["gamma"] = second["gamma"] = x["gamma"]
    kw = dict(gamma=x["gamma"], normalize=normalize, eps=1e-3)
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"], **kw)
    _, st1 = run(first, w, normalize=normalize, eps=1e-3)
    o2, st2 = run(second, w, normalize=normalize, eps=1e-3, state_in=st1)
    check(o2, st2, o_ref[:, :, cut:], st_ref, w, TOL_F32, "fwd3 resume", normalize)
    _, so1 = oracle.forward3(first["q"], first["k"], first["v"], **kw)
    o3, st3 = run(second, w, normalize=normalize, eps=1e-3, state_in=state_dev(so1, w.B * w.H, w.d, w.dv, normalize))
    check(o3, st3, o_ref[:, :, cut:], st_ref, w, TOL_F32, "fwd3 resume from the oracle's state", normalize)


def test_forward3_decay_on_the_tensor_core_shape():
    """bf16 at d = dv = chunk = 64 runs the CUDA-core kernels when decay is on; the
    tensor-core result without decay stays as it was (gamma = 1 for every head gives the
    same numbers as no decay within the tolerance)."""
    w = small(B=2, H=2, n=300, d=64, dv=64, chunk=64, dtype="bf16", seed=54)
    x = W.make_inputs(w)
    o, st = run(x, w)
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"], gamma=x["gamma"])
    check(o, st, o_ref, st_ref, w, TOL_BF16, "fwd3 decay bf16 64/64/64", False)
    x1 = dict(x, gamma=np.ones_like(x["gamma"]))
    o1, _ = run(x1, w)
    o0, _ = run(dict(x, gamma=None), w)
    assert per_pair_errors(o1, o0).max() <= TOL_BF16


def test_forward3_normalised_no_tokens_copies_state():
    units, d, dv = 2, 16, 16
    z = lambda *s: torch.randn(*s, device="cuda")
    st_in = hla.State3(z(units, d, d), z(units, d, dv), z(units, d, dv), z(units, d), z(units, d))
    q = torch.empty((1, 2, 0, d), device="cuda")
    v = torch.empty((1, 2, 0, dv), device="cuda")
    o, st = hla.forward3(q, q, v, chunk=16, state_in=st_in, return_state=True, normalize=True, eps=0.1)
    hla.hla_sync_status()
    for a, b in ((st.S, st_in.S), (st.P, st_in.P), (st.T, st_in.T), (st.m, st_in.m), (st.h, st_in.h)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("normalize", [False, True])
@pytest.mark.parametrize("d,dv,dtype", [(16, 16, "f32"), (64, 128, "bf16"), (128, 32, "f32")])
def test_decode3_decay_continues_forward(normalize, d, dv, dtype):
    """Prefix through the oracle's state, then decode steps on the GPU; outputs against
    the oracle's serial recurrence over the joined sequence."""
    B, H, n0, steps = 2, 2, 40, 6
    w = small(B=B, H=H, n=n0 + steps, d=d, dv=dv, dtype=dtype, chunk=16, qk="elu1" if normalize else "l2",
              seed=55)
    x = W.make_inputs(w)
    kw = dict(gamma=x["gamma"], normalize=normalize, eps=1e-2)
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"], **kw)
    _, st0 = oracle.forward3(x["q"][:, :, :n0], x["k"][:, :, :n0], x["v"][:, :, :n0], **kw)
    units = B * H
    st = state_dev(st0, units, d, dv, normalize)
    g = gamma_dev(x)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    for s in range(steps):
        t = n0 + s
        q, k, v = (to_dev(np.ascontiguousarray(x[nm][:, :, t].reshape(units, -1)), dtype) for nm in ("q", "k", "v"))
        o = hla.decode3_step(st, q, k, v, H=H, gamma=g, normalize=normalize, eps=1e-2)
        hla.hla_sync_status()
        got = o.float().cpu().numpy().reshape(B, H, 1, dv)
        e = per_pair_errors(got, o_ref[:, :, t:t + 1]).max()
        assert e <= tol, f"decode3 step {s}: {e:.3e}"
    P, T = np.asarray(st_ref["P"]).reshape(units, d, -1), np.asarray(st_ref["T"]).reshape(units, d, -1)
    pairs = [(st.S, np.asarray(st_ref["SK"]).reshape(units, d, d)), (st.P, P[:, :, :dv]), (st.T, T[:, :, :dv])]
    if normalize:
        pairs += [(st.m, P[:, :, dv]), (st.h, T[:, :, dv])]
    for got, ref in pairs:
        gg = got.double().cpu().numpy().reshape(units, 1, -1)
        assert per_pair_errors(gg, ref.reshape(units, 1, -1)).max() <= max(tol, 1e-5)
