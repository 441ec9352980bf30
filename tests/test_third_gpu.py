"""GPU parity of masked third-order HLA: the CUDA forward and decode step (through the
C ABI) against the fp64 oracle (hla_oracle3.c, serial recurrence in the moments and
cross summaries) on the same seeded inputs.  Tolerance per (b,h) relative L2: 1e-4 for
fp32 inputs, 2e-2 for bf16 inputs and outputs (fp32 state and arithmetic)."""
import numpy as np
import pytest
import torch

import causal_prefix_scan_gb300 as hla
import oracle
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import TOL_BF16, TOL_F32, per_pair_errors, to_dev

pytestmark = pytest.mark.gpu


def small(**kw):
    base = dict(B=1, H=2, n=256, d=64, dv=64, chunk=64, dtype="bf16", qk="l2", seed=41)
    base.update(kw)
    return W.Workload("fwd3", **base)


def state3_dev(st, units, d, dv):
    f = lambda a, s: torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.float32).reshape(s))).cuda()
    return hla.State3(f(st["SK"], (units, d, d)), f(st["P"], (units, d, dv)), f(st["T"], (units, d, dv)))


def run3(x, dtype, chunk, state_in=None):
    q, k, v = (to_dev(x[n], dtype) for n in ("q", "k", "v"))
    o, st = hla.forward3(q, k, v, chunk=chunk, state_in=state_in, return_state=True)
    hla.hla_sync_status()
    return o.float().cpu().numpy(), {n: getattr(st, n).double().cpu().numpy() for n in ("S", "P", "T")}


def check(o, st, o_ref, st_ref, tol, what):
    assert np.all(np.isfinite(o)), f"{what}: non-finite outputs"
    e = per_pair_errors(o, o_ref).max()
    assert e <= tol, f"{what}: output max per-(b,h) rel L2 {e:.3e} > {tol}"
    B, H = o_ref.shape[:2]
    for mine, theirs in (("S", "SK"), ("P", "P"), ("T", "T")):
        got = st[mine].reshape((B, H) + st[mine].shape[1:])
        ref = st_ref[theirs].reshape((B, H) + st_ref[theirs].shape[1:])
        es = per_pair_errors(got, ref).max()
        assert es <= tol, f"{what}: state {mine} max per-(b,h) rel L2 {es:.3e} > {tol}"
    return float(e)


@pytest.mark.parametrize("d,dv,chunk,n", [(16, 32, 16, 100), (32, 32, 32, 33), (64, 64, 64, 130), (64, 16, 16, 7),
                                          (16, 64, 64, 200), (32, 16, 32, 1), (64, 32, 32, 96)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_forward3_shapes(d, dv, chunk, n, dtype):
    w = small(d=d, dv=dv, chunk=chunk, n=n, dtype=dtype)
    x = W.make_inputs(w)
    o, st = run3(x, dtype, chunk)
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"])
    check(o, st, o_ref, st_ref, TOL_F32 if dtype == "f32" else TOL_BF16, f"fwd3 {dtype} d{d} dv{dv} c{chunk} n{n}")


def test_forward3_many_pairs_and_chunks():
    w = small(B=2, H=3, n=16 * 21 + 5, d=32, dv=64, chunk=16, dtype="f32", qk="scaled")
    x = W.make_inputs(w)
    o, st = run3(x, "f32", 16)
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"])
    check(o, st, o_ref, st_ref, TOL_F32, "fwd3 B2H3 many chunks")


def test_forward3_resume_from_state():
    w = small(n=300, d=32, dv=32, chunk=32, dtype="f32")
    x = W.make_inputs(w)
    cut = 137
    first = {n: x[n][:, :, :cut] for n in ("q", "k", "v")}
    second = {n: x[n][:, :, cut:] for n in ("q", "k", "v")}
    _, st1 = run3(first, "f32", 32)
    units = w.B * w.H
    sin = hla.State3(*(torch.from_numpy(st1[n].astype(np.float32)).cuda() for n in ("S", "P", "T")))
    o2, st2 = run3(second, "f32", 32, state_in=sin)
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"])
    check(o2, st2, o_ref[:, :, cut:], st_ref, TOL_F32, "fwd3 resume")
    # from the oracle's own state of the first part
    _, so1 = oracle.forward3(first["q"], first["k"], first["v"])
    o3, st3 = run3(second, "f32", 32, state_in=state3_dev(so1, units, w.d, w.dv))
    check(o3, st3, o_ref[:, :, cut:], st_ref, TOL_F32, "fwd3 resume from oracle state")


def test_forward3_chunk_lengths_agree():
    w = small(n=192, d=32, dv=32, dtype="f32", qk="scaled")
    x = W.make_inputs(w)
    res = [run3(x, "f32", c)[0] for c in (16, 32, 64)]
    for other in res[1:]:
        assert per_pair_errors(other, res[0]).max() <= 1e-5


def test_forward3_no_tokens_copies_state():
    units, d, dv = 2, 16, 16
    st_in = hla.State3(*(torch.randn(s, device="cuda") for s in ((units, d, d), (units, d, dv), (units, d, dv))))
    q = torch.empty((1, 2, 0, d), device="cuda")
    v = torch.empty((1, 2, 0, dv), device="cuda")
    o, st = hla.forward3(q, q, v, chunk=16, state_in=st_in, return_state=True)
    hla.hla_sync_status()
    for a, b in ((st.S, st_in.S), (st.P, st_in.P), (st.T, st_in.T)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("d,dv,dtype", [(16, 16, "f32"), (64, 64, "f32"), (64, 128, "bf16"), (128, 128, "bf16"),
                                        (128, 32, "f32")])
def test_decode3_continues_forward(d, dv, dtype):
    """Prefix through the oracle's state, then decode steps on the GPU; outputs against
    the oracle's serial recurrence over the joined sequence."""
    B, H, n0, steps = 2, 2, 40, 6
    w = small(B=B, H=H, n=n0 + steps, d=d, dv=dv, dtype=dtype, chunk=16, qk="l2")
    x = W.make_inputs(w)
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"])
    _, st0 = oracle.forward3(x["q"][:, :, :n0], x["k"][:, :, :n0], x["v"][:, :, :n0])
    units = B * H
    st = state3_dev(st0, units, d, dv)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    for s in range(steps):
        t = n0 + s
        q, k, v = (to_dev(np.ascontiguousarray(x[nm][:, :, t].reshape(units, -1)), dtype) for nm in ("q", "k", "v"))
        o = hla.decode3_step(st, q, k, v)
        hla.hla_sync_status()
        got = o.float().cpu().numpy().reshape(B, H, 1, dv)
        e = per_pair_errors(got, o_ref[:, :, t:t + 1]).max()
        assert e <= tol, f"decode3 step {s}: {e:.3e}"
    for mine, theirs in (("S", "SK"), ("P", "P"), ("T", "T")):
        got = getattr(st, mine).double().cpu().numpy()
        assert per_pair_errors(got[:, None], st_ref[theirs][:, None]).max() <= max(tol, 1e-5), mine


def test_forward3_full_workload():
    w = W.FWD3_BF16
    x = W.make_inputs(w)
    o, st = run3(x, w.dtype, w.chunk)
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"])
    err = check(o, st, o_ref, st_ref, TOL_BF16, w.name)
    print(f"{w.name}: max per-(b,h) rel L2 {err:.3e}")


def test_forward3_tensor_core_resume_and_pairs():
    """The tensor-core pipeline (bf16, d = dv = chunk = 64): several pairs, a split in the
    middle of a chunk, state_out of the first part fed back as state_in."""
    w = small(B=2, H=3, n=300, d=64, dv=64, chunk=64, dtype="bf16", seed=43)
    x = W.make_inputs(w)
    cut = 157
    first = {n: x[n][:, :, :cut] for n in ("q", "k", "v")}
    second = {n: x[n][:, :, cut:] for n in ("q", "k", "v")}
    o1, st1 = run3(first, "bf16", 64)
    sin = hla.State3(*(torch.from_numpy(st1[n].astype(np.float32)).cuda() for n in ("S", "P", "T")))
    o2, st2 = run3(second, "bf16", 64, state_in=sin)
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"])
    _, st1_ref = oracle.forward3(first["q"], first["k"], first["v"])
    check(o1, st1, o_ref[:, :, :cut], st1_ref, TOL_BF16, "fwd3 tc first part")
    check(o2, st2, o_ref[:, :, cut:], st_ref, TOL_BF16, "fwd3 tc resumed")


@pytest.mark.parametrize("n", [1, 5, 64, 65])
def test_forward3_tensor_core_short_sequences(n):
    w = small(n=n, d=64, dv=64, chunk=64, dtype="bf16", seed=44)
    x = W.make_inputs(w)
    o, st = run3(x, "bf16", 64)
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"])
    check(o, st, o_ref, st_ref, TOL_BF16, f"fwd3 tc n{n}")
