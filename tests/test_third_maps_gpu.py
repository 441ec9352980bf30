"""GPU parity of the third-order segment maps and concatenation (section 4, "Derde-orde
scans"): the maps S^Q, M^QP, M^KQ (and mqm, the M^QP of a unit value) that the forward
writes with its state, and hla_state3_combine, against the fp64 oracle's chunked scan
(whose state carries the same maps) and its concatenation rule.  Tolerance per (b,h)
relative L2: 1e-4 (fp32 inputs and state)."""
import numpy as np
import pytest
import torch

import causal_prefix_scan_gb300 as hla
import oracle
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import TOL_F32, per_pair_errors, to_dev

pytestmark = pytest.mark.gpu


def small(**kw):
    base = dict(B=1, H=3, n=170, d=32, dv=16, chunk=32, dtype="f32", qk="l2", seed=81, decay=True,
                gamma_lo=0.8, gamma_hi=0.99)
    base.update(kw)
    return W.Workload("maps3", **base)


def gamma_dev(g):
    return None if g is None else torch.from_numpy(np.asarray(g, np.float32)).cuda()


def gpu3(x, w, normalize, state_in=None, eps=1e-3):
    q, k, v = (to_dev(x[n], "f32") for n in ("q", "k", "v"))
    o, st = hla.forward3(q, k, v, chunk=w.chunk, gamma=gamma_dev(x["gamma"]), normalize=normalize, eps=eps,
                         state_in=state_in, return_state=True, maps=True)
    hla.hla_sync_status()
    return o.float().cpu().numpy(), st


def expect(st_ref, units, d, dv, normalize):
    """The oracle's state (value columns; the unit column when normalising) per field."""
    r = lambda n: np.asarray(st_ref[n])
    P, T, MQP = (r(n).reshape(units, d, -1) for n in ("P", "T", "MQP"))
    out = {"S": r("SK").reshape(units, d, d), "P": P[:, :, :dv], "T": T[:, :, :dv], "SQ": r("SQ").reshape(units, d, d),
           "MQP": MQP[:, :, :dv], "MKQ": r("MKQ").reshape(units, d, d)}
    if normalize:
        out.update(m=P[:, :, dv], h=T[:, :, dv], mqm=MQP[:, :, dv])
    return out


def check_state(st, ref, what):
    for name, want in ref.items():
        got = getattr(st, name).double().cpu().numpy().reshape(want.shape[0], 1, -1)
        e = per_pair_errors(got, want.reshape(want.shape[0], 1, -1)).max()
        assert e <= TOL_F32, f"{what}: {name} max per-(b,h) rel L2 {e:.3e}"


@pytest.mark.parametrize("d,dv,chunk,n", [(16, 32, 16, 100), (32, 16, 32, 170), (64, 64, 64, 130), (32, 32, 16, 33)])
@pytest.mark.parametrize("decay", [False, True])
@pytest.mark.parametrize("normalize", [False, True])
def test_forward3_writes_the_segment_maps(d, dv, chunk, n, decay, normalize):
    w = small(d=d, dv=dv, chunk=chunk, n=n, decay=decay, qk="elu1" if normalize else "l2")
    x = W.make_inputs(w)
    o, st = gpu3(x, w, normalize)
    _, st_ref = oracle.forward3(x["q"], x["k"], x["v"], chunk=chunk, gamma=x["gamma"], normalize=normalize,
                                eps=1e-3)
    check_state(st, expect(st_ref, w.B * w.H, d, dv, normalize), f"fwd3 maps d{d} dv{dv} c{chunk}")


@pytest.mark.parametrize("normalize", [False, True])
def test_concatenation_of_two_forwards(normalize):
    """Two segments summarised independently from zero, concatenated on the GPU (decay
    factor gamma^(tokens of the second)), equal the summary of the joined sequence; a
    third part continued from the concatenation gives the joined sequence's outputs."""
    w = small(n=260, qk="elu1" if normalize else "l2", seed=82)
    x = W.make_inputs(w)
    cut1, cut2 = 97, 201
    part = lambda a, b: {n: np.ascontiguousarray(x[n][:, :, a:b]) for n in ("q", "k", "v")} | {"gamma": x["gamma"]}
    _, A = gpu3(part(0, cut1), w, normalize)
    _, Bs = gpu3(part(cut1, cut2), w, normalize)
    units = w.B * w.H
    g = np.asarray(x["gamma"], np.float64)
    fpow = torch.from_numpy((g[np.arange(units) % w.H] ** (cut2 - cut1)).astype(np.float32)).cuda()
    AB = hla.state3_combine(A, Bs, decay_pow=fpow, normalize=normalize)
    hla.hla_sync_status()
    o_ref, st_ref = oracle.forward3(x["q"][:, :, :cut2], x["k"][:, :, :cut2], x["v"][:, :, :cut2], chunk=16,
                                    gamma=x["gamma"], normalize=normalize, eps=1e-3)
    check_state(AB, expect(st_ref, units, w.d, w.dv, normalize), "combine")
    # in place: out aliases A
    hla.state3_combine(A, Bs, decay_pow=fpow, normalize=normalize, out=A)
    hla.hla_sync_status()
    check_state(A, expect(st_ref, units, w.d, w.dv, normalize), "combine into A")
    # continue from the concatenation
    o3, _ = gpu3(part(cut2, w.n), w, normalize, state_in=AB)
    o_all, _ = oracle.forward3(x["q"], x["k"], x["v"], gamma=x["gamma"], normalize=normalize, eps=1e-3)
    e = per_pair_errors(o3, o_all[:, :, cut2:]).max()
    assert e <= TOL_F32, f"continued outputs: {e:.3e}"


def test_resumed_forward_composes_the_maps():
    w = small(n=150, seed=83)
    x = W.make_inputs(w)
    cut = 61
    first = {n: np.ascontiguousarray(x[n][:, :, :cut]) for n in ("q", "k", "v")} | {"gamma": x["gamma"]}
    second = {n: np.ascontiguousarray(x[n][:, :, cut:]) for n in ("q", "k", "v")} | {"gamma": x["gamma"]}
    _, s1 = gpu3(first, w, False)
    _, s2 = gpu3(second, w, False, state_in=s1)
    _, st_ref = oracle.forward3(x["q"], x["k"], x["v"], chunk=16, gamma=x["gamma"])
    check_state(s2, expect(st_ref, w.B * w.H, w.d, w.dv, False), "resumed maps")
