"""GPU parity of the third-order forward at dv = 128 and with 128-token chunks (section 4,
"Derde-orde scans"): dv = 128 runs as two 64-column halves of the values (the output's
column j and the state's P, T, M^QP columns j depend on the values' column j only), a
128-token chunk as two of 64 tokens.  Outputs, the state and the segment maps against
the fp64 oracle; tolerance per (b,h) relative L2: 1e-4 for fp32, 2e-2 for bf16."""
import numpy as np
import pytest
import torch

import causal_prefix_scan_gb300 as hla
import oracle
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import TOL_BF16, TOL_F32, per_pair_errors, to_dev

pytestmark = pytest.mark.gpu


def case(d, chunk, n, dtype, decay, normalize, seed):
    w = W.Workload("wide3", B=1, H=2, n=n, d=d, dv=128, chunk=chunk, dtype=dtype,
                   qk="elu1" if normalize else "l2", seed=seed, decay=decay, gamma_lo=0.8, gamma_hi=0.99)
    return w, W.make_inputs(w)


def gpu3(x, w, normalize, part=None, state_in=None, eps=1e-3):
    a, b = part if part else (0, w.n)
    q, k, v = (to_dev(np.ascontiguousarray(x[n][:, :, a:b]), w.dtype) for n in ("q", "k", "v"))
    g = None if x["gamma"] is None else torch.from_numpy(np.asarray(x["gamma"], np.float32)).cuda()
    o, st = hla.forward3(q, k, v, chunk=w.chunk, gamma=g, normalize=normalize, eps=eps, state_in=state_in,
                         return_state=True, maps=True)
    hla.hla_sync_status()
    return o.float().cpu().numpy(), st


def expect(st_ref, units, d, dv, normalize):
    r = lambda n: np.asarray(st_ref[n])
    P, T, MQP = (r(n).reshape(units, d, -1) for n in ("P", "T", "MQP"))
    out = {"S": r("SK").reshape(units, d, d), "P": P[:, :, :dv], "T": T[:, :, :dv], "SQ": r("SQ").reshape(units, d, d),
           "MQP": MQP[:, :, :dv], "MKQ": r("MKQ").reshape(units, d, d)}
    if normalize:
        out.update(m=P[:, :, dv], h=T[:, :, dv], mqm=MQP[:, :, dv])
    return out


def check(o, o_ref, st, st_ref, w, normalize, tol, what):
    e = per_pair_errors(o, o_ref).max()
    assert e <= tol, f"{what}: outputs {e:.3e}"
    for name, want in expect(st_ref, w.B * w.H, w.d, 128, normalize).items():
        got = getattr(st, name).double().cpu().numpy().reshape(want.shape[0], 1, -1)
        e = per_pair_errors(got, want.reshape(want.shape[0], 1, -1)).max()
        assert e <= TOL_F32 if w.dtype == "f32" else e <= tol, f"{what}: {name} {e:.3e}"


@pytest.mark.parametrize("d,chunk,dtype", [(64, 64, "bf16"), (32, 32, "f32"), (64, 128, "bf16"), (16, 16, "f32")])
@pytest.mark.parametrize("decay,normalize", [(False, False), (True, False), (False, True), (True, True)])
def test_forward3_value_width_128(d, chunk, dtype, decay, normalize):
    w, x = case(d, chunk, 2 * 64 + 29, dtype, decay, normalize, 91)
    o, st = gpu3(x, w, normalize)
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"], chunk=16, gamma=x["gamma"], normalize=normalize, eps=1e-3)
    check(o, o_ref, st, st_ref, w, normalize, TOL_F32 if dtype == "f32" else TOL_BF16,
          f"fwd3 dv128 {dtype} d{d} c{chunk} decay={decay} norm={normalize}")


@pytest.mark.parametrize("normalize", [False, True])
def test_forward3_value_width_128_resumed(normalize):
    """A forward continued from the state (with its maps) that the first part left:
    state_in's value-column halves are gathered for each half problem."""
    w, x = case(32, 32, 170, "f32", True, normalize, 92)
    cut = 77
    _, s1 = gpu3(x, w, normalize, part=(0, cut))
    o2, s2 = gpu3(x, w, normalize, part=(cut, w.n), state_in=s1)
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"], chunk=16, gamma=x["gamma"], normalize=normalize, eps=1e-3)
    check(o2, o_ref[:, :, cut:], s2, st_ref, w, normalize, TOL_F32, "fwd3 dv128 resumed")


def test_forward3_chunk_128_is_chunk_64():
    """A 128-token chunk runs as two of 64 tokens: outputs and state bit for bit, the
    segment maps up to the order of their atomic sums."""
    w, x = case(64, 128, 300, "bf16", True, True, 93)
    o128, s128 = gpu3(x, w, True)
    w64 = W.Workload("wide3", B=1, H=2, n=300, d=64, dv=128, chunk=64, dtype="bf16", qk="elu1", seed=93, decay=True,
                     gamma_lo=0.8, gamma_hi=0.99)
    o64, s64 = gpu3(x, w64, True)
    assert np.array_equal(o128, o64)
    for name in ("S", "P", "T", "m", "h"):
        assert torch.equal(getattr(s128, name), getattr(s64, name)), name
    # the maps sum the chunks' parts with atomic adds, in no fixed order
    for name in ("SQ", "MQP", "MKQ", "mqm"):
        a, b = getattr(s128, name).double(), getattr(s64, name).double()
        assert float((a - b).norm() / b.norm()) < 1e-6, name


@pytest.mark.parametrize("normalize", [False, True])
def test_concatenation_at_value_width_128(normalize):
    """Two dv = 128 segments summarised independently (with their maps) and concatenated on
    the GPU equal the summary of the joined sequence."""
    w, x = case(32, 32, 190, "f32", True, normalize, 94)
    cut = 83
    _, A = gpu3(x, w, normalize, part=(0, cut))
    _, Bs = gpu3(x, w, normalize, part=(cut, w.n))
    units = w.B * w.H
    g = np.asarray(x["gamma"], np.float64)
    fpow = torch.from_numpy((g[np.arange(units) % w.H] ** (w.n - cut)).astype(np.float32)).cuda()
    AB = hla.state3_combine(A, Bs, decay_pow=fpow, normalize=normalize)
    hla.hla_sync_status()
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"], chunk=16, gamma=x["gamma"], normalize=normalize, eps=1e-3)
    for name, want in expect(st_ref, units, w.d, 128, normalize).items():
        got = getattr(AB, name).double().cpu().numpy().reshape(want.shape[0], 1, -1)
        e = per_pair_errors(got, want.reshape(want.shape[0], 1, -1)).max()
        assert e <= TOL_F32, f"combine dv128: {name} {e:.3e}"
