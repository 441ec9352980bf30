"""GPU parity of the third-order forward and concatenation at key width d = 128 (section 3
"Derde-orde HLA", section 4 "Derde-orde scans"): the CUDA-core kernels in 16-token chunks
over slices of at most 32 value columns (the output's column j and the state's P, T, M^QP
columns j depend on the values' column j only), the segment maps, and
hla_state3_combine's two-phase d = 128 kernel.  Against the fp64 oracle; tolerance per
(b,h) relative L2: 1e-4 for fp32, 2e-2 for bf16 outputs (the fp32 state and maps at 1e-4
with fp32 inputs)."""
import numpy as np
import pytest
import torch

import causal_prefix_scan_gb300 as hla
import oracle
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import TOL_BF16, TOL_F32, per_pair_errors, to_dev

pytestmark = pytest.mark.gpu


def case(dv, chunk, n, dtype, decay, normalize, seed, **kw):
    base = dict(B=1, H=2, n=n, d=128, dv=dv, chunk=chunk, dtype=dtype, qk="elu1" if normalize else "l2", seed=seed,
                decay=decay, gamma_lo=0.8, gamma_hi=0.99)
    base.update(kw)
    w = W.Workload("d128_3", **base)
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


def check_state(st, st_ref, w, normalize, tol, what):
    for name, want in expect(st_ref, w.B * w.H, w.d, w.dv, normalize).items():
        got = getattr(st, name).double().cpu().numpy().reshape(want.shape[0], 1, -1)
        e = per_pair_errors(got, want.reshape(want.shape[0], 1, -1)).max()
        assert e <= tol, f"{what}: {name} {e:.3e}"


def oracle3(x, normalize, n=None):
    sl = (lambda a: a[:, :, :n]) if n else (lambda a: a)
    return oracle.forward3(sl(x["q"]), sl(x["k"]), sl(x["v"]), chunk=16, gamma=x["gamma"], normalize=normalize,
                           eps=1e-3)


@pytest.mark.parametrize("dv,chunk,n", [(16, 16, 70), (32, 64, 53), (64, 128, 90), (128, 64, 41)])
@pytest.mark.parametrize("decay,normalize", [(False, False), (True, False), (False, True), (True, True)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_forward3_key_width_128(dv, chunk, n, decay, normalize, dtype):
    w, x = case(dv, chunk, n, dtype, decay, normalize, seed=151 + n)
    o, st = gpu3(x, w, normalize)
    o_ref, st_ref = oracle3(x, normalize)
    e = per_pair_errors(o, o_ref).max()
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    assert e <= tol, f"fwd3 d128 dv{dv} {dtype}: outputs {e:.3e}"
    check_state(st, st_ref, w, normalize, TOL_F32 if dtype == "f32" else TOL_BF16, f"fwd3 d128 dv{dv} {dtype}")


@pytest.mark.parametrize("dv", [32, 128])
def test_forward3_key_width_128_resumed(dv):
    """Continued from the state (with its maps) that a first part left."""
    w, x = case(dv, 32, 120, "f32", True, True, seed=160)
    cut = 45
    _, s1 = gpu3(x, w, True, part=(0, cut))
    o2, s2 = gpu3(x, w, True, part=(cut, w.n), state_in=s1)
    o_ref, st_ref = oracle3(x, True)
    assert per_pair_errors(o2, o_ref[:, :, cut:]).max() <= TOL_F32
    check_state(s2, st_ref, w, True, TOL_F32, f"fwd3 d128 dv{dv} resumed")


def test_forward3_key_width_128_chunk_lengths_agree():
    """Every chunk length runs as 16-token chunks: outputs and state bit for bit."""
    w, x = case(64, 16, 77, "bf16", True, False, seed=161)
    res = []
    for c in (16, 32, 64, 128):
        wc = W.Workload("d128_3", B=1, H=2, n=77, d=128, dv=64, chunk=c, dtype="bf16", qk="l2", seed=161,
                        decay=True, gamma_lo=0.8, gamma_hi=0.99)
        res.append(gpu3(x, wc, False))
    for o, st in res[1:]:
        assert np.array_equal(o, res[0][0])
        for name in ("S", "P", "T"):
            assert torch.equal(getattr(st, name), getattr(res[0][1], name)), name


@pytest.mark.parametrize("dv", [16, 32, 64, 128])
@pytest.mark.parametrize("normalize", [False, True])
def test_concatenation_at_key_width_128(dv, normalize):
    """Two segments summarised independently (with their maps) and concatenated on the
    GPU equal the summary of the joined sequence; also in place (out = A, out = B)."""
    w, x = case(dv, 16, 100, "f32", True, normalize, seed=170 + dv)
    cut = 37
    units = w.B * w.H
    g = np.asarray(x["gamma"], np.float64)
    fpow = torch.from_numpy((g[np.arange(units) % w.H] ** (w.n - cut)).astype(np.float32)).cuda()
    _, st_ref = oracle3(x, normalize)
    for where in ("new", "A", "B"):
        _, A = gpu3(x, w, normalize, part=(0, cut))
        _, Bs = gpu3(x, w, normalize, part=(cut, w.n))
        out = {"new": None, "A": A, "B": Bs}[where]
        AB = hla.state3_combine(A, Bs, decay_pow=fpow, normalize=normalize, out=out)
        hla.hla_sync_status()
        check_state(AB, st_ref, w, normalize, TOL_F32, f"combine d128 dv{dv} into {where}")


@pytest.mark.parametrize("n", [1, 15, 16, 17])
def test_forward3_key_width_128_short_sequences(n):
    """One token, shorter than the 16-token inner chunk, exactly one and one token more."""
    w, x = case(64, 64, n, "f32", True, True, seed=260 + n)
    o, st = gpu3(x, w, True)
    o_ref, st_ref = oracle3(x, True)
    assert per_pair_errors(o, o_ref).max() <= TOL_F32
    check_state(st, st_ref, w, True, TOL_F32, f"fwd3 d128 n{n}")
