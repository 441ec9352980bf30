"""GPU parity of the third-order forward with key/value heads shared by groups of query
heads (query head h reads key/value head h / (H / Hkv); the state, with its segment
maps, stays per query head): the tensor-core shape, the CUDA-core shapes, value halves
at dv = 128 and d = 128, plain, with decay and ratio-normalised.  Against the fp64
oracle; tolerance per (b,h) relative L2: 1e-4 for fp32, 2e-2 for bf16 outputs."""
import numpy as np
import pytest
import torch

import causal_prefix_scan_gb300 as hla
import oracle
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import TOL_BF16, TOL_F32, per_pair_errors, to_dev

pytestmark = pytest.mark.gpu


def case(d, dv, chunk, n, dtype, decay, normalize, Hkv, seed):
    w = W.Workload("kv3", B=2, H=4, n=n, d=d, dv=dv, chunk=chunk, dtype=dtype, qk="elu1" if normalize else "l2",
                   seed=seed, decay=decay, gamma_lo=0.8, gamma_hi=0.99, Hkv=Hkv)
    return w, W.make_inputs(w)


def gpu3(x, w, normalize, part=None, state_in=None, eps=1e-3):
    a, b = part if part else (0, w.n)
    q, k, v = (to_dev(np.ascontiguousarray(x[n][:, :, a:b]), w.dtype) for n in ("q", "k", "v"))
    g = None if x["gamma"] is None else torch.from_numpy(np.asarray(x["gamma"], np.float32)).cuda()
    o, st = hla.forward3(q, k, v, chunk=w.chunk, gamma=g, normalize=normalize, eps=eps, state_in=state_in,
                         return_state=True, maps=True)
    hla.hla_sync_status()
    return o.float().cpu().numpy(), st


def check(o, o_ref, st, st_ref, w, normalize, what):
    tol = TOL_F32 if w.dtype == "f32" else TOL_BF16
    e = per_pair_errors(o, o_ref).max()
    assert e <= tol, f"{what}: outputs {e:.3e}"
    units, d, dv = w.B * w.H, w.d, w.dv
    r = lambda n: np.asarray(st_ref[n])
    P, T, MQP = (r(n).reshape(units, d, -1) for n in ("P", "T", "MQP"))
    want = {"S": r("SK").reshape(units, d, d), "P": P[:, :, :dv], "T": T[:, :, :dv], "SQ": r("SQ").reshape(units, d, d),
            "MQP": MQP[:, :, :dv], "MKQ": r("MKQ").reshape(units, d, d)}
    if normalize:
        want.update(m=P[:, :, dv], h=T[:, :, dv], mqm=MQP[:, :, dv])
    for name, ref in want.items():
        got = getattr(st, name).double().cpu().numpy().reshape(units, 1, -1)
        e = per_pair_errors(got, ref.reshape(units, 1, -1)).max()
        assert e <= tol, f"{what}: {name} {e:.3e}"


# the tensor-core shape (bf16 64/64/64, no decay), CUDA-core shapes, dv = 128 halves, d = 128
@pytest.mark.parametrize("d,dv,chunk,dtype,decay", [(64, 64, 64, "bf16", False), (32, 16, 32, "f32", True),
                                                    (64, 128, 64, "bf16", False), (128, 32, 16, "f32", True),
                                                    (16, 64, 128, "f32", False)])
@pytest.mark.parametrize("Hkv", [2, 1])
@pytest.mark.parametrize("normalize", [False, True])
def test_forward3_shared_kv_heads(d, dv, chunk, dtype, decay, Hkv, normalize):
    w, x = case(d, dv, chunk, 2 * chunk + 19, dtype, decay, normalize, Hkv, seed=180 + d + dv)
    o, st = gpu3(x, w, normalize)
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"], chunk=16, gamma=x["gamma"], normalize=normalize,
                                    eps=1e-3)
    check(o, o_ref, st, st_ref, w, normalize, f"fwd3 H4 Hkv{Hkv} d{d} dv{dv} c{chunk} {dtype}")


def test_forward3_shared_kv_heads_resumed():
    w, x = case(32, 32, 32, 150, "f32", True, True, 2, seed=190)
    cut = 61
    _, s1 = gpu3(x, w, True, part=(0, cut))
    o2, s2 = gpu3(x, w, True, part=(cut, w.n), state_in=s1)
    o_ref, st_ref = oracle.forward3(x["q"], x["k"], x["v"], chunk=16, gamma=x["gamma"], normalize=True, eps=1e-3)
    check(o2, o_ref[:, :, cut:], s2, st_ref, w, True, "fwd3 shared heads resumed")
