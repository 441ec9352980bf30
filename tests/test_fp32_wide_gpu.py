"""GPU parity of the CUDA-core forward at the widths the tensor-core kernels leave to it:
fp32 inputs at d, dv, chunk up to 128 (and bf16 shapes outside the tensor-core set),
and of the ratio-normalised backward at d = 128, whose fp32 chain runs that forward.
One CTA per pair keeps the pair's state in shared memory; where that leaves little room
a chunk runs as several shorter ones (the chunk length changes only the rounding).
Against the fp64 oracle (section 1 recurrence, "Normalisatie"); tolerance per (b,h)
relative L2: 1e-4 for fp32 inputs, 2e-2 for bf16 inputs and outputs."""
import numpy as np
import pytest
import torch

import causal_prefix_scan_gb300 as hla
import oracle
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import TOL_BF16, TOL_F32, assert_parity, per_pair_errors, run_forward, run_oracle, to_dev

pytestmark = pytest.mark.gpu


def wl(**kw):
    base = dict(B=1, H=2, n=150, d=128, dv=128, chunk=128, dtype="f32", qk="l2", seed=111, gamma_lo=0.85,
                gamma_hi=0.999)
    base.update(kw)
    return W.Workload("wide", **base)


# d = 128 at every value width (chunk caps 64, 32, 32, 8), dv = 128 at narrow keys,
# 128-token chunks at d <= 64 (run as 64)
@pytest.mark.parametrize("d,dv,chunk,n", [(128, 16, 64, 150), (128, 32, 128, 77), (128, 64, 64, 100),
                                          (128, 128, 128, 70), (64, 128, 128, 140), (16, 128, 32, 50),
                                          (32, 64, 128, 200)])
@pytest.mark.parametrize("decay,normalize", [(False, False), (True, True)])
def test_fp32_forward_wide(d, dv, chunk, n, decay, normalize):
    w = wl(d=d, dv=dv, chunk=chunk, n=n, decay=decay, qk="elu1" if normalize else "l2", seed=111 + n)
    x = W.make_inputs(w)
    o, st = run_forward(x, "f32", chunk, normalize=normalize, eps=1e-6)
    o_ref, st_ref = run_oracle(x, normalize=normalize, eps=1e-6)
    assert_parity(o, o_ref, st, st_ref, tol=TOL_F32, what=f"fp32 d{d} dv{dv} c{chunk} n{n}")


def test_fp32_forward_d128_resumed_and_shared_heads():
    """Keys and values shared by pairs of query heads, continued from the oracle's state
    of a first part."""
    w = wl(B=2, H=4, Hkv=2, n=190, dv=64, chunk=64, decay=True, seed=120)
    x = W.make_inputs(w)
    cut = 71
    first = {k: x[k][:, :, :cut] for k in ("q", "k", "v")} | {"gamma": x["gamma"]}
    second = {k: x[k][:, :, cut:] for k in ("q", "k", "v")} | {"gamma": x["gamma"]}
    _, st1 = run_oracle(first)
    o2, st2 = run_forward(second, "f32", 64, state_in=st1)
    o_ref, st_ref = run_oracle(x)
    assert_parity(o2, o_ref[:, :, cut:], st2, st_ref, tol=TOL_F32, what="fp32 d128 resumed, shared heads")


def test_fp32_chunk_128_is_chunk_64():
    """At d <= 64 a 128-token chunk runs as two of 64: the same result bit for bit."""
    w = wl(d=64, dv=64, chunk=128, n=300, decay=True, seed=121)
    x = W.make_inputs(w)
    a = run_forward(x, "f32", 128)
    b = run_forward(x, "f32", 64)
    assert np.array_equal(a[0], b[0])
    for name in ("S", "C", "m", "G", "h"):
        assert np.array_equal(getattr(a[1], name), getattr(b[1], name)), name


def test_bf16_outside_tensor_core_shapes():
    """bf16 at d = 128, dv = 32 (no tensor-core form): the CUDA-core kernel."""
    w = wl(dv=32, chunk=64, n=130, dtype="bf16", decay=True, seed=122)
    x = W.make_inputs(w)
    q = to_dev(x["q"], "bf16")
    v = to_dev(x["v"], "bf16")
    assert hla.hla_forward_kernel(hla.make_params(q, v, 64, torch.ones(2, device="cuda"))) == "fwd_simt_kernel"
    o, st = run_forward(x, "bf16", 64)
    o_ref, st_ref = run_oracle(x)
    assert_parity(o, o_ref, st, st_ref, tol=TOL_BF16, what="bf16 d128 dv32")


def bwd(w, x, g, eps):
    q, k, v = (to_dev(x[n], w.dtype) for n in ("q", "k", "v"))
    dout = to_dev(g, w.dtype)
    gam = None if x.get("gamma") is None else torch.from_numpy(np.asarray(x["gamma"], np.float32)).cuda()
    dq, dk, dv = hla.backward(q, k, v, dout, chunk=w.chunk, gamma=gam, normalize=True, eps=eps)
    hla.hla_sync_status()
    return tuple(t.float().cpu().numpy() for t in (dq, dk, dv))


@pytest.mark.parametrize("dv,chunk,n,dtype", [(32, 64, 90, "f32"), (128, 128, 70, "bf16"), (16, 16, 45, "f32"),
                                              (64, 32, 33, "bf16")])
@pytest.mark.parametrize("decay", [False, True])
def test_backward_normalised_key_width_128(dv, chunk, n, dtype, decay):
    """The normalised gradient at d = 128: the fp32 chain (two forwards, the upstream
    kernel, two backwards) on 16-token chunks over value slices of at most 32 columns."""
    w = wl(dv=dv, chunk=chunk, n=n, dtype=dtype, decay=decay, qk="elu1", seed=130 + n)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    got = bwd(w, x, g, 1e-3)
    gam = None if x.get("gamma") is None else np.asarray(x["gamma"], np.float64)
    ref = oracle.backward(x["q"], x["k"], x["v"], g, gam, normalize=True, eps=1e-3)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        assert np.all(np.isfinite(a)), name
        e = per_pair_errors(a, b).max()
        assert e <= tol, f"norm bwd d128 dv{dv} {dtype}: {name} {e:.3e}"


@pytest.mark.parametrize("n", [1, 5, 32, 33])
def test_fp32_forward_d128_short_sequences(n):
    """d = dv = 128 (8-token inner chunks) and d = 128, dv = 64 (32-token) on sequences of
    one token, shorter than a chunk, one chunk and one token more."""
    for dv in (128, 64):
        w = wl(dv=dv, chunk=64, n=n, decay=True, qk="elu1", seed=250 + n + dv)
        x = W.make_inputs(w)
        o, st = run_forward(x, "f32", 64, normalize=True, eps=1e-6)
        o_ref, st_ref = run_oracle(x, normalize=True, eps=1e-6)
        assert_parity(o, o_ref, st, st_ref, tol=TOL_F32, what=f"fp32 d128 dv{dv} n{n}")
