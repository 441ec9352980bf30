"""GPU parity of the backward pass at key width d = 128, the width of the decay workload
B1H32n32768d128 (section 4 motivates chunk-parallel training at the forward's shapes; the
gradient is reverse-mode differentiation of the section 1 recurrence).  The CUDA-core
kernels run it in 16-token chunks over slices of at most 32 value columns: the loss is a
sum over value columns and column j of the output depends on column j of the values
only, so dq and dk add over the slices and dv is the slices side by side.  Against the
fp64 oracle's gradient on the same seeded inputs; tolerance per (b,h) relative L2: 1e-4
for fp32 inputs, 2e-2 for bf16 inputs and outputs."""
import numpy as np
import pytest
import torch

import causal_prefix_scan_gb300 as hla
import oracle
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import TOL_BF16, TOL_F32, per_pair_errors, to_dev

pytestmark = pytest.mark.gpu


def case(dv, chunk, n, dtype, decay, seed, **kw):
    base = dict(B=1, H=2, n=n, d=128, dv=dv, chunk=chunk, dtype=dtype, qk="l2", seed=seed, decay=decay,
                gamma_lo=0.85, gamma_hi=0.999)
    base.update(kw)
    w = W.Workload("bwd128", **base)
    return w, W.make_inputs(w), W.make_dout(w)


def gamma_dev(x):
    return None if x.get("gamma") is None else torch.from_numpy(np.asarray(x["gamma"], np.float32)).cuda()


def gpu_grads(w, x, g, state_in=None, want_dstate=False):
    q, k, v = (to_dev(x[n], w.dtype) for n in ("q", "k", "v"))
    dout = to_dev(g, w.dtype)
    res = hla.backward(q, k, v, dout, chunk=w.chunk, gamma=gamma_dev(x), state_in=state_in, want_dstate=want_dstate)
    hla.hla_sync_status()
    grads = tuple(t.float().cpu().numpy() for t in res[:3])
    return (grads, res[3]) if want_dstate else grads


def check(got, ref, tol, what):
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        assert np.all(np.isfinite(a)), f"{what}: non-finite {name}"
        e = per_pair_errors(a, b).max()
        assert e <= tol, f"{what}: {name} max per-(b,h) rel L2 {e:.3e} > {tol}"


def oracle_grads(x, g, **kw):
    gam = None if x.get("gamma") is None else np.asarray(x["gamma"], np.float64)
    return oracle.backward(x["q"], x["k"], x["v"], g, gam, **kw)


# value widths 16 and 32 (one slice), 64 and 128 (two and four slices); every chunk length,
# ragged tails, a sequence shorter than one chunk
@pytest.mark.parametrize("dv,chunk,n", [(16, 16, 100), (32, 64, 77), (64, 128, 150), (128, 128, 129), (128, 32, 5)])
@pytest.mark.parametrize("decay", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_key_width_128(dv, chunk, n, decay, dtype):
    w, x, g = case(dv, chunk, n, dtype, decay, seed=41 + n)
    check(gpu_grads(w, x, g), oracle_grads(x, g), TOL_F32 if dtype == "f32" else TOL_BF16,
          f"bwd d128 {dtype} dv{dv} c{chunk} n{n} decay={decay}")


def test_backward_key_width_128_many_chunks():
    """63 chunks of 16 tokens per pair, distinct decay rates per head."""
    w, x, g = case(32, 64, 1000, "f32", True, seed=47, H=3)
    check(gpu_grads(w, x, g), oracle_grads(x, g), TOL_F32, "bwd d128 many chunks")


def test_backward_key_width_128_chunk_lengths_agree():
    """Every chunk length runs as 16-token chunks: the same gradient bit for bit."""
    w, x, g = case(64, 16, 140, "bf16", True, seed=48)
    res = []
    for c in (16, 32, 64, 128):
        wc = W.Workload("bwd128", B=1, H=2, n=140, d=128, dv=64, chunk=c, dtype="bf16", qk="l2", seed=48,
                        decay=True, gamma_lo=0.85, gamma_hi=0.999)
        res.append(gpu_grads(wc, x, g))
    for other in res[1:]:
        for a, b in zip(res[0], other):
            assert np.array_equal(a, b)


@pytest.mark.parametrize("dv", [32, 128])
def test_backward_key_width_128_shared_kv_heads(dv):
    """Four query heads on two key/value heads: dk, dv summed over each group."""
    w, x, g = case(dv, 64, 90, "bf16", True, seed=49, B=2, H=4, Hkv=2)
    check(gpu_grads(w, x, g), oracle_grads(x, g), TOL_BF16, f"bwd d128 dv{dv} shared heads")


@pytest.mark.parametrize("decay", [False, True])
def test_backward_key_width_128_from_state(decay):
    """dv = 32 (no split): the backward from a given state, with the state's gradient."""
    w, x, g = case(32, 16, 70, "f32", decay, seed=50)
    units, d, dv = w.B * w.H, 128, 32
    rng = np.random.default_rng(51)
    a = rng.standard_normal((units, d, d)) * 0.3
    st = oracle.State(a @ a.transpose(0, 2, 1) / d + np.eye(d), rng.standard_normal((units, d, dv)) * 0.3,
                      rng.standard_normal((units, d)) * 0.3, rng.standard_normal((units, d, dv)) * 0.3,
                      rng.standard_normal((units, d)) * 0.3)
    f = lambda z: torch.from_numpy(np.ascontiguousarray(np.asarray(z, np.float32))).cuda()
    grads, ds = gpu_grads(w, x, g, state_in=hla.State(*(f(z) for z in st.astuple())), want_dstate=True)
    dq, dk, dv_, ds_ref = oracle_grads(x, g, state_in=st, want_dstate=True)
    check(grads, (dq, dk, dv_), TOL_F32, "bwd d128 from state")
    for name in ("S", "C", "G"):
        got = getattr(ds, name).double().cpu().numpy().reshape(units, 1, -1)
        e = per_pair_errors(got, getattr(ds_ref, name).reshape(units, 1, -1)).max()
        assert e <= TOL_F32, f"d{name}: {e:.3e}"


def test_backward_key_width_128_empty_sequence():
    w, x, g = case(64, 64, 0, "bf16", False, seed=52)
    dq, dk, dv = gpu_grads(w, x, g)
    assert dq.shape == (1, 2, 0, 128) and dv.shape == (1, 2, 0, 64)


@pytest.mark.parametrize("n", [1, 15, 16, 17])
def test_backward_key_width_128_short_sequences(n):
    """One token, shorter than the 16-token inner chunk, exactly one and one token more."""
    w, x, g = case(64, 64, n, "f32", True, seed=270 + n)
    check(gpu_grads(w, x, g), oracle_grads(x, g), TOL_F32, f"bwd d128 n{n}")
