"""GPU parity of the backward pass: dq, dk, dv from the CUDA kernels (through the C
ABI) against the fp64 oracle's reverse-mode gradient on the same seeded inputs, plus
a directional-derivative check against the library's own forward.  Tolerance per
(b,h) relative L2: 1e-4 for fp32 inputs, 2e-2 for bf16 inputs and outputs."""
import numpy as np
import pytest
import torch

import causal_prefix_scan_gb300 as hla
import oracle
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import TOL_BF16, TOL_F32, per_pair_errors, to_dev

pytestmark = pytest.mark.gpu


def small(**kw):
    base = dict(B=1, H=2, n=256, d=64, dv=64, chunk=64, dtype="bf16", qk="l2", seed=31, gamma_lo=0.85,
                gamma_hi=0.999)
    base.update(kw)
    return W.Workload("bwd", **base)


def run_backward(x, g, dtype, chunk, eps=None):
    q, k, v = (to_dev(x[n], dtype) for n in ("q", "k", "v"))
    dout = to_dev(g, dtype)
    gam = None if x.get("gamma") is None else torch.from_numpy(np.asarray(x["gamma"], np.float32)).cuda()
    dq, dk, dv = hla.backward(q, k, v, dout, chunk=chunk, gamma=gam, normalize=eps is not None,
                              eps=0.0 if eps is None else eps)
    hla.hla_sync_status()
    return tuple(t.float().cpu().numpy() for t in (dq, dk, dv))


def run_oracle(x, g, eps=None):
    gam = None if x.get("gamma") is None else np.asarray(x["gamma"], np.float64)
    if eps is None:
        return oracle.backward(x["q"], x["k"], x["v"], g, gam)
    return oracle.backward(x["q"], x["k"], x["v"], g, gam, normalize=True, eps=eps)


def check(got, ref, tol, what):
    worst = 0.0
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        assert np.all(np.isfinite(a)), f"{what}: non-finite {name}"
        e = per_pair_errors(a, b).max()
        assert e <= tol, f"{what}: {name} max per-(b,h) rel L2 {e:.3e} > {tol}"
        worst = max(worst, float(e))
    return worst


@pytest.mark.parametrize("d,dv,chunk,n", [(16, 32, 16, 100), (32, 32, 32, 33), (64, 64, 64, 130),
                                          (64, 16, 16, 7), (16, 64, 64, 200), (32, 16, 32, 1), (64, 32, 32, 96)])
@pytest.mark.parametrize("decay", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_shapes(d, dv, chunk, n, decay, dtype):
    w = small(d=d, dv=dv, chunk=chunk, n=n, decay=decay, dtype=dtype)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    got = run_backward(x, g, dtype, chunk)
    check(got, run_oracle(x, g), TOL_F32 if dtype == "f32" else TOL_BF16,
          f"bwd {dtype} d{d} dv{dv} c{chunk} n{n} decay={decay}")


def test_backward_many_pairs_and_chunks():
    # several (b,h) pairs with distinct decay rates, many chunks, ragged tail
    w = small(B=2, H=3, n=16 * 21 + 5, d=32, dv=64, chunk=16, decay=True, dtype="f32")
    x = W.make_inputs(w)
    g = W.make_dout(w)
    check(run_backward(x, g, "f32", 16), run_oracle(x, g), TOL_F32, "bwd B2H3 many chunks")


def test_backward_chunk_lengths_agree():
    w = small(n=192, d=32, dv=32, dtype="f32", decay=True)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    res = [run_backward(x, g, "f32", c) for c in (16, 32, 64)]
    for other in res[1:]:
        for a, b in zip(res[0], other):
            assert per_pair_errors(a, b).max() <= 1e-5


def test_backward_is_gradient_of_forward():
    """<dq, e_q> + <dk, e_k> + <dv, e_v> equals the derivative in s of
    f(s) = sum(dout * forward(q + s e_q, k + s e_k, v + s e_v)), with the library's
    fp32 forward.  Along a line the output is a polynomial of degree 5 in s (q enters
    twice, k twice, v once), so the seven-point central difference, exact for degree
    <= 6, leaves only rounding error."""
    w = small(n=80, d=16, dv=16, chunk=16, dtype="f32", decay=True, qk="scaled")
    x = W.make_inputs(w)
    g = W.make_dout(w)
    rng = np.random.default_rng(5)
    dirs = [rng.standard_normal(x[n].shape).astype(np.float32) for n in ("q", "k", "v")]
    dq, dk, dv = run_backward(x, g, "f32", 16)
    want = sum(float(np.sum(a.astype(np.float64) * e)) for a, e in zip((dq, dk, dv), dirs))
    gam = torch.from_numpy(x["gamma"]).cuda()
    gd = to_dev(g, "f32").double()

    def f(s):
        q, k, v = (to_dev(x[n] + s * e, "f32") for n, e in zip(("q", "k", "v"), dirs))
        o = hla.forward(q, k, v, chunk=16, gamma=gam)
        hla.hla_sync_status()
        return float((o.double() * gd).sum())

    s = 0.1
    F = {j: f(j * s) for j in (-3, -2, -1, 1, 2, 3)}
    fd = (45 * (F[1] - F[-1]) - 9 * (F[2] - F[-2]) + (F[3] - F[-3])) / (60 * s)
    assert abs(fd - want) <= 1e-3 * abs(want), (fd, want)


def test_backward_empty_sequence():
    q = torch.empty((1, 2, 0, 32), device="cuda")
    v = torch.empty((1, 2, 0, 32), device="cuda")
    dq, dk, dv = hla.backward(q, q, v, v, chunk=32)
    hla.hla_sync_status()
    assert dq.shape == q.shape and dv.shape == v.shape


def test_backward_full_workload():
    w = W.BWD_BF16
    x = W.make_inputs(w)
    g = W.make_dout(w)
    err = check(run_backward(x, g, w.dtype, w.chunk), run_oracle(x, g), TOL_BF16, w.name)
    print(f"{w.name}: max per-(b,h) rel L2 {err:.3e}")


def test_backward_tensor_core_pairs_with_decay():
    """The tensor-core pipeline (bf16, d = dv = chunk = 64) over several pairs with
    distinct per-head decay rates and a ragged final chunk."""
    w = small(B=2, H=3, n=64 * 5 + 21, d=64, dv=64, chunk=64, decay=True, dtype="bf16", seed=37)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    check(run_backward(x, g, "bf16", 64), run_oracle(x, g), TOL_BF16, "bwd tc B2H3 decay")


@pytest.mark.parametrize("n", [1, 5, 64, 65])
def test_backward_tensor_core_short_sequences(n):
    w = small(n=n, d=64, dv=64, chunk=64, decay=True, dtype="bf16", seed=38)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    check(run_backward(x, g, "bf16", 64), run_oracle(x, g), TOL_BF16, f"bwd tc n{n}")


@pytest.mark.parametrize("n", [2, 5, 64, 65])
@pytest.mark.parametrize("Hkv", [2, 1])
def test_backward_normalised_tensor_core_short_sequences(n, Hkv):
    """The tensor-core normalised backward on sequences of one partial chunk, one full chunk
    and a chunk plus one token (the TMA tiles past the sequence read as zeros).  Not n = 1:
    a single token's normalised output is its own value up to eps, so dq and dk are
    O(eps) remainders of O(1) parts and no relative bound applies to them."""
    w = small(n=n, d=64, dv=64, chunk=64, decay=True, dtype="bf16", qk="elu1", Hkv=Hkv, seed=39)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    check(run_backward(x, g, "bf16", 64, eps=1e-3), run_oracle(x, g, eps=1e-3), TOL_BF16, f"bwd norm tc n{n} Hkv{Hkv}")


@pytest.mark.parametrize("d,dv,chunk,dtype", [(64, 64, 64, "bf16"), (32, 16, 32, "f32")])
@pytest.mark.parametrize("Hkv", [1, 2])
def test_backward_shared_kv_heads(d, dv, chunk, dtype, Hkv):
    """Keys and values shared by groups of query heads: dk, dv summed over each group."""
    w = small(B=2, H=4, Hkv=Hkv, n=2 * chunk + 9, d=d, dv=dv, chunk=chunk, decay=True, dtype=dtype, seed=39)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    check(run_backward(x, g, dtype, chunk), run_oracle(x, g), TOL_F32 if dtype == "f32" else TOL_BF16,
          f"bwd {dtype} H4 Hkv{Hkv}")


@pytest.mark.parametrize("d,dv,chunk,n,dtype", [(64, 64, 64, 64 * 3 + 17, "bf16"), (32, 16, 32, 100, "f32"),
                                                (16, 32, 16, 45, "bf16"), (64, 32, 64, 70, "f32")])
@pytest.mark.parametrize("decay", [False, True])
def test_backward_normalised(d, dv, chunk, n, dtype, decay):
    """Gradient through o = n / (den + eps) with positive features (den > 0)."""
    w = small(B=2, H=2, n=n, d=d, dv=dv, chunk=chunk, decay=decay, dtype=dtype, qk="elu1", seed=41)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    check(run_backward(x, g, dtype, chunk, eps=1e-3), run_oracle(x, g, eps=1e-3),
          TOL_F32 if dtype == "f32" else TOL_BF16, f"bwd norm {dtype} d{d} dv{dv} c{chunk} n{n} decay={decay}")


@pytest.mark.parametrize("d,dv,chunk,dtype", [(64, 64, 64, "bf16"), (32, 16, 32, "f32")])
def test_backward_normalised_shared_kv_heads(d, dv, chunk, dtype):
    w = small(B=1, H=4, Hkv=2, n=2 * chunk + 5, d=d, dv=dv, chunk=chunk, decay=True, dtype=dtype, qk="elu1",
              seed=42)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    check(run_backward(x, g, dtype, chunk, eps=0.5), run_oracle(x, g, eps=0.5),
          TOL_F32 if dtype == "f32" else TOL_BF16, f"bwd norm {dtype} H4 Hkv2")


@pytest.mark.parametrize("decay", [False, True])
@pytest.mark.parametrize("Hkv", [2, 1])
def test_backward_normalised_values_with_a_common_offset(decay, Hkv):
    """Values with a large common mean (3 + N(0,1)): every output is then close to every
    value, and the two parts of the gradient (through the values and through the
    denominator) are each 20-30 times their sum.  Rounding the upstream gradients or
    the outputs to bf16 alone costs ~5% here (fp64 check of the same case), so this
    holds the tensor-core path's mixed products to fp32-level accuracy."""
    w = small(B=1, H=2, Hkv=Hkv, n=64 * 4 + 9, decay=decay, qk="elu1", seed=45)
    x = W.make_inputs(w)
    x["v"] = W.round_bf16(x["v"] + np.float32(3.0))
    g = W.make_dout(w)
    err = check(run_backward(x, g, "bf16", 64, eps=1e-3), run_oracle(x, g, eps=1e-3), TOL_BF16,
                f"bwd norm offset values decay={decay} Hkv={Hkv}")
    print(f"offset values decay={decay} Hkv={Hkv}: max per-(b,h) rel L2 {err:.3e}")


@pytest.mark.parametrize("d,chunk,dtype", [(64, 64, "bf16"), (32, 32, "f32"), (64, 128, "bf16"), (16, 16, "bf16")])
@pytest.mark.parametrize("decay,normalize", [(False, False), (True, False), (False, True), (True, True)])
def test_backward_value_width_128(d, chunk, dtype, decay, normalize):
    """dv = 128 as two 64-column halves of the values (dq, dk summed in fp32, dv side by
    side; normalised, each half keeps the whole denominator), and a 128-token chunk as two
    of 64 tokens, against the oracle's gradient."""
    w = small(B=1, H=2, n=2 * 64 + 37, d=d, dv=128, chunk=chunk, decay=decay, dtype=dtype,
              qk="elu1" if normalize else "l2", seed=46)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    eps = 1e-3 if normalize else None
    check(run_backward(x, g, dtype, chunk, eps=eps), run_oracle(x, g, eps=eps), TOL_F32 if dtype == "f32" else TOL_BF16,
          f"bwd dv128 {dtype} d{d} c{chunk} decay={decay} norm={normalize}")


def test_backward_value_width_128_shared_heads_at_size():
    """The backward shape of the d = 64, dv = 128 forward workload (ratio-normalised, bf16)
    at 2048 tokens on four pairs, with two query heads per key/value head."""
    w = small(B=1, H=4, Hkv=2, n=2048, d=64, dv=128, chunk=64, dtype="bf16", qk="elu1", seed=47)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    err = check(run_backward(x, g, "bf16", 64, eps=1e-6), run_oracle(x, g, eps=1e-6), TOL_BF16, "bwd dv128 n2048")
    print(f"bwd dv128 n2048 Hkv2: max per-(b,h) rel L2 {err:.3e}")


@pytest.mark.parametrize("normalize", [False, True])
def test_backward_chunk_128_is_chunk_64(normalize):
    """The backward runs a 128-token chunk as two 64-token chunks: the same result, bit
    for bit."""
    w = small(B=1, H=2, n=300, qk="elu1" if normalize else "l2", decay=True, seed=48)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    eps = 1e-3 if normalize else None
    a = run_backward(x, g, "bf16", 128, eps=eps)
    b = run_backward(x, g, "bf16", 64, eps=eps)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_backward_normalised_is_gradient_of_forward():
    """The normalised backward against central differences of the library's own
    normalised fp32 forward along a random direction.  Along the line the output is a
    rational function of s; with directions of scale 0.1 the seven-point stencil's
    O(s^6) truncation error is below 1e-10 relative at s = 0.1 (fp64 check of the same
    case), so the fp32 rounding of the forward sets the tolerance."""
    w = small(n=70, d=16, dv=16, chunk=16, dtype="f32", decay=True, qk="elu1", seed=43)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    rng = np.random.default_rng(6)
    dirs = [0.1 * rng.standard_normal(x[n].shape).astype(np.float32) for n in ("q", "k", "v")]
    dq, dk, dv = run_backward(x, g, "f32", 16, eps=1e-3)
    want = sum(float(np.sum(a.astype(np.float64) * e)) for a, e in zip((dq, dk, dv), dirs))
    gam = torch.from_numpy(x["gamma"]).cuda()
    gd = to_dev(g, "f32").double()

    def f(s):
        q, k, v = (to_dev(x[n] + s * e, "f32") for n, e in zip(("q", "k", "v"), dirs))
        o = hla.forward(q, k, v, chunk=16, gamma=gam, normalize=True, eps=1e-3)
        hla.hla_sync_status()
        return float((o.double() * gd).sum())

    s = 0.1
    F = {j: f(j * s) for j in (-3, -2, -1, 1, 2, 3)}
    fd = (45 * (F[1] - F[-1]) - 9 * (F[2] - F[-2]) + (F[3] - F[-3])) / (60 * s)
    assert abs(fd - want) <= 2e-3 * abs(want), (fd, want)


@pytest.mark.parametrize("d,dv,chunk,n,dtype,decay", [(32, 16, 16, 256, "f32", True), (64, 64, 64, 1024, "bf16", True),
                                                      (16, 32, 16, 96, "f32", False), (64, 32, 32, 512, "bf16", False)])
def test_backward_normalised_segmented(d, dv, chunk, n, dtype, decay):
    """Long enough sequences that the fp32 forwards run as 4-16 segments per sequence
    (forward from zero, exclusive scan of the segment states, forward from the prefixes)."""
    w = small(B=1, H=2, n=n, d=d, dv=dv, chunk=chunk, decay=decay, dtype=dtype, qk="elu1", seed=44)
    x = W.make_inputs(w)
    g = W.make_dout(w)
    check(run_backward(x, g, dtype, chunk, eps=1e-3), run_oracle(x, g, eps=1e-3),
          TOL_F32 if dtype == "f32" else TOL_BF16, f"bwd norm segmented {dtype} d{d} dv{dv} c{chunk} n{n} decay={decay}")


def test_backward_normalised_full_workload():
    """The normalised backward at the size its bench leg times (B4 H8 n2048 d = dv = 64,
    bf16, 16 segments per sequence in the forwards), against the oracle's gradient."""
    w = W.BWD_NORM
    x = W.make_inputs(w)
    g = W.make_dout(w)
    err = check(run_backward(x, g, w.dtype, w.chunk, eps=w.eps), run_oracle(x, g, eps=w.eps), TOL_BF16, w.name)
    print(f"{w.name}: max per-(b,h) rel L2 {err:.3e}")
