"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs.  Tolerance per (b,h) relative L2: 1e-4 for fp32 inputs,
2e-2 for bf16 inputs with fp32 state."""
import numpy as np
import pytest
import torch

import causal_prefix_scan_gb300 as hla
import oracle
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import (TOL_BF16, TOL_F32, assert_parity, per_pair_errors, rel_l2, run_forward, run_oracle,
                         state_errors, state_to_dev, state_to_np, to_dev)

pytestmark = pytest.mark.gpu


def small(name, **kw):
    base = dict(B=1, H=2, n=256, d=64, dv=64, chunk=64, dtype="bf16", qk="l2", seed=21)
    base.update(kw)
    return W.Workload(name, **base)


# ------------------------------------------------------------------ fp32 path
def test_small_f32_workload():
    w = W.SMALL_F32
    x = W.make_inputs(w)
    o, st = run_forward(x, "f32", w.chunk)
    o_ref, st_ref = run_oracle(x)
    assert_parity(o, o_ref, st, st_ref, tol=TOL_F32, what="fp32 B1H2n256d16")


@pytest.mark.parametrize("d,dv,chunk,n", [(16, 32, 16, 100), (32, 32, 32, 33), (64, 64, 64, 130), (64, 16, 16, 7)])
@pytest.mark.parametrize("decay,normalize", [(False, False), (True, True)])
def test_simt_shapes(d, dv, chunk, n, decay, normalize):
    for dtype in ("f32", "bf16"):
        w = small("simt", d=d, dv=dv, chunk=chunk, n=n, dtype=dtype, decay=decay, qk="elu1" if normalize else "l2")
        x = W.make_inputs(w)
        o, st = run_forward(x, dtype, chunk, normalize=normalize, eps=1e-6)
        o_ref, st_ref = run_oracle(x, normalize=normalize, eps=1e-6)
        assert_parity(o, o_ref, st, st_ref, tol=TOL_F32 if dtype == "f32" else TOL_BF16, what=f"simt {dtype}")


# ------------------------------------------------------------ tensor-core path
TC_SHAPES = [(64, 64, 64), (64, 64, 128), (128, 128, 128), (128, 64, 64), (64, 128, 128), (128, 128, 64)]


@pytest.mark.parametrize("chunk,d,dv", TC_SHAPES)
@pytest.mark.parametrize("decay,normalize", [(False, False), (False, True), (True, False), (True, True)])
def test_tc_variants(chunk, d, dv, decay, normalize):
    # few (b,h) pairs -> several segments per sequence; ragged final chunk
    n = 5 * chunk + 17
    w = small("tc", d=d, dv=dv, chunk=chunk, n=n, decay=decay, qk="elu1" if normalize else "l2",
              gamma_lo=0.9, gamma_hi=0.999)
    x = W.make_inputs(w)
    o, st = run_forward(x, "bf16", chunk, normalize=normalize, eps=1e-6)
    o_ref, st_ref = run_oracle(x, normalize=normalize, eps=1e-6)
    assert_parity(o, o_ref, st, st_ref, what=f"tc c{chunk} d{d} dv{dv} decay={decay} norm={normalize}")


@pytest.mark.parametrize("chunk,d,dv", [(64, 64, 64), (128, 128, 128), (64, 64, 128)])
def test_tc_state_in_resume(chunk, d, dv):
    w = small("resume", d=d, dv=dv, chunk=chunk, n=3 * chunk + 5, decay=True, B=2, H=2)
    x = W.make_inputs(w)
    n1 = 2 * chunk + 9
    x1 = {kk: (vv[:, :, :n1] if kk != "gamma" else vv) for kk, vv in x.items()}
    x2 = {kk: (vv[:, :, n1:] if kk != "gamma" else vv) for kk, vv in x.items()}
    _, st1_ref = run_oracle(x1)
    o2, st2 = run_forward(x2, "bf16", chunk, state_in=st1_ref)
    o2_ref, st2_ref = run_oracle(x2, state_in=st1_ref)
    assert_parity(o2, o2_ref, st2, st2_ref, what="resume from state_in")
    # the full run equals the split run
    o_full, _ = run_oracle(x)
    assert per_pair_errors(o2, o_full[:, :, n1:]).max() <= TOL_BF16


@pytest.mark.parametrize("n", [1, 2, 63, 64, 65])
def test_tc_short_sequences(n):
    w = small("short", n=n, B=3, H=1, decay=True)
    x = W.make_inputs(w)
    o, st = run_forward(x, "bf16", 64)
    o_ref, st_ref = run_oracle(x)
    assert_parity(o, o_ref, st, st_ref, what=f"n={n}")


def test_tc_many_pairs_single_segment():
    # B*H above the SM count: each CTA's run holds several whole sequences
    w = small("wide", B=20, H=10, n=150, d=64, dv=64)
    x = W.make_inputs(w)
    o, st = run_forward(x, "bf16", 64)
    o_ref, st_ref = run_oracle(x)
    assert_parity(o, o_ref, st, st_ref, what="B*H=200")


@pytest.mark.parametrize("B,H,n,chunk,d,dv,decay,normalize", [
    (1, 3, 8192, 64, 64, 128, False, True),    # long sequences; runs end inside sequences
    (2, 40, 200, 64, 64, 128, True, False),    # 4 chunks per sequence, runs of a few chunks
    (1, 400, 40, 64, 64, 64, True, True),      # one chunk per sequence: runs of several whole sequences
    (1, 7, 4990, 128, 128, 128, True, False),  # 39 chunks per sequence
])
def test_tc_runs_cross_sequences(B, H, n, chunk, d, dv, decay, normalize):
    # The chunks of all sequences, end to end, are split into equal runs, one per
    # CTA; with these sizes (and any SM count) some runs hold pieces of two or more
    # sequences, and some sequences start or end inside a run.
    w = small("runs", B=B, H=H, n=n, chunk=chunk, d=d, dv=dv, decay=decay, qk="elu1" if normalize else "l2",
              gamma_lo=0.9, gamma_hi=0.999)
    x = W.make_inputs(w)
    o, st = run_forward(x, "bf16", chunk, normalize=normalize, eps=1e-6)
    o_ref, st_ref = run_oracle(x, normalize=normalize, eps=1e-6)
    assert_parity(o, o_ref, st, st_ref, what=f"runs B{B}H{H}n{n}")


def test_empty_sequence_passes_state_through():
    w = small("empty", n=7)
    x = W.make_inputs(w)
    _, st_ref = run_oracle(x)
    x0 = {kk: (vv[:, :, :0] if kk != "gamma" else vv) for kk, vv in x.items()}
    o, st = run_forward(x0, "bf16", 64, state_in=st_ref)
    assert o.shape[2] == 0
    state_errors(st, st_ref, 1e-6, "empty sequence")


def test_tc_causality():
    w = small("causal", n=300, decay=True)
    x = W.make_inputs(w)
    o, _ = run_forward(x, "bf16", 64, return_state=False)
    t = 150
    y = {kk: (vv.copy() if kk != "gamma" else vv) for kk, vv in x.items()}
    for kk in ("q", "k", "v"):
        y[kk][:, :, t + 1:] = W.round_bf16(y[kk][:, :, t + 1:] * 2 + 0.5)
    o2, _ = run_forward(y, "bf16", 64, return_state=False)
    assert np.array_equal(o2[:, :, : t + 1], o[:, :, : t + 1])
    assert not np.allclose(o2[:, :, t + 1:], o[:, :, t + 1:])


def test_tc_deterministic():
    w = small("det", n=500, decay=True)
    x = W.make_inputs(w)
    a, sa = run_forward(x, "bf16", 64)
    b, sb = run_forward(x, "bf16", 64)
    assert np.array_equal(a, b)
    for p, q in zip(sa.astuple(), sb.astuple()):
        assert np.array_equal(p, q)


# ------------------------------------------- unmasked variant, shared key/value heads
@pytest.mark.parametrize("chunk,d,dv", TC_SHAPES)
@pytest.mark.parametrize("decay,normalize", [(False, False), (False, True), (True, False), (True, True)])
def test_tc_unmasked_variants(chunk, d, dv, decay, normalize):
    n = 5 * chunk + 17
    w = small("unm", d=d, dv=dv, chunk=chunk, n=n, decay=decay, qk="elu1" if normalize else "l2",
              gamma_lo=0.9, gamma_hi=0.999, seed=23)
    x = W.make_inputs(w)
    o, st = run_forward(x, "bf16", chunk, normalize=normalize, eps=1e-6, unmasked=True)
    o_ref, st_ref = run_oracle(x, normalize=normalize, eps=1e-6, unmasked=True)
    assert_parity(o, o_ref, st, st_ref, what=f"unmasked c{chunk} d{d} dv{dv} decay={decay} norm={normalize}")


@pytest.mark.parametrize("d,dv,chunk,n", [(16, 32, 16, 100), (64, 64, 64, 130), (32, 16, 32, 45)])
@pytest.mark.parametrize("decay,normalize", [(False, False), (True, True)])
def test_simt_unmasked(d, dv, chunk, n, decay, normalize):
    for dtype in ("f32", "bf16"):
        w = small("simt_unm", d=d, dv=dv, chunk=chunk, n=n, dtype=dtype, decay=decay,
                  qk="elu1" if normalize else "l2")
        x = W.make_inputs(w)
        o, st = run_forward(x, dtype, chunk, normalize=normalize, eps=1e-6, unmasked=True)
        o_ref, st_ref = run_oracle(x, normalize=normalize, eps=1e-6, unmasked=True)
        assert_parity(o, o_ref, st, st_ref, tol=TOL_F32 if dtype == "f32" else TOL_BF16, what=f"simt unm {dtype}")


@pytest.mark.parametrize("B,H,n,chunk,d,dv", [(1, 3, 8192, 64, 64, 128), (1, 400, 40, 64, 64, 64),
                                              (1, 7, 4990, 128, 128, 128)])
def test_tc_unmasked_runs_and_resume(B, H, n, chunk, d, dv):
    w = small("unm_runs", B=B, H=H, n=n, chunk=chunk, d=d, dv=dv, decay=True, qk="elu1", seed=24)
    x = W.make_inputs(w)
    o, st = run_forward(x, "bf16", chunk, normalize=True, eps=1e-6, unmasked=True)
    o_ref, st_ref = run_oracle(x, normalize=True, eps=1e-6, unmasked=True)
    assert_parity(o, o_ref, st, st_ref, what=f"unmasked runs B{B}H{H}n{n}")
    # resume from a state in the middle of the sequence
    n1 = (n // 3) + 5
    x1 = {kk: (vv[:, :, :n1] if kk != "gamma" else vv) for kk, vv in x.items()}
    x2 = {kk: (vv[:, :, n1:] if kk != "gamma" else vv) for kk, vv in x.items()}
    _, st1 = run_oracle(x1, normalize=True, eps=1e-6, unmasked=True)
    o2, st2 = run_forward(x2, "bf16", chunk, normalize=True, eps=1e-6, state_in=st1, unmasked=True)
    o2_ref, st2_ref = run_oracle(x2, normalize=True, eps=1e-6, state_in=st1, unmasked=True)
    assert_parity(o2, o2_ref, st2, st2_ref, what="unmasked resume")


@pytest.mark.parametrize("unmasked", [False, True])
@pytest.mark.parametrize("chunk,d,dv,dtype", [(64, 64, 64, "bf16"), (128, 128, 128, "bf16"), (64, 64, 128, "bf16"),
                                              (32, 32, 16, "f32")])
def test_shared_kv_heads(unmasked, chunk, d, dv, dtype):
    # 8 query heads reading 2 key/value heads; several pieces per sequence
    w = small("kv2", B=2, H=8, Hkv=2, n=6 * chunk + 9, chunk=chunk, d=d, dv=dv, dtype=dtype, decay=True,
              qk="elu1", seed=25)
    x = W.make_inputs(w)
    assert x["k"].shape[1] == 2 and x["v"].shape[1] == 2
    o, st = run_forward(x, dtype, chunk, normalize=True, eps=1e-6, unmasked=unmasked)
    o_ref, st_ref = run_oracle(x, normalize=True, eps=1e-6, unmasked=unmasked)
    assert_parity(o, o_ref, st, st_ref, tol=TOL_F32 if dtype == "f32" else TOL_BF16,
                  what=f"shared kv unmasked={unmasked} c{chunk} d{d} dv{dv}")


# ------------------------------------------------------- asymmetric variant (AHLA)
@pytest.mark.parametrize("d,dv,chunk,n", [(16, 32, 16, 100), (64, 64, 64, 130), (32, 16, 32, 45), (64, 32, 64, 200)])
@pytest.mark.parametrize("decay,normalize", [(False, False), (True, False), (True, True)])
def test_asym_forward(d, dv, chunk, n, decay, normalize):
    for dtype in ("f32", "bf16"):
        w = small("asym", d=d, dv=dv, chunk=chunk, n=n, dtype=dtype, decay=decay,
                  qk="elu1" if normalize else "l2", seed=27)
        x = W.make_inputs(w)
        o, st = run_forward(x, dtype, chunk, normalize=normalize, eps=1e-6, asymmetric=True)
        o_ref, st_ref = run_oracle(x, normalize=normalize, eps=1e-6, asymmetric=True)
        assert_parity(o, o_ref, st, st_ref, tol=TOL_F32 if dtype == "f32" else TOL_BF16,
                      what=f"asym {dtype} d{d} dv{dv}", asymmetric=True)


TC_SHAPES_ASYM = [sh for sh in TC_SHAPES if sh[2] <= sh[1]]  # (chunk, d, dv) with dv <= d


@pytest.mark.parametrize("chunk,d,dv", TC_SHAPES_ASYM)
@pytest.mark.parametrize("decay,normalize", [(False, False), (False, True), (True, False), (True, True)])
def test_tc_asym_variants(chunk, d, dv, decay, normalize):
    n = 5 * chunk + 17
    w = small("asym_tc", d=d, dv=dv, chunk=chunk, n=n, decay=decay, qk="elu1" if normalize else "l2",
              gamma_lo=0.9, gamma_hi=0.999, seed=29)
    x = W.make_inputs(w)
    o, st = run_forward(x, "bf16", chunk, normalize=normalize, eps=1e-6, asymmetric=True)
    o_ref, st_ref = run_oracle(x, normalize=normalize, eps=1e-6, asymmetric=True)
    assert_parity(o, o_ref, st, st_ref, what=f"asym tc c{chunk} d{d} dv{dv} decay={decay} norm={normalize}",
                  asymmetric=True)


@pytest.mark.parametrize("B,H,Hkv,n,chunk,d,dv", [(1, 3, 3, 8192, 64, 64, 64), (1, 400, 400, 40, 64, 64, 64),
                                                  (1, 8, 2, 4990, 128, 128, 128)])
def test_tc_asym_runs_resume_shared_kv(B, H, Hkv, n, chunk, d, dv):
    w = small("asym_runs", B=B, H=H, Hkv=Hkv, n=n, chunk=chunk, d=d, dv=dv, decay=True, qk="elu1", seed=30)
    x = W.make_inputs(w)
    o, st = run_forward(x, "bf16", chunk, normalize=True, eps=1e-6, asymmetric=True)
    o_ref, st_ref = run_oracle(x, normalize=True, eps=1e-6, asymmetric=True)
    assert_parity(o, o_ref, st, st_ref, what=f"asym runs B{B}H{H}n{n}", asymmetric=True)
    n1 = n // 3 + 5
    x1 = {kk: (vv[:, :, :n1] if kk != "gamma" else vv) for kk, vv in x.items()}
    x2 = {kk: (vv[:, :, n1:] if kk != "gamma" else vv) for kk, vv in x.items()}
    _, st1 = run_oracle(x1, normalize=True, eps=1e-6, asymmetric=True)
    o2, st2 = run_forward(x2, "bf16", chunk, normalize=True, eps=1e-6, state_in=st1, asymmetric=True)
    o2_ref, st2_ref = run_oracle(x2, normalize=True, eps=1e-6, state_in=st1, asymmetric=True)
    assert_parity(o2, o2_ref, st2, st2_ref, what="asym resume", asymmetric=True)


def test_asym_resume_and_shared_kv():
    w = small("asym_kv", B=2, H=4, Hkv=2, n=300, d=64, dv=64, chunk=64, dtype="f32", decay=True, qk="elu1",
              seed=28)
    x = W.make_inputs(w)
    n1 = 117
    x1 = {kk: (vv[:, :, :n1] if kk != "gamma" else vv) for kk, vv in x.items()}
    x2 = {kk: (vv[:, :, n1:] if kk != "gamma" else vv) for kk, vv in x.items()}
    _, st1 = run_oracle(x1, normalize=True, eps=1e-6, asymmetric=True)
    o2, st2 = run_forward(x2, "f32", 64, normalize=True, eps=1e-6, state_in=st1, asymmetric=True)
    o2_ref, st2_ref = run_oracle(x2, normalize=True, eps=1e-6, state_in=st1, asymmetric=True)
    assert_parity(o2, o2_ref, st2, st2_ref, tol=TOL_F32, what="asym resume, shared kv", asymmetric=True)


# ------------------------------------------------------------------ combine
@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (16, 32), (64, 128)])
def test_state_combine(d, dv):
    rng = np.random.default_rng(5)
    cnt = 6
    qa, ka, va = (rng.standard_normal((1, cnt, 13, s)) for s in (d, d, dv))
    qb, kb, vb = (rng.standard_normal((1, cnt, 9, s)) for s in (d, d, dv))
    gamma = rng.uniform(0.8, 1.0, cnt)
    _, A = oracle.forward(qa, ka, va, gamma=gamma)
    _, Bs = oracle.forward(qb, kb, vb, gamma=gamma)
    f = gamma ** 9
    ref = oracle.combine(A, Bs, f)
    dA, dB = state_to_dev(A), state_to_dev(Bs)
    df = torch.from_numpy(f.astype(np.float32)).cuda()
    out = hla.state_combine(dA, dB, df)
    got = state_to_np(out, cnt, d, dv)
    state_errors(got, ref, 1e-5, "combine")
    # in place: out aliases A
    hla.state_combine(dA, dB, df, out=dA)
    state_errors(state_to_np(dA, cnt, d, dv), ref, 1e-5, "combine in place")


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("d,dv", [(128, 128), (64, 128), (32, 16)])
@pytest.mark.parametrize("decay,normalize", [(False, False), (True, True)])
def test_decode_steps(d, dv, decay, normalize):
    seqs, H, steps = 8, 4, 3
    N = seqs * H
    rng = np.random.default_rng(9)
    gamma = np.exp(rng.uniform(np.log(0.9), np.log(0.999), H)) if decay else None
    pre = W.make_inputs(W.Workload("pre", seqs, H, 40, d, dv, 64, "bf16", "elu1" if normalize else "l2", seed=31))
    _, st = oracle.forward(pre["q"], pre["k"], pre["v"], gamma=gamma)
    st32 = oracle.State(*(np.asarray(a, np.float32).astype(np.float64) for a in st.astuple()))
    dst = state_to_dev(st32)
    toks = W.make_decode_tokens(seqs, H, d, dv, steps, seed=32)
    if normalize:
        toks["q"], toks["k"] = np.abs(toks["q"]), np.abs(toks["k"])
    g = torch.from_numpy(gamma.astype(np.float32)).cuda() if decay else None
    ref = st32.copy()
    for s in range(steps):
        q, k, v = (to_dev(toks[kk][s], "bf16") for kk in ("q", "k", "v"))
        o = hla.decode_step(dst, q, k, v, H, gamma=g, normalize=normalize, eps=1e-6)
        o_ref = oracle.decode_step(ref, toks["q"][s], toks["k"][s], toks["v"][s], H,
                                   gamma=None if gamma is None else gamma.astype(np.float32).astype(np.float64),
                                   normalize=normalize, eps=1e-6)
        hla.hla_sync_status()
        og = o.float().cpu().numpy()
        errs = [rel_l2(og[u], o_ref[u]) for u in range(N)]
        assert max(errs) <= TOL_BF16, f"step {s}: {max(errs):.3e}"
    state_errors(state_to_np(dst, N, d, dv), ref, 1e-5, "decode state")


@pytest.mark.parametrize("unmasked,Hkv", [(True, 4), (False, 2), (True, 1)])
def test_decode_unmasked_and_shared_heads(unmasked, Hkv):
    seqs, H, d, dv, steps = 6, 4, 128, 64, 3
    N = seqs * H
    rng = np.random.default_rng(19)
    gamma = np.exp(rng.uniform(np.log(0.9), np.log(0.999), H))
    pre = W.make_inputs(W.Workload("pre", seqs, H, 40, d, dv, 64, "bf16", "elu1", seed=33, Hkv=Hkv))
    _, st = oracle.forward(pre["q"], pre["k"], pre["v"], gamma=gamma, unmasked=unmasked)
    st32 = oracle.State(*(np.asarray(a, np.float32).astype(np.float64) for a in st.astuple()))
    dst = state_to_dev(st32)
    g = torch.from_numpy(gamma.astype(np.float32)).cuda()
    g64 = gamma.astype(np.float32).astype(np.float64)
    ref = st32.copy()
    for s in range(steps):
        toks = W.make_decode_tokens(seqs, H, d, dv, 1, seed=40 + s)
        qn = np.abs(toks["q"][0])
        kn = np.abs(toks["k"][0]).reshape(seqs, H, d)[:, :Hkv].reshape(seqs * Hkv, d)
        vn = toks["v"][0].reshape(seqs, H, dv)[:, :Hkv].reshape(seqs * Hkv, dv)
        kn, vn = np.ascontiguousarray(kn), np.ascontiguousarray(vn)
        q, k, v = to_dev(qn, "bf16"), to_dev(kn, "bf16"), to_dev(vn, "bf16")
        o = hla.decode_step(dst, q, k, v, H, gamma=g, normalize=True, eps=1e-6, unmasked=unmasked)
        o_ref = oracle.decode_step(ref, qn, kn, vn, H, gamma=g64, normalize=True, eps=1e-6, unmasked=unmasked)
        hla.hla_sync_status()
        og = o.float().cpu().numpy()
        assert max(rel_l2(og[u], o_ref[u]) for u in range(N)) <= TOL_BF16, f"step {s}"
    got = state_to_np(dst, N, d, dv)
    if unmasked:  # G, h are neither read nor written by the unmasked step
        got.G[...] = ref.G
        got.h[...] = ref.h
    state_errors(got, ref, 1e-5, "decode state")


@pytest.mark.parametrize("d,dv,Hkv", [(128, 128, 4), (64, 64, 2), (32, 16, 1)])
def test_decode_asym(d, dv, Hkv):
    seqs, H, steps = 6, 4, 3
    N = seqs * H
    rng = np.random.default_rng(21)
    gamma = np.exp(rng.uniform(np.log(0.9), np.log(0.999), H))
    pre = W.make_inputs(W.Workload("pre", seqs, H, 40, d, dv, 64, "bf16", "elu1", seed=35, Hkv=Hkv))
    _, st = oracle.forward(pre["q"], pre["k"], pre["v"], gamma=gamma, asymmetric=True)
    st32 = oracle.State(*(np.asarray(a, np.float32).astype(np.float64) for a in st.astuple()))
    dst = state_to_dev(st32)
    g = torch.from_numpy(gamma.astype(np.float32)).cuda()
    g64 = gamma.astype(np.float32).astype(np.float64)
    ref = st32.copy()
    for s in range(steps):
        toks = W.make_decode_tokens(seqs, H, d, dv, 1, seed=50 + s)
        qn = np.abs(toks["q"][0])
        kn = np.ascontiguousarray(np.abs(toks["k"][0]).reshape(seqs, H, d)[:, :Hkv].reshape(seqs * Hkv, d))
        vn = np.ascontiguousarray(toks["v"][0].reshape(seqs, H, dv)[:, :Hkv].reshape(seqs * Hkv, dv))
        q, k, v = to_dev(qn, "bf16"), to_dev(kn, "bf16"), to_dev(vn, "bf16")
        o = hla.decode_step(dst, q, k, v, H, gamma=g, normalize=True, eps=1e-6, asymmetric=True)
        o_ref = oracle.decode_step(ref, qn, kn, vn, H, gamma=g64, normalize=True, eps=1e-6, asymmetric=True)
        hla.hla_sync_status()
        og = o.float().cpu().numpy()
        assert max(rel_l2(og[u], o_ref[u]) for u in range(N)) <= TOL_BF16, f"step {s}"
    state_errors(state_to_np(dst, N, d, dv), ref, 1e-5, "asym decode state", asymmetric=True)


@pytest.mark.parametrize("variant", ["unmasked", "asymmetric"])
def test_state_combine_variants(variant):
    d, dv, cnt = 64, 32, 6
    rng = np.random.default_rng(22)
    kw = {variant: True}
    wa = W.Workload("ca", 1, cnt, 30, d, dv, 64, "f32", "l2", seed=36)
    wb = W.Workload("cb", 1, cnt, 23, d, dv, 64, "f32", "l2", seed=37)
    xa, xb = W.make_inputs(wa), W.make_inputs(wb)
    gamma = rng.uniform(0.9, 0.99, cnt)
    _, A = oracle.forward(xa["q"], xa["k"], xa["v"], gamma=gamma, **kw)
    _, B = oracle.forward(xb["q"], xb["k"], xb["v"], gamma=gamma, **kw)
    f = gamma ** 23
    ref = oracle.combine(A, B, f, asymmetric=(variant == "asymmetric"))
    if variant == "unmasked":
        ref.G[...] = 0.0
        ref.h[...] = 0.0
    f32 = lambda st: oracle.State(*(np.asarray(a, np.float32).astype(np.float64) for a in st.astuple()))
    dA, dB = state_to_dev(f32(A)), state_to_dev(f32(B))
    df = torch.from_numpy(f.astype(np.float32)).cuda()
    out = hla.state_combine(dA, dB, df, **kw)
    hla.hla_sync_status()
    state_errors(state_to_np(out, cnt, d, dv), ref, 1e-5, f"combine {variant}", asymmetric=True)


# ---------------------------------------------------- full-size workloads
@pytest.mark.parametrize("w", [W.FWD_BF16, W.FWD_NORM, W.FWD_DECAY, W.FWD_UNMASKED, W.FWD_SHARED_KV, W.FWD_ASYM],
                         ids=lambda w: w.name)
def test_full_workload(w):
    x = W.make_inputs(w)
    kw = dict(normalize=w.normalize, eps=w.eps, unmasked=w.unmasked, asymmetric=w.asymmetric)
    o, st = run_forward(x, w.dtype, w.chunk, **kw)
    o_ref, st_ref = run_oracle(x, **kw)
    err = assert_parity(o, o_ref, st, st_ref, what=w.name, asymmetric=w.asymmetric)
    print(f"{w.name}: max per-(b,h) rel L2 {err:.3e}")
