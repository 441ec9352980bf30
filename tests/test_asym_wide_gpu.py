"""GPU parity of the asymmetric variant AHLA (section 2) and of the unmasked variant at
value width dv = 128 with d <= 64 where no kernel takes the shape whole: two problems
over the value columns [0, 64) and [64, 128) (the output's column j and the state's
value-width columns j depend on column j of v only, the rest on none).  Each half takes
the tensor-core path (bf16, d = 64) or the CUDA-core one.  Against the fp64 oracle;
tolerance per (b,h) relative L2: 1e-4 for fp32 inputs, 2e-2 for bf16."""
import numpy as np
import pytest
import torch

import causal_prefix_scan_gb300 as hla
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import TOL_BF16, TOL_F32, assert_parity, run_forward, run_oracle, to_dev

pytestmark = pytest.mark.gpu


def wl(**kw):
    base = dict(B=1, H=2, n=200, d=64, dv=128, chunk=64, dtype="bf16", qk="elu1", seed=201, gamma_lo=0.9,
                gamma_hi=0.999)
    base.update(kw)
    return W.Workload("asym128", **base)


@pytest.mark.parametrize("d,chunk,dtype", [(64, 64, "bf16"), (64, 128, "bf16"), (32, 32, "f32"), (16, 64, "bf16")])
@pytest.mark.parametrize("decay,normalize", [(False, False), (True, False), (True, True)])
def test_asym_value_width_128(d, chunk, dtype, decay, normalize):
    w = wl(d=d, chunk=chunk, dtype=dtype, decay=decay, n=3 * chunk + 21, seed=201 + d)
    x = W.make_inputs(w)
    o, st = run_forward(x, dtype, chunk, normalize=normalize, eps=1e-6, asymmetric=True)
    o_ref, st_ref = run_oracle(x, normalize=normalize, eps=1e-6, asymmetric=True)
    assert_parity(o, o_ref, st, st_ref, tol=TOL_F32 if dtype == "f32" else TOL_BF16,
                  what=f"asym dv128 d{d} c{chunk} {dtype}", asymmetric=True)


def test_asym_value_width_128_resumed_shared_heads():
    """Four query heads on two key/value heads, continued from the oracle's state."""
    w = wl(B=2, H=4, Hkv=2, n=330, decay=True, seed=210)
    x = W.make_inputs(w)
    n1 = 131
    x1 = {kk: (vv[:, :, :n1] if kk != "gamma" else vv) for kk, vv in x.items()}
    x2 = {kk: (vv[:, :, n1:] if kk != "gamma" else vv) for kk, vv in x.items()}
    _, st1 = run_oracle(x1, normalize=True, eps=1e-6, asymmetric=True)
    o2, st2 = run_forward(x2, "bf16", 64, normalize=True, eps=1e-6, state_in=st1, asymmetric=True)
    o2_ref, st2_ref = run_oracle(x2, normalize=True, eps=1e-6, state_in=st1, asymmetric=True)
    assert_parity(o2, o2_ref, st2, st2_ref, what="asym dv128 resumed, shared heads", asymmetric=True)


def test_asym_value_width_128_kernel_name():
    q = to_dev(np.zeros((1, 2, 64, 64), np.float32), "bf16")
    v = to_dev(np.zeros((1, 2, 64, 128), np.float32), "bf16")
    p = hla.make_params(q, v, 64, None, False, 0.0, False, True)
    assert hla.hla_forward_kernel(p) == "fwd_tc_kernel"
    assert hla.hla_forward_workspace_size(p) > 0


@pytest.mark.parametrize("d,dtype", [(64, "f32"), (32, "f32"), (32, "bf16")])
@pytest.mark.parametrize("decay,normalize", [(False, False), (True, True)])
def test_unmasked_value_width_128(d, dtype, decay, normalize):
    w = wl(d=d, chunk=32, dtype=dtype, decay=decay, n=117, seed=220 + d, qk="elu1" if normalize else "l2")
    x = W.make_inputs(w)
    o, st = run_forward(x, dtype, 32, normalize=normalize, eps=1e-6, unmasked=True)
    o_ref, st_ref = run_oracle(x, normalize=normalize, eps=1e-6, unmasked=True)
    assert_parity(o, o_ref, st, st_ref, tol=TOL_F32 if dtype == "f32" else TOL_BF16,
                  what=f"unmasked dv128 d{d} {dtype}")


@pytest.mark.parametrize("n", [1, 7, 64, 65])
def test_asym_value_width_128_short_sequences(n):
    """Sequences of one token, shorter than a chunk, exactly one chunk and one token more."""
    w = wl(n=n, decay=True, seed=230 + n)
    x = W.make_inputs(w)
    o, st = run_forward(x, "bf16", 64, normalize=True, eps=1e-6, asymmetric=True)
    o_ref, st_ref = run_oracle(x, normalize=True, eps=1e-6, asymmetric=True)
    assert_parity(o, o_ref, st, st_ref, tol=TOL_BF16, what=f"asym dv128 n{n}", asymmetric=True)


def test_asym_value_width_128_empty_sequence_copies_the_state():
    """n = 0: state_out is state_in, all 128 value columns."""
    w = wl(n=40, decay=True, seed=240)
    x = W.make_inputs(w)
    _, st1 = run_oracle(x, normalize=True, eps=1e-6, asymmetric=True)
    empty = {kk: (vv[:, :, :0] if kk != "gamma" else vv) for kk, vv in x.items()}
    o, st = run_forward(empty, "bf16", 64, normalize=True, eps=1e-6, state_in=st1, asymmetric=True)
    assert o.shape == (1, 2, 0, 128)
    for name in ("S", "C", "m", "G", "h"):
        a, b = getattr(st, name), np.asarray(getattr(st1, name), np.float32)
        assert np.array_equal(np.asarray(a, np.float32).reshape(b.shape), b), name
