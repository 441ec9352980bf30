"""GPU parity of the 128-token forward (d = dv = 64, bf16, no decay) on shapes with many
(b,h) pairs of a few pieces each (up to eight pieces of one to three chunks, ragged
tails), plain and normalised, with a state carried in and out.  Against the fp64
oracle, per (b,h) relative L2 <= 2e-2."""
import numpy as np
import pytest

import causal_prefix_scan_gb300 as hla
import oracle
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import TOL_BF16, assert_parity, run_forward, run_oracle

pytestmark = pytest.mark.gpu


def wl(**kw):
    base = dict(B=4, H=8, n=2048, d=64, dv=64, chunk=64, dtype="bf16", qk="l2", seed=71)
    base.update(kw)
    return W.Workload("pairs", **base)


# (B, H, n): 7 pieces of 2 chunks and the last piece split in two of 1; 7 pieces of one
# chunk with a ragged tail; 3 pieces of 3 chunks; 2 pieces (one of 2 chunks, one of 1);
# 15 pieces of 2 chunks and two of 1; 7 pieces of 4 chunks and two of 2
SHAPES = [(4, 8, 2048), (2, 12, 777), (8, 12, 1100), (10, 14, 300), (2, 8, 4096), (4, 8, 4096)]


@pytest.mark.parametrize("B,H,n", SHAPES)
@pytest.mark.parametrize("normalize", [False, True])
def test_many_pairs_forward(B, H, n, normalize):
    w = wl(B=B, H=H, n=n, qk="elu1" if normalize else "l2")
    x = W.make_inputs(w)
    o, st = run_forward(x, "bf16", 64, normalize=normalize, eps=1e-6)
    o_ref, st_ref = run_oracle(x, normalize=normalize, eps=1e-6)
    assert_parity(o, o_ref, st, st_ref, TOL_BF16, f"pairs B{B}H{H}n{n} norm={normalize}")


@pytest.mark.parametrize("B,H,n", [(4, 8, 2048), (2, 12, 777), (2, 8, 4096)])
def test_many_pairs_forward_resume(B, H, n):
    """state_in from the oracle's state of a first part (piece 0 folds it in), no state out."""
    w = wl(B=B, H=H, n=n + 333, seed=72)
    x = W.make_inputs(w)
    first = {k: x[k][:, :, :333] for k in ("q", "k", "v")}
    second = {k: x[k][:, :, 333:] for k in ("q", "k", "v")}
    first["gamma"] = second["gamma"] = None
    _, st1 = run_oracle(first)
    o_ref, st_ref = run_oracle(x)
    o2, st2 = run_forward(second, "bf16", 64, state_in=st1)
    assert_parity(o2, o_ref[:, :, 333:], st2, st_ref, TOL_BF16, "resume")
    o3, _ = run_forward(second, "bf16", 64, state_in=st1, return_state=False)
    assert_parity(o3, o_ref[:, :, 333:], tol=TOL_BF16, what="resume, no state out")


def test_dispatch_names_the_128_token_kernel():
    import torch
    for B, H, n in SHAPES:
        q = torch.empty((B, H, n, 64), dtype=torch.bfloat16, device="cuda")
        assert hla.hla_forward_kernel(hla.make_params(q, q, 64)) == "fwd_ws2_kernel"
