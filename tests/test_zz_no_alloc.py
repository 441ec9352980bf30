"""The no-alloc forward entry point, for callers that cannot allocate device
memory (code inside an allocator hook, allocation-free real-time loops, hosts
that hand out device memory only up front).  It must give the same results as
the ordinary forward, which takes a caller-allocated workspace, on two calls in
a row that share its fixed scratch array.

This file is collected last, so a run that stops at its first failure has run
every other test before this one."""
import ctypes

import numpy as np
import pytest
import torch

import causal_prefix_scan_gb300 as hla
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import TOL_BF16, per_pair_errors, state_errors, state_to_np, to_dev

pytestmark = pytest.mark.gpu


def _inputs(w):
    x = W.make_inputs(w)
    q, k, v = to_dev(x["q"], "bf16"), to_dev(x["k"], "bf16"), to_dev(x["v"], "bf16")
    g = torch.from_numpy(x["gamma"]).cuda() if x["gamma"] is not None else None
    return q, k, v, g


@pytest.mark.parametrize("w", [
    W.Workload("noalloc_small", 1, 2, 5 * 64 + 17, 64, 64, 64, "bf16", "l2", decay=True, seed=41),
    W.Workload("noalloc_norm", 2, 2, 3 * 128 + 5, 128, 128, 128, "bf16", "elu1", normalize=True, eps=1e-6, seed=42),
    W.FWD_BF16,
], ids=lambda w: w.name)
def test_noalloc_matches_workspace_forward_twice(w):
    q, k, v, g = _inputs(w)
    units = w.B * w.H
    # reference: the ordinary entry point with a caller workspace
    o_ref, st_ref = hla.forward(q, k, v, chunk=w.chunk, gamma=g, normalize=w.normalize, eps=w.eps,
                                return_state=True)
    hla.hla_sync_status()
    o_ref = o_ref.float().cpu().numpy()
    st_ref = state_to_np(st_ref, units, w.d, w.dv)
    p = hla.make_params(q, v, w.chunk, g, w.normalize, w.eps)
    assert 0 < hla.hla_forward_workspace_size(p) <= 32 << 20
    for call in range(2):
        o = torch.full(q.shape[:3] + (w.dv,), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = hla.State.empty(units, w.d, w.dv)
        hla.hla_forward_chunked_noalloc(p, q, k, v, o, None, st)
        hla.hla_sync_status()
        og = o.float().cpu().numpy()
        assert np.all(np.isfinite(og)), f"call {call}: non-finite outputs"
        assert per_pair_errors(og, o_ref).max() <= TOL_BF16, f"call {call}"
        state_errors(state_to_np(st, units, w.d, w.dv), st_ref, TOL_BF16, f"no-alloc call {call}")


def test_noalloc_rejects_oversized_problem():
    # 64000 (b,h) pairs at d = dv = 128 need far more scratch than the fixed array
    p = hla.hla_params(2000, 32, 64, 128, 128, 128, hla.HLA_BF16, 0, 0.0, None)
    need = hla.hla_forward_workspace_size(p)
    assert need > 32 << 20
    st = hla.library().hla_forward_chunked_noalloc(ctypes.byref(p), 16, 16, 16, 16, None, None, None)
    assert st == hla.HLA_ERR_UNSUPPORTED
    assert "scratch" in hla.hla_last_error()


def test_noalloc_split_call():
    """The AHLA forward at dv = 128 (two value-half launches) through the no-alloc entry:
    the same results, bit for bit, as with a caller workspace, on two calls in a row."""
    w = W.Workload("noalloc_asym", 1, 2, 3 * 64 + 9, 64, 128, 64, "bf16", "elu1", normalize=True, eps=1e-6, seed=43,
                   decay=True, asymmetric=True)
    q, k, v, g = _inputs(w)
    units = w.B * w.H
    o_ref, st_ref = hla.forward(q, k, v, chunk=64, gamma=g, normalize=True, eps=1e-6, return_state=True,
                                asymmetric=True)
    hla.hla_sync_status()
    p = hla.make_params(q, v, 64, g, True, 1e-6, False, True)
    assert 0 < hla.hla_forward_workspace_size(p) <= 32 << 20
    for call in range(2):
        o = torch.full(q.shape[:3] + (w.dv,), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = hla.State.empty(units, w.d, w.dv)
        hla.hla_forward_chunked_noalloc(p, q, k, v, o, None, st)
        hla.hla_sync_status()
        assert torch.equal(o, o_ref), f"call {call}"
        assert all(torch.equal(a, b) for a, b in zip(st.astuple(), st_ref.astuple())), f"call {call}"
