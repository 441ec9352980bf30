"""The forward's workspace between calls (include/hla.h, hla_forward_chunked): the
ordering header carries a call generation, the release flags carry the tag of the call
that wrote them, and nothing else in the workspace is read before this call writes it.
So one workspace serves calls of any shape in turn without clearing, whatever earlier
calls left in it, and the one call whose tag is the largest 32-bit value zeroes the
header and flags for the calls after it."""
import numpy as np
import pytest
import torch

import causal_prefix_scan_gb300 as hla
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu

# one shape per forward kernel: fwd_ws2_kernel, fwd_ws_kernel, fwd_tc_kernel
SHAPES = [
    dict(d=64, dv=64, chunk=64, n=900, decay=False, normalize=False),
    dict(d=64, dv=128, chunk=64, n=700, decay=False, normalize=True),
    dict(d=128, dv=128, chunk=64, n=650, decay=True, normalize=False),
]


def case(i, seed):
    s = SHAPES[i]
    w = W.Workload("ws", B=2, H=3, n=s["n"], d=s["d"], dv=s["dv"], chunk=s["chunk"], dtype="bf16",
                   qk="elu1" if s["normalize"] else "l2", seed=seed, decay=s["decay"], gamma_lo=0.9, gamma_hi=0.999)
    x = W.make_inputs(w)
    q, k, v = (to_dev(x[n], "bf16") for n in ("q", "k", "v"))
    g = None if x.get("gamma") is None else torch.from_numpy(np.asarray(x["gamma"], np.float32)).cuda()
    return dict(q=q, k=k, v=v, chunk=s["chunk"], gamma=g, normalize=s["normalize"], eps=1e-6)


def run(c, ws=None):
    o, st = hla.forward(c["q"], c["k"], c["v"], chunk=c["chunk"], gamma=c["gamma"], normalize=c["normalize"],
                        eps=c["eps"], return_state=True, workspace=ws)
    hla.hla_sync_status()
    return [o] + list(st.astuple())


def need(c):
    p = hla.make_params(c["q"], c["v"], c["chunk"], c["gamma"], c["normalize"], c["eps"], False, False)
    return hla.hla_forward_workspace_size(p)


def header(ws):
    h = ws[:12].cpu().numpy().view(np.uint32)
    return int(h[0]), int(h[1]), int(h[2])  # tickets taken, generation, finish counter


def same(a, b):
    return all(torch.equal(x, y) for x, y in zip(a, b))


def test_generation_counts_calls_and_tickets_return_to_zero():
    c = case(0, 91)
    ws = hla.new_workspace(need(c))
    for i in range(1, 4):
        run(c, ws)
        assert header(ws) == (0, i, 0)


def test_one_workspace_serves_every_kernel_in_turn():
    """Results on one shared workspace equal those on a fresh one, bit for bit, over
    calls of the three kernels interleaved."""
    cases = [case(i, 92 + i) for i in range(3)]
    fresh = [run(c) for c in cases]
    ws = hla.new_workspace(max(need(c) for c in cases))
    for rep in range(2):
        for c, ref in zip(cases, fresh):
            assert same(run(c, ws), ref)
    assert header(ws) == (0, 6, 0)


@pytest.mark.parametrize("i", range(3))
def test_contents_other_than_the_header_are_ignored(i):
    """Random bytes everywhere after the header (any flag value except this call's tag):
    the call reads nothing it has not written itself."""
    c = case(i, 95 + i)
    ref = run(c)
    ws = hla.new_workspace(need(c))
    gen = 12345
    rng = np.random.default_rng(7 + i)
    words = rng.integers(0, 2**32, size=ws.numel() // 4, dtype=np.uint64).astype(np.uint32)
    words[words == gen + 1] = 0
    words[:64] = 0
    words[1] = gen
    ws.copy_(torch.from_numpy(words.view(np.uint8)).to(ws.device))
    assert same(run(c, ws), ref)
    assert header(ws) == (0, gen + 1, 0)


@pytest.mark.parametrize("i", range(3))
def test_the_last_tag_clears_header_and_flags(i):
    c = case(i, 98 + i)
    ref = run(c)
    ws = hla.new_workspace(need(c))
    ws[4:8] = torch.from_numpy(np.array([0xFFFFFFFE], np.uint32).view(np.uint8).copy()).to(ws.device)
    assert header(ws) == (0, 0xFFFFFFFE, 0)
    assert same(run(c, ws), ref)
    assert header(ws) == (0, 0, 0)
    assert same(run(c, ws), ref)
    assert header(ws) == (0, 1, 0)


def test_split_call_shares_the_workspace_across_the_generation_wrap():
    """The AHLA forward at dv = 128 runs two tensor-core launches per call on the same
    workspace (one per value half): results equal those on a fresh workspace, bit for bit,
    also when the first half's launch carries the last 32-bit tag."""
    w = W.Workload("ws_asym", B=2, H=3, n=500, d=64, dv=128, chunk=64, dtype="bf16", qk="elu1", seed=111,
                   decay=True, gamma_lo=0.9, gamma_hi=0.999, asymmetric=True)
    x = W.make_inputs(w)
    q, k, v = (to_dev(x[n], "bf16") for n in ("q", "k", "v"))
    g = torch.from_numpy(np.asarray(x["gamma"], np.float32)).cuda()

    def run_asym(ws=None):
        o, st = hla.forward(q, k, v, chunk=64, gamma=g, normalize=True, eps=1e-6, return_state=True, workspace=ws,
                            asymmetric=True)
        hla.hla_sync_status()
        return [o] + list(st.astuple())

    ref = run_asym()
    p = hla.make_params(q, v, 64, g, True, 1e-6, False, True)
    ws = hla.new_workspace(hla.hla_forward_workspace_size(p))
    assert same(run_asym(ws), ref)
    assert same(run_asym(ws), ref)
    assert header(ws) == (0, 4, 0)  # two calls of two launches
    ws[4:8] = torch.from_numpy(np.array([0xFFFFFFFE], np.uint32).view(np.uint8).copy()).to(ws.device)
    assert same(run_asym(ws), ref)
    assert header(ws) == (0, 1, 0)  # the first half's launch cleared the header, the second took generation 1
