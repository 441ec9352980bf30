"""The streaming decode workload at its stated size against the fp64 oracle.

256 sequences x 32 heads at d = dv = 128: the fp32 state (S, C, m, G, h) is
prefilled by the chunked forward over a seeded 4096-token prefix, then 1024
consecutive decode steps update it in place (gist.science summary of the paper,
section 1, "Onderhoud van de toestand", "Strenge causaliteit",
"Outputformulering"; constant state per "Complexiteit").  The oracle cannot
afford all 8192 pairs, so a seeded sample of 64 pairs is checked:

* the prefill state against the oracle's serial recurrence over the same
  (device-drawn, copied back) prefix tokens;
* every decode output row of the sampled pairs, and their final state, against
  the oracle's decode step continued from the exact fp32 device state after the
  prefill, with the same tokens.

The 1024 in-place fp32 updates are where drift of the device state would show;
the bf16 tolerance (per-pair relative L2 <= 2e-2) applies throughout."""
import numpy as np
import pytest
import torch

import causal_prefix_scan_gb300 as hla
import oracle
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import TOL_BF16, rel_l2, state_errors

pytestmark = pytest.mark.gpu

SAMPLE = 64


def _host(t, idx):
    return t.index_select(0, idx).double().cpu().numpy()


def test_decode_workload_full_size():
    dw = W.DECODE
    dev = torch.device("cuda", 0)
    N, H, d, dv = dw.seqs * dw.H, dw.H, dw.d, dw.dv
    idx = np.sort(np.random.default_rng(dw.seed + 500).choice(N, SAMPLE, replace=False))
    ti = torch.from_numpy(idx).to(dev)

    # ---- prefill: the forward over the workload's seeded prefix, block by block;
    # the sampled pairs' prefix tokens are copied back for the oracle
    st = hla.State.empty(N, d, dv, device=dev)
    pq = np.zeros((1, SAMPLE, dw.prefix, d))
    pk = np.zeros_like(pq)
    pv = np.zeros((1, SAMPLE, dw.prefix, dv))
    for b0, pw in W.decode_prefix_blocks(dw):
        px = W.make_inputs_device(pw, device=dev)
        u0, u1 = b0 * H, (b0 + pw.B) * H
        sub = hla.State(*(a[u0:u1] for a in st.astuple()))
        p = hla.make_params(px["q"], px["v"], dw.chunk)
        need = hla.hla_forward_workspace_size(p)
        ws = hla.new_workspace(need, dev)
        o = torch.empty_like(px["v"])
        hla.hla_forward_chunked(p, px["q"], px["k"], px["v"], o, None, sub, ws, need)
        for j in np.nonzero((idx >= u0) & (idx < u1))[0]:
            b, h = divmod(int(idx[j]) - u0, H)
            pq[0, j] = px["q"][b, h].double().cpu().numpy()
            pk[0, j] = px["k"][b, h].double().cpu().numpy()
            pv[0, j] = px["v"][b, h].double().cpu().numpy()
        del px, o, ws
    torch.cuda.synchronize()
    hla.hla_sync_status()

    _, st_pre = oracle.forward(pq, pk, pv)
    got_pre = oracle.State(*(_host(a, ti) for a in st.astuple()))
    pre_err = state_errors(got_pre, st_pre, TOL_BF16, "decode prefill state")

    # ---- 1024 decode steps on all pairs; the sampled pairs' outputs are gathered on the device
    T = 64
    toks = W.decode_tokens_device(dw, T, device=dev)
    outs = torch.empty((dw.steps, SAMPLE, dv), dtype=torch.bfloat16, device=dev)
    o = torch.empty((N, dv), dtype=torch.bfloat16, device=dev)
    for i in range(dw.steps):
        q, k, v = toks[i % T]
        hla.hla_decode_step(N, H, 0, d, dv, hla.HLA_BF16, 0, 0.0, None, st, q, k, v, o, None)
        outs[i].copy_(o.index_select(0, ti))
    torch.cuda.synchronize()
    hla.hla_sync_status()

    # ---- the oracle continues from the exact fp32 state after the prefill
    ref = got_pre.copy()
    sets = [tuple(t.index_select(0, ti).double().cpu().numpy() for t in ts) for ts in toks]
    outs = outs.float().cpu().numpy()
    worst, worst_step = 0.0, -1
    for i in range(dw.steps):
        q, k, v = sets[i % T]
        o_ref = oracle.decode_step(ref, q, k, v, 1)
        e = max(rel_l2(outs[i, j], o_ref[j]) for j in range(SAMPLE))
        if e > worst:
            worst, worst_step = e, i
    assert np.all(np.isfinite(outs))
    assert worst <= TOL_BF16, f"decode output rel L2 {worst:.3e} at step {worst_step}"
    got_end = oracle.State(*(_host(a, ti) for a in st.astuple()))
    end_err = state_errors(got_end, ref, TOL_BF16, "decode final state")
    print(f"\ndecode workload: prefill state {pre_err}; outputs max rel L2 {worst:.3e} (step {worst_step}); "
          f"final state {end_err}")
