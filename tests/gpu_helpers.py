"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and compare with the fp64 oracle per (b,h)."""
import numpy as np
import torch

import causal_prefix_scan_gb300 as hla
import oracle

# Tolerances on the per-(b,h) relative L2 error (relative to the oracle's norm).
TOL_F32 = 1e-4      # fp32 inputs, fp32 arithmetic
TOL_BF16 = 2e-2     # bf16 inputs, fp32 state and accumulation


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def per_pair_errors(got, ref):
    """got, ref: [B,H,...]; returns the array of per-(b,h) relative L2 errors."""
    B, H = ref.shape[:2]
    return np.array([[rel_l2(got[b, h], ref[b, h]) for h in range(H)] for b in range(B)])


def to_dev(x, dtype):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(tdt).contiguous()


def state_to_dev(st: "oracle.State"):
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    return hla.State(*(f(a) for a in st.astuple()))


def state_to_np(st: "hla.State", units, d, dv):
    shapes = [(units, d, d), (units, d, dv), (units, d), (units, d, dv), (units, d)]
    return oracle.State(*(x.double().cpu().numpy().reshape(s) for x, s in zip(st.astuple(), shapes)))


def run_forward(x, dtype, chunk, normalize=False, eps=0.0, state_in=None, return_state=True, unmasked=False,
                asymmetric=False):
    q, k, v = to_dev(x["q"], dtype), to_dev(x["k"], dtype), to_dev(x["v"], dtype)
    g = None if x.get("gamma") is None else torch.from_numpy(np.asarray(x["gamma"], np.float32)).cuda()
    sin = state_to_dev(state_in) if state_in is not None else None
    res = hla.forward(q, k, v, chunk=chunk, gamma=g, normalize=normalize, eps=eps, state_in=sin,
                      return_state=return_state, unmasked=unmasked, asymmetric=asymmetric)
    hla.hla_sync_status()
    if return_state:
        o, st = res
        B, H, n, d = x["q"].shape
        return o.float().cpu().numpy(), state_to_np(st, B * H, d, x["v"].shape[-1])
    return res.float().cpu().numpy(), None


def run_oracle(x, normalize=False, eps=0.0, state_in=None, unmasked=False, asymmetric=False):
    g = None if x.get("gamma") is None else np.asarray(x["gamma"], np.float64)
    return oracle.forward(x["q"], x["k"], x["v"], gamma=g, normalize=normalize, eps=eps, state_in=state_in,
                          unmasked=unmasked, asymmetric=asymmetric)


def assert_parity(o, o_ref, st=None, st_ref=None, tol=TOL_BF16, what="", asymmetric=False):
    e = per_pair_errors(o, o_ref)
    assert np.all(np.isfinite(o)), f"{what}: non-finite outputs"
    assert e.max() <= tol, f"{what}: max per-(b,h) output rel L2 {e.max():.3e} > {tol}"
    if st is not None:
        state_errors(st, st_ref, tol, what, asymmetric=asymmetric)
    return float(e.max())


def state_errors(st, st_ref, tol, what="", asymmetric=False):
    """Per-pair relative L2 error of each summary.  G and h are differences of
    larger terms (G_t = S_t C_t - (S_t C_t - G_t)); their error is measured
    against the larger of |G| and |S C| (|h| and |S m|), so that an exactly zero
    reference (e.g. one token: no earlier query/value index) is well posed.  The
    asymmetric variant's E and n (in G, h) are plain sums: relative to themselves."""
    worst = {}
    for u in range(st_ref.S.shape[0]):
        S, C, m = st_ref.S[u], st_ref.C[u], st_ref.m[u]
        scale = {} if asymmetric else {"G": max(np.linalg.norm(st_ref.G[u]), np.linalg.norm(S @ C)),
                                       "h": max(np.linalg.norm(st_ref.h[u]), np.linalg.norm(S @ m))}
        for name, a, b in zip("SCmGh", st.astuple(), st_ref.astuple()):
            den = scale.get(name, np.linalg.norm(b[u]))
            err = float(np.linalg.norm(a[u] - b[u]) / max(den, 1e-30))
            worst[name] = max(worst.get(name, 0.0), err)
    for name, err in worst.items():
        assert err <= tol, f"{what}: state {name} rel L2 {err:.3e} > {tol}"
    return worst
