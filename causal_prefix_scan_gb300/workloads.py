"""Seeded synthetic inputs for the HLA forward and decode workloads.

This module holds only random draws and input preprocessing (row L2
normalisation, elu+1 features, the per-head decay draw, bf16 rounding); none of
the attention arithmetic.  Both the oracle side (tests, CPU baseline) and the
CUDA side (tests, benchmark) take their inputs from here, so they see the same
values.

Recipe: numpy ``default_rng(seed)``, draws in the order q, k, v, gamma, each as
float32 standard normals of the full [B,H,n,d] / [B,Hkv,n,d] / [B,Hkv,n,dv] shape
(Hkv = H unless keys and values are shared by head groups), then the
workload's preprocessing, then rounding to the input dtype (round to nearest
even for bf16).  The oracle reads the rounded values exactly.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    n: int
    d: int
    dv: int
    chunk: int
    dtype: str                # "f32" or "bf16": the input / output element type
    qk: str                   # "scaled" N(0,1)/sqrt(d), "l2" row-normalised N(0,1), "elu1" elu(x)+1
    normalize: bool = False
    eps: float = 0.0
    decay: bool = False       # per-head gamma, log-uniform in [gamma_lo, gamma_hi]
    gamma_lo: float = 0.9
    gamma_hi: float = 0.999
    seed: int = 0
    note: str = field(default="", compare=False)
    unmasked: bool = False    # unmasked variant o = q^T S C
    asymmetric: bool = False  # asymmetric variant AHLA, o = q^T E
    Hkv: int = 0              # key/value heads (0: H); query head h reads head h // (H // Hkv)

    @property
    def kv_heads(self) -> int:
        return self.Hkv or self.H

    @property
    def tokens(self) -> int:
        return self.B * self.n

    @property
    def token_heads(self) -> int:
        return self.B * self.H * self.n

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads the method is measured on.  The first is the small fp32
# case the oracle finishes in well under a second; 2-4 are forward workloads;
# DECODE describes the streaming decode workload.
SMALL_F32 = Workload("fwd_f32_B1H2n256d16", 1, 2, 256, 16, 16, 32, "f32", "scaled", seed=1)
FWD_BF16 = Workload("fwd_bf16_B4H8n2048d64", 4, 8, 2048, 64, 64, 64, "bf16", "l2", seed=2)
FWD_NORM = Workload("fwd_bf16_norm_B2H16n8192d64dv128", 2, 16, 8192, 64, 128, 64, "bf16", "elu1",
                    normalize=True, eps=1e-6, seed=3)
FWD_DECAY = Workload("fwd_bf16_decay_B1H32n32768d128", 1, 32, 32768, 128, 128, 128, "bf16", "l2",
                     decay=True, seed=4)
# Widening beyond the masked forward: the unmasked variant, keys/values shared by
# groups of query heads, and the asymmetric variant, on the shape of the
# B4H8n2048d64 workload.
FWD_UNMASKED = Workload("fwd_bf16_unmasked_B4H8n2048d64", 4, 8, 2048, 64, 64, 64, "bf16", "l2", seed=6,
                        unmasked=True)
FWD_SHARED_KV = Workload("fwd_bf16_kv2_B4H8n2048d64", 4, 8, 2048, 64, 64, 64, "bf16", "l2", seed=7, Hkv=2)
FWD_ASYM = Workload("fwd_bf16_asym_B4H8n2048d64", 4, 8, 2048, 64, 64, 64, "bf16", "l2", seed=8, asymmetric=True)
# The backward pass (training) on the same shape: q, k, v as above plus the
# gradient of the output from make_dout.
BWD_BF16 = Workload("bwd_bf16_B4H8n2048d64", 4, 8, 2048, 64, 64, 64, "bf16", "l2", seed=9)
# Backward through the ratio normalisation: positive (elu+1) features as in the
# normalised forward workload, on the backward workload's shape.
BWD_NORM = Workload("bwd_bf16_norm_B4H8n2048d64", 4, 8, 2048, 64, 64, 64, "bf16", "elu1", normalize=True, eps=1e-6,
                    seed=11)
# Masked third-order HLA on the same shape.
FWD3_BF16 = Workload("fwd3_bf16_B4H8n2048d64", 4, 8, 2048, 64, 64, 64, "bf16", "l2", seed=10)
WORKLOADS = {w.name: w for w in (SMALL_F32, FWD_BF16, FWD_NORM, FWD_DECAY, FWD_UNMASKED, FWD_SHARED_KV, FWD_ASYM,
                                 BWD_BF16, BWD_NORM, FWD3_BF16)}


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    seqs: int
    H: int
    d: int
    dv: int
    prefix: int
    steps: int
    chunk: int
    seed: int
    order: int = 2            # 3: third-order decode on the state (S^K, P, T)


DECODE = DecodeWorkload("decode_256x32_d128_prefix4096_steps1024", 256, 32, 128, 128, 4096, 1024, 128, seed=5)
# Third-order decode on the same pairs and widths.  Its state is drawn (seeded, on the
# device) instead of prefilled: the forward covers widths up to 64, and the cost of a
# step does not depend on the state's values.
DECODE3 = DecodeWorkload("decode3_256x32_d128_steps1024", 256, 32, 128, 128, 0, 1024, 0, seed=12, order=3)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returned as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _rows_l2(x: np.ndarray) -> np.ndarray:
    return x / np.linalg.norm(x, axis=-1, keepdims=True).astype(np.float32)


def _elu1(x: np.ndarray) -> np.ndarray:
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0))).astype(np.float32)


def _features(x: np.ndarray, kind: str, d: int) -> np.ndarray:
    if kind == "scaled":
        return (x / np.float32(np.sqrt(d))).astype(np.float32)
    if kind == "l2":
        return _rows_l2(x)
    if kind == "elu1":
        return _elu1(x)
    raise ValueError(kind)


def make_inputs(w: Workload):
    """Return dict(q, k, v, gamma) as float32 numpy arrays holding exactly the
    values of the input dtype (bf16-rounded for bf16 workloads); gamma is [H]
    float32 or None."""
    rng = np.random.default_rng(w.seed)
    q = rng.standard_normal((w.B, w.H, w.n, w.d), dtype=np.float32)
    k = rng.standard_normal((w.B, w.kv_heads, w.n, w.d), dtype=np.float32)
    v = rng.standard_normal((w.B, w.kv_heads, w.n, w.dv), dtype=np.float32)
    gamma = None
    if w.decay:
        lo, hi = np.log(w.gamma_lo), np.log(w.gamma_hi)
        gamma = np.exp(rng.uniform(lo, hi, size=w.H)).astype(np.float32)
    q = _features(q, w.qk, w.d)
    k = _features(k, w.qk, w.d)
    if w.dtype == "bf16":
        q, k, v = round_bf16(q), round_bf16(k), round_bf16(v)
    return {"q": q, "k": k, "v": v, "gamma": gamma}


def make_dout(w: Workload) -> np.ndarray:
    """The gradient of the output for a backward workload: float32 standard normals
    of shape [B,H,n,dv] from default_rng(seed + 1000), rounded like the inputs."""
    rng = np.random.default_rng(w.seed + 1000)
    g = rng.standard_normal((w.B, w.H, w.n, w.dv), dtype=np.float32)
    return round_bf16(g) if w.dtype == "bf16" else g


def make_decode_tokens(seqs: int, H: int, d: int, dv: int, steps: int, seed: int):
    """Per-step decode tokens [steps, seqs*H, d|dv], L2-normalised q, k, bf16-rounded."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((steps, seqs * H, d), dtype=np.float32)
    k = rng.standard_normal((steps, seqs * H, d), dtype=np.float32)
    v = rng.standard_normal((steps, seqs * H, dv), dtype=np.float32)
    return {"q": round_bf16(_rows_l2(q)), "k": round_bf16(_rows_l2(k)), "v": round_bf16(v)}


# Sequences per prefill launch of a decode workload (bounds the device memory of
# the drawn prefix: 32 sequences x 32 heads x 4096 tokens x 128 is 1 GiB per bf16 tensor).
DECODE_PREFILL_ROWS = 32


def decode_prefix_blocks(dw: DecodeWorkload):
    """The prefill of a second-order decode workload as forward workloads over
    blocks of at most DECODE_PREFILL_ROWS sequences.  Yields (b0, Workload): the
    block's first sequence and its recipe, drawn on the device by
    make_inputs_device (L2-normalised q, k, v ~ N(0,1), bf16, seed dw.seed * 1000 + b0)."""
    base = Workload("decode_prefix", dw.seqs, dw.H, dw.prefix, dw.d, dw.dv, max(dw.chunk, 64), "bf16", "l2",
                    seed=dw.seed)
    for b0 in range(0, dw.seqs, DECODE_PREFILL_ROWS):
        yield b0, base.with_(B=min(DECODE_PREFILL_ROWS, dw.seqs - b0), seed=dw.seed * 1000 + b0)


def decode_tokens_device(dw: DecodeWorkload, count: int, device="cuda"):
    """`count` token sets of a decode workload, drawn on the device with torch's
    generator seeded by dw.seed: per set q [seqs*H, d], k [seqs*H, d] (N(0,1),
    rows L2-normalised) and v [seqs*H, dv] (N(0,1)), in that order, as bf16.
    Step i of the workload uses set i % count."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(dw.seed)
    N = dw.seqs * dw.H

    def draw(shape):
        x = torch.randn(shape, generator=g, device=device)
        return (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)

    return [(draw((N, dw.d)), draw((N, dw.d)),
             torch.randn((N, dw.dv), generator=g, device=device).to(torch.bfloat16)) for _ in range(count)]


def make_inputs_device(w: Workload, device="cuda"):
    """Same recipe drawn on the device with torch's seeded generator, for
    workloads too large to draw on the host (the decode prefix).  Returns
    torch tensors in the input dtype.  Values differ from make_inputs (another
    generator); whoever checks against the oracle copies the drawn values back."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def draw(shape, kind, dim):
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if kind == "l2":
            x = x / x.norm(dim=-1, keepdim=True)
        elif kind == "scaled":
            x = x / dim ** 0.5
        elif kind == "elu1":
            x = torch.nn.functional.elu(x) + 1.0
        return x.to(dt)

    q = draw((w.B, w.H, w.n, w.d), w.qk, w.d)
    k = draw((w.B, w.kv_heads, w.n, w.d), w.qk, w.d)
    v = draw((w.B, w.kv_heads, w.n, w.dv), "none", w.dv)
    gamma = None
    if w.decay:
        u = torch.rand((w.H,), generator=g, device=device, dtype=torch.float64)
        lo, hi = np.log(w.gamma_lo), np.log(w.gamma_hi)
        gamma = torch.exp(lo + (hi - lo) * u).to(torch.float32)
    return {"q": q, "k": k, "v": v, "gamma": gamma}
