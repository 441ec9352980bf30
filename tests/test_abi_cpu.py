"""C-ABI checks that need no GPU: the library loads, exports every function that
include/hla.h declares, and rejects bad arguments with a status code before any
CUDA work."""
import ctypes
import os
import re

import pytest

import causal_prefix_scan_gb300 as hla
from causal_prefix_scan_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "hla.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return hla.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hla_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(hla.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_has_no_oracle_symbols(lib):
    for name in ("hla_oracle_forward", "hla_oracle_combine"):
        with pytest.raises(AttributeError):
            getattr(lib, name)


def test_status_strings(lib):
    for s in range(5):
        assert hla.hla_status_string(s)


def _params(**kw):
    base = dict(B=1, H=2, n=128, d=64, dv=64, chunk=64, in_dtype=hla.HLA_BF16, flags=0, eps=0.0, gamma=None, Hkv=0)
    base.update(kw)
    return hla.hla_params(**base)


def _call(p, q=16, k=16, v=16, o=16, sin=None, sout=None, ws=None, ws_bytes=0):
    return hla.library().hla_forward_chunked(ctypes.byref(p) if p is not None else None, q, k, v, o, sin, sout,
                                             ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), hla.HLA_ERR_ARG),
    (dict(H=0), hla.HLA_ERR_ARG),
    (dict(n=-1), hla.HLA_ERR_ARG),
    (dict(in_dtype=7), hla.HLA_ERR_ARG),
    (dict(flags=16), hla.HLA_ERR_ARG),
    (dict(flags=hla.HLA_UNMASKED | hla.HLA_ASYMMETRIC), hla.HLA_ERR_ARG),
    (dict(flags=hla.HLA_ASYMMETRIC, d=128, dv=96), hla.HLA_ERR_UNSUPPORTED),
    (dict(H=6, Hkv=4), hla.HLA_ERR_ARG),                    # key/value heads must divide H
    (dict(Hkv=-1), hla.HLA_ERR_ARG),
    (dict(flags=hla.HLA_DECAY), hla.HLA_ERR_ARG),          # decay without gamma
    (dict(flags=hla.HLA_NORMALIZE, eps=-1.0), hla.HLA_ERR_ARG),
    (dict(d=48), hla.HLA_ERR_UNSUPPORTED),
    (dict(chunk=256), hla.HLA_ERR_UNSUPPORTED),
    (dict(in_dtype=hla.HLA_F32, d=128, flags=hla.HLA_UNMASKED), hla.HLA_ERR_UNSUPPORTED),
    (dict(in_dtype=hla.HLA_F32, dv=96), hla.HLA_ERR_UNSUPPORTED),
])
def test_forward_rejects_bad_params(lib, kw, status):
    assert _call(_params(**kw)) == status
    assert hla.hla_last_error()


def test_forward_asymmetric_value_halves(lib):
    """AHLA at dv = 128, d <= 64 runs as two 64-column value halves: the half problem's
    workspace, then the gathered value half, the output half (input type) and the C, G
    halves of state_in and state_out (fp32), in 256-byte aligned regions."""
    al = lambda x: -(-x // 256) * 256
    for dt, el in ((hla.HLA_F32, 4), (hla.HLA_BF16, 2)):
        for d in (16, 32, 64):
            B, H, Hkv, n = 2, 4, 2, 100
            kw = dict(B=B, H=H, Hkv=Hkv, n=n, d=d, chunk=64, in_dtype=dt, flags=hla.HLA_ASYMMETRIC)
            inner = hla.hla_forward_workspace_size(_params(dv=64, **kw))
            rq, rkv, cg = B * H * n, B * Hkv * n, B * H * d * 64 * 4
            want = al(inner) + al(rkv * 64 * el) + al(rq * 64 * el) + 2 * al(2 * cg)
            assert hla.hla_forward_workspace_size(_params(dv=128, **kw)) == want
            assert hla.hla_forward_kernel(_params(dv=128, **kw)) == hla.hla_forward_kernel(_params(dv=64, **kw))
    assert _call(_params(flags=hla.HLA_ASYMMETRIC, dv=128), ws=16, ws_bytes=1 << 40) == hla.HLA_ERR_ARG
    assert "256" in hla.hla_last_error()
    # the unmasked variant splits only where no kernel takes the shape whole
    um = dict(flags=hla.HLA_UNMASKED, dv=128, n=100)
    assert hla.hla_forward_workspace_size(_params(d=64, **um)) == \
        hla.hla_forward_workspace_size(_params(d=64, **um, in_dtype=hla.HLA_BF16))  # tensor cores, no split
    for d in (16, 32, 64):
        assert hla.hla_forward_workspace_size(_params(d=d, in_dtype=hla.HLA_F32, **um)) > 0


def test_forward_rejects_null_and_misaligned(lib):
    assert _call(None) == hla.HLA_ERR_ARG
    assert _call(_params(), q=None) == hla.HLA_ERR_ARG
    assert _call(_params(), v=8) == hla.HLA_ERR_ARG  # not 16-byte aligned
    # tensor-core shape with no workspace
    assert _call(_params()) == hla.HLA_ERR_ARG
    assert "workspace" in hla.hla_last_error()
    bad = hla.hla_state(16, 16, None, 16, 16)
    assert _call(_params(), sout=ctypes.pointer(bad)) == hla.HLA_ERR_ARG


def test_combine_and_decode_reject_bad_args(lib):
    L = hla.library()
    st = hla.hla_state(16, 16, 16, 16, 16)
    sp = ctypes.pointer(st)
    assert L.hla_state_combine(-1, 64, 64, 0, sp, sp, sp, None, None) == hla.HLA_ERR_ARG
    assert L.hla_state_combine(1, 48, 64, 0, sp, sp, sp, None, None) == hla.HLA_ERR_UNSUPPORTED
    assert L.hla_state_combine(1, 64, 64, 0, None, sp, sp, None, None) == hla.HLA_ERR_ARG
    assert L.hla_state_combine(1, 64, 64, hla.HLA_UNMASKED | hla.HLA_ASYMMETRIC, sp, sp, sp, None,
                               None) == hla.HLA_ERR_ARG
    assert L.hla_decode_step(5, 2, 0, 64, 64, hla.HLA_BF16, 0, 0.0, None, sp, 16, 16, 16, 16, None) == hla.HLA_ERR_ARG
    assert L.hla_decode_step(4, 2, 0, 64, 64, hla.HLA_BF16, hla.HLA_DECAY, 0.0, None, sp, 16, 16, 16, 16,
                             None) == hla.HLA_ERR_ARG
    assert L.hla_decode_step(4, 2, 0, 64, 64, 9, 0, 0.0, None, sp, 16, 16, 16, 16, None) == hla.HLA_ERR_ARG
    assert L.hla_decode_step(4, 2, 0, 64, 64, hla.HLA_BF16, 0, 0.0, None, None, 16, 16, 16, 16,
                             None) == hla.HLA_ERR_ARG
    # key/value heads must divide the query heads; flag bits above HLA_ASYMMETRIC are unknown
    assert L.hla_decode_step(6, 3, 2, 64, 64, hla.HLA_BF16, 0, 0.0, None, sp, 16, 16, 16, 16, None) == hla.HLA_ERR_ARG
    assert L.hla_decode_step(4, 2, 0, 64, 64, hla.HLA_BF16, 16, 0.0, None, sp, 16, 16, 16, 16, None) == hla.HLA_ERR_ARG
    assert L.hla_decode_step(4, 2, 0, 64, 64, hla.HLA_BF16, hla.HLA_UNMASKED | hla.HLA_ASYMMETRIC, 0.0, None, sp,
                             16, 16, 16, 16, None) == hla.HLA_ERR_ARG
    # the unmasked state needs S, C, m only
    um = hla.hla_state(16, 16, None, None, None)
    assert L.hla_decode_step(4, 2, 0, 64, 64, hla.HLA_BF16, hla.HLA_UNMASKED, 0.0, None, ctypes.pointer(um),
                             16, 16, 16, 16, None) == hla.HLA_ERR_ARG


def test_workspace_size_zero_for_invalid(lib):
    assert hla.hla_forward_workspace_size(_params(d=48)) == 0
    assert hla.hla_forward_workspace_size(_params(in_dtype=hla.HLA_F32, d=16, dv=16, chunk=32)) == 0


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(hla, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        hla.library(str(tmp_path / "nope.so"))


def _bcall(p, ptrs=(16,) * 7, ws=16, ws_bytes=1 << 40):
    q, k, v, do, dq, dk, dv = ptrs
    return hla.library().hla_backward_chunked(ctypes.byref(p) if p is not None else None, q, k, v, do, dq, dk, dv,
                                              ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), hla.HLA_ERR_ARG),
    (dict(n=-1), hla.HLA_ERR_ARG),
    (dict(flags=16), hla.HLA_ERR_ARG),
    (dict(flags=hla.HLA_DECAY), hla.HLA_ERR_ARG),            # decay without gamma
    (dict(flags=hla.HLA_NORMALIZE, eps=-1.0), hla.HLA_ERR_ARG),
    (dict(flags=hla.HLA_UNMASKED), hla.HLA_ERR_UNSUPPORTED),
    (dict(flags=hla.HLA_ASYMMETRIC), hla.HLA_ERR_UNSUPPORTED),
    (dict(H=6, Hkv=4), hla.HLA_ERR_ARG),
    (dict(dv=96), hla.HLA_ERR_UNSUPPORTED),
    (dict(chunk=256), hla.HLA_ERR_UNSUPPORTED),
    (dict(d=48), hla.HLA_ERR_UNSUPPORTED),
])
def test_backward_rejects_bad_params(lib, kw, status):
    assert _bcall(_params(**kw)) == status
    assert hla.hla_last_error()
    assert hla.hla_backward_workspace_size(_params(**kw)) == 0


def test_backward_rejects_null_misaligned_and_short_workspace(lib):
    assert _bcall(None) == hla.HLA_ERR_ARG
    assert _bcall(_params(), ptrs=(16, 16, 16, None, 16, 16, 16)) == hla.HLA_ERR_ARG
    assert _bcall(_params(), ptrs=(16, 16, 16, 16, 16, 8, 16)) == hla.HLA_ERR_ARG
    need = hla.hla_backward_workspace_size(_params())
    assert _bcall(_params(), ws_bytes=need - 1) == hla.HLA_ERR_ARG
    assert "workspace" in hla.hla_last_error()
    assert _bcall(_params(), ws=None) == hla.HLA_ERR_ARG
    assert _bcall(_params(), ws=8) == hla.HLA_ERR_ARG


def test_backward_workspace_size_and_empty_sequence(lib):
    # per (b,h, chunk): six local sums and four states; per (b,h) the adjoints at the
    # first token (Lam d x dv, Om d x d) for the gradient of a given state; fp32
    for B, H, n, d, dv, c in [(1, 2, 128, 64, 64, 64), (2, 3, 100, 32, 16, 32), (1, 1, 1, 16, 64, 16)]:
        nch = -(-n // c)
        want = (B * H * nch * (4 * d * d + 6 * d * dv) + B * H * (d * dv + d * d)) * 4
        got = hla.hla_backward_workspace_size(_params(B=B, H=H, n=n, d=d, dv=dv, chunk=c, in_dtype=hla.HLA_F32))
        assert got == want
    # shared key/value heads: plus the fp32 dk, dv of every query head before the group sum
    B, H, n, d, dv, c = 2, 4, 100, 32, 16, 32
    nch = -(-n // c)
    base = (B * H * nch * (4 * d * d + 6 * d * dv) + B * H * (d * dv + d * d)) * 4
    assert hla.hla_backward_workspace_size(_params(B=B, H=H, Hkv=2, n=n, d=d, dv=dv, chunk=c,
                                                   in_dtype=hla.HLA_F32)) == base + B * H * n * (d + dv) * 4
    # no tokens: nothing to compute, no pointer needed
    assert _bcall(_params(n=0), ptrs=(None,) * 7, ws=None, ws_bytes=0) == hla.HLA_OK
    assert _bcall(_params(n=0, flags=hla.HLA_NORMALIZE), ptrs=(None,) * 7, ws=None, ws_bytes=0) == hla.HLA_OK


def test_backward_normalised_workspace(lib):
    # two unnormalised fp32 backwards and forwards share the scratch: at least the
    # backward workspace plus the fp32 outputs of both forwards and the upstream gradients
    for dt in (hla.HLA_F32, hla.HLA_BF16):
        B, H, n, d, dv, c = 2, 3, 100, 32, 16, 32
        plain = hla.hla_backward_workspace_size(_params(B=B, H=H, n=n, d=d, dv=dv, chunk=c, in_dtype=dt))
        norm = hla.hla_backward_workspace_size(_params(B=B, H=H, n=n, d=d, dv=dv, chunk=c, in_dtype=dt,
                                                       flags=hla.HLA_NORMALIZE, eps=1e-3))
        rows = B * H * n
        assert norm >= plain + rows * 4 * (2 * dv + 3 * 16 + 2 * d)
        assert norm % 256 == 0
    assert hla.hla_backward_workspace_size(_params(n=0, flags=hla.HLA_NORMALIZE)) == 0
    # the tensor-core shape (bf16, d = dv = chunk = 64) also covers that path's layout: per
    # chunk six 64 x 64 local sums and four vectors, four states and two vectors; r and c
    # per token; with shared key/value heads the per-query-head dk, dv
    for Hkv in (3, 1):
        B, H, n = 2, 3, 100
        units, nch = B * H, -(-n // 64)
        need = 4 * (units * nch * ((6 * 4096 + 4 * 64) + (4 * 4096 + 2 * 64)) + 2 * units * n
                    + (2 * units * n * 64 if Hkv < H else 0))
        got = hla.hla_backward_workspace_size(_params(B=B, H=H, Hkv=Hkv, n=n, d=64, dv=64, chunk=64,
                                                      in_dtype=hla.HLA_BF16, flags=hla.HLA_NORMALIZE, eps=1e-3))
        assert got >= need and got % 256 == 0
    # the scratch must be 256-byte aligned with HLA_NORMALIZE
    p = _params(flags=hla.HLA_NORMALIZE, eps=1e-3)
    assert _bcall(p, ws=16) == hla.HLA_ERR_ARG
    assert "256" in hla.hla_last_error()


def test_backward_traced_rejects_missing_events(lib):
    p = _params()
    ev = (ctypes.c_void_p * 4)(16, 16, None, 16)
    assert hla.library().hla_backward_chunked_traced(ctypes.byref(p), 16, 16, 16, 16, 16, 16, 16, 16, 1 << 40, None,
                                                     ev) == hla.HLA_ERR_ARG
    assert "event" in hla.hla_last_error()


def _f3call(p, ptrs=(16,) * 4, sin=None, sout=None, ws=16, ws_bytes=1 << 40):
    q, k, v, o = ptrs
    return hla.library().hla_forward3_chunked(ctypes.byref(p) if p is not None else None, q, k, v, o, sin, sout, ws,
                                              ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), hla.HLA_ERR_ARG),
    (dict(n=-1), hla.HLA_ERR_ARG),
    (dict(flags=16), hla.HLA_ERR_ARG),
    (dict(flags=hla.HLA_NORMALIZE, eps=-1.0), hla.HLA_ERR_ARG),
    (dict(flags=hla.HLA_DECAY), hla.HLA_ERR_ARG),  # decay without rates
    (dict(flags=hla.HLA_UNMASKED), hla.HLA_ERR_UNSUPPORTED),
    (dict(flags=hla.HLA_ASYMMETRIC), hla.HLA_ERR_UNSUPPORTED),
    (dict(H=6, Hkv=4), hla.HLA_ERR_ARG),
    (dict(d=48), hla.HLA_ERR_UNSUPPORTED),
    (dict(chunk=256), hla.HLA_ERR_UNSUPPORTED),
    (dict(dv=48), hla.HLA_ERR_UNSUPPORTED),
    (dict(dv=96), hla.HLA_ERR_UNSUPPORTED),
])
def test_forward3_rejects_bad_params(lib, kw, status):
    assert _f3call(_params(**kw)) == status
    assert hla.hla_last_error()
    assert hla.hla_forward3_workspace_size(_params(**kw)) == 0


def test_forward3_value_halves_and_long_chunks(lib):
    """dv = 128 runs as two 64-column halves: the half problem's workspace, the value and
    output halves (input type) and the P, T, M^QP halves of state_in and state_out (fp32),
    in 256-byte aligned regions; a 128-token chunk as two of 64 tokens (the same workspace)."""
    al = lambda x: -(-x // 256) * 256
    for dt, el in ((hla.HLA_F32, 4), (hla.HLA_BF16, 2)):
        for flags in (0, hla.HLA_NORMALIZE):
            B, H, n, d, c = 2, 3, 100, 32, 32
            kw = dict(B=B, H=H, n=n, d=d, chunk=c, in_dtype=dt, flags=flags, eps=1e-3)
            inner = hla.hla_forward3_workspace_size(_params(dv=64, **kw))
            rows, half = B * H * n, B * H * d * 64 * 4
            want = al(inner) + 2 * al(rows * 64 * el) + 2 * al(3 * half)
            assert hla.hla_forward3_workspace_size(_params(dv=128, **kw)) == want
        assert hla.hla_forward3_workspace_size(_params(chunk=128, in_dtype=dt)) == \
            hla.hla_forward3_workspace_size(_params(chunk=64, in_dtype=dt))
    assert _f3call(_params(dv=128), ws=16) == hla.HLA_ERR_ARG
    assert "256" in hla.hla_last_error()


def test_forward3_key_width_128(lib):
    """d = 128 runs in 16-token chunks over slices of at most 32 value columns: dv <= 32
    is the plain layout at chunk 16 (whatever chunk is asked for), wider values split like
    dv = 128 at d <= 64 with 32-column slices."""
    al = lambda x: -(-x // 256) * 256
    B, H, n, d = 1, 2, 100, 128
    for dv in (16, 32):
        want = B * H * (-(-n // 16)) * (4 * d * d + 5 * d * dv) * 4
        for c in (16, 32, 64, 128):
            assert hla.hla_forward3_workspace_size(_params(B=B, H=H, n=n, d=d, dv=dv, chunk=c)) == want
    for dt, el in ((hla.HLA_F32, 4), (hla.HLA_BF16, 2)):
        inner = hla.hla_forward3_workspace_size(_params(B=B, H=H, n=n, d=d, dv=32, chunk=16, in_dtype=dt))
        rows, part = B * H * n, B * H * d * 32 * 4
        for dv in (64, 128):
            want = al(inner) + 2 * al(rows * 32 * el) + 2 * al(3 * part)
            assert hla.hla_forward3_workspace_size(_params(B=B, H=H, n=n, d=d, dv=dv, chunk=64, in_dtype=dt)) == want


def test_forward3_rejects_null_misaligned_short_workspace_and_aliasing(lib):
    assert _f3call(None) == hla.HLA_ERR_ARG
    assert _f3call(_params(), ptrs=(16, None, 16, 16)) == hla.HLA_ERR_ARG
    assert _f3call(_params(), ptrs=(16, 16, 8, 16)) == hla.HLA_ERR_ARG
    need = hla.hla_forward3_workspace_size(_params())
    assert _f3call(_params(), ws_bytes=need - 1) == hla.HLA_ERR_ARG
    s3 = hla.hla_state3(16, 16, 16)
    assert _f3call(_params(), sin=ctypes.pointer(s3), sout=ctypes.pointer(s3)) == hla.HLA_ERR_ARG
    bad = hla.hla_state3(16, None, 16)
    assert _f3call(_params(), sout=ctypes.pointer(bad)) == hla.HLA_ERR_ARG
    # ratio normalisation: the state needs m and h; the workspace 256-byte alignment
    pn = _params(flags=hla.HLA_NORMALIZE)
    assert _f3call(pn, sout=ctypes.pointer(hla.hla_state3(16, 16, 16))) == hla.HLA_ERR_ARG
    assert _f3call(pn, ws=272) == hla.HLA_ERR_ARG
    # no tokens and no state: nothing to do
    assert _f3call(_params(n=0), ptrs=(None,) * 4, ws=None, ws_bytes=0) == hla.HLA_OK


def test_forward3_workspace_size(lib):
    # per (b,h, chunk): local sums 3d^2 + 3 d dv and prefix state d^2 + 2 d dv, fp32
    for B, H, n, d, dv, c in [(1, 2, 128, 64, 64, 64), (2, 3, 100, 32, 16, 32)]:
        nch = -(-n // c)
        want = B * H * nch * (4 * d * d + 5 * d * dv) * 4
        assert hla.hla_forward3_workspace_size(_params(B=B, H=H, n=n, d=d, dv=dv, chunk=c)) == want


def test_backward_value_halves_and_long_chunks(lib):
    """dv = 128 runs as two 64-column halves: the half problem's workspace, then the two
    gathered halves, the half's dq, dk, dv and the fp32 sums of dq, dk (256-byte aligned
    regions).  A 128-token chunk runs as two 64-token ones: the same workspace as chunk 64."""
    al = lambda x: -(-x // 256) * 256
    for dt, el in ((hla.HLA_F32, 4), (hla.HLA_BF16, 2)):
        for flags in (0, hla.HLA_NORMALIZE):
            B, H, Hkv, n, d, c = 2, 4, 2, 100, 32, 32
            kw = dict(B=B, H=H, Hkv=Hkv, n=n, d=d, chunk=c, in_dtype=dt, flags=flags, eps=1e-3)
            inner = hla.hla_backward_workspace_size(_params(dv=64, **kw))
            rq, rkv = B * H * n, B * Hkv * n
            want = al(inner) + al(rkv * 64 * el) + al(rq * 64 * el) + al(rq * d * el) + al(rkv * d * el) \
                + al(rkv * 64 * el) + al(rq * d * 4) + al(rkv * d * 4)
            assert hla.hla_backward_workspace_size(_params(dv=128, **kw)) == want
    for flags in (0, hla.HLA_NORMALIZE):
        a = hla.hla_backward_workspace_size(_params(chunk=128, flags=flags, eps=1e-3))
        assert a > 0 and a == hla.hla_backward_workspace_size(_params(chunk=64, flags=flags, eps=1e-3))
    # the split needs a 256-byte aligned workspace, and supports no given state
    assert _bcall(_params(dv=128), ws=16) == hla.HLA_ERR_ARG
    good = ctypes.pointer(hla.hla_state(256, 256, 256, 256, 256))
    assert hla.library().hla_backward_chunked_state(ctypes.byref(_params(dv=128)), 16, 16, 16, 16, good, 16, 16, 16,
                                                    None, 256, 1 << 40, None) == hla.HLA_ERR_UNSUPPORTED
    assert "dv = 128" in hla.hla_last_error()


def test_backward_key_width_128(lib):
    """d = 128 runs in 16-token chunks over slices of at most 32 value columns: dv <= 32
    is the plain layout at chunk 16 (whatever chunk is asked for); wider values are split
    like dv = 128 at d <= 64, with 32-column slices."""
    al = lambda x: -(-x // 256) * 256
    B, H, n, d = 1, 2, 100, 128
    for dv in (16, 32):
        nch = -(-n // 16)
        want = (B * H * nch * (4 * d * d + 6 * d * dv) + B * H * (d * dv + d * d)) * 4
        for c in (16, 32, 64, 128):
            assert hla.hla_backward_workspace_size(_params(B=B, H=H, n=n, d=d, dv=dv, chunk=c,
                                                           in_dtype=hla.HLA_F32)) == want
    for dt, el in ((hla.HLA_F32, 4), (hla.HLA_BF16, 2)):
        inner = hla.hla_backward_workspace_size(_params(B=B, H=H, n=n, d=d, dv=32, chunk=16, in_dtype=dt))
        rq = B * H * n
        for dv in (64, 128):
            want = al(inner) + al(rq * 32 * el) + al(rq * 32 * el) + al(rq * d * el) + al(rq * d * el) \
                + al(rq * 32 * el) + al(rq * d * 4) + al(rq * d * 4)
            assert hla.hla_backward_workspace_size(_params(B=B, H=H, n=n, d=d, dv=dv, chunk=64, in_dtype=dt)) == want
    # a split supports no given state; dv <= 32 does
    good = ctypes.pointer(hla.hla_state(256, 256, 256, 256, 256))
    assert hla.library().hla_backward_chunked_state(ctypes.byref(_params(d=128, dv=64)), 16, 16, 16, 16, good, 16,
                                                    16, 16, None, 256, 1 << 40, None) == hla.HLA_ERR_UNSUPPORTED
    assert "d = 128 with dv > 32" in hla.hla_last_error()
    assert hla.hla_backward_workspace_size(_params(d=128, dv=128, chunk=128, flags=hla.HLA_DECAY, gamma=16)) > 0
    assert hla.hla_backward_workspace_size(_params(d=128, dv=128, chunk=64, flags=hla.HLA_NORMALIZE, eps=1e-3)) > 0


def test_backward_state_rejects_bad_args(lib):
    L = hla.library()
    good = ctypes.pointer(hla.hla_state(16, 16, 16, 16, 16))
    call = lambda p, sin=good, dst=good: L.hla_backward_chunked_state(ctypes.byref(p), 16, 16, 16, 16, sin, 16, 16,
                                                                       16, dst, 16, 1 << 40, None)
    assert call(_params(flags=hla.HLA_NORMALIZE, eps=-1.0)) == hla.HLA_ERR_ARG
    assert call(_params(), sin=ctypes.pointer(hla.hla_state(16, None, 16, 16, 16))) == hla.HLA_ERR_ARG
    assert call(_params(), dst=ctypes.pointer(hla.hla_state(16, 16, 8, 16, 16))) == hla.HLA_ERR_ARG
    assert call(_params(d=48)) == hla.HLA_ERR_UNSUPPORTED


def test_state3_combine_rejects_bad_args(lib):
    L = hla.library()
    full = ctypes.pointer(hla.hla_state3(16, 16, 16, 16, 16, 16, 16, 16, 16))
    nomaps = ctypes.pointer(hla.hla_state3(16, 16, 16, 16, 16))
    call = lambda count=2, d=64, dv=64, fl=0, A=full, B=full, out=full: L.hla_state3_combine(count, d, dv, fl, A, B,
                                                                                             out, None, None)
    assert call(count=-1) == hla.HLA_ERR_ARG
    assert call(d=48) == hla.HLA_ERR_UNSUPPORTED
    assert call(d=128, dv=96) == hla.HLA_ERR_UNSUPPORTED
    assert call(fl=hla.HLA_DECAY) == hla.HLA_ERR_UNSUPPORTED
    assert call(A=None) == hla.HLA_ERR_ARG
    assert call(B=nomaps) == hla.HLA_ERR_ARG
    assert call(count=0) == hla.HLA_OK  # nothing to do
    # a forward that wants the maps needs them on a given state_in too
    sout = ctypes.pointer(hla.hla_state3(16, 16, 16, 16, 16, 16, 16, 16, 16))
    assert _f3call(_params(), sin=nomaps, sout=sout) == hla.HLA_ERR_ARG


def test_decode3_rejects_bad_args(lib):
    L = hla.library()
    s3 = ctypes.pointer(hla.hla_state3(16, 16, 16))
    call = lambda N=4, H=1, d=64, dv=64, dt=hla.HLA_BF16, fl=0, eps=0.0, g=None, st=s3: L.hla_decode3_step(
        N, H, d, dv, dt, fl, eps, g, st, 16, 16, 16, 16, None)
    assert call(N=-1) == hla.HLA_ERR_ARG
    assert call(H=0) == hla.HLA_ERR_ARG
    assert call(d=48) == hla.HLA_ERR_UNSUPPORTED
    assert call(dt=9) == hla.HLA_ERR_ARG
    assert call(st=None) == hla.HLA_ERR_ARG
    assert call(st=ctypes.pointer(hla.hla_state3(16, 8, 16))) == hla.HLA_ERR_ARG
    assert call(fl=hla.HLA_UNMASKED) == hla.HLA_ERR_UNSUPPORTED
    assert call(fl=hla.HLA_DECAY) == hla.HLA_ERR_ARG  # no rates
    assert call(fl=hla.HLA_NORMALIZE) == hla.HLA_ERR_ARG  # no m, h
    assert call(fl=hla.HLA_NORMALIZE, eps=-1.0, st=ctypes.pointer(hla.hla_state3(16, 16, 16, 16, 16))) == hla.HLA_ERR_ARG
