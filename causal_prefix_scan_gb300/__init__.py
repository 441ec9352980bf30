"""GB300-native second-order Higher-order Linear Attention (HLA): masked, unmasked and
the asymmetric variant AHLA, the backward pass of the masked forward, and masked
third-order HLA (forward and decode).

Thin ctypes binding over the C ABI in ``include/hla.h`` (library
``_lib/libhla_gb300.so``, built for sm_103a by ``_build.build()``).  Functions named
like the C entry points take device pointers (ints) or torch CUDA tensors and only
marshal arguments; every step of the computation runs in the library's kernels.
PyTorch is used for device memory and streams only.

If the library has not been built, every call raises ``RuntimeError``: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

from ._build import LIB_PATH

HLA_OK, HLA_ERR_ARG, HLA_ERR_UNSUPPORTED, HLA_ERR_CUDA, HLA_ERR_TIMEOUT = 0, 1, 2, 3, 4
HLA_F32, HLA_BF16 = 0, 1
HLA_NORMALIZE, HLA_DECAY, HLA_UNMASKED, HLA_ASYMMETRIC = 1, 2, 4, 8

__all__ = [
    "HLA_OK", "HLA_ERR_ARG", "HLA_ERR_UNSUPPORTED", "HLA_ERR_CUDA", "HLA_ERR_TIMEOUT",
    "HLA_F32", "HLA_BF16", "HLA_NORMALIZE", "HLA_DECAY", "HLA_UNMASKED", "HLA_ASYMMETRIC",
    "HlaError", "hla_params", "hla_state", "library", "EXPORTS",
    "hla_forward_workspace_size", "hla_forward_kernel", "hla_forward_chunked", "hla_state_combine",
    "hla_decode_step", "hla_sync_status", "hla_status_string", "hla_last_error", "hla_forward_chunked_noalloc",
    "hla_backward_workspace_size", "hla_backward_chunked", "hla_backward_chunked_traced",
    "hla_backward_chunked_state", "hla_state3", "hla_state3_combine", "state3_combine", "hla_forward3_workspace_size", "hla_forward3_chunked", "hla_forward3_chunked_traced",
    "hla_decode3_step", "State3", "forward3", "decode3_step", "hla_selftest_expired_wait",
    "State", "new_workspace", "forward", "state_combine", "decode_step", "backward",
]

# Every symbol include/hla.h declares.
EXPORTS = ("hla_forward_workspace_size", "hla_forward_chunked", "hla_state_combine", "hla_decode_step",
           "hla_sync_status", "hla_status_string", "hla_last_error", "hla_forward_chunked_noalloc",
           "hla_backward_workspace_size", "hla_backward_chunked", "hla_backward_chunked_traced",
           "hla_forward3_workspace_size", "hla_forward3_chunked", "hla_forward3_chunked_traced", "hla_decode3_step",
           "hla_selftest_expired_wait", "hla_forward_kernel", "hla_backward_chunked_state", "hla_state3_combine")


class HlaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


class hla_params(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("n", ctypes.c_int), ("d", ctypes.c_int),
                ("dv", ctypes.c_int), ("chunk", ctypes.c_int), ("in_dtype", ctypes.c_int),
                ("flags", ctypes.c_uint), ("eps", ctypes.c_float), ("gamma", ctypes.c_void_p),
                ("Hkv", ctypes.c_int)]


class hla_state(ctypes.Structure):
    _fields_ = [("S", ctypes.c_void_p), ("C", ctypes.c_void_p), ("m", ctypes.c_void_p),
                ("G", ctypes.c_void_p), ("h", ctypes.c_void_p)]


class hla_state3(ctypes.Structure):
    _fields_ = [("S", ctypes.c_void_p), ("P", ctypes.c_void_p), ("T", ctypes.c_void_p),
                ("m", ctypes.c_void_p), ("h", ctypes.c_void_p),
                ("SQ", ctypes.c_void_p), ("MQP", ctypes.c_void_p), ("MKQ", ctypes.c_void_p), ("mqm", ctypes.c_void_p)]


_lib = None


def library(path: str | None = None):
    """Load libhla_gb300.so (raises RuntimeError if it was never built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, S, vp, sz = ctypes.POINTER(hla_params), ctypes.POINTER(hla_state), ctypes.c_void_p, ctypes.c_size_t
    i, u, f = ctypes.c_int, ctypes.c_uint, ctypes.c_float
    lib.hla_forward_workspace_size.argtypes = [P]
    lib.hla_forward_workspace_size.restype = sz
    lib.hla_forward_kernel.argtypes = [P]
    lib.hla_forward_kernel.restype = ctypes.c_char_p
    lib.hla_forward_chunked.argtypes = [P, vp, vp, vp, vp, S, S, vp, sz, vp]
    lib.hla_forward_chunked_noalloc.argtypes = [P, vp, vp, vp, vp, S, S, vp]
    lib.hla_forward_chunked_noalloc.restype = ctypes.c_int
    lib.hla_state_combine.argtypes = [i, i, i, u, S, S, S, vp, vp]
    lib.hla_decode_step.argtypes = [i, i, i, i, i, i, u, f, vp, S, vp, vp, vp, vp, vp]
    lib.hla_backward_workspace_size.argtypes = [P]
    lib.hla_backward_workspace_size.restype = sz
    lib.hla_backward_chunked.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.hla_backward_chunked_traced.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp,
                                                ctypes.POINTER(ctypes.c_void_p)]
    lib.hla_backward_chunked_state.argtypes = [P, vp, vp, vp, vp, ctypes.POINTER(hla_state), vp, vp, vp,
                                               ctypes.POINTER(hla_state), vp, sz, vp]
    S3 = ctypes.POINTER(hla_state3)
    lib.hla_forward3_workspace_size.argtypes = [P]
    lib.hla_forward3_workspace_size.restype = sz
    lib.hla_forward3_chunked.argtypes = [P, vp, vp, vp, vp, S3, S3, vp, sz, vp]
    lib.hla_forward3_chunked_traced.argtypes = [P, vp, vp, vp, vp, S3, S3, vp, sz, vp,
                                                ctypes.POINTER(ctypes.c_void_p)]
    lib.hla_decode3_step.argtypes = [i, i, i, i, i, u, f, vp, S3, vp, vp, vp, vp, vp]
    lib.hla_state3_combine.argtypes = [i, i, i, u, S3, S3, S3, vp, vp]
    lib.hla_sync_status.argtypes = [vp]
    lib.hla_selftest_expired_wait.argtypes = [vp]
    for fn in (lib.hla_forward_chunked, lib.hla_state_combine, lib.hla_decode_step, lib.hla_sync_status,
               lib.hla_backward_chunked, lib.hla_backward_chunked_traced, lib.hla_forward3_chunked,
               lib.hla_forward3_chunked_traced, lib.hla_decode3_step, lib.hla_selftest_expired_wait,
               lib.hla_state3_combine):
        fn.restype = ctypes.c_int
    lib.hla_status_string.argtypes = [ctypes.c_int]
    lib.hla_status_string.restype = ctypes.c_char_p
    lib.hla_last_error.argtypes = []
    lib.hla_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int):
    if status != HLA_OK:
        lib = library()
        raise HlaError(status, lib.hla_last_error().decode() or lib.hla_status_string(status).decode())


def _state_struct(st):
    if st is None:
        return None
    if isinstance(st, hla_state):
        return ctypes.pointer(st)
    return ctypes.pointer(hla_state(_ptr(st.S), _ptr(st.C), _ptr(st.m), _ptr(st.G), _ptr(st.h)))


# --------------------------------------------------------------------- raw ABI
def hla_status_string(status: int) -> str:
    return library().hla_status_string(status).decode()


def hla_last_error() -> str:
    return library().hla_last_error().decode()


def hla_forward_workspace_size(params: hla_params) -> int:
    return library().hla_forward_workspace_size(ctypes.byref(params))


def hla_forward_kernel(params: hla_params):
    """Name of the kernel the forward launches for these parameters (None: no launch)."""
    r = library().hla_forward_kernel(ctypes.byref(params))
    return r.decode() if r else None


def hla_forward_chunked(params: hla_params, q, k, v, o, state_in=None, state_out=None, workspace=None,
                        workspace_bytes: int = 0, stream=None) -> None:
    _check(library().hla_forward_chunked(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                         _state_struct(state_in), _state_struct(state_out), _ptr(workspace),
                                         workspace_bytes, _stream(stream)))


def hla_forward_chunked_noalloc(params: hla_params, q, k, v, o, state_in=None, state_out=None,
                                stream=None) -> None:
    """The forward without a caller workspace, for callers that cannot allocate
    device memory (the scratch is a fixed array inside the library; see hla.h)."""
    _check(library().hla_forward_chunked_noalloc(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                                 _state_struct(state_in), _state_struct(state_out),
                                                 _stream(stream)))


def hla_state_combine(count: int, d: int, dv: int, flags: int, A, B, out, decay_pow=None, stream=None) -> None:
    _check(library().hla_state_combine(count, d, dv, flags, _state_struct(A), _state_struct(B), _state_struct(out),
                                       _ptr(decay_pow), _stream(stream)))


def hla_decode_step(N: int, H: int, Hkv: int, d: int, dv: int, dtype: int, flags: int, eps: float, gamma,
                    state, q, k, v, o, stream=None) -> None:
    _check(library().hla_decode_step(N, H, Hkv, d, dv, dtype, flags, eps, _ptr(gamma), _state_struct(state),
                                     _ptr(q), _ptr(k), _ptr(v), _ptr(o), _stream(stream)))


def hla_backward_workspace_size(params: hla_params) -> int:
    return library().hla_backward_workspace_size(ctypes.byref(params))


def hla_backward_chunked(params: hla_params, q, k, v, dout, dq, dk, dv, workspace, workspace_bytes: int,
                         stream=None) -> None:
    _check(library().hla_backward_chunked(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq),
                                          _ptr(dk), _ptr(dv), _ptr(workspace), workspace_bytes, _stream(stream)))


def hla_backward_chunked_state(params: hla_params, q, k, v, dout, state_in, dq, dk, dv, d_state_in, workspace,
                               workspace_bytes: int, stream=None) -> None:
    _check(library().hla_backward_chunked_state(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                                _state_struct(state_in), _ptr(dq), _ptr(dk), _ptr(dv),
                                                _state_struct(d_state_in), _ptr(workspace), workspace_bytes,
                                                _stream(stream)))


def hla_backward_chunked_traced(params: hla_params, q, k, v, dout, dq, dk, dv, workspace, workspace_bytes: int,
                                stream=None, events=None) -> None:
    """hla_backward_chunked recording four events (torch.cuda.Event that have been
    recorded once, or raw cudaEvent_t ints) at its phase boundaries."""
    arr = None
    if events is not None:
        hs = [e if isinstance(e, int) else e.cuda_event for e in events]
        assert len(hs) == 4 and all(hs), "four created events are needed"
        arr = (ctypes.c_void_p * 4)(*hs)
    _check(library().hla_backward_chunked_traced(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                                 _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), workspace_bytes,
                                                 _stream(stream), arr))


def _state3_struct(st):
    if st is None:
        return None
    return ctypes.byref(hla_state3(*(_ptr(x) for x in (st.S, st.P, st.T, st.m, st.h, st.SQ, st.MQP, st.MKQ,
                                                         st.mqm))))


def _events(events):
    if events is None:
        return None
    hs = [e if isinstance(e, int) else e.cuda_event for e in events]
    assert len(hs) == 4 and all(hs), "four created events are needed"
    return (ctypes.c_void_p * 4)(*hs)


def hla_forward3_workspace_size(params: hla_params) -> int:
    return library().hla_forward3_workspace_size(ctypes.byref(params))


def hla_forward3_chunked(params: hla_params, q, k, v, o, state_in=None, state_out=None, workspace=None,
                         workspace_bytes: int = 0, stream=None) -> None:
    _check(library().hla_forward3_chunked(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                          _state3_struct(state_in), _state3_struct(state_out), _ptr(workspace),
                                          workspace_bytes, _stream(stream)))


def hla_forward3_chunked_traced(params: hla_params, q, k, v, o, state_in=None, state_out=None, workspace=None,
                                workspace_bytes: int = 0, stream=None, events=None) -> None:
    _check(library().hla_forward3_chunked_traced(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                                 _state3_struct(state_in), _state3_struct(state_out),
                                                 _ptr(workspace), workspace_bytes, _stream(stream),
                                                 _events(events)))


def hla_decode3_step(N: int, H: int, d: int, dv: int, dtype: int, flags: int, eps: float, gamma, state, q, k, v, o,
                     stream=None) -> None:
    _check(library().hla_decode3_step(N, H, d, dv, dtype, flags, eps, _ptr(gamma), _state3_struct(state), _ptr(q),
                                      _ptr(k), _ptr(v), _ptr(o), _stream(stream)))


def hla_state3_combine(count: int, d: int, dv: int, flags: int, A, B, out, decay_pow=None, stream=None) -> None:
    _check(library().hla_state3_combine(count, d, dv, flags, _state3_struct(A), _state3_struct(B),
                                        _state3_struct(out), _ptr(decay_pow), _stream(stream)))


def hla_selftest_expired_wait(stream=None) -> None:
    """Launch the failure-path self-test (a bounded wait that expires); the next
    hla_sync_status reports HLA_ERR_TIMEOUT."""
    _check(library().hla_selftest_expired_wait(_stream(stream)))


def hla_sync_status(stream=None) -> None:
    _check(library().hla_sync_status(_stream(stream)))


# ------------------------------------------------------- tensor-level helpers
@dataclass
class State:
    """Five fp32 summaries of `units` pairs: S [U,d,d], C [U,d,dv], m [U,d], G [U,d,dv], h [U,d]."""
    S: object
    C: object
    m: object
    G: object
    h: object

    @staticmethod
    def empty(units: int, d: int, dv: int, device="cuda") -> "State":
        import torch
        z = lambda *s: torch.empty(*s, dtype=torch.float32, device=device)
        return State(z(units, d, d), z(units, d, dv), z(units, d), z(units, d, dv), z(units, d))

    @staticmethod
    def zeros(units: int, d: int, dv: int, device="cuda") -> "State":
        import torch
        z = lambda *s: torch.zeros(*s, dtype=torch.float32, device=device)
        return State(z(units, d, d), z(units, d, dv), z(units, d), z(units, d, dv), z(units, d))

    def astuple(self):
        return (self.S, self.C, self.m, self.G, self.h)


@dataclass
class State3:
    """Third-order streaming state of `units` pairs, fp32: S [U,d,d] (key moment S^K),
    P [U,d,dv] (key-value moment), T [U,d,dv] (masked third-order accumulator); with
    ratio normalisation also m [U,d] (key mass) and h [U,d] (T of a unit value); with
    the segment maps (for state3_combine) SQ [U,d,d], MQP [U,d,dv], MKQ [U,d,d] and,
    normalised, mqm [U,d]."""
    S: object
    P: object
    T: object
    m: object = None
    h: object = None
    SQ: object = None
    MQP: object = None
    MKQ: object = None
    mqm: object = None

    @staticmethod
    def _make(z, units, d, dv, normalize, maps):
        mh = (z(units, d), z(units, d)) if normalize else (None, None)
        mp = (z(units, d, d), z(units, d, dv), z(units, d, d), z(units, d) if normalize else None) if maps else \
            (None,) * 4
        return State3(z(units, d, d), z(units, d, dv), z(units, d, dv), *mh, *mp)

    @staticmethod
    def empty(units: int, d: int, dv: int, device="cuda", normalize: bool = False, maps: bool = False) -> "State3":
        import torch
        return State3._make(lambda *s: torch.empty(*s, dtype=torch.float32, device=device), units, d, dv, normalize,
                            maps)

    @staticmethod
    def zeros(units: int, d: int, dv: int, device="cuda", normalize: bool = False, maps: bool = False) -> "State3":
        import torch
        return State3._make(lambda *s: torch.zeros(*s, dtype=torch.float32, device=device), units, d, dv, normalize,
                            maps)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return HLA_F32
    if t.dtype == torch.bfloat16:
        return HLA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _variant_flags(unmasked: bool, asymmetric: bool) -> int:
    return (HLA_UNMASKED if unmasked else 0) | (HLA_ASYMMETRIC if asymmetric else 0)


def make_params(q, v, chunk: int, gamma=None, normalize: bool = False, eps: float = 0.0,
                unmasked: bool = False, asymmetric: bool = False) -> hla_params:
    """Parameters for q [B,H,n,d] and v [B,Hkv,n,dv] (Hkv = H, or a divisor of H when
    key/value heads are shared)."""
    B, H, n, d = q.shape
    flags = (HLA_NORMALIZE if normalize else 0) | (HLA_DECAY if gamma is not None else 0) | \
        _variant_flags(unmasked, asymmetric)
    return hla_params(B, H, n, d, v.shape[-1], chunk, _dtype_code(q), flags, float(eps), _ptr(gamma),
                      v.shape[1])


def new_workspace(nbytes: int, device="cuda"):
    """A zeroed device workspace of `nbytes` (each forward call leaves it ready for the next)."""
    import torch
    return torch.zeros(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def forward(q, k, v, chunk: int, gamma=None, normalize: bool = False, eps: float = 0.0, state_in=None,
            return_state: bool = False, out=None, workspace=None, stream=None, unmasked: bool = False,
            asymmetric: bool = False):
    """2nd-order HLA forward (masked; unmasked with ``unmasked=True``; the asymmetric
    variant AHLA with ``asymmetric=True``, state R, P, m^K, E, n).  q [B,H,n,d],
    k [B,Hkv,n,d], v [B,Hkv,n,dv] contiguous CUDA tensors (bf16 or fp32; Hkv divides H);
    gamma [H] fp32 or None.  Returns o (and the final State)."""
    import torch
    p = make_params(q, v, chunk, gamma, normalize, eps, unmasked, asymmetric)
    o = out if out is not None else torch.empty(q.shape[:3] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    need = hla_forward_workspace_size(p)
    if workspace is None and need:
        workspace = new_workspace(need, q.device)
    st = State.empty(p.B * p.H, p.d, p.dv, device=q.device) if return_state else None
    hla_forward_chunked(p, q, k, v, o, state_in, st, workspace, need if workspace is not None else 0, stream)
    return (o, st) if return_state else o


def state_combine(A: State, B: State, decay_pow=None, out: State | None = None, stream=None,
                  unmasked: bool = False, asymmetric: bool = False) -> State:
    count, d, dv = A.C.shape
    out = out if out is not None else State.empty(count, d, dv, device=A.S.device)
    hla_state_combine(count, d, dv, _variant_flags(unmasked, asymmetric), A, B, out, decay_pow, stream)
    return out


def decode_step(state: State, q, k, v, H: int, gamma=None, normalize: bool = False, eps: float = 0.0,
                out=None, stream=None, unmasked: bool = False, asymmetric: bool = False):
    """One decode step for N pairs (q [N,d]; k [N/H*Hkv,d], v [N/H*Hkv,dv]); state
    updated in place."""
    import torch
    N, d = q.shape
    dv = v.shape[-1]
    Hkv = k.shape[0] * H // N if N else H
    o = out if out is not None else torch.empty((N, dv), dtype=q.dtype, device=q.device)
    flags = (HLA_NORMALIZE if normalize else 0) | (HLA_DECAY if gamma is not None else 0) | \
        _variant_flags(unmasked, asymmetric)
    hla_decode_step(N, H, Hkv, d, dv, _dtype_code(q), flags, float(eps), gamma, state, q, k, v, o, stream)
    return o


def backward(q, k, v, dout, chunk: int, gamma=None, workspace=None, out=None, stream=None,
             normalize: bool = False, eps: float = 0.0, state_in: State | None = None, want_dstate: bool = False):
    """Gradients (dq, dk, dv) of sum(dout * o) for the masked forward o of q, k, v from a
    zero state, or from ``state_in`` (with ``normalize=True`` the ratio-normalised o).  q [B,H,n,d], k [B,Hkv,n,d], v [B,Hkv,n,dv], dout [B,H,n,dv]
    contiguous CUDA tensors of one dtype (bf16 or fp32); gamma [H] fp32 or None.
    ``out`` may hold three preallocated result tensors.  ``want_dstate``: also return the
    gradient with respect to the initial state (a State)."""
    import torch
    p = make_params(q, v, chunk, gamma, normalize, eps)
    need = hla_backward_workspace_size(p)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    dq, dk, dv = out if out is not None else (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    if state_in is None and not want_dstate:
        hla_backward_chunked(p, q, k, v, dout, dq, dk, dv, workspace, need if workspace is not None else 0, stream)
        return dq, dk, dv
    dst = State.empty(p.B * p.H, p.d, p.dv, device=q.device) if want_dstate else None
    hla_backward_chunked_state(p, q, k, v, dout, state_in, dq, dk, dv, dst, workspace,
                               need if workspace is not None else 0, stream)
    return (dq, dk, dv, dst) if want_dstate else (dq, dk, dv)


def forward3(q, k, v, chunk: int, state_in: State3 | None = None, return_state: bool = False, out=None,
             workspace=None, stream=None, gamma=None, normalize: bool = False, eps: float = 0.0, maps: bool = False):
    """Masked third-order HLA forward.  q, k [B,H,n,d], v [B,H,n,dv] contiguous CUDA
    tensors (bf16 or fp32); gamma: [H] fp32 CUDA tensor of decay rates or None;
    normalize: o = num / (den + eps).  Returns o (and the final State3)."""
    import torch
    p = make_params(q, v, chunk, gamma, normalize, eps)
    o = out if out is not None else torch.empty(q.shape[:3] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    need = hla_forward3_workspace_size(p)
    if workspace is None and need:
        workspace = new_workspace(need, device=q.device)
    st = State3.empty(p.B * p.H, p.d, p.dv, device=q.device, normalize=normalize, maps=maps) if return_state else None
    hla_forward3_chunked(p, q, k, v, o, state_in, st, workspace, need if workspace is not None else 0, stream)
    return (o, st) if return_state else o


def state3_combine(A: State3, B: State3, decay_pow=None, normalize: bool = False, out: State3 | None = None,
                   stream=None) -> State3:
    """Concatenation (A before B) of third-order states with their segment maps, item by
    item; decay_pow [U] fp32 = gamma^(tokens of B) or None."""
    units, d, dv = A.P.shape
    if out is None:
        out = State3.empty(units, d, dv, device=A.P.device, normalize=normalize, maps=True)
    hla_state3_combine(units, d, dv, HLA_NORMALIZE if normalize else 0, A, B, out, decay_pow, stream)
    return out


def decode3_step(state: State3, q, k, v, out=None, stream=None, H: int = 1, gamma=None, normalize: bool = False,
                 eps: float = 0.0):
    """One third-order decode step for N pairs (q, k [N,d], v [N,dv]); state updated in
    place.  gamma: [H] decay rates (pair i uses gamma[i % H]) or None."""
    import torch
    N, d = q.shape
    dv = v.shape[-1]
    o = out if out is not None else torch.empty((N, dv), dtype=q.dtype, device=q.device)
    flags = (HLA_DECAY if gamma is not None else 0) | (HLA_NORMALIZE if normalize else 0)
    hla_decode3_step(N, H, d, dv, _dtype_code(q), flags, float(eps), gamma, state, q, k, v, o, stream)
    return o
