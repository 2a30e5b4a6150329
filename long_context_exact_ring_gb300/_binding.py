"""ctypes binding of libringattn.so -- argument marshalling only.

Every function here checks shapes and dtypes, allocates outputs with torch
(device-memory plumbing), passes raw device pointers and the current CUDA
stream to the C ABI (include/ring_attn.h), and raises on a non-zero status.
All arithmetic runs in the library's CUDA kernels; there is no fallback: if
the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libringattn.so")

RA_OK = 0
RA_ERR_INVALID_ARG = -1
RA_ERR_UNSUPPORTED = -2
RA_ERR_CUDA = -3
RA_ERR_DEVICE_TIMEOUT = -4

EXPORTED = (
    "ring_attn_fwd",
    "ring_attn_fwd_gqa",
    "ring_attn_bwd_gqa",
    "ring_attn_fwd_strided",
    "ring_attn_bwd_strided",
    "ring_attn_fwd_f32",
    "ring_attn_fwd_f32_workspace_size",
    "ring_attn_fwd_ulysses_emulated",
    "ring_attn_fwd_ulysses_workspace_size",
    "ring_attn_bwd_workspace_size",
    "ring_attn_fwd_emulated",
    "ring_attn_fwd_emulated_workspace_size",
    "ring_attn_bwd",
    "ring_attn_bwd_noalloc",
    "attn_merge_partials",
    "ring_attn_schedule",
    "ring_attn_check_status",
    "ring_attn_status_string",
    "ring_attn_last_error",
    "ring_attn_set_wait_limit_ns",
    "ring_attn_trace_visits",
    "ring_attn_profile_enable",
    "ring_attn_profile_reset",
    "ring_attn_profile_read",
)

_lock = threading.Lock()
_lib = None


class RingAttnError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        msg = f"{what} failed: {status_string(status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libringattn.so (raises OSError if it is absent)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise OSError(f"{p} not found: build it with python -m long_context_exact_ring_gb300.build")
        lib = ctypes.CDLL(p)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        ip = ctypes.POINTER(ctypes.c_int)
        lib.ring_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
        lib.ring_attn_fwd.restype = i
        lib.ring_attn_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
        llp = ctypes.POINTER(ctypes.c_longlong)
        lib.ring_attn_fwd_strided.argtypes = [vp, llp, vp, llp, vp, llp, vp, llp, vp, i, i, i, i, i, i,
                                              i, f, vp]
        lib.ring_attn_fwd_strided.restype = i
        lib.ring_attn_bwd_strided.argtypes = [vp, llp, vp, llp, vp, llp, vp, llp, vp, vp, llp, vp, llp,
                                              vp, llp, vp, llp, i, i, i, i, i, i, i, f, vp, sz, vp]
        lib.ring_attn_bwd_strided.restype = i
        lib.ring_attn_fwd_f32_workspace_size.argtypes = [i, i, i, i, i]
        lib.ring_attn_fwd_f32_workspace_size.restype = sz
        lib.ring_attn_fwd_f32.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp, sz, vp]
        lib.ring_attn_fwd_f32.restype = i
        lib.ring_attn_fwd_ulysses_workspace_size.argtypes = [i, i, i, i, i]
        lib.ring_attn_fwd_ulysses_workspace_size.restype = sz
        lib.ring_attn_fwd_ulysses_emulated.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp,
                                                       sz, vp]
        lib.ring_attn_fwd_ulysses_emulated.restype = i
        lib.ring_attn_fwd_gqa.restype = i
        lib.ring_attn_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i,
                                          f, vp, sz, vp]
        lib.ring_attn_bwd_gqa.restype = i
        lib.ring_attn_fwd_emulated.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp, sz, i, vp]
        lib.ring_attn_fwd_emulated.restype = i
        lib.ring_attn_fwd_emulated_workspace_size.argtypes = [i, i, i, i]
        lib.ring_attn_fwd_emulated_workspace_size.restype = sz
        lib.ring_attn_bwd_workspace_size.argtypes = [i, i, i, i]
        lib.ring_attn_bwd_workspace_size.restype = sz
        lib.ring_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f,
                                      vp, sz, vp]
        lib.ring_attn_bwd.restype = i
        lib.ring_attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i,
                                              f, vp]
        lib.ring_attn_bwd_noalloc.restype = i
        lib.attn_merge_partials.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, vp]
        lib.attn_merge_partials.restype = i
        lib.ring_attn_schedule.argtypes = [i, i, i, ip, ip, i]
        lib.ring_attn_schedule.restype = i
        lib.ring_attn_check_status.argtypes = [vp]
        lib.ring_attn_check_status.restype = i
        lib.ring_attn_status_string.argtypes = [i]
        lib.ring_attn_status_string.restype = ctypes.c_char_p
        lib.ring_attn_last_error.argtypes = []
        lib.ring_attn_last_error.restype = ctypes.c_char_p
        lib.ring_attn_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
        lib.ring_attn_set_wait_limit_ns.restype = i
        lib.ring_attn_trace_visits.argtypes = [vp, ctypes.c_longlong]
        lib.ring_attn_trace_visits.restype = i
        lib.ring_attn_profile_enable.argtypes = [i]
        lib.ring_attn_profile_enable.restype = i
        lib.ring_attn_profile_reset.argtypes = []
        lib.ring_attn_profile_reset.restype = i
        lib.ring_attn_profile_read.argtypes = [ctypes.c_char_p, ctypes.POINTER(ctypes.c_double),
                                               ctypes.POINTER(ctypes.c_longlong)]
        lib.ring_attn_profile_read.restype = i
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load_library().ring_attn_status_string(status).decode()
    except OSError:
        return str(status)


def _check(status: int, what: str):
    if status != RA_OK:
        detail = ""
        if status == RA_ERR_CUDA:
            detail = load_library().ring_attn_last_error().decode()
        raise RingAttnError(status, what, detail)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _need(t: torch.Tensor, name: str, dtype, shape=None, rows_ok: bool = False):
    """Type, device and shape checks.  rows_ok: any [B, heads, S, d] view whose
    d-element rows are contiguous is accepted (the library takes its strides);
    otherwise the tensor must be contiguous."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if rows_ok:
        if t.dim() != 4 or (t.numel() > 0 and t.stride(3) != 1):
            raise ValueError(f"{name} must be [B, heads, S, d] with contiguous d-element rows")
    elif not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _strides(t: torch.Tensor):
    """(batch, head, position) element strides of a [B, heads, S, d] view, as
    the C array the *_strided entry points take."""
    return (ctypes.c_longlong * 3)(t.stride(0), t.stride(1), t.stride(2))


def _all_contiguous(*ts) -> bool:
    return all(t.is_contiguous() for t in ts)


def _kv_heads(q, k, v):
    """H_kv from k / v shaped [B, H_kv, S, d] with H % H_kv == 0."""
    B, H, S, d = q.shape
    if k.dim() != 4 or k.shape[0] != B or k.shape[2:] != q.shape[2:]:
        raise ValueError(f"k has shape {tuple(k.shape)}, expected [B, H_kv, S, d] matching q")
    H_kv = k.shape[1]
    if H_kv < 1 or H % H_kv:
        raise ValueError(f"query heads ({H}) must be a multiple of key/value heads ({H_kv})")
    _need(k, "k", torch.bfloat16, (B, H_kv, S, d), rows_ok=True)
    _need(v, "v", torch.bfloat16, (B, H_kv, S, d), rows_ok=True)
    return H_kv


def ring_attn_fwd(q, k, v, P: int, causal: bool, scale: float | None = None, *,
                  o=None, lse=None, stream=None):
    """O, LSE = exact ring attention of bf16 [B, H, S, d] q over P chunks.
    k, v are [B, H_kv, S, d]; H_kv < H is grouped-query attention (query
    head h reads key/value head h // (H / H_kv)).  q, k, v and o may be
    strided views whose d-element rows are contiguous -- [B, S, H, d]
    storage is x.transpose(1, 2) -- and o defaults to q's layout."""
    _need(q, "q", torch.bfloat16, rows_ok=True)
    B, H, S, d = q.shape
    H_kv = _kv_heads(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    _need(o, "o", torch.bfloat16, q.shape, rows_ok=True)
    _need(lse, "lse", torch.float32, (B, H, S))
    lib = load_library()
    if not _all_contiguous(q, k, v, o):
        rc = lib.ring_attn_fwd_strided(q.data_ptr(), _strides(q), k.data_ptr(), _strides(k),
                                       v.data_ptr(), _strides(v), o.data_ptr(), _strides(o),
                                       lse.data_ptr(), B, H, H_kv, S, d, int(P), int(bool(causal)),
                                       float(scale), _stream(stream))
    elif H_kv == H:
        rc = lib.ring_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), B, H, S, d, int(P), int(bool(causal)),
                               float(scale), _stream(stream))
    else:
        rc = lib.ring_attn_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, H_kv, S, d, int(P), int(bool(causal)),
                                   float(scale), _stream(stream))
    _check(rc, "ring_attn_fwd")
    return o, lse


def fwd_f32_workspace_size(B: int, H: int, H_kv: int, S: int, d: int) -> int:
    return int(load_library().ring_attn_fwd_f32_workspace_size(B, H, H_kv, S, d))


def ring_attn_fwd_f32(q, k, v, P: int, causal: bool, scale: float | None = None, *,
                      o=None, lse=None, workspace=None, stream=None):
    """O (fp32), LSE of exact ring attention from fp32 [B, H, S, d] q and
    [B, H_kv, S, d] k, v: the inputs are rounded to bf16 on the GPU and the
    products accumulate in fp32; O is returned without bf16 rounding."""
    _need(q, "q", torch.float32)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, S, d]")
    B, H, S, d = q.shape
    if k.dim() != 4 or k.shape[0] != B or k.shape[2:] != q.shape[2:]:
        raise ValueError(f"k has shape {tuple(k.shape)}, expected [B, H_kv, S, d] matching q")
    H_kv = k.shape[1]
    _need(k, "k", torch.float32, (B, H_kv, S, d))
    _need(v, "v", torch.float32, (B, H_kv, S, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None else lse
    _need(o, "o", torch.float32, q.shape)
    _need(lse, "lse", torch.float32, (B, H, S))
    need = fwd_f32_workspace_size(B, H, H_kv, S, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8)
    rc = load_library().ring_attn_fwd_f32(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                          lse.data_ptr(), B, H, H_kv, S, d, int(P),
                                          int(bool(causal)), float(scale), workspace.data_ptr(),
                                          workspace.numel(), _stream(stream))
    _check(rc, "ring_attn_fwd_f32")
    return o, lse


def ulysses_workspace_size(B: int, H: int, H_kv: int, S: int, d: int) -> int:
    return int(load_library().ring_attn_fwd_ulysses_workspace_size(B, H, H_kv, S, d))


def ring_attn_fwd_ulysses_emulated(q, k, v, P: int, causal: bool, scale: float | None = None, *,
                                   o=None, lse=None, workspace=None, stream=None):
    """The Ulysses layout path with P logical ranks on one GPU: an all-to-all
    from token chunks to head groups, full-sequence attention per head group,
    and an all-to-all back.  Needs H and H_kv divisible by P."""
    _need(q, "q", torch.bfloat16)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, S, d]")
    B, H, S, d = q.shape
    H_kv = _kv_heads(q, k, v)
    for t, n in ((k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None else lse
    _need(o, "o", torch.bfloat16, q.shape)
    _need(lse, "lse", torch.float32, (B, H, S))
    need = ulysses_workspace_size(B, H, H_kv, S, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8)
    rc = load_library().ring_attn_fwd_ulysses_emulated(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, H_kv, S, d,
        int(P), int(bool(causal)), float(scale), workspace.data_ptr(), workspace.numel(),
        _stream(stream))
    _check(rc, "ring_attn_fwd_ulysses_emulated")
    return o, lse


def emulated_workspace_size(B: int, H: int, S: int, d: int) -> int:
    return int(load_library().ring_attn_fwd_emulated_workspace_size(B, H, S, d))


def ring_attn_fwd_emulated(q, k, v, P: int, causal: bool, scale: float | None = None, *,
                           overlap: bool = True, o=None, lse=None, workspace=None, stream=None):
    """The ring protocol with P logical ranks on one GPU: per-step partials
    merged with the LSE merge while a copy stream rotates each rank's K/V
    chunk to the next rank (overlap=False puts the copies between steps)."""
    _need(q, "q", torch.bfloat16)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, S, d]")
    B, H, S, d = q.shape
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None else lse
    _need(o, "o", torch.bfloat16, q.shape)
    _need(lse, "lse", torch.float32, (B, H, S))
    need = emulated_workspace_size(B, H, S, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8)
    rc = load_library().ring_attn_fwd_emulated(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                               o.data_ptr(), lse.data_ptr(), B, H, S, d, int(P),
                                               int(bool(causal)), float(scale), workspace.data_ptr(),
                                               workspace.numel(), int(bool(overlap)),
                                               _stream(stream))
    _check(rc, "ring_attn_fwd_emulated")
    return o, lse


def bwd_workspace_size(B: int, H: int, S: int, d: int) -> int:
    return int(load_library().ring_attn_bwd_workspace_size(B, H, S, d))


def ring_attn_bwd(q, k, v, o, lse, dO, P: int, causal: bool, scale: float | None = None, *,
                  dq=None, dk=None, dv=None, workspace=None, stream=None):
    """dQ, dK, dV of exact ring attention (P recomputed from the saved LSE).
    With grouped-query k, v ([B, H_kv, S, d]) dk and dv have that shape.
    Every bf16 tensor may be a strided view with contiguous d-element rows;
    dq, dk and dv default to the layouts of q, k and v."""
    _need(q, "q", torch.bfloat16, rows_ok=True)
    B, H, S, d = q.shape
    H_kv = _kv_heads(q, k, v)
    for t, n in ((o, "o"), (dO, "dO")):
        _need(t, n, torch.bfloat16, q.shape, rows_ok=True)
    _need(lse, "lse", torch.float32, (B, H, S))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _need(dq, "dq", torch.bfloat16, q.shape, rows_ok=True)
    _need(dk, "dk", torch.bfloat16, k.shape, rows_ok=True)
    _need(dv, "dv", torch.bfloat16, v.shape, rows_ok=True)
    need = bwd_workspace_size(B, H, S, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8)
    lib = load_library()
    if not _all_contiguous(q, k, v, o, dO, dq, dk, dv):
        rc = lib.ring_attn_bwd_strided(q.data_ptr(), _strides(q), k.data_ptr(), _strides(k),
                                       v.data_ptr(), _strides(v), o.data_ptr(), _strides(o),
                                       lse.data_ptr(), dO.data_ptr(), _strides(dO), dq.data_ptr(),
                                       _strides(dq), dk.data_ptr(), _strides(dk), dv.data_ptr(),
                                       _strides(dv), B, H, H_kv, S, d, int(P), int(bool(causal)),
                                       float(scale), workspace.data_ptr(), workspace.numel(),
                                       _stream(stream))
    elif H_kv == H:
        rc = lib.ring_attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), dO.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                               dv.data_ptr(), B, H, S, d, int(P), int(bool(causal)),
                               float(scale), workspace.data_ptr(), workspace.numel(),
                               _stream(stream))
    else:
        rc = lib.ring_attn_bwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), dO.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                   dv.data_ptr(), B, H, H_kv, S, d, int(P), int(bool(causal)),
                                   float(scale), workspace.data_ptr(), workspace.numel(),
                                   _stream(stream))
    _check(rc, "ring_attn_bwd")
    return dq, dk, dv


NOALLOC_SCRATCH_BYTES = 64 << 20


def ring_attn_bwd_noalloc(q, k, v, o, lse, dO, P: int, causal: bool, scale: float | None = None,
                          *, dq, dk, dv, stream=None):
    """ring_attn_bwd for callers that cannot allocate device memory: the
    library's fixed static scratch replaces the workspace, and the caller
    passes preallocated dq, dk, dv.  Calls that overlap on the GPU race on
    the shared scratch."""
    _need(q, "q", torch.bfloat16)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, S, d]")
    B, H, S, d = q.shape
    for t, n in ((k, "k"), (v, "v"), (o, "o"), (dO, "dO"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _need(t, n, torch.bfloat16, q.shape)
    _need(lse, "lse", torch.float32, (B, H, S))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rc = load_library().ring_attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                              o.data_ptr(), lse.data_ptr(), dO.data_ptr(),
                                              dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, S,
                                              d, int(P), int(bool(causal)), float(scale),
                                              _stream(stream))
    _check(rc, "ring_attn_bwd_noalloc")
    return dq, dk, dv


def attn_merge_partials(o_a, lse_a, o_b, lse_b, *, o_out=None, lse_out=None, stream=None):
    """LSE merge of two fp32 partials [B, H, S, d] / [B, H, S]."""
    _need(o_a, "o_a", torch.float32)
    if o_a.dim() != 4:
        raise ValueError("o_a must be [B, H, S, d]")
    B, H, S, d = o_a.shape
    _need(o_b, "o_b", torch.float32, o_a.shape)
    _need(lse_a, "lse_a", torch.float32, (B, H, S))
    _need(lse_b, "lse_b", torch.float32, (B, H, S))
    o_out = torch.empty_like(o_a) if o_out is None else o_out
    lse_out = torch.empty_like(lse_a) if lse_out is None else lse_out
    _need(o_out, "o_out", torch.float32, o_a.shape)
    _need(lse_out, "lse_out", torch.float32, (B, H, S))
    rc = load_library().attn_merge_partials(o_a.data_ptr(), lse_a.data_ptr(), o_b.data_ptr(),
                                            lse_b.data_ptr(), o_out.data_ptr(), lse_out.data_ptr(),
                                            B, H, S, d, _stream(stream))
    _check(rc, "attn_merge_partials")
    return o_out, lse_out


def ring_schedule(P: int, causal: bool, i: int):
    """Chunk-level visit list of query chunk i: [(j, kind)], kind 0 local, 1 full."""
    lib = load_library()
    n = lib.ring_attn_schedule(P, int(bool(causal)), i, None, None, 0)
    if n < 0:
        raise RingAttnError(n, "ring_attn_schedule")
    js = (ctypes.c_int * n)()
    ks = (ctypes.c_int * n)()
    m = lib.ring_attn_schedule(P, int(bool(causal)), i, js, ks, n)
    if m != n:
        raise RingAttnError(m, "ring_attn_schedule")
    return [(js[t], ks[t]) for t in range(n)]


def check_status(stream=None) -> int:
    """Synchronize and return (and clear) the device status (0 = OK)."""
    return int(load_library().ring_attn_check_status(_stream(stream)))


def set_wait_limit_ns(ns: int) -> None:
    load_library().ring_attn_set_wait_limit_ns(int(ns))


def trace_visits(buf=None) -> None:
    """Record the ring visits of later forward / backward launches into
    ``buf`` (an int32 CUDA tensor; see ring_attn_trace_visits in the header
    for the slot layout), or stop recording with ``None``."""
    if buf is None:
        _check(load_library().ring_attn_trace_visits(None, 0), "ring_attn_trace_visits")
        return
    _need(buf, "buf", torch.int32)
    _check(load_library().ring_attn_trace_visits(buf.data_ptr(), buf.numel()), "ring_attn_trace_visits")


KERNELS = ("ring_fwd_kernel", "ring_bwd_kernel", "bwd_prep_kernel", "dq_convert_kernel",
           "merge_partials_kernel", "f32_to_bf16_kernel")


def profile_enable(on: bool = True) -> None:
    load_library().ring_attn_profile_enable(int(bool(on)))


def profile_reset() -> None:
    load_library().ring_attn_profile_reset()


def profile_read() -> dict:
    """{kernel: (launches, total_ms)} for the library's kernels since the last reset."""
    lib = load_library()
    out = {}
    for name in KERNELS:
        ms = ctypes.c_double()
        n = ctypes.c_longlong()
        rc = lib.ring_attn_profile_read(name.encode(), ctypes.byref(ms), ctypes.byref(n))
        _check(rc, "ring_attn_profile_read")
        out[name] = (int(n.value), float(ms.value))
    return out
