"""ctypes binding to libevo_attn.so — argument marshalling only.

Every step of the attention runs in the library's sm_103a kernels; this module
checks tensor properties, allocates outputs with PyTorch when the caller does
not pass them, and forwards raw device pointers, sizes and the current CUDA
stream to the C ABI declared in include/evo_attn.h.  There is no CPU or
PyTorch fallback: if the library is missing, every call raises.

Names follow the C ABI: ``evo_attn_fwd``, ``evo_attn_bwd``, ``evo_attn_bwd_ex``,
``evo_attn_fwd_strided``, ``evo_attn_bwd_strided``, ``evo_attn_fwd_opts``,
``evo_attn_bwd_opts``, ``evo_attn_bwd_status``, ``evo_attn_bwd_workspace_bytes``,
``evo_attn_device_status``, ``evo_attn_selftest_wait_timeout``.  Every tensor of a
call must live on the current CUDA device (the library launches there); a tensor
on another device is refused with ValueError before anything reaches the library.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libevo_attn.so")

EVO_OK = 0
EVO_ERR_CUDA = 7
STATUS_NAMES = {
    0: "EVO_OK", 1: "EVO_ERR_NULL_POINTER", 2: "EVO_ERR_BAD_SHAPE", 3: "EVO_ERR_BAD_DTYPE",
    4: "EVO_ERR_MISALIGNED", 5: "EVO_ERR_WORKSPACE_TOO_SMALL", 6: "EVO_ERR_ARCH", 7: "EVO_ERR_CUDA",
    8: "EVO_ERR_DEVICE_TIMEOUT", 9: "EVO_ERR_ALIASING", 10: "EVO_ERR_BAD_ARGUMENT",
    11: "EVO_ERR_SCRATCH_LIMIT", 12: "EVO_ERR_BAD_LAYOUT",
}
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024
EXPORTED = ("evo_attn_abi_version", "evo_status_string", "evo_attn_fwd", "evo_attn_bwd_workspace_bytes",
            "evo_attn_bwd", "evo_attn_device_status", "evo_attn_selftest_wait_timeout",
            "evo_attn_step_host_arena_bytes", "evo_attn_step_host", "evo_attn_bwd_noalloc", "evo_attn_bwd_ex",
            "evo_attn_last_error_detail", "evo_attn_fwd_strided", "evo_attn_bwd_strided", "evo_attn_fwd_opts",
            "evo_attn_bwd_opts", "evo_attn_bwd_status")
OPT_SKIP_MASKED_TILES, OPT_NO_DBIAS2 = 1, 2  # evo_options_t flags

_DTYPE_CODE = {torch.float16: 0, torch.bfloat16: 1}


class EvoShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("N", ctypes.c_int64), ("L", ctypes.c_int64),
                ("H", ctypes.c_int64), ("D", ctypes.c_int64)]


class EvoStrides(ctypes.Structure):
    """Element strides of the B, N and L dimensions of one [B,N,L,H,D] tensor."""
    _fields_ = [("b", ctypes.c_int64), ("n", ctypes.c_int64), ("l", ctypes.c_int64)]


LAYOUT_FIELDS = ("q", "k", "v", "out", "dout", "dq", "dk", "dv")


class EvoLayout(ctypes.Structure):
    _fields_ = [(n, EvoStrides) for n in LAYOUT_FIELDS]


class EvoOptions(ctypes.Structure):
    """evo_options_t: the per-call options of evo_attn_fwd_opts / evo_attn_bwd_opts."""
    _fields_ = [("size", ctypes.c_uint32), ("flags", ctypes.c_uint32), ("skip_threshold", ctypes.c_float),
                ("reserved", ctypes.c_uint32), ("wait_limit_ns", ctypes.c_uint64), ("status", ctypes.c_void_p),
                ("events", ctypes.POINTER(ctypes.c_void_p)), ("num_events", ctypes.c_int32)]


def make_options(skip_masked_tiles: bool = False, skip_threshold: float = -1.0e4, wait_limit_ns: int = 0,
                 status: Optional[torch.Tensor] = None, events=None, no_dbias2: bool = False):
    """An EvoOptions (and the event-handle array it points to, which the caller keeps
    alive for the call).  ``status``: a CUDA int32 tensor of one element; ``events``:
    torch.cuda.Event objects created with enable_timing=True."""
    o = EvoOptions()
    o.size = ctypes.sizeof(EvoOptions)
    o.flags = (OPT_SKIP_MASKED_TILES if skip_masked_tiles else 0) | (OPT_NO_DBIAS2 if no_dbias2 else 0)
    o.skip_threshold = float(skip_threshold)
    o.wait_limit_ns = int(wait_limit_ns)
    if status is not None:
        if not status.is_cuda or status.dtype != torch.int32 or status.numel() < 1:
            raise ValueError("status must be a CUDA int32 tensor")
        o.status = status.data_ptr()
    arr = None
    if events:
        for e in events:
            if e.cuda_event == 0:  # torch creates the CUDA event lazily
                e.record()
        arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
        o.events = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
        o.num_events = len(events)
    return o, arr


class EvoAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        msg = f"{where}: {name}"
        try:
            msg += f" ({load().evo_status_string(status).decode()})"
            if status == EVO_ERR_CUDA:
                msg += f" [{load().evo_attn_last_error_detail().decode()}]"
        except Exception:  # pragma: no cover
            pass
        super().__init__(msg)


_lib = None


def load(path: Optional[str] = None):
    """Load libevo_attn.so (built by memory_efficient_biased_gb300.build); raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libevo_attn.so not built at {p}: run `python -m memory_efficient_biased_gb300.build`")
    lib = ctypes.CDLL(p)
    vp, sz, i32, u64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint64
    lib.evo_attn_abi_version.restype = i32
    lib.evo_status_string.restype = ctypes.c_char_p
    lib.evo_status_string.argtypes = [i32]
    lib.evo_attn_fwd.restype = i32
    lib.evo_attn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, EvoShape, i32, vp]
    lib.evo_attn_bwd_workspace_bytes.restype = sz
    lib.evo_attn_bwd_workspace_bytes.argtypes = [EvoShape, i32, i32]
    lib.evo_attn_bwd.restype = i32
    lib.evo_attn_bwd.argtypes = [vp] * 12 + [vp, sz, EvoShape, i32, vp]
    lib.evo_attn_device_status.restype = i32
    lib.evo_attn_device_status.argtypes = [vp]
    lib.evo_attn_selftest_wait_timeout.restype = i32
    lib.evo_attn_selftest_wait_timeout.argtypes = [u64, vp, vp]
    lib.evo_attn_step_host_arena_bytes.restype = sz
    lib.evo_attn_step_host_arena_bytes.argtypes = [EvoShape, i32, i32, i32]
    lib.evo_attn_step_host.restype = i32
    lib.evo_attn_step_host.argtypes = [vp] * 13 + [sz, EvoShape, i32, vp]
    lib.evo_attn_bwd_noalloc.restype = i32
    lib.evo_attn_bwd_noalloc.argtypes = [vp] * 12 + [EvoShape, i32, vp]
    lib.evo_attn_last_error_detail.restype = ctypes.c_char_p
    lib.evo_attn_last_error_detail.argtypes = []
    lib.evo_attn_bwd_ex.restype = i32
    lib.evo_attn_bwd_ex.argtypes = [vp] * 14 + [sz, EvoShape, i32, vp]
    lib.evo_attn_fwd_strided.restype = i32
    lib.evo_attn_fwd_strided.argtypes = [vp] * 7 + [EvoShape, i32, ctypes.POINTER(EvoLayout), vp]
    lib.evo_attn_bwd_strided.restype = i32
    lib.evo_attn_bwd_strided.argtypes = [vp] * 14 + [sz, EvoShape, i32, ctypes.POINTER(EvoLayout), vp]
    lib.evo_attn_fwd_opts.restype = i32
    lib.evo_attn_fwd_opts.argtypes = [vp] * 7 + [EvoShape, i32, ctypes.POINTER(EvoLayout),
                                                 ctypes.POINTER(EvoOptions), vp]
    lib.evo_attn_bwd_opts.restype = i32
    lib.evo_attn_bwd_opts.argtypes = [vp] * 14 + [sz, EvoShape, i32, ctypes.POINTER(EvoLayout),
                                                  ctypes.POINTER(EvoOptions), vp]
    lib.evo_attn_bwd_status.restype = i32
    lib.evo_attn_bwd_status.argtypes = [vp, vp]
    if path is None:
        _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    elif stream.device.index != torch.cuda.current_device():
        raise ValueError(f"stream is on cuda:{stream.device.index}, the current device is "
                         f"cuda:{torch.cuda.current_device()}")
    return ctypes.c_void_p(stream.cuda_stream)


def _on_current_device(t: torch.Tensor, name: str):
    """The library launches on the current device and addresses every buffer there."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    cur = torch.cuda.current_device()
    if t.device.index != cur:
        raise ValueError(f"{name} is on cuda:{t.device.index}, the current device is cuda:{cur}; "
                         f"call under torch.cuda.device({t.device.index})")


def _check(t: Optional[torch.Tensor], name: str, shape=None, dtype=None):
    if t is None:
        return
    _on_current_device(t, name)
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")


def row_strided(t: torch.Tensor) -> bool:
    """A [B,N,L,H,D] tensor whose H*D elements per token are packed (any B, N, L strides)."""
    H, D = t.shape[3], t.shape[4]
    return (D == 1 or t.stride(4) == 1) and (H == 1 or t.stride(3) == D)


def _check_rows(t: Optional[torch.Tensor], name: str, shape, dtype):
    if t is None:
        return
    _on_current_device(t, name)
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not row_strided(t):
        raise ValueError(f"{name} must have packed (H, D) dimensions")


def layout_of(**tensors) -> EvoLayout:
    """EvoLayout from the strides of the given tensors (q=, k=, ...); packed for the rest."""
    lay = EvoLayout()
    for name in LAYOUT_FIELDS:
        t = tensors.get(name)
        if t is not None:
            setattr(lay, name, EvoStrides(t.stride(0), t.stride(1), t.stride(2)))
        else:
            B, N, L, H, D = next(x for x in tensors.values() if x is not None).shape
            setattr(lay, name, EvoStrides(N * L * H * D, L * H * D, H * D))
    return lay


def shape_of(q: torch.Tensor) -> EvoShape:
    B, N, L, H, D = q.shape
    return EvoShape(B, N, L, H, D)


def evo_attn_fwd(q, k, v, bias1=None, bias2=None, out=None, lse=None, stream=None):
    """O = softmax(Q Kᵀ D^-1/2 + bias1 + bias2) V and the fp32 lse [B,N,H,L]."""
    if q.dim() != 5:
        raise ValueError("q must be [B, N, L, H, D]")
    B, N, L, H, D = q.shape
    dt = q.dtype
    if dt not in _DTYPE_CODE:
        raise ValueError("inputs must be float16 or bfloat16")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, q.shape, dt)
    _check(bias1, "bias1", (B, N, 1, 1, L), dt)
    _check(bias2, "bias2", (B, 1, H, L, L), dt)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, N, H, L), dtype=torch.float32, device=q.device)
    _check(out, "out", q.shape, dt)
    _check(lse, "lse", (B, N, H, L), torch.float32)
    st = load().evo_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(bias1), _ptr(bias2), _ptr(out), _ptr(lse),
                             shape_of(q), _DTYPE_CODE[dt], _stream_ptr(stream))
    if st != EVO_OK:
        raise EvoAttnError(st, "evo_attn_fwd")
    return out, lse


WS_BIAS2, WS_DBIAS1, WS_NO_DBIAS2 = 1, 2, 4  # flags of evo_attn_bwd_workspace_bytes


def evo_attn_bwd_workspace_bytes(shape, dtype, has_bias2: bool, want_dbias1: bool = False) -> int:
    flags = (WS_BIAS2 if has_bias2 else 0) | (WS_DBIAS1 if want_dbias1 else 0)
    return int(load().evo_attn_bwd_workspace_bytes(EvoShape(*shape), _DTYPE_CODE[dtype], flags))


def evo_attn_bwd(q, k, v, bias1, bias2, out, lse, dout, dq=None, dk=None, dv=None, dbias2=None,
                 workspace=None, stream=None):
    """dQ, dK, dV (and dbias2 when bias2 is given); returns (dq, dk, dv, dbias2)."""
    B, N, L, H, D = q.shape
    dt = q.dtype
    if dt not in _DTYPE_CODE:
        raise ValueError("inputs must be float16 or bfloat16")
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _check(t, n, q.shape, dt)
    _check(bias1, "bias1", (B, N, 1, 1, L), dt)
    _check(bias2, "bias2", (B, 1, H, L, L), dt)
    _check(lse, "lse", (B, N, H, L), torch.float32)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    if bias2 is not None and dbias2 is None:
        dbias2 = torch.empty_like(bias2)
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check(t, n, q.shape, dt)
    _check(dbias2, "dbias2", (B, 1, H, L, L), dt)
    need = evo_attn_bwd_workspace_bytes(tuple(q.shape), dt, bias2 is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace")
    st = load().evo_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(bias1), _ptr(bias2), _ptr(out), _ptr(lse),
                             _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias2), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), shape_of(q), _DTYPE_CODE[dt],
                             _stream_ptr(stream))
    if st != EVO_OK:
        raise EvoAttnError(st, "evo_attn_bwd")
    return dq, dk, dv, dbias2


def evo_attn_bwd_ex(q, k, v, bias1, bias2, out, lse, dout, dq=None, dk=None, dv=None, dbias1=None, dbias2=None,
                    workspace=None, stream=None, want_dbias1=True):
    """evo_attn_bwd plus the key-mask gradient dbias1 [B,N,1,1,L] (requires bias1);
    returns (dq, dk, dv, dbias1, dbias2)."""
    B, N, L, H, D = q.shape
    dt = q.dtype
    if dt not in _DTYPE_CODE:
        raise ValueError("inputs must be float16 or bfloat16")
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _check(t, n, q.shape, dt)
    _check(bias1, "bias1", (B, N, 1, 1, L), dt)
    _check(bias2, "bias2", (B, 1, H, L, L), dt)
    _check(lse, "lse", (B, N, H, L), torch.float32)
    if want_dbias1 and bias1 is None:
        raise ValueError("dbias1 needs bias1")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    if want_dbias1 and dbias1 is None:
        dbias1 = torch.empty_like(bias1)
    if bias2 is not None and dbias2 is None:
        dbias2 = torch.empty_like(bias2)
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check(t, n, q.shape, dt)
    _check(dbias1, "dbias1", (B, N, 1, 1, L), dt)
    _check(dbias2, "dbias2", (B, 1, H, L, L), dt)
    need = evo_attn_bwd_workspace_bytes(tuple(q.shape), dt, bias2 is not None, dbias1 is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace")
    st = load().evo_attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(bias1), _ptr(bias2), _ptr(out), _ptr(lse),
                                _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias1), _ptr(dbias2),
                                _ptr(workspace), workspace.numel() * workspace.element_size(), shape_of(q),
                                _DTYPE_CODE[dt], _stream_ptr(stream))
    if st != EVO_OK:
        raise EvoAttnError(st, "evo_attn_bwd_ex")
    return dq, dk, dv, dbias1, dbias2


def evo_attn_fwd_strided(q, k, v, bias1=None, bias2=None, out=None, lse=None, stream=None):
    """evo_attn_fwd on tensors with any B, N, L strides (H and D packed), e.g. the
    transposed view of column-wise MSA or ending-node triangle attention; the
    tensors are read in place.  ``out`` defaults to a new packed tensor."""
    if q.dim() != 5:
        raise ValueError("q must be [B, N, L, H, D]")
    B, N, L, H, D = q.shape
    dt = q.dtype
    if dt not in _DTYPE_CODE:
        raise ValueError("inputs must be float16 or bfloat16")
    if out is None:
        out = torch.empty(q.shape, dtype=dt, device=q.device)
    if lse is None:
        lse = torch.empty((B, N, H, L), dtype=torch.float32, device=q.device)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _check_rows(t, n, q.shape, dt)
    _check(bias1, "bias1", (B, N, 1, 1, L), dt)
    _check(bias2, "bias2", (B, 1, H, L, L), dt)
    _check(lse, "lse", (B, N, H, L), torch.float32)
    lay = layout_of(q=q, k=k, v=v, out=out)
    st = load().evo_attn_fwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(bias1), _ptr(bias2), _ptr(out), _ptr(lse),
                                     shape_of(q), _DTYPE_CODE[dt], ctypes.byref(lay), _stream_ptr(stream))
    if st != EVO_OK:
        raise EvoAttnError(st, "evo_attn_fwd_strided")
    return out, lse


def evo_attn_bwd_strided(q, k, v, bias1, bias2, out, lse, dout, dq=None, dk=None, dv=None, dbias1=None,
                         dbias2=None, workspace=None, stream=None, want_dbias1=False):
    """evo_attn_bwd_ex on tensors with any B, N, L strides (H and D packed); missing
    gradient outputs are allocated packed.  Returns (dq, dk, dv, dbias1, dbias2)."""
    B, N, L, H, D = q.shape
    dt = q.dtype
    if dt not in _DTYPE_CODE:
        raise ValueError("inputs must be float16 or bfloat16")
    if want_dbias1 and bias1 is None:
        raise ValueError("dbias1 needs bias1")
    dq = torch.empty(q.shape, dtype=dt, device=q.device) if dq is None else dq
    dk = torch.empty(q.shape, dtype=dt, device=q.device) if dk is None else dk
    dv = torch.empty(q.shape, dtype=dt, device=q.device) if dv is None else dv
    if want_dbias1 and dbias1 is None:
        dbias1 = torch.empty_like(bias1)
    if bias2 is not None and dbias2 is None:
        dbias2 = torch.empty_like(bias2)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check_rows(t, n, q.shape, dt)
    _check(bias1, "bias1", (B, N, 1, 1, L), dt)
    _check(bias2, "bias2", (B, 1, H, L, L), dt)
    _check(lse, "lse", (B, N, H, L), torch.float32)
    _check(dbias1, "dbias1", (B, N, 1, 1, L), dt)
    _check(dbias2, "dbias2", (B, 1, H, L, L), dt)
    need = evo_attn_bwd_workspace_bytes(tuple(q.shape), dt, bias2 is not None, dbias1 is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace")
    lay = layout_of(q=q, k=k, v=v, out=out, dout=dout, dq=dq, dk=dk, dv=dv)
    st = load().evo_attn_bwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(bias1), _ptr(bias2), _ptr(out), _ptr(lse),
                                     _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias1), _ptr(dbias2),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(), shape_of(q),
                                     _DTYPE_CODE[dt], ctypes.byref(lay), _stream_ptr(stream))
    if st != EVO_OK:
        raise EvoAttnError(st, "evo_attn_bwd_strided")
    return dq, dk, dv, dbias1, dbias2


def evo_attn_device_status(stream=None) -> int:
    return int(load().evo_attn_device_status(_stream_ptr(stream)))


def evo_attn_selftest_wait_timeout(limit_ns: int, status: Optional[torch.Tensor] = None, stream=None) -> int:
    """Launch the bounded-wait self-test; the timeout lands in ``status`` (a CUDA int32
    tensor) or, without one, in the fallback word (evo_attn_device_status)."""
    if status is not None:
        _check(status, "status", dtype=torch.int32)
    return int(load().evo_attn_selftest_wait_timeout(int(limit_ns), _ptr(status), _stream_ptr(stream)))


def evo_attn_fwd_opts(q, k, v, bias1=None, bias2=None, out=None, lse=None, stream=None, *,
                      skip_masked_tiles: bool = False, skip_threshold: float = -1.0e4, wait_limit_ns: int = 0,
                      status: Optional[torch.Tensor] = None, events=None):
    """evo_attn_fwd_strided with per-call options (evo_options_t): masked key-tile
    skipping, the wait limit, a status word of the caller's and profiling events."""
    if q.dim() != 5:
        raise ValueError("q must be [B, N, L, H, D]")
    B, N, L, H, D = q.shape
    dt = q.dtype
    if dt not in _DTYPE_CODE:
        raise ValueError("inputs must be float16 or bfloat16")
    if out is None:
        out = torch.empty(q.shape, dtype=dt, device=q.device)
    if lse is None:
        lse = torch.empty((B, N, H, L), dtype=torch.float32, device=q.device)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _check_rows(t, n, q.shape, dt)
    _check(bias1, "bias1", (B, N, 1, 1, L), dt)
    _check(bias2, "bias2", (B, 1, H, L, L), dt)
    _check(lse, "lse", (B, N, H, L), torch.float32)
    if status is not None:
        _check(status, "status", dtype=torch.int32)
    lay = layout_of(q=q, k=k, v=v, out=out)
    opts, keep = make_options(skip_masked_tiles, skip_threshold, wait_limit_ns, status, events)
    st = load().evo_attn_fwd_opts(_ptr(q), _ptr(k), _ptr(v), _ptr(bias1), _ptr(bias2), _ptr(out), _ptr(lse),
                                  shape_of(q), _DTYPE_CODE[dt], ctypes.byref(lay), ctypes.byref(opts),
                                  _stream_ptr(stream))
    del keep
    if st != EVO_OK:
        raise EvoAttnError(st, "evo_attn_fwd_opts")
    return out, lse


def evo_attn_bwd_opts(q, k, v, bias1, bias2, out, lse, dout, dq=None, dk=None, dv=None, dbias1=None,
                      dbias2=None, workspace=None, stream=None, *, want_dbias1: bool = False,
                      want_dbias2: bool = True, skip_masked_tiles: bool = False, skip_threshold: float = -1.0e4,
                      wait_limit_ns: int = 0, status: Optional[torch.Tensor] = None, events=None):
    """evo_attn_bwd_strided with per-call options (evo_options_t).  Without ``status``,
    a timeout lands in the workspace's own word: read it with evo_attn_bwd_status.
    ``want_dbias2=False`` skips the pair-bias gradient (EVO_OPT_NO_DBIAS2).
    Returns (dq, dk, dv, dbias1, dbias2)."""
    B, N, L, H, D = q.shape
    dt = q.dtype
    if dt not in _DTYPE_CODE:
        raise ValueError("inputs must be float16 or bfloat16")
    if want_dbias1 and bias1 is None:
        raise ValueError("dbias1 needs bias1")
    want_db2 = bias2 is not None and want_dbias2
    dq = torch.empty(q.shape, dtype=dt, device=q.device) if dq is None else dq
    dk = torch.empty(q.shape, dtype=dt, device=q.device) if dk is None else dk
    dv = torch.empty(q.shape, dtype=dt, device=q.device) if dv is None else dv
    if want_dbias1 and dbias1 is None:
        dbias1 = torch.empty_like(bias1)
    if want_db2 and dbias2 is None:
        dbias2 = torch.empty_like(bias2)
    if not want_db2:
        dbias2 = None
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check_rows(t, n, q.shape, dt)
    _check(bias1, "bias1", (B, N, 1, 1, L), dt)
    _check(bias2, "bias2", (B, 1, H, L, L), dt)
    _check(lse, "lse", (B, N, H, L), torch.float32)
    _check(dbias1, "dbias1", (B, N, 1, 1, L), dt)
    _check(dbias2, "dbias2", (B, 1, H, L, L), dt)
    if status is not None:
        _check(status, "status", dtype=torch.int32)
    flags = (WS_BIAS2 if bias2 is not None else 0) | (WS_DBIAS1 if dbias1 is not None else 0) | \
        (WS_NO_DBIAS2 if bias2 is not None and not want_db2 else 0)
    need = int(load().evo_attn_bwd_workspace_bytes(shape_of(q), _DTYPE_CODE[dt], flags))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace")
    lay = layout_of(q=q, k=k, v=v, out=out, dout=dout, dq=dq, dk=dk, dv=dv)
    opts, keep = make_options(skip_masked_tiles, skip_threshold, wait_limit_ns, status, events,
                              no_dbias2=bias2 is not None and not want_db2)
    st = load().evo_attn_bwd_opts(_ptr(q), _ptr(k), _ptr(v), _ptr(bias1), _ptr(bias2), _ptr(out), _ptr(lse),
                                  _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias1), _ptr(dbias2),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(), shape_of(q),
                                  _DTYPE_CODE[dt], ctypes.byref(lay), ctypes.byref(opts), _stream_ptr(stream))
    del keep
    if st != EVO_OK:
        raise EvoAttnError(st, "evo_attn_bwd_opts")
    return dq, dk, dv, dbias1, dbias2


def evo_attn_bwd_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and read the status word of a workspace last used by
    evo_attn_bwd_opts (0 = ok, 8 = a device-side wait ran out)."""
    _check(workspace, "workspace")
    return int(load().evo_attn_bwd_status(_ptr(workspace), _stream_ptr(stream)))


def evo_attn_step_host_arena_bytes(shape, dtype, has_bias1: bool, has_bias2: bool) -> int:
    return int(load().evo_attn_step_host_arena_bytes(EvoShape(*shape), _DTYPE_CODE[dtype], int(bool(has_bias1)),
                                                     int(bool(has_bias2))))


def evo_attn_step_host(q, k, v, bias1, bias2, dout, out, lse, dq, dk, dv, dbias2, arena, stream=None):
    """Forward + backward from and to host (ideally pinned) CPU tensors through
    a caller-owned device arena; queued on ``stream`` (synchronise before use)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout"), (out, "out"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous host tensor")
    if not arena.is_cuda:
        raise ValueError("arena must be a CUDA tensor")
    st = load().evo_attn_step_host(_ptr(q), _ptr(k), _ptr(v), _ptr(bias1), _ptr(bias2), _ptr(dout), _ptr(out),
                                   _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias2), _ptr(arena),
                                   arena.numel() * arena.element_size(), shape_of(q), _DTYPE_CODE[q.dtype],
                                   _stream_ptr(stream))
    if st != EVO_OK:
        raise EvoAttnError(st, "evo_attn_step_host")


def evo_attn_bwd_noalloc(q, k, v, bias1, bias2, out, lse, dout, dq, dk, dv, dbias2=None, stream=None):
    """The backward for callers that cannot allocate device memory: no
    workspace argument; the library's fixed 16 MiB scratch array is used
    instead (see include/evo_attn.h).  Output tensors must be passed in.
    Calls on one device must not overlap on the GPU: they share the scratch."""
    B, N, L, H, D = q.shape
    dt = q.dtype
    if dt not in _DTYPE_CODE:
        raise ValueError("inputs must be float16 or bfloat16")
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check(t, n, q.shape, dt)
    _check(bias1, "bias1", (B, N, 1, 1, L), dt)
    _check(bias2, "bias2", (B, 1, H, L, L), dt)
    _check(dbias2, "dbias2", (B, 1, H, L, L), dt)
    _check(lse, "lse", (B, N, H, L), torch.float32)
    st = load().evo_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(bias1), _ptr(bias2), _ptr(out), _ptr(lse),
                                     _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias2), shape_of(q),
                                     _DTYPE_CODE[dt], _stream_ptr(stream))
    if st != EVO_OK:
        raise EvoAttnError(st, "evo_attn_bwd_noalloc")
    return dq, dk, dv, dbias2
