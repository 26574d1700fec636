"""Python binding of libssd: the Mamba-2 SSD layer forward scan (and its
backward) on one B300.

Thin ctypes marshalling over the C ABI declared in ``include/ssd.h``; every
step of the computation runs in the library's CUDA kernels.  PyTorch is used
for device memory and streams only.  The functions carry the C names:

    ssd_fwd, ssd_fwd_ws, ssd_fwd_host, ssd_fwd_pre, ssd_fwd_varlen, ssd_fwd_noalloc, ssd_fwd_workspace_size,
    ssd_fwd_path, ssd_fwd_block, ssd_step, ssd_fwd_kernels, ssd_bwd, ssd_bwd_workspace_size, ssd_bwd_kernels,
    ssd_profile_events, ssd_test_set_fault,
    ssd_check_device_status, ssd_status_string, ssd_last_error_detail, ssd_version

Layouts: x, y [batch, seqlen, nheads, headdim]; dt [batch, seqlen, nheads];
A, D [nheads]; B, C [batch, seqlen, ngroups, dstate]; states
[batch, nheads, headdim, dstate].  x, B, C, y share one dtype (float32 or
bfloat16); dt, A, D and the states are float32.

There is no fallback: if ``libssd.so`` is missing or cannot be loaded, the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssd.so")

SSD_OK, SSD_ERR_INVALID_ARG, SSD_ERR_UNSUPPORTED, SSD_ERR_CUDA, SSD_ERR_NO_MEMORY, SSD_ERR_TIMEOUT = range(6)
SSD_DTYPE_F32, SSD_DTYPE_BF16 = 0, 1
SSD_PRE_SOFTPLUS, SSD_PRE_ZOH = 1, 2
SSD_PATH_NONE, SSD_PATH_SIMT, SSD_PATH_TCGEN05, SSD_PATH_TCGEN05_FUSED = -1, 0, 1, 2
PATH_NAMES = {SSD_PATH_NONE: "none", SSD_PATH_SIMT: "simt", SSD_PATH_TCGEN05: "tcgen05",
              SSD_PATH_TCGEN05_FUSED: "tcgen05_fused"}

# Every function declared in include/ssd.h, with its ctypes signature.
_P, _I, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_DIMS = [_I] * 8  # batch, seqlen, nheads, headdim, ngroups, dstate, chunk, dtype
_FWD = [_P] * 9 + _DIMS
SIGNATURES = {
    "ssd_fwd": (_I, _FWD + [_P]),
    "ssd_fwd_ws": (_I, _FWD + [_P, _S, _P]),
    "ssd_fwd_host": (_I, _FWD + [_P]),
    "ssd_fwd_noalloc": (_I, _FWD + [_P]),
    "ssd_step": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "ssd_fwd_pre": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "ssd_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, ctypes.POINTER(ctypes.c_int), _I, _P, _P, _P, _I, _I, _I, _I, _I,
                            _I, _P]),
    "ssd_bwd": (_I, [_P] * 16 + [_I] * 7 + [_P]),
    "ssd_bwd_workspace_size": (_I, [_I] * 7 + [ctypes.POINTER(ctypes.c_size_t)]),
    "ssd_bwd_kernels": (_I, [_I] * 7 + [ctypes.c_char_p, _S]),
    "ssd_fwd_workspace_size": (_I, _DIMS + [ctypes.POINTER(ctypes.c_size_t)]),
    "ssd_fwd_path": (_I, _DIMS),
    "ssd_fwd_block": (_I, _DIMS),
    "ssd_fwd_kernels": (_I, _DIMS + [ctypes.c_char_p, _S]),
    "ssd_profile_events": (_I, [ctypes.POINTER(_P), _I]),
    "ssd_check_device_status": (_I, [_P]),
    "ssd_test_set_fault": (_I, [ctypes.c_ulonglong, ctypes.c_longlong]),
    "ssd_status_string": (ctypes.c_char_p, [_I]),
    "ssd_last_error_detail": (ctypes.c_char_p, []),
    "ssd_version": (ctypes.c_char_p, []),
}

_lock = threading.Lock()
_lib = None


class SsdError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{_status_string(status)} ({detail})" if detail else _status_string(status))


def lib() -> ctypes.CDLL:
    """The loaded libssd (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise ImportError(f"libssd.so not built at {LIB_PATH}; run "
                                      "`python -m structured_state_space_03_b300.build`")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def _status_string(st: int) -> str:
    return lib().ssd_status_string(st).decode()


def ssd_status_string(status: int) -> str:
    return _status_string(status)


def ssd_last_error_detail() -> str:
    return lib().ssd_last_error_detail().decode()


def ssd_version() -> str:
    return lib().ssd_version().decode()


def _check(st: int):
    if st != SSD_OK:
        raise SsdError(st, ssd_last_error_detail())


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return SSD_DTYPE_F32
    if t == torch.bfloat16:
        return SSD_DTYPE_BF16
    raise TypeError(f"x, B, C must be float32 or bfloat16, got {t}")


def _dims(x, B):
    if x.dim() != 4 or B.dim() != 4:
        raise ValueError("x must be [batch, seqlen, nheads, headdim] and B, C [batch, seqlen, ngroups, dstate]")
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    return b, L, H, P, G, N


def _validate(x, dt, A, B, C, D, init_state, device_kind):
    el = x.dtype
    b, L, H, P, G, N = _dims(x, B)
    for name, t, shape, dtype in (("dt", dt, (b, L, H), torch.float32), ("A", A, (H,), torch.float32),
                                  ("B", B, (b, L, G, N), el), ("C", C, (b, L, G, N), el),
                                  ("D", D, (H,), torch.float32),
                                  ("init_state", init_state, (b, H, P, N), torch.float32)):
        if t is None:
            continue
        if tuple(t.shape) != shape or t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype} of shape {shape}, got {t.dtype} {tuple(t.shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device.type != device_kind:
            raise ValueError(f"{name} must be on {device_kind}")
    if not x.is_contiguous() or x.device.type != device_kind:
        raise ValueError(f"x must be contiguous and on {device_kind}")
    return b, L, H, P, G, N


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _outputs(x, b, H, P, N, y, final_state, return_final):
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and return_final:
        final_state = torch.empty(b, H, P, N, dtype=torch.float32, device=x.device)
    for name, t, ref in (("y", y, x),):
        if t.shape != ref.shape or t.dtype != ref.dtype or not t.is_contiguous() or t.device != ref.device:
            raise ValueError(f"{name} must be a contiguous tensor like x")
    if final_state is not None and (tuple(final_state.shape) != (b, H, P, N) or final_state.dtype != torch.float32
                                    or not final_state.is_contiguous()):
        raise ValueError("final_state must be contiguous float32 [batch, nheads, headdim, dstate]")
    return y, final_state


def ssd_fwd(x, dt, A, B, C, D=None, init_state=None, *, chunk: int, y=None, final_state=None,
            return_final: bool = True, stream=None):
    """SSD forward on CUDA tensors; enqueued on ``stream`` (default: current).

    Returns ``(y, final_state)`` (``final_state`` is None when not requested).
    """
    b, L, H, P, G, N = _validate(x, dt, A, B, C, D, init_state, "cuda")
    y, final_state = _outputs(x, b, H, P, N, y, final_state, return_final)
    _check(lib().ssd_fwd(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init_state), _ptr(y),
                         _ptr(final_state), b, L, H, P, G, N, chunk, _dtype_code(x.dtype),
                         _stream_handle(stream)))
    return y, final_state


def ssd_fwd_noalloc(x, dt, A, B, C, D=None, init_state=None, *, chunk: int, y=None, final_state=None,
                    return_final: bool = True, stream=None):
    """SSD forward that allocates nothing on the device side of the call: the
    library's fixed 32 MiB scratch replaces the workspace (see include/ssd.h for
    who needs this and its limits).  ``y``/``final_state`` may be passed in to
    avoid allocating outputs here as well."""
    b, L, H, P, G, N = _validate(x, dt, A, B, C, D, init_state, "cuda")
    y, final_state = _outputs(x, b, H, P, N, y, final_state, return_final)
    _check(lib().ssd_fwd_noalloc(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init_state),
                                 _ptr(y), _ptr(final_state), b, L, H, P, G, N, chunk, _dtype_code(x.dtype),
                                 _stream_handle(stream)))
    return y, final_state


def ssd_fwd_pre(x, dt, A, B, C, D=None, init_state=None, *, chunk: int, dt_bias=None, softplus: bool = False,
                zoh: bool = False, y=None, final_state=None, return_final: bool = True, stream=None):
    """ssd_fwd with the device-side pre-step of dt: dt_eff = softplus(dt + dt_bias)
    (``softplus``) or dt + dt_bias, and the zero-order-hold input scale
    expm1(dt_eff A) / A in place of dt_eff (``zoh``)."""
    b, L, H, P, G, N = _validate(x, dt, A, B, C, D, init_state, "cuda")
    if dt_bias is not None and (tuple(dt_bias.shape) != (H,) or dt_bias.dtype != torch.float32
                                or not dt_bias.is_contiguous() or dt_bias.device.type != "cuda"):
        raise ValueError(f"dt_bias must be a contiguous CUDA float32 tensor of shape ({H},)")
    y, final_state = _outputs(x, b, H, P, N, y, final_state, return_final)
    flags = (SSD_PRE_SOFTPLUS if softplus else 0) | (SSD_PRE_ZOH if zoh else 0)
    _check(lib().ssd_fwd_pre(_ptr(x), _ptr(dt), _ptr(dt_bias), flags, _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                             _ptr(init_state), _ptr(y), _ptr(final_state), b, L, H, P, G, N, chunk,
                             _dtype_code(x.dtype), _stream_handle(stream)))
    return y, final_state


def ssd_fwd_varlen(x, dt, A, B, C, D=None, init_state=None, *, cu_seqlens, chunk: int, y=None, final_state=None,
                   return_final: bool = True, stream=None):
    """ssd_fwd over packed variable-length sequences on CUDA tensors.

    x [total, nheads, headdim]; dt [total, nheads] float32; B, C [total, ngroups,
    dstate]; ``cu_seqlens`` (host: a sequence of ints or a CPU tensor) holds the
    nseq + 1 offsets of the sequences in the packed token dimension; init_state
    and final_state are [nseq, nheads, headdim, dstate] float32.  Each sequence
    is its own recurrence.  Returns (y, final_state).
    """
    cu = [int(v) for v in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    nseq = len(cu) - 1
    if nseq < 1:
        raise ValueError("cu_seqlens needs at least two offsets")
    if x.dim() != 3 or B.dim() != 3:
        raise ValueError("x must be [total, nheads, headdim] and B, C [total, ngroups, dstate]")
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    el = x.dtype
    for name, t, shape, dtype in (("dt", dt, (T, H), torch.float32), ("A", A, (H,), torch.float32),
                                  ("B", B, (T, G, N), el), ("C", C, (T, G, N), el), ("D", D, (H,), torch.float32),
                                  ("init_state", init_state, (nseq, H, P, N), torch.float32)):
        if t is None:
            continue
        if tuple(t.shape) != shape or t.dtype != dtype or not t.is_contiguous() or t.device.type != "cuda":
            raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor of shape {shape}")
    if not x.is_contiguous() or x.device.type != "cuda":
        raise ValueError("x must be a contiguous CUDA tensor")
    if cu[-1] != T:
        raise ValueError(f"cu_seqlens must end at the packed token count {T}")
    if y is None:
        y = torch.empty_like(x)
    elif y.shape != x.shape or y.dtype != el or not y.is_contiguous():
        raise ValueError("y must be a contiguous tensor like x")
    if final_state is None and return_final:
        final_state = torch.empty(nseq, H, P, N, dtype=torch.float32, device=x.device)
    offs = (ctypes.c_int * (nseq + 1))(*cu)
    _check(lib().ssd_fwd_varlen(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), offs, nseq, _ptr(init_state),
                                _ptr(y), _ptr(final_state), H, P, G, N, chunk, _dtype_code(el),
                                _stream_handle(stream)))
    return y, final_state


def ssd_step(x, dt, A, B, C, D=None, *, state, y=None, stream=None):
    """One recurrent step for one new token per sequence on CUDA tensors.

    x [batch, nheads, headdim]; dt [batch, nheads] float32; A, D [nheads]
    float32; B, C [batch, ngroups, dstate]; ``state`` [batch, nheads, headdim,
    dstate] float32 is updated in place.  x, B, C, y share one dtype.  Returns y.
    """
    if x.dim() != 3 or B.dim() != 3:
        raise ValueError("x must be [batch, nheads, headdim] and B, C [batch, ngroups, dstate]")
    b, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    el = x.dtype
    for name, t, shape, dtype in (("dt", dt, (b, H), torch.float32), ("A", A, (H,), torch.float32),
                                  ("B", B, (b, G, N), el), ("C", C, (b, G, N), el), ("D", D, (H,), torch.float32),
                                  ("state", state, (b, H, P, N), torch.float32)):
        if t is None:
            continue
        if tuple(t.shape) != shape or t.dtype != dtype or not t.is_contiguous() or t.device.type != "cuda":
            raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor of shape {shape}")
    if not x.is_contiguous() or x.device.type != "cuda":
        raise ValueError("x must be a contiguous CUDA tensor")
    if y is None:
        y = torch.empty_like(x)
    elif y.shape != x.shape or y.dtype != el or not y.is_contiguous():
        raise ValueError("y must be a contiguous tensor like x")
    _check(lib().ssd_step(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(state), _ptr(y), b, H, P, G, N,
                          _dtype_code(el), _stream_handle(stream)))
    return y


def ssd_bwd(x, dt, A, B, C, D=None, init_state=None, *, dy, dfinal_state=None, want_dD: bool = True,
            want_dinit: bool = True, stream=None):
    """Backward of ssd_fwd on CUDA tensors: gradients of a loss given ``dy``
    (like x) and ``dfinal_state`` (float32 [batch, nheads, headdim, dstate] or
    None).  Returns a dict of float32 tensors dx, ddt, dA, dB, dC, dD and
    dinit_state (the last two None when not wanted)."""
    b, L, H, P, G, N = _validate(x, dt, A, B, C, D, init_state, "cuda")
    if tuple(dy.shape) != tuple(x.shape) or dy.dtype != x.dtype or not dy.is_contiguous() or dy.device != x.device:
        raise ValueError("dy must be a contiguous tensor like x")
    if dfinal_state is not None and (tuple(dfinal_state.shape) != (b, H, P, N) or dfinal_state.dtype != torch.float32
                                     or not dfinal_state.is_contiguous() or dfinal_state.device != x.device):
        raise ValueError("dfinal_state must be contiguous float32 [batch, nheads, headdim, dstate] on x's device")
    f32 = dict(dtype=torch.float32, device=x.device)
    out = {"dx": torch.empty(b, L, H, P, **f32), "ddt": torch.empty(b, L, H, **f32), "dA": torch.empty(H, **f32),
           "dB": torch.empty(b, L, G, N, **f32), "dC": torch.empty(b, L, G, N, **f32),
           "dD": torch.empty(H, **f32) if want_dD else None,
           "dinit_state": torch.empty(b, H, P, N, **f32) if want_dinit else None}
    _check(lib().ssd_bwd(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init_state), _ptr(dy),
                         _ptr(dfinal_state), _ptr(out["dx"]), _ptr(out["ddt"]), _ptr(out["dA"]), _ptr(out["dB"]),
                         _ptr(out["dC"]), _ptr(out["dD"]), _ptr(out["dinit_state"]), b, L, H, P, G, N,
                         _dtype_code(x.dtype), _stream_handle(stream)))
    return out


def ssd_bwd_workspace_size(batch, seqlen, nheads, headdim, ngroups, dstate, dtype) -> int:
    code = _dtype_code(dtype) if isinstance(dtype, torch.dtype) else int(dtype)
    out = ctypes.c_size_t(0)
    _check(lib().ssd_bwd_workspace_size(batch, seqlen, nheads, headdim, ngroups, dstate, code, ctypes.byref(out)))
    return out.value


def ssd_bwd_kernels(batch, seqlen, nheads, headdim, ngroups, dstate, dtype) -> list:
    """Names of the kernels one ssd_bwd launches for these sizes, in order."""
    code = _dtype_code(dtype) if isinstance(dtype, torch.dtype) else int(dtype)
    buf = ctypes.create_string_buffer(512)
    n = lib().ssd_bwd_kernels(batch, seqlen, nheads, headdim, ngroups, dstate, code, buf, 512)
    if n < 0:
        raise SsdError(SSD_ERR_INVALID_ARG, "sizes rejected")
    names = buf.value.decode().split(",") if n else []
    assert len(names) == n
    return names


def ssd_fwd_workspace_size(batch, seqlen, nheads, headdim, ngroups, dstate, chunk, dtype) -> int:
    code = _dtype_code(dtype) if isinstance(dtype, torch.dtype) else int(dtype)
    out = ctypes.c_size_t(0)
    _check(lib().ssd_fwd_workspace_size(batch, seqlen, nheads, headdim, ngroups, dstate, chunk, code,
                                        ctypes.byref(out)))
    return out.value


def ssd_fwd_ws(x, dt, A, B, C, D=None, init_state=None, *, chunk: int, workspace, y=None, final_state=None,
               return_final: bool = True, stream=None):
    """SSD forward with a caller-provided device workspace (a uint8 CUDA tensor)."""
    b, L, H, P, G, N = _validate(x, dt, A, B, C, D, init_state, "cuda")
    y, final_state = _outputs(x, b, H, P, N, y, final_state, return_final)
    _check(lib().ssd_fwd_ws(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init_state), _ptr(y),
                            _ptr(final_state), b, L, H, P, G, N, chunk, _dtype_code(x.dtype),
                            _ptr(workspace), workspace.numel() * workspace.element_size(),
                            _stream_handle(stream)))
    return y, final_state


def ssd_fwd_host(x, dt, A, B, C, D=None, init_state=None, *, chunk: int, y=None, final_state=None,
                 return_final: bool = True, stream=None):
    """SSD forward on CPU tensors: copies in, runs, copies out, synchronises."""
    b, L, H, P, G, N = _validate(x, dt, A, B, C, D, init_state, "cpu")
    y, final_state = _outputs(x, b, H, P, N, y, final_state, return_final)
    _check(lib().ssd_fwd_host(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init_state), _ptr(y),
                              _ptr(final_state), b, L, H, P, G, N, chunk, _dtype_code(x.dtype),
                              _stream_handle(stream)))
    return y, final_state


def ssd_fwd_path(batch, seqlen, nheads, headdim, ngroups, dstate, chunk, dtype) -> str:
    code = _dtype_code(dtype) if isinstance(dtype, torch.dtype) else int(dtype)
    return PATH_NAMES[lib().ssd_fwd_path(batch, seqlen, nheads, headdim, ngroups, dstate, chunk, code)]


def ssd_fwd_block(batch, seqlen, nheads, headdim, ngroups, dstate, chunk, dtype) -> int:
    """The chunk length ssd_fwd evaluates for these sizes (-1 when they are rejected)."""
    code = _dtype_code(dtype) if isinstance(dtype, torch.dtype) else int(dtype)
    return int(lib().ssd_fwd_block(batch, seqlen, nheads, headdim, ngroups, dstate, chunk, code))


def ssd_fwd_kernels(batch, seqlen, nheads, headdim, ngroups, dstate, chunk, dtype) -> list:
    """Names of the kernels one ssd_fwd launches for these sizes, in order."""
    code = _dtype_code(dtype) if isinstance(dtype, torch.dtype) else int(dtype)
    buf = ctypes.create_string_buffer(512)
    n = lib().ssd_fwd_kernels(batch, seqlen, nheads, headdim, ngroups, dstate, chunk, code, buf, 512)
    if n < 0:
        raise SsdError(SSD_ERR_INVALID_ARG, "sizes rejected")
    names = buf.value.decode().split(",") if n else []
    assert len(names) == n
    return names


def ssd_profile_events(events):
    """Install (list of recorded torch.cuda.Event) or clear (None) the per-kernel
    timing hook for forwards issued from this thread."""
    if not events:
        _check(lib().ssd_profile_events(None, 0))
        return
    arr = (_P * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(lib().ssd_profile_events(arr, len(events)))


def ssd_test_set_fault(wait_limit_ns: int = 0, withhold_unit: int = -1):
    """Failure-detection test hook (this thread's later forwards): bounded waits
    of the fused kernels give up after ``wait_limit_ns`` (0: the 2 s default)
    and unit ``withhold_unit`` (-1: none) never publishes its chunk state."""
    _check(lib().ssd_test_set_fault(int(wait_limit_ns), int(withhold_unit)))


def ssd_check_device_status(stream=None):
    """Synchronise the stream and raise if a kernel reported an error."""
    _check(lib().ssd_check_device_status(_stream_handle(stream)))
