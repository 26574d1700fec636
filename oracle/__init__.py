"""fp64 CPU oracle for the Mamba-2 SSD layer forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The CUDA library (``structured_state_space_03_b300``) never uses
it, and it shares no code with that library.

The arithmetic lives in ``ssd_oracle.c`` (plain C, fp64); this module compiles
it with gcc on first use and marshals numpy / torch CPU arrays into it.

What is computed (recurrent form, "Mamba模型：线性复杂度序列建模的革命性突破"
§2.2, "Mamba 模型" §2.3.1, "深挖-Mamba" core concepts §1, with the SSD layer's
scalar-per-head A and input scaling dt*B):

    s_t = exp(dt_t A_h) s_{t-1} + dt_t x_t[p] B_t       (per head h, row p)
    y_t[p] = C_t . s_t + D_h x_t[p]

``recurrence`` is the sequential definition (O1).  ``quadratic`` evaluates the
semiseparable matrix form of "Mamba 模型" §4.1 by brute force (O2) and
``assoc_scan`` evaluates the same map by a Blelloch scan over (decay, input)
pairs ("Mamba 模型" §3.4) (O3); both exist to pin O1, not to replace it.

``backward`` (O4) returns the gradients of sum(dy * y) + sum(dfinal * final)
with respect to every input, by the reverse-time adjoint of the recurrence with
each row's states recomputed ("Mamba 模型" §3.4 on recomputation in the
backward pass); tests/test_oracle_backward.py pins it by central differences of
O1, torch autodiff of the written-out recurrence and closed forms.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None

IN_F32 = 0
IN_BF16 = 1


def compile_library(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile an oracle C source into a shared library with gcc."""
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
           *extra_flags, "-o", out, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True, capture_output=True)
    return out


def _bind(lib):
    p = ctypes.c_void_p
    L = ctypes.c_long
    common = [p, p, p, p, p, p, p, ctypes.c_int, L, L, L, L, L, L]
    lib.oracle_ssd_recurrence.argtypes = common + [p, L, p, p, ctypes.c_int]
    lib.oracle_ssd_recurrence.restype = ctypes.c_int
    if hasattr(lib, "oracle_ssd_recurrence_pre"):
        lib.oracle_ssd_recurrence_pre.argtypes = [p, p, p, ctypes.c_int] + common[2:] + [p, L, p, p, ctypes.c_int]
        lib.oracle_ssd_recurrence_pre.restype = ctypes.c_int
    if hasattr(lib, "oracle_ssd_backward"):
        lib.oracle_ssd_backward.argtypes = common + [p, p, p, p, p, p, p, p, p, ctypes.c_int]
        lib.oracle_ssd_backward.restype = ctypes.c_int
    for name in ("oracle_ssd_quadratic", "oracle_ssd_assoc_scan"):
        fn = getattr(lib, name)
        fn.argtypes = common + [p, p]
        fn.restype = ctypes.c_int
    return lib


def load_library(path: str | None = None):
    """Load (building if needed) the oracle library; a path loads a variant."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                compile_library()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def default_threads() -> int:
    return len(os.sched_getaffinity(0))


def _as_input(a, name, allow_bf16):
    """Return (contiguous numpy array, in_dtype) for x/B/C or an fp32 array."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                if not allow_bf16:
                    raise TypeError(f"{name} must be fp32")
                return a.view(torch.int16).numpy().view(np.uint16), IN_BF16
            a = a.numpy()
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16 and allow_bf16:
        return a, IN_BF16
    if a.dtype != np.float32:
        raise TypeError(f"{name} must be float32 (got {a.dtype})")
    return a, IN_F32


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _prepare(x, dt, A, B, C, D, init_state):
    xa, xd = _as_input(x, "x", True)
    Ba, bd = _as_input(B, "B", True)
    Ca, cd = _as_input(C, "C", True)
    if not (xd == bd == cd):
        raise TypeError("x, B and C must share one element type")
    dta, _ = _as_input(dt, "dt", False)
    Aa, _ = _as_input(A, "A", False)
    Da = None if D is None else _as_input(D, "D", False)[0]
    ia = None if init_state is None else _as_input(init_state, "init_state", False)[0]
    if xa.ndim != 4 or Ba.ndim != 4 or Ca.ndim != 4:
        raise ValueError("x must be [b,L,H,P]; B, C must be [b,L,G,N]")
    b, L, H, P = xa.shape
    G, N = Ba.shape[2], Ba.shape[3]
    if Ba.shape != (b, L, G, N) or Ca.shape != (b, L, G, N):
        raise ValueError("B and C must both be [b,L,G,N]")
    if dta.shape != (b, L, H) or Aa.shape != (H,):
        raise ValueError("dt must be [b,L,H] and A must be [H]")
    if Da is not None and Da.shape != (H,):
        raise ValueError("D must be [H]")
    if ia is not None and ia.shape != (b, H, P, N):
        raise ValueError("init_state must be [b,H,P,N]")
    dims = (b, L, H, P, G, N)
    return (xa, dta, Aa, Ba, Ca, Da, ia), xd, dims


def recurrence(x, dt, A, B, C, D=None, init_state=None, rows=None, nthreads=None):
    """Sequential fp64 recurrence (O1).

    With ``rows=None`` returns ``(y [b,L,H,P], final_state [b,H,P,N])`` in fp64.
    With ``rows`` (flat ids ``(b*H + h)*P + p``) returns
    ``(y_rows [nrows, L], final_rows [nrows, N])`` for those rows only.
    """
    arrs, xd, (b, L, H, P, G, N) = _prepare(x, dt, A, B, C, D, init_state)
    lib = load_library()
    if rows is None:
        nrows = b * H * P
        ra = None
    else:
        ra = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = ra.shape[0]
    y = np.empty((nrows, L), np.float64)
    fin = np.empty((nrows, N), np.float64)
    rc = lib.oracle_ssd_recurrence(*[_ptr(a) for a in arrs], xd, b, L, H, P, G, N,
                                   _ptr(ra), nrows, _ptr(y), _ptr(fin),
                                   int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_ssd_recurrence failed with {rc}")
    if rows is not None:
        return y, fin
    return (y.reshape(b, H, P, L).transpose(0, 3, 1, 2).copy(),
            fin.reshape(b, H, P, N))


def _full_rows_call(fn_name, x, dt, A, B, C, D, init_state, lib=None):
    arrs, xd, (b, L, H, P, G, N) = _prepare(x, dt, A, B, C, D, init_state)
    lib = lib or load_library()
    y = np.empty((b * H * P, L), np.float64)
    fin = np.empty((b * H * P, N), np.float64)
    rc = getattr(lib, fn_name)(*[_ptr(a) for a in arrs], xd, b, L, H, P, G, N, _ptr(y), _ptr(fin))
    if rc != 0:
        raise RuntimeError(f"{fn_name} failed with {rc}")
    return (y.reshape(b, H, P, L).transpose(0, 3, 1, 2).copy(), fin.reshape(b, H, P, N))


def quadratic(x, dt, A, B, C, D=None, init_state=None):
    """Brute-force semiseparable-matrix form (O2); O(L^3) -- tiny inputs only."""
    return _full_rows_call("oracle_ssd_quadratic", x, dt, A, B, C, D, init_state)


def assoc_scan(x, dt, A, B, C, D=None, init_state=None):
    """Blelloch associative scan over (decay, input) pairs (O3)."""
    return _full_rows_call("oracle_ssd_assoc_scan", x, dt, A, B, C, D, init_state)


def recurrence_with(lib, x, dt, A, B, C, D=None, init_state=None):
    """O1 through an explicitly loaded library (used to test planted mistakes)."""
    arrs, xd, (b, L, H, P, G, N) = _prepare(x, dt, A, B, C, D, init_state)
    nrows = b * H * P
    y = np.empty((nrows, L), np.float64)
    fin = np.empty((nrows, N), np.float64)
    rc = lib.oracle_ssd_recurrence(*[_ptr(a) for a in arrs], xd, b, L, H, P, G, N,
                                   None, nrows, _ptr(y), _ptr(fin), 1)
    if rc != 0:
        raise RuntimeError(f"oracle_ssd_recurrence failed with {rc}")
    return (y.reshape(b, H, P, L).transpose(0, 3, 1, 2).copy(), fin.reshape(b, H, P, N))


def backward(x, dt, A, B, C, D=None, init_state=None, dy=None, dfinal=None, nthreads=None, lib=None):
    """Gradients of  sum(dy * y) + sum(dfinal * final_state)  through the
    recurrence (fp64, reverse-time adjoint with each row's states recomputed).
    ``dy`` [b,L,H,P] and ``dfinal`` [b,H,P,N] (or None) are taken as fp64.
    Returns a dict of fp64 arrays: dx [b,L,H,P], ddt [b,L,H], dA [H], dB and
    dC [b,L,G,N], dD [H], dinit [b,H,P,N]."""
    arrs, xd, (b, L, H, P, G, N) = _prepare(x, dt, A, B, C, D, init_state)
    lib = lib or load_library()
    dya = np.ascontiguousarray(np.asarray(dy, dtype=np.float64))
    if dya.shape != (b, L, H, P):
        raise ValueError("dy must be [b,L,H,P]")
    dfa = None if dfinal is None else np.ascontiguousarray(np.asarray(dfinal, dtype=np.float64))
    if dfa is not None and dfa.shape != (b, H, P, N):
        raise ValueError("dfinal must be [b,H,P,N]")
    out = {"dx": np.empty((b, L, H, P)), "ddt": np.empty((b, L, H)), "dA": np.empty(H), "dB": np.empty((b, L, G, N)),
           "dC": np.empty((b, L, G, N)), "dD": np.empty(H), "dinit": np.empty((b, H, P, N))}
    rc = lib.oracle_ssd_backward(*[_ptr(a) for a in arrs], xd, b, L, H, P, G, N, _ptr(dya), _ptr(dfa),
                                 _ptr(out["dx"]), _ptr(out["ddt"]), _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]),
                                 _ptr(out["dD"]), _ptr(out["dinit"]), int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_ssd_backward failed with {rc}")
    return out


PRE_SOFTPLUS, PRE_ZOH = 1, 2


def recurrence_pre(x, dt, A, B, C, D=None, init_state=None, dt_bias=None, softplus=False, zoh=False, rows=None,
                   nthreads=None, lib=None):
    """O1 with the pre-step of dt: d = dt + dt_bias, through a softplus when
    ``softplus``, decay exp(d A), and the input scale (exp(d A) - 1) / A when
    ``zoh`` (d otherwise).  Same returns as ``recurrence``."""
    arrs, xd, (b, L, H, P, G, N) = _prepare(x, dt, A, B, C, D, init_state)
    xa, dta, Aa, Ba, Ca, Da, ia = arrs
    ba = None if dt_bias is None else _as_input(dt_bias, "dt_bias", False)[0]
    if ba is not None and ba.shape != (H,):
        raise ValueError("dt_bias must be [H]")
    lib = lib or load_library()
    if rows is None:
        nrows = b * H * P
        ra = None
    else:
        ra = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = ra.shape[0]
    y = np.empty((nrows, L), np.float64)
    fin = np.empty((nrows, N), np.float64)
    flags = (PRE_SOFTPLUS if softplus else 0) | (PRE_ZOH if zoh else 0)
    rc = lib.oracle_ssd_recurrence_pre(_ptr(xa), _ptr(dta), _ptr(ba), flags, _ptr(Aa), _ptr(Ba), _ptr(Ca),
                                       _ptr(Da), _ptr(ia), xd, b, L, H, P, G, N, _ptr(ra), nrows, _ptr(y),
                                       _ptr(fin), int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_ssd_recurrence_pre failed with {rc}")
    if rows is not None:
        return y, fin
    return (y.reshape(b, H, P, L).transpose(0, 3, 1, 2).copy(), fin.reshape(b, H, P, N))


def recurrence_varlen(x, dt, A, B, C, D=None, init_state=None, cu_seqlens=None, nthreads=None):
    """O1 over packed variable-length sequences ("Mamba-2架构深度解析" §5, dynamic
    sequence packing; reading: every packed sequence is its own recurrence, so
    the state restarts from that sequence's initial state at its first token).

    x [T, H, P], dt [T, H], B and C [T, G, N] hold the sequences back to back;
    sequence s owns tokens cu_seqlens[s] .. cu_seqlens[s+1]-1 (cu_seqlens[0] = 0,
    nondecreasing, last = T; empty sequences allowed).  init_state is
    [nseq, H, P, N] or None (zero).  Returns (y [T, H, P], final_state
    [nseq, H, P, N]) in fp64; an empty sequence's final state is its initial
    state.
    """
    cu = [int(v) for v in cu_seqlens]
    if not cu or cu[0] != 0 or any(b < a for a, b in zip(cu, cu[1:])):
        raise ValueError("cu_seqlens must start at 0 and be nondecreasing")
    T, H, P = (int(v) for v in x.shape)
    if cu[-1] != T:
        raise ValueError("cu_seqlens must end at the packed token count")
    N = int(B.shape[2])
    nseq = len(cu) - 1
    y = np.zeros((T, H, P), np.float64)
    fin = np.zeros((nseq, H, P, N), np.float64)
    for s in range(nseq):
        a, e = cu[s], cu[s + 1]
        h0 = None if init_state is None else init_state[s:s + 1]
        if e == a:
            if h0 is not None:
                fin[s] = np.asarray(_as_input(h0, "init_state", False)[0], np.float64)[0]
            continue
        ys, fs = recurrence(x[None, a:e], dt[None, a:e], A, B[None, a:e], C[None, a:e], D, h0, nthreads=nthreads)
        y[a:e] = ys[0]
        fin[s] = fs[0]
    return y, fin
