"""Pins for the fp64 oracle's sequential recurrence.

Each ``pin_*`` takes a recurrence callable ``rec(x, dt, A, B, C, D, init) ->
(y [b,L,H,P], final [b,H,P,N])`` and raises AssertionError when it disagrees
with something fixed independently of the recurrence: the brute-force
semiseparable-matrix form, a different (associative-scan) evaluation order, a
textbook special case evaluated with numpy/scipy routines, or a hand-derived
example.  The same pins run against deliberately broken builds of the oracle
(see test_oracle_mutants.py) to show that each plausible mistake is caught.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import scipy.signal
import torch

import oracle
from structured_state_space_03_b300.workloads import make_inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rms(a):
    return float(np.sqrt(np.mean(np.square(a)))) or 1.0


def _close(got, want, rel, what):
    err = float(np.max(np.abs(got - want))) / _rms(want)
    assert err <= rel, f"{what}: max-abs error {err:.3e} x RMS exceeds {rel:.1e}"


def _np(t):
    return None if t is None else t.detach().double().numpy()


def _small(seed, b=2, L=37, H=4, P=3, N=5, G=2, with_init=True, dt_range=(1e-2, 5e-1)):
    return make_inputs(b, L, H, P, N, G, "f32", seed=seed, dt_range=dt_range, with_init=with_init)


def _call(rec, inp):
    return rec(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["init_state"])


# -- brute force and a second evaluation order --------------------------------

def pin_quadratic_form(rec):
    """Semiseparable matrix M_ij = C_i.B_j exp(A sum_{k=j+1..i} dt_k), y = M(dt x) + D x
    ("Mamba 模型" §4.1), brute force with and without an init state."""
    for seed, with_init in ((1, True), (2, False)):
        inp = _small(seed, with_init=with_init)
        y, f = _call(rec, inp)
        yq, fq = oracle.quadratic(**inp)
        _close(y, yq, 1e-12, "y vs quadratic form")
        _close(f, fq, 1e-12, "final state vs quadratic form")


def pin_assoc_scan(rec):
    """Blelloch scan over (decay, input) pairs ("Mamba 模型" §3.4)."""
    inp = _small(3, L=50)
    y, f = _call(rec, inp)
    ys, fs = oracle.assoc_scan(**inp)
    _close(y, ys, 1e-12, "y vs associative scan")
    _close(f, fs, 1e-12, "final state vs associative scan")


# -- closed forms and textbook reductions -------------------------------------

def pin_A_zero_linear_attention(rec):
    """A = 0 removes all decay: the layer is causal linear attention,
    y = tril(C B^T) (dt x) + D x ("Mamba 模型" §4.2, structured masked attention)."""
    inp = _small(4, with_init=False)
    inp["A"] = torch.zeros_like(inp["A"])
    y, _ = _call(rec, inp)
    x, dt, B, C, D = (_np(inp[k]) for k in ("x", "dt", "B", "C", "D"))
    b, L, H, P = x.shape
    G = B.shape[2]
    want = np.empty_like(y)
    for bb in range(b):
        for h in range(H):
            g = h // (H // G)
            mask = np.tril(C[bb, :, g, :] @ B[bb, :, g, :].T)
            want[bb, :, h, :] = mask @ (dt[bb, :, h, None] * x[bb, :, h, :]) + D[h] * x[bb, :, h, :]
    _close(y, want, 1e-12, "A=0 vs linear attention")


def pin_dt_zero(rec):
    """dt = 0: no decay and no input, so every state equals the init state:
    y = C.h0 + D x, final = h0."""
    inp = _small(5)
    inp["dt"] = torch.zeros_like(inp["dt"])
    y, f = _call(rec, inp)
    x, B, C, D, h0 = (_np(inp[k]) for k in ("x", "B", "C", "D", "init_state"))
    H = x.shape[2]
    G = C.shape[2]
    Ch = np.einsum("blhn,bhpn->blhp", np.repeat(C, H // G, axis=2), h0)
    _close(y, Ch + D[None, None, :, None] * x, 1e-12, "dt=0 output")
    _close(f, h0, 0.0, "dt=0 final state")


def pin_impulse(rec):
    """One nonzero input x[t0] at zero init: y_t = 0 before t0, then
    (C_t.B_t0) dt_t0 x_t0 exp(A (cumdt_t - cumdt_t0)) (+ D x at t0)."""
    inp = _small(6, b=1, L=40, H=2, P=2, N=4, G=1, with_init=False)
    t0, h, p = 11, 1, 1
    x = torch.zeros_like(inp["x"])
    x[0, t0, h, p] = 1.75
    inp["x"] = x
    y, f = _call(rec, inp)
    dt, A, B, C, D = (_np(inp[k]) for k in ("dt", "A", "B", "C", "D"))
    cum = np.cumsum(dt[0, :, h])
    want = np.zeros(40)
    for t in range(t0, 40):
        want[t] = (C[0, t, 0] @ B[0, t0, 0]) * dt[0, t0, h] * 1.75 * math.exp(A[h] * (cum[t] - cum[t0]))
    want[t0] += D[h] * 1.75
    _close(y[0, :, h, p], want, 1e-12, "impulse response")
    others = np.delete(y.reshape(40, -1), h * 2 + p, axis=1)
    assert np.all(others == 0.0), "impulse leaked into another (head, row)"
    fin = B[0, t0, 0] * dt[0, t0, h] * 1.75 * math.exp(A[h] * (cum[-1] - cum[t0]))
    _close(f[0, h, p], fin, 1e-12, "impulse final state")


def pin_lti_iir(rec):
    """Constant dt, B, C: each (head, row) is the first-order IIR filter
    z_t = a z_{t-1} + (C.B) dt x_t with z = C.s, a = exp(dt A), evaluated by
    scipy.signal.lfilter; an init state enters as the filter's initial condition
    ("Mamba 模型" §2.3.2, the LTI special case)."""
    inp = _small(7, b=1, L=64, H=2, P=3, N=4, G=1)
    L = 64
    inp["dt"][:] = inp["dt"][:, :1, :]
    inp["B"][:] = inp["B"][:, :1]
    inp["C"][:] = inp["C"][:, :1]
    y, _ = _call(rec, inp)
    x, dt, A, B, C, D, h0 = (_np(inp[k]) for k in ("x", "dt", "A", "B", "C", "D", "init_state"))
    for h in range(2):
        a = math.exp(dt[0, 0, h] * A[h])
        cb = float(C[0, 0, 0] @ B[0, 0, 0])
        for p in range(3):
            z0 = float(C[0, 0, 0] @ h0[0, h, p])
            z, _ = scipy.signal.lfilter([cb * dt[0, 0, h]], [1.0, -a], x[0, :, h, p], zi=[a * z0])
            _close(y[0, :, h, p], z + D[h] * x[0, :, h, p], 1e-12, "LTI vs lfilter")
    assert L == y.shape[1]


def pin_geometric_limit(rec):
    """Constant x, dt, B, C: the state converges to the geometric-series limit,
    y_inf = D x + (C.B) dt x / (1 - exp(dt A))."""
    inp = _small(8, b=1, L=600, H=1, P=1, N=3, G=1, with_init=False)
    inp["dt"][:] = 0.25
    inp["A"][:] = -0.5
    inp["x"][:] = 0.75
    inp["B"][:] = inp["B"][:, :1]
    inp["C"][:] = inp["C"][:, :1]
    y, _ = _call(rec, inp)
    B, C, D = _np(inp["B"]), _np(inp["C"]), _np(inp["D"])
    a = math.exp(0.25 * -0.5)
    want = D[0] * 0.75 + float(C[0, 0, 0] @ B[0, 0, 0]) * 0.25 * 0.75 / (1.0 - a)
    assert abs(y[0, -1, 0, 0] - want) <= 1e-9 * max(1.0, abs(want)), (y[0, -1, 0, 0], want)


def pin_state_split(rec):
    """Running [0, L1) and feeding its final state as the init state of
    [L1, L) reproduces one run over [0, L): the state is the whole carry."""
    inp = _small(9, L=45)
    y, f = _call(rec, inp)
    L1 = 19
    first = {k: (v[:, :L1] if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    y1, f1 = _call(rec, first)
    second = {k: (v[:, L1:] if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    second["init_state"] = torch.from_numpy(f1.astype(np.float32))
    # the carried state is rounded to fp32 by the interface; compare loosely
    y2, f2 = _call(rec, second)
    _close(y1, y[:, :L1], 1e-13, "prefix run")
    _close(np.concatenate([y1, y2], axis=1), y, 1e-6, "split run")
    _close(f2, f, 1e-6, "split final state")


def pin_groups(rec):
    """Heads map to B/C groups contiguously (g = h // (H/G)); G groups give
    the same result as G = H with each group's B, C repeated per head."""
    inp = _small(10, H=4, G=2)
    y, f = _call(rec, inp)
    rep = dict(inp)
    rep["B"] = inp["B"].repeat_interleave(2, dim=2)
    rep["C"] = inp["C"].repeat_interleave(2, dim=2)
    yr, fr = _call(rec, rep)
    _close(y, yr, 1e-14, "grouped vs replicated B/C")
    _close(f, fr, 1e-14, "grouped vs replicated final state")
    zero = dict(inp)
    zero["B"] = inp["B"].clone()
    zero["B"][:, :, 1] = 0
    zero["init_state"] = None
    yz, _ = _call(rec, zero)
    x, D = _np(inp["x"]), _np(inp["D"])
    _close(yz[:, :, 2:], D[None, None, 2:, None] * x[:, :, 2:], 0.0, "group 1 heads see only D x")
    assert np.max(np.abs(yz[:, :, :2] - D[None, None, :2, None] * x[:, :, :2])) > 1e-3


def pin_hand_example(rec):
    """Three-token example worked out by hand (tests/golden/hand_example.json)."""
    with open(os.path.join(GOLDEN, "hand_example.json")) as fh:
        g = json.load(fh)
    f32 = lambda v, shape: torch.tensor(v, dtype=torch.float32).reshape(shape)
    y, f = rec(f32(g["x"], (1, 3, 1, 1)), f32(g["dt"], (1, 3, 1)), f32(g["A"], (1,)),
               f32(g["B"], (1, 3, 1, 2)), f32(g["C"], (1, 3, 1, 2)), f32(g["D"], (1,)),
               f32(g["init_state"], (1, 1, 1, 2)))
    np.testing.assert_allclose(y.reshape(-1), g["y"], rtol=g["rtol"], atol=0)
    np.testing.assert_allclose(f.reshape(-1), g["final_state"], rtol=g["rtol"], atol=0)


def pin_bf16_widening(rec):
    """bf16 inputs are widened exactly: the result equals the fp32 run on the
    same (bf16-representable) values."""
    inp = _small(11, with_init=False)
    bf = dict(inp)
    for k in ("x", "B", "C"):
        bf[k] = inp[k].to(torch.bfloat16)
    f32 = dict(bf)
    for k in ("x", "B", "C"):
        f32[k] = bf[k].float()
    y1, f1 = _call(rec, bf)
    y2, f2 = _call(rec, f32)
    _close(y1, y2, 0.0, "bf16 vs widened fp32")
    _close(f1, f2, 0.0, "bf16 vs widened fp32 final")


PINS = [pin_quadratic_form, pin_assoc_scan, pin_A_zero_linear_attention, pin_dt_zero, pin_impulse,
        pin_lti_iir, pin_geometric_limit, pin_state_split, pin_groups, pin_hand_example,
        pin_bf16_widening]
