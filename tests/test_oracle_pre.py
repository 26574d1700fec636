"""Pins of the oracle's pre-step of dt (softplus, bias, zero-order hold), on
the CPU, plus planted mistakes in it that the pins must catch.

Each pin rests on something other than the oracle's own formula: numpy's
logaddexp and expm1 as library routines, the A = 0 limit of the zero-order
hold (it becomes the plain input dt B), and the zero-order hold's closed-form
steady state -x B / A under constant inputs.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from structured_state_space_03_b300.workloads import make_inputs


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.sqrt(np.mean(b * b)), 1e-300))


def pin_softplus_bias_is_logaddexp(rec):
    inp = make_inputs(2, 40, 3, 4, 8, 1, "f32", seed=201, with_init=True)
    bias = torch.tensor([-1.5, 0.25, 2.0])
    y, f = rec(**inp, dt_bias=bias, softplus=True)
    dt2 = torch.from_numpy(np.logaddexp(0.0, inp["dt"].numpy().astype(np.float64) + bias.numpy()).astype(np.float32))
    y0, f0 = oracle.recurrence(**dict(inp, dt=dt2))
    assert _rel(y, y0) < 1e-6 and _rel(f, f0) < 1e-6


def pin_bias_without_softplus_shifts_dt(rec):
    inp = make_inputs(1, 30, 2, 4, 8, 1, "f32", seed=202, with_init=True)
    bias = torch.tensor([0.5, 0.125])
    y, f = rec(**inp, dt_bias=bias)
    y0, f0 = oracle.recurrence(**dict(inp, dt=inp["dt"] + bias))  # dt + bias rounded once to fp32 here
    assert _rel(y, y0) < 1e-6 and _rel(f, f0) < 1e-6


def pin_zoh_at_A_zero_is_plain(rec):
    inp = make_inputs(1, 30, 2, 4, 8, 1, "f32", seed=203, with_init=True)
    inp["A"] = torch.zeros(2)
    y, f = rec(**inp, zoh=True)
    y0, f0 = oracle.recurrence(**inp)
    assert _rel(y, y0) < 1e-14 and _rel(f, f0) < 1e-14


def pin_zoh_one_step_is_expm1(rec):
    inp = make_inputs(1, 1, 2, 3, 5, 1, "f32", seed=204)
    y, f = rec(**inp, zoh=True)
    dt = inp["dt"][0, 0].numpy().astype(np.float64)
    A = inp["A"].numpy().astype(np.float64)
    x = inp["x"][0, 0].numpy().astype(np.float64)
    B = inp["B"][0, 0, 0].numpy().astype(np.float64)
    C = inp["C"][0, 0, 0].numpy().astype(np.float64)
    u = np.expm1(dt * A) / A
    want_f = u[:, None, None] * x[:, :, None] * B[None, None, :]
    want_y = np.einsum("hpn,n->hp", want_f, C) + inp["D"].numpy()[:, None] * x
    assert _rel(f[0], want_f) < 1e-12 and _rel(y[0, 0], want_y) < 1e-12


def pin_zoh_steady_state(rec):
    """Constant dt, x and B with A < 0: the zero-order-hold state tends to
    -x B / A for any dt (the continuous system's fixed point)."""
    b, L, H, P, N = 1, 80, 2, 3, 4
    x = torch.tensor([[0.5, -1.0, 2.0], [1.5, 0.25, -0.75]]).expand(b, L, H, P).contiguous()
    B = torch.tensor([1.0, -2.0, 0.5, 3.0]).expand(b, L, 1, N).contiguous()
    C = torch.ones(b, L, 1, N)
    A = torch.tensor([-2.0, -0.75])
    dt = torch.tensor([0.5, 1.25]).expand(b, L, H).contiguous()
    _, f = rec(x, dt, A, B, C, zoh=True)
    want = -(x[0, 0].numpy().astype(np.float64)[:, :, None] * B[0, 0, 0].numpy()[None, None, :]) / A.numpy()[:, None, None]
    assert _rel(f[0], want) < 1e-9


PINS = [pin_softplus_bias_is_logaddexp, pin_bias_without_softplus_shifts_dt, pin_zoh_at_A_zero_is_plain,
        pin_zoh_one_step_is_expm1, pin_zoh_steady_state]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pre_step_pin(pin):
    pin(oracle.recurrence_pre)


SRC = os.path.join(os.path.dirname(oracle.__file__), "ssd_oracle.c")
MUTANTS = {
    "zoh_sign": ("(decay - 1.0) / A_h : d) : d;", "(1.0 - decay) / A_h : d) : d;"),
    "zoh_missing": ("const double u = (pr->pre_flags & ORACLE_PRE_ZOH)", "const double u = 0 && (pr->pre_flags & ORACLE_PRE_ZOH)"),
    "no_softplus": ("            d = log(1.0 + exp(d));", "            d = d;"),
    "bias_ignored": ("const double bias = pr->dt_bias ? (double)pr->dt_bias[h] : 0.0;", "const double bias = 0.0;"),
    "softplus_sign": ("            d = log(1.0 + exp(d));", "            d = log(1.0 + exp(-d));"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pre_step_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.load_library(oracle.compile_library(str(path), str(tmp_path / "libmutant.so")))
    rec = lambda *a, **k: oracle.recurrence_pre(*a, lib=lib, **k)
    caught = []
    for pin in PINS:
        try:
            pin(rec)
        except (AssertionError, RuntimeError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
