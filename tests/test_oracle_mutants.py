"""Planted mistakes in the oracle's recurrence must each fail at least one pin.

Each mutant is a copy of the oracle's C source with one plausible mistake
(a dropped term, a wrong sign, a wrong index, swapped operands), compiled to a
temporary library; the pins of oracle_pins.py run against it on the CPU.
"""
import os

import pytest

import oracle
from oracle_pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssd_oracle.c")

MUTANTS = {
    "decay_sign": ("const double decay = exp(dt_t * A_h);", "const double decay = exp(-dt_t * A_h);"),
    "no_dt_on_input": ("s[n] = decay * s[n] + dt_t * x_t * widen(pr->B, bc + n, pr->in_dtype);",
                       "s[n] = decay * s[n] + x_t * widen(pr->B, bc + n, pr->in_dtype);"),
    "decay_after_input": ("s[n] = decay * s[n] + dt_t * x_t * widen(pr->B, bc + n, pr->in_dtype);",
                          "s[n] = decay * (s[n] + dt_t * x_t * widen(pr->B, bc + n, pr->in_dtype));"),
    "no_D_term": ("y_row[t] = acc + D_h * x_t;", "y_row[t] = acc;"),
    "output_before_update": (
        "            s[n] = decay * s[n] + dt_t * x_t * widen(pr->B, bc + n, pr->in_dtype);\n"
        "            acc += widen(pr->C, bc + n, pr->in_dtype) * s[n];",
        "            acc += widen(pr->C, bc + n, pr->in_dtype) * s[n];\n"
        "            s[n] = decay * s[n] + dt_t * x_t * widen(pr->B, bc + n, pr->in_dtype);"),
    "B_C_swapped": (
        "            s[n] = decay * s[n] + dt_t * x_t * widen(pr->B, bc + n, pr->in_dtype);\n"
        "            acc += widen(pr->C, bc + n, pr->in_dtype) * s[n];",
        "            s[n] = decay * s[n] + dt_t * x_t * widen(pr->C, bc + n, pr->in_dtype);\n"
        "            acc += widen(pr->B, bc + n, pr->in_dtype) * s[n];"),
    "group_modulo": ("*g = *h / (pr->nheads / pr->ngroups);", "*g = *h % pr->ngroups;"),
    "init_ignored": ("s[n] = pr->init ? (double)pr->init[((b * H + h) * P + p) * N + n] : 0.0;", "s[n] = 0.0;"),
    "dt_previous_token": ("const double dt_t = (double)pr->dt[(b * L + t) * H + h];",
                          "const double dt_t = (double)pr->dt[(b * L + (t > 0 ? t - 1 : 0)) * H + h];"),
    "x_head_row_transposed": ("const double x_t = widen(pr->x, ((b * L + t) * H + h) * P + p, pr->in_dtype);",
                              "const double x_t = widen(pr->x, ((b * L + t) * P + (p % P)) * H + (h % H), pr->in_dtype);"),
    "init_transposed": ("s[n] = pr->init ? (double)pr->init[((b * H + h) * P + p) * N + n] : 0.0;",
                        "s[n] = pr->init ? (double)pr->init[((b * H + h) * N + (n % N)) * P + (p % P)] : 0.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(SRC) as fh:
        src = fh.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.load_library(oracle.compile_library(str(path), str(tmp_path / "libmutant.so")))
    rec = lambda *a: oracle.recurrence_with(lib, *a)
    caught = []
    for pin in PINS:
        try:
            pin(rec)
        except (AssertionError, RuntimeError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
