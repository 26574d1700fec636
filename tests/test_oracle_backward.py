"""Pins for the oracle's backward (the adjoint of the recurrence).

The loss is  L = sum(dy * y) + sum(dfinal * final_state); ``oracle.backward``
returns dL/d(every input).  Each ``pin_*`` takes a backward callable and checks
it against something derived independently of the adjoint recurrence:

* central differences of the (separately pinned) fp64 forward along random
  directions, one input at a time, with inputs and steps on a dyadic grid so
  that every perturbed fp32 input is exact and the difference quotient needs no
  rounding allowance;
* reverse-mode autodiff of the recurrence written out with torch fp64 ops;
* closed forms: with dy = 0 only the decay products reach x and the initial
  state; Euler's theorem for the parts of L that are linear (x and the initial
  state jointly; C; D; B).

Planted mistakes in the backward's C source must each fail one of them.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
from structured_state_space_03_b300.workloads import make_inputs

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssd_oracle.c")
KEYS = ("x", "dt", "A", "B", "C", "D", "init_state")
GRAD = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "init_state": "dinit"}


def _dyadic(inp):
    """Round every input to a multiple of 2^-10 (dt: 2^-12) so that adding a
    multiple of 2^-20 keeps it exact in fp32 (all magnitudes are below 16)."""
    out = {}
    for k in KEYS:
        v = inp[k]
        if v is None:
            out[k] = None
            continue
        q = 2.0 ** -12 if k == "dt" else 2.0 ** -10
        a = np.round(v.double().numpy() / q) * q
        assert np.all(np.abs(a) < 16.0)
        out[k] = torch.from_numpy(a.astype(np.float32))
    assert torch.all(out["dt"] > 0)
    return out


def _case(seed, b=2, L=23, H=4, P=3, N=5, G=2, with_init=True):
    inp = _dyadic(make_inputs(b, L, H, P, N, G, "f32", seed=seed, dt_range=(2e-2, 5e-1), with_init=with_init))
    rng = np.random.default_rng(seed)
    dy = np.round(rng.standard_normal((b, L, H, P)) * 64) / 64
    dfinal = np.round(rng.standard_normal((b, H, P, N)) * 64) / 64
    return inp, dy, dfinal


def _loss(inp, dy, dfinal):
    y, f = oracle.recurrence(**inp)
    return float(np.sum(dy * y)) + (float(np.sum(dfinal * f)) if dfinal is not None else 0.0)


def _rel(got, want):
    scale = float(np.max(np.abs(want))) or 1.0
    return float(np.max(np.abs(np.asarray(got) - np.asarray(want)))) / scale


# -- pins -----------------------------------------------------------------------

def pin_central_differences(bwd):
    """dL along a random direction of one input = <grad, direction>, for every input."""
    inp, dy, dfinal = _case(5)
    g = bwd(inp, dy, dfinal)
    rng = np.random.default_rng(11)
    for k in KEYS:
        base = inp[k].double().numpy()
        step = rng.integers(-3, 4, size=base.shape).astype(np.float64) * 2.0 ** -20
        if k == "dt":
            step *= 0.25
        plus, minus = dict(inp), dict(inp)
        plus[k] = torch.from_numpy((base + step).astype(np.float32))
        minus[k] = torch.from_numpy((base - step).astype(np.float32))
        # the perturbed fp32 inputs hold base +- step exactly
        assert np.array_equal(plus[k].double().numpy() - base, step)
        assert np.array_equal(base - minus[k].double().numpy(), step)
        fd = (_loss(plus, dy, dfinal) - _loss(minus, dy, dfinal)) / 2.0
        lin = float(np.sum(g[GRAD[k]] * step))
        scale = float(np.sum(np.abs(g[GRAD[k]] * step)))
        assert abs(fd - lin) <= 1e-6 * scale, f"d{k}: difference {fd:.12e} vs gradient {lin:.12e}"


def _torch_loss(inp, dy, dfinal):
    """The recurrence written out with torch fp64 ops, for autograd."""
    x, dt, A, B, C, D, s0 = (inp[k] for k in KEYS)
    b, L, H, P = x.shape
    G = B.shape[2]
    hpg = H // G
    s = s0.clone()
    loss = torch.zeros((), dtype=torch.float64)
    for t in range(L):
        Bt = B[:, t].repeat_interleave(hpg, dim=1)  # [b,H,N]
        Ct = C[:, t].repeat_interleave(hpg, dim=1)
        a = torch.exp(dt[:, t] * A)  # [b,H]
        s = a[:, :, None, None] * s + (dt[:, t, :, None] * x[:, t])[..., None] * Bt[:, :, None, :]
        y = torch.einsum("bhpn,bhn->bhp", s, Ct) + D[None, :, None] * x[:, t]
        loss = loss + torch.sum(torch.from_numpy(dy[:, t]) * y)
    return loss + torch.sum(torch.from_numpy(dfinal) * s)


def pin_autograd(bwd):
    """Gradients of the written-out recurrence by torch reverse-mode autodiff."""
    inp, dy, dfinal = _case(6, b=1, L=9, H=6, P=2, N=3, G=3)
    g = bwd(inp, dy, dfinal)
    leaves = {k: inp[k].double().clone().requires_grad_(True) for k in KEYS}
    _torch_loss(leaves, dy, dfinal).backward()
    for k in KEYS:
        err = _rel(g[GRAD[k]], leaves[k].grad.numpy())
        assert err <= 1e-12, f"d{k} vs autograd: {err:.3e}"


def pin_final_gradient_only(bwd):
    """dy = 0: dinit = exp(A sum_t dt_t) dfinal, dx_t = dt_t exp(A sum_{u>t} dt_u) (B_t . dfinal),
    and nothing reaches C or D."""
    inp, _, dfinal = _case(7)
    x, dt, A, B = (inp[k].double().numpy() for k in ("x", "dt", "A", "B"))
    b, L, H, P = x.shape
    G = B.shape[2]
    g = bwd(inp, np.zeros((b, L, H, P)), dfinal)
    after = np.cumsum(dt[:, ::-1], axis=1)[:, ::-1] - dt  # sum over u > t, [b,L,H]
    total = dt.sum(axis=1)  # [b,H]
    np.testing.assert_allclose(g["dinit"], np.exp(A * total)[:, :, None, None] * dfinal, rtol=1e-13, atol=0)
    Bh = np.repeat(B, H // G, axis=2)  # [b,L,H,N]
    want = dt[..., None] * np.exp(A * after)[..., None] * np.einsum("blhn,bhpn->blhp", Bh, dfinal)
    assert _rel(g["dx"], want) <= 1e-13, "dx with dy = 0"
    assert np.all(g["dC"] == 0) and np.all(g["dD"] == 0)


def pin_linear_parts(bwd):
    """Euler's theorem on the parts of L that are linear:
    y and the final state are linear in (x, init) jointly, y is linear in C
    (the final state does not see C), and the input term is bilinear in x and B."""
    inp, dy, dfinal = _case(8)
    g = bwd(inp, dy, dfinal)
    x, C, B, D, s0 = (inp[k].double().numpy() for k in ("x", "C", "B", "D", "init_state"))
    y, f = oracle.recurrence(**inp)
    L_total = float(np.sum(dy * y) + np.sum(dfinal * f))
    lhs = float(np.sum(g["dx"] * x) + np.sum(g["dinit"] * s0))
    assert abs(lhs - L_total) <= 1e-12 * (abs(L_total) + 1.0), "<dx,x> + <dinit,init> != L"
    y_no_D = y - D[None, None, :, None] * x
    want = float(np.sum(dy * y_no_D))
    assert abs(float(np.sum(g["dC"] * C)) - want) <= 1e-12 * (abs(want) + 1.0), "<dC,C> != <dy, y - D x>"
    want = float(np.sum(g["dD"] * D) + np.sum(g["dB"] * B))
    assert abs(float(np.sum(g["dx"] * x)) - want) <= 1e-12 * (abs(want) + 1.0), "<dx,x> != <dD,D> + <dB,B>"


PINS = [pin_central_differences, pin_autograd, pin_final_gradient_only, pin_linear_parts]


def _bwd_with(lib):
    return lambda inp, dy, dfinal: oracle.backward(**inp, dy=dy, dfinal=dfinal, lib=lib)


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_backward_pin(pin):
    pin(_bwd_with(None))


def test_threads_and_missing_optionals():
    inp, dy, dfinal = _case(9, b=3, G=4, H=8)
    one = oracle.backward(**inp, dy=dy, dfinal=dfinal, nthreads=1)
    many = oracle.backward(**inp, dy=dy, dfinal=dfinal, nthreads=5)
    for k in one:
        assert np.array_equal(one[k], many[k]), k
    # no D, no init state, no final-state gradient: the same as zeros for each
    bare = dict(inp, D=None, init_state=None)
    g0 = oracle.backward(**bare, dy=dy, dfinal=None)
    z = dict(inp, D=torch.zeros_like(inp["D"]), init_state=torch.zeros_like(inp["init_state"]))
    g1 = oracle.backward(**z, dy=dy, dfinal=np.zeros_like(dfinal))
    for k in ("dx", "ddt", "dA", "dB", "dC", "dinit"):
        assert np.array_equal(g0[k], g1[k]), k


def test_rejects_bad_shapes():
    inp, dy, dfinal = _case(10)
    with pytest.raises(ValueError):
        oracle.backward(**inp, dy=dy[:, :-1], dfinal=dfinal)
    with pytest.raises(ValueError):
        oracle.backward(**inp, dy=dy, dfinal=dfinal[..., :-1])


MUTANTS = {
    "dC_previous_state": ("job->dC[bc + n] += dy_t * s_all[(t + 1) * N + n];",
                          "job->dC[bc + n] += dy_t * s_all[t * N + n];"),
    "dB_no_dt": ("job->dB[bc + n] += dt_t * x_t * lam[n];", "job->dB[bc + n] += x_t * lam[n];"),
    "ddt_no_decay_term": ("job->ddt[ti] += x_t * b_lam + A_h * a_t * lam_sprev;", "job->ddt[ti] += x_t * b_lam;"),
    "ddt_no_input_term": ("job->ddt[ti] += x_t * b_lam + A_h * a_t * lam_sprev;",
                          "job->ddt[ti] += A_h * a_t * lam_sprev;"),
    "dA_factor_A": ("job->dA_part[bg * H + h] += dt_t * a_t * lam_sprev;",
                    "job->dA_part[bg * H + h] += A_h * a_t * lam_sprev;"),
    "dx_no_D": ("job->dx[xi] = D_h * dy_t + dt_t * b_lam;", "job->dx[xi] = dt_t * b_lam;"),
    "dinit_missing_first_decay": ("lam[n] *= a_t;  /* a_t lam_t", "lam[n] *= (t > 0 ? a_t : 1.0);  /* a_t lam_t"),
    "decay_uses_current_state": ("lam_sprev += lam[n] * s_all[t * N + n];",
                                 "lam_sprev += lam[n] * s_all[(t + 1) * N + n];"),
    "dfinal_ignored": ("lam[n] = job->dfinal ? job->dfinal[((b * H + h) * P + p) * N + n] : 0.0;", "lam[n] = 0.0;"),
    "dD_scaled_by_dt": ("job->dD_part[bg * H + h] += dy_t * x_t;", "job->dD_part[bg * H + h] += dy_t * dt_t * x_t;"),
    "heads_strided_over_groups": ("for (long h = g * hpg; h < (g + 1) * hpg; ++h) {\n        const double A_h",
                                  "for (long h = g; h < H; h += G) {\n        const double A_h"),
    "B_read_as_C": ("const double B_n = widen(pr->B, bc + n, pr->in_dtype);",
                    "const double B_n = widen(pr->C, bc + n, pr->in_dtype);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_backward_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(SRC) as fh:
        src = fh.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.load_library(oracle.compile_library(str(path), str(tmp_path / "libmutant.so")))
    caught = []
    for pin in PINS:
        try:
            pin(_bwd_with(lib))
        except (AssertionError, RuntimeError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
