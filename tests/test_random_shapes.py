"""Seeded random shapes through every forward path and the backward, each
compared element by element with the oracle.

The fixed cases elsewhere pin known corners; these draw batch, length, heads,
headdim, state size, groups, chunk and dtype from each path's supported set
(seeded, so a failure reproduces), with ragged lengths and optional initial
states, so that an index that is only right for the usual shapes shows up.
"""
import numpy as np
import pytest
import torch

import oracle
import structured_state_space_03_b300 as ssd
from structured_state_space_03_b300.workloads import make_cotangents, make_inputs
from parity import STORAGE_U, TOL, assert_close, rel_err, to_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    ssd.lib()


def _draw_forward(rng):
    """One random forward problem: (b, L, H, P, N, G, Q, dtype, with_init)."""
    kind = rng.integers(0, 4)
    if kind == 0:  # fused (bf16, headdim 64/128, dstate 64/128, chunk <= 128)
        P = int(rng.choice([64, 128]))
        N = int(rng.choice([64, 128]))
        Q = int(rng.choice([64, 96, 100, 128]))
        hb = 128 // P
        G = int(rng.integers(1, 4))
        H = G * hb * int(rng.integers(1, 4))
        dt = "bf16"
    elif kind == 1:  # multi-kernel tcgen05 (dstate 256 or chunk 256)
        P = int(rng.choice([64, 128]))
        N, Q = (256, int(rng.choice([64, 128, 256]))) if rng.integers(0, 2) else (int(rng.choice([64, 128])), 256)
        hb = 128 // P
        G = int(rng.integers(1, 3))
        H = G * hb * int(rng.integers(1, 3))
        dt = "bf16"
    elif kind == 2:  # fp32 FMA path
        P = int(rng.choice([16, 24, 32, 64]))
        N = int(rng.choice([16, 20, 64]))
        Q = int(rng.choice([32, 64, 100]))
        G = int(rng.integers(1, 3))
        H = G * int(rng.integers(1, 4))
        dt = "f32"
    else:  # bf16 on the fp32 FMA path (headdim outside 64/128)
        P = int(rng.choice([16, 32, 48]))
        N = int(rng.choice([32, 64]))
        Q = int(rng.choice([64, 128]))
        G = int(rng.integers(1, 3))
        H = G * int(rng.integers(1, 3))
        dt = "bf16"
    b = int(rng.integers(1, 4))
    L = int(rng.integers(1, 3 * Q + 7))
    return b, L, H, P, N, G, Q, dt, bool(rng.integers(0, 2))


@pytest.mark.parametrize("seed", range(24))
def test_random_forward_matches_oracle(seed):
    rng = np.random.default_rng(9000 + seed)
    b, L, H, P, N, G, Q, dt, with_init = _draw_forward(rng)
    inp = make_inputs(b, L, H, P, N, G, dt, seed=9000 + seed, with_init=with_init)
    c = to_cuda(inp)
    y, f = ssd.ssd_fwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init_state"], chunk=Q)
    ssd.ssd_check_device_status()
    yr, fr = oracle.recurrence(**inp)
    el = c["x"].dtype
    what = f"b{b} L{L} H{H} P{P} N{N} G{G} Q{Q} {dt} init={with_init} path={ssd.ssd_fwd_path(b, L, H, P, G, N, Q, el)}"
    assert_close(y.float().cpu().numpy(), yr, TOL[el], "y " + what, STORAGE_U[el])
    assert_close(f.cpu().numpy(), fr, TOL[el], "final state " + what)


@pytest.mark.parametrize("seed", range(12))
def test_random_backward_matches_oracle(seed):
    rng = np.random.default_rng(9500 + seed)
    if rng.integers(0, 2):  # the tensor-core in-chunk kernel
        P, N, dt = 64, 64, "bf16"
    else:
        P, N = int(rng.choice([16, 40, 64, 128])), int(rng.choice([16, 24, 64, 128, 256]))
        dt = str(rng.choice(["f32", "bf16"]))
    G = int(rng.integers(1, 4))
    H = G * int(rng.integers(1, 4))
    b, L = int(rng.integers(1, 3)), int(rng.integers(1, 400))
    with_init, with_dfinal = bool(rng.integers(0, 2)), bool(rng.integers(0, 2))
    inp = make_inputs(b, L, H, P, N, G, dt, seed=9500 + seed, with_init=with_init)
    dy, dfinal = make_cotangents(b, L, H, P, N, dt, seed=9500 + seed, with_dfinal=with_dfinal)
    c = to_cuda(inp)
    g = ssd.ssd_bwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init_state"], dy=dy.cuda(),
                    dfinal_state=None if dfinal is None else dfinal.cuda())
    ssd.ssd_check_device_status()
    ref = oracle.backward(**inp, dy=dy.double().numpy(), dfinal=None if dfinal is None else dfinal.double().numpy())
    what = f"b{b} L{L} H{H} P{P} N{N} G{G} {dt} kernels={ssd.ssd_bwd_kernels(b, L, H, P, G, N, c['x'].dtype)}"
    for k, rk in (("dx", "dx"), ("ddt", "ddt"), ("dA", "dA"), ("dB", "dB"), ("dC", "dC"), ("dD", "dD"),
                  ("dinit_state", "dinit")):
        err = rel_err(g[k].double().cpu().numpy(), ref[rk])
        assert err <= 1e-4, f"{k}: {err:.2e} x RMS ({what})"
