"""ssd_step, the recurrent single-token form, on the GPU through the C ABI.

One step is the layer's recurrence for one token with the state carried in
and out, so it is checked (1) against the fp64 oracle run over that one token
with the same entry state, and (2) as a continuation: a prefix through ssd_fwd
followed by single steps must reproduce ssd_fwd over the whole sequence and
the oracle's outputs token by token.
"""
import numpy as np
import pytest
import torch

import oracle
import structured_state_space_03_b300 as ssd
from structured_state_space_03_b300.workloads import make_inputs
from parity import STORAGE_U, TOL, assert_close, to_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    ssd.lib()


def _token(inp, t):
    """Token t of a sequence input set, in the step layouts."""
    return (inp["x"][:, t].contiguous(), inp["dt"][:, t].contiguous(), inp["B"][:, t].contiguous(),
            inp["C"][:, t].contiguous())


# (batch, nheads, headdim, dstate, ngroups)
SHAPES = [(2, 80, 64, 64, 1), (3, 8, 16, 48, 2), (1, 4, 128, 256, 4), (2, 6, 33, 20, 3),
          (5, 3, 8, 64, 1), (2, 3, 1, 16, 1)]  # the last two: few rows per head (partly idle blocks)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_one_step_matches_oracle(shape, dtype):
    b, H, P, N, G = shape
    inp = make_inputs(b, 1, H, P, N, G, dtype, seed=40 + N, with_init=True)
    yr, fr = oracle.recurrence(**inp)  # [b,1,H,P], [b,H,P,N]
    c = to_cuda(inp)
    state = c["init_state"].clone()
    x, dt, B, C = _token(c, 0)
    y = ssd.ssd_step(x, dt, c["A"], B, C, c["D"], state=state)
    ssd.ssd_check_device_status()
    el = torch.float32 if dtype == "f32" else torch.bfloat16
    assert_close(y.float().cpu().numpy(), yr[:, 0], TOL[el], "y (one step)", STORAGE_U[el])
    assert_close(state.cpu().numpy(), fr, TOL[el], "state after one step")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_steps_continue_a_prefix(dtype):
    """ssd_fwd over a prefix, then one step per token: every y_t and the final
    state agree with the oracle over the whole sequence, and y_t agrees with
    ssd_fwd run over the whole sequence."""
    b, L0, T, H, P, N, G = 2, 200, 12, 8, 64, 64, 2
    inp = make_inputs(b, L0 + T, H, P, N, G, dtype, seed=51, with_init=True)
    el = inp["x"].dtype
    yr, fr = oracle.recurrence(**inp)
    c = to_cuda(inp)
    pre = {k: (v[:, :L0].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in c.items()}
    _, state = ssd.ssd_fwd(pre["x"], pre["dt"], pre["A"], pre["B"], pre["C"], pre["D"], pre["init_state"], chunk=64)
    y_full, f_full = ssd.ssd_fwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init_state"], chunk=64)
    ys = []
    for t in range(L0, L0 + T):
        x, dt, B, C = _token(c, t)
        ys.append(ssd.ssd_step(x, dt, c["A"], B, C, c["D"], state=state))
    ssd.ssd_check_device_status()
    y_steps = torch.stack(ys, dim=1).float().cpu().numpy()
    assert_close(y_steps, yr[:, L0:], TOL[el], "y of the steps vs oracle", STORAGE_U[el])
    assert_close(state.cpu().numpy(), fr, TOL[el], "state after the steps vs oracle")
    assert_close(y_steps, y_full[:, L0:].float().cpu().numpy(), TOL[el], "y of the steps vs ssd_fwd",
                 2 * STORAGE_U[el])
    assert_close(state.cpu().numpy(), f_full.cpu().numpy(), TOL[el], "state vs ssd_fwd final_state")


def test_zero_dt_keeps_state_and_reads_it_out():
    """dt = 0: the state is untouched and y = C . h + D x (a closed form)."""
    b, H, P, N, G = 2, 4, 16, 32, 2
    inp = make_inputs(b, 1, H, P, N, G, "f32", seed=61, with_init=True)
    c = to_cuda(inp)
    x, dt, B, C = _token(c, 0)
    dt.zero_()
    state = c["init_state"].clone()
    y = ssd.ssd_step(x, dt, c["A"], B, C, c["D"], state=state)
    ssd.ssd_check_device_status()
    assert torch.equal(state, c["init_state"])
    g = torch.arange(H, device="cuda") // (H // G)
    want = torch.einsum("bhpn,bhn->bhp", c["init_state"].double(), C[:, g].double()) + c["D"].double()[None, :, None] * x.double()
    assert_close(y.cpu().numpy(), want.cpu().numpy(), 1e-6, "y at dt = 0")


def test_without_D():
    b, H, P, N, G = 1, 4, 32, 64, 1
    inp = make_inputs(b, 1, H, P, N, G, "f32", seed=62, with_init=True, with_D=False)
    yr, fr = oracle.recurrence(**inp)
    c = to_cuda(inp)
    state = c["init_state"].clone()
    x, dt, B, C = _token(c, 0)
    y = ssd.ssd_step(x, dt, c["A"], B, C, None, state=state)
    ssd.ssd_check_device_status()
    assert_close(y.cpu().numpy(), yr[:, 0], TOL[torch.float32], "y (no D)", STORAGE_U[torch.float32])
    assert_close(state.cpu().numpy(), fr, TOL[torch.float32], "state (no D)")
