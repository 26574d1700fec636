"""ssd_fwd_pre on the GPU through the C ABI: the dt pre-step (softplus of
dt + bias, zero-order-hold input scale) against the oracle's recurrence with
the same pre-step, on every path of the library."""
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


# b, L, H, P, N, G, Q, dtype, expected path
CASES = [
    (2, 600, 8, 64, 64, 2, 128, "bf16", "tcgen05_fused"),   # persistent fused kernel
    (1, 400, 2, 128, 128, 1, 128, "bf16", "tcgen05_fused"),  # one-unit fused kernel
    (1, 500, 4, 64, 256, 1, 256, "bf16", "tcgen05"),         # three-kernel tensor-core path (dstate 256)
    (1, 500, 4, 64, 128, 1, 256, "bf16", "tcgen05"),         # dstate 128 at chunk 256: three kernels
    (1, 500, 4, 64, 64, 1, 256, "bf16", "tcgen05_fused"),    # dstate 64: chunk 256 as two 128-token blocks
    (2, 300, 6, 32, 48, 3, 100, "f32", "simt"),             # fp32 path
]
MODES = [dict(softplus=True, bias=True), dict(zoh=True), dict(softplus=True, bias=True, zoh=True)]


@pytest.mark.parametrize("mode", MODES, ids=["softplus_bias", "zoh", "softplus_bias_zoh"])
@pytest.mark.parametrize("case", CASES, ids=[c[8] + f"_N{c[4]}Q{c[6]}" for c in CASES])
def test_pre_step_matches_oracle(case, mode):
    b, L, H, P, N, G, Q, dtype, path = case
    el = torch.float32 if dtype == "f32" else torch.bfloat16
    assert ssd.ssd_fwd_path(b, L, H, P, G, N, Q, el) == path
    # raw dt around zero so that the softplus matters; |A| in [1, 16]
    inp = make_inputs(b, L, H, P, N, G, dtype, seed=300 + N + Q, dt_range=(1e-3, 1e-1), with_init=True)
    if mode.get("softplus"):
        inp["dt"] = (torch.log(inp["dt"]) * 0.5).contiguous()  # mostly negative: softplus keeps it positive
    bias = torch.linspace(-2.0, -0.5, H) if mode.get("bias") else None
    yr, fr = oracle.recurrence_pre(**inp, dt_bias=bias, softplus=mode.get("softplus", False),
                                   zoh=mode.get("zoh", False))
    c = to_cuda(inp)
    y, f = ssd.ssd_fwd_pre(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init_state"], chunk=Q,
                           dt_bias=None if bias is None else bias.cuda(), softplus=mode.get("softplus", False),
                           zoh=mode.get("zoh", False))
    ssd.ssd_check_device_status()
    assert_close(y.float().cpu().numpy(), yr, TOL[el], "y", STORAGE_U[el])
    assert_close(f.cpu().numpy(), fr, TOL[el], "final_state")


def test_no_pre_step_is_ssd_fwd():
    inp = make_inputs(2, 500, 8, 64, 64, 2, "bf16", seed=320, with_init=True)
    c = to_cuda(inp)
    y0, f0 = ssd.ssd_fwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init_state"], chunk=128)
    y1, f1 = ssd.ssd_fwd_pre(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init_state"], chunk=128)
    ssd.ssd_check_device_status()
    assert torch.equal(y0, y1) and torch.equal(f0, f1)
