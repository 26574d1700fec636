"""Failure detection of the fused kernels, tested without any GPU fault.

The fused kernels resolve the chunk-to-chunk recurrence ("Mamba 模型" §4.1:
the off-diagonal blocks pass through the hidden state) by waiting inside the
kernel for the chunk states other units publish.  Every such wait is bounded:
one that runs out sets the library's device error word and the kernel gives
up instead of hanging.  Here a unit's publication is withheld through the
library's test hook (ssd_test_set_fault), so the waits of the units after it
wait for a flag that nothing sets; with a 1 ms limit they give up, the call
ends, ssd_check_device_status reports SSD_ERR_TIMEOUT, and the next ordinary
call on the same context is correct again.
"""
import time

import pytest
import torch

import structured_state_space_03_b300 as ssd
from structured_state_space_03_b300.workloads import make_inputs
from parity import check_full, to_cuda

pytestmark = pytest.mark.gpu

# (b, L, H, P, N, G, Q): the sequence-pipelined dstate-64 kernel (few sequences), the
# persistent look-back dstate-64 kernel (40 sequences), the one-unit dstate-128 kernel
FUSED = [(2, 1000, 8, 64, 64, 2, 128), (1, 700, 80, 64, 64, 1, 128), (1, 700, 4, 128, 128, 1, 100)]
KERNELS = ["ssd_seq_pipe_tc", "ssd_fused_pipe_tc", "ssd_fused_tc"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    ssd.lib()
    yield
    ssd.ssd_test_set_fault(0, -1)


@pytest.fixture(autouse=True)
def _reset_hook():
    yield
    ssd.ssd_test_set_fault(0, -1)


@pytest.mark.parametrize("case,kernel", list(zip(FUSED, KERNELS)), ids=KERNELS)
def test_withheld_state_times_out_then_recovers(case, kernel):
    b, L, H, P, N, G, Q = case
    assert ssd.ssd_fwd_kernels(b, L, H, P, G, N, Q, torch.bfloat16) == [kernel]
    inp = make_inputs(b, L, H, P, N, G, "bf16", seed=71 + N, with_init=True)
    c = to_cuda(inp)
    ssd.ssd_check_device_status()  # start from a clear error word
    ssd.ssd_test_set_fault(1_000_000, 0)  # 1 ms waits; unit 0 (chunk 0 of the first sequence) withheld
    t0 = time.perf_counter()
    ssd.ssd_fwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init_state"], chunk=Q)
    with pytest.raises(ssd.SsdError) as err:
        ssd.ssd_check_device_status()
    elapsed = time.perf_counter() - t0
    assert err.value.status == ssd.SSD_ERR_TIMEOUT, str(err.value)
    assert elapsed < 10.0, f"the failing call took {elapsed:.1f} s"
    # the error word was read and cleared; the context is usable and correct again
    ssd.ssd_test_set_fault(0, -1)
    ssd.ssd_check_device_status()
    check_full(inp, Q)


def test_short_limit_alone_changes_nothing():
    # a limit far above any legitimate wait, with nothing withheld: ordinary results
    b, L, H, P, N, G, Q = FUSED[0]
    inp = make_inputs(b, L, H, P, N, G, "bf16", seed=75, with_init=True)
    ssd.ssd_test_set_fault(50_000_000, -1)
    check_full(inp, Q)


def test_hook_is_per_thread():
    # a setting made on another thread does not reach this thread's forwards
    import threading
    b, L, H, P, N, G, Q = FUSED[0]
    inp = make_inputs(b, L, H, P, N, G, "bf16", seed=76)
    t = threading.Thread(target=lambda: ssd.ssd_test_set_fault(1_000_000, 0))
    t.start()
    t.join()
    check_full(inp, Q)
