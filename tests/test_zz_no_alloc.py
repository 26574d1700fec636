"""ssd_fwd_noalloc: the forward for callers that may not allocate device memory.

Some callers cannot call the CUDA allocator at all: processes that hand all
device memory to a framework-owned pool, plugins hosted by such runtimes, and
latency-critical loops for which an allocator call (which can synchronise the
device or fail under memory pressure) is not acceptable.  For them the library
has one entry point whose scratch is a fixed 32 MiB array compiled into the
library.  These tests call it through the C ABI and check it against the
regular entry point, ssd_fwd, on two calls in a row (the scratch is shared and
keeps the previous call's contents, so the second call must not be polluted by
the first).

The file is named so that pytest collects it last.
"""
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


def _regular(c, chunk):
    y, f = ssd.ssd_fwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init_state"], chunk=chunk)
    ssd.ssd_check_device_status()
    return y, f


def _noalloc(c, chunk):
    y, f = ssd.ssd_fwd_noalloc(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init_state"], chunk=chunk)
    ssd.ssd_check_device_status()
    return y, f


def test_noalloc_matches_regular_entry_twice_in_a_row():
    # Two different problems (the persistent dstate-64 kernel and the one-unit
    # dstate-128 kernel) through the no-allocation entry back to back, with no
    # synchronisation in between, then the same pair again.  Both entries run
    # the same deterministic kernels, so each result must equal ssd_fwd's bit
    # for bit: a scratch left polluted by the previous call would show here.
    cases = [(2, 1000, 8, 64, 64, 2, 128, 31), (1, 700, 4, 128, 128, 1, 100, 32)]
    data, refs = [], []
    for b, L, H, P, N, G, Q, seed in cases:
        inp = make_inputs(b, L, H, P, N, G, "bf16", seed=seed, with_init=True)
        c = to_cuda(inp)
        assert ssd.ssd_fwd_workspace_size(b, L, H, P, G, N, Q, torch.bfloat16) <= 32 << 20
        data.append((inp, c, Q))
        refs.append(_regular(c, Q))
    for rep in range(2):
        outs = []
        for inp, c, Q in data:
            outs.append(ssd.ssd_fwd_noalloc(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init_state"],
                                            chunk=Q))
        ssd.ssd_check_device_status()
        for (y, f), (y_ref, f_ref) in zip(outs, refs):
            assert torch.equal(y, y_ref), f"y differs from ssd_fwd (call pair {rep})"
            assert torch.equal(f, f_ref), f"final state differs from ssd_fwd (call pair {rep})"
    # and against the oracle, within the library's tolerance
    inp, c, Q = data[0]
    yr, fr = oracle.recurrence(**inp)
    y, f = outs[0]
    assert_close(y.float().cpu().numpy(), yr, TOL[torch.bfloat16], "y, no-alloc vs oracle", STORAGE_U[torch.bfloat16])
    assert_close(f.cpu().numpy(), fr, TOL[torch.bfloat16], "final state, no-alloc vs oracle")


def test_noalloc_long_chunk_at_dstate_128():
    # ssd_fwd takes a 256-token chunk at dstate 128 on the three-kernel path; the
    # no-allocation entry runs the fused kernel only and evaluates it as two 128-token
    # blocks: the same result up to rounding, so it agrees with the oracle
    inp = make_inputs(1, 600, 4, 64, 128, 1, "bf16", seed=35, with_init=True)
    c = to_cuda(inp)
    assert ssd.ssd_fwd_path(1, 600, 4, 64, 1, 128, 256, torch.bfloat16) == "tcgen05"
    y, f = _noalloc(c, 256)
    yr, fr = oracle.recurrence(**inp)
    assert_close(y.float().cpu().numpy(), yr, TOL[torch.bfloat16], "y, no-alloc chunk 256", STORAGE_U[torch.bfloat16])
    assert_close(f.cpu().numpy(), fr, TOL[torch.bfloat16], "final state, no-alloc chunk 256")


def test_noalloc_rejects_what_it_cannot_hold():
    # larger than the fixed scratch: a clear error, nothing enqueued.  (At dstate
    # 64 the scratch is one state slot per CTA, at most 16 MiB, so every size
    # fits; at dstate 128 it grows with the number of (chunk, head block) units.)
    c = to_cuda(make_inputs(1, 64, 2, 64, 64, 1, "bf16", seed=33))
    big = dict(b=1, L=8192, H=16, P=64, N=128, G=1, Q=128)
    need = ssd.ssd_fwd_workspace_size(big["b"], big["L"], big["H"], big["P"], big["G"], big["N"], big["Q"],
                                      torch.bfloat16)
    assert need > 32 << 20
    x = torch.empty(big["b"], big["L"], big["H"], big["P"], dtype=torch.bfloat16, device="cuda")
    dt = torch.empty(big["b"], big["L"], big["H"], dtype=torch.float32, device="cuda")
    A = torch.empty(big["H"], dtype=torch.float32, device="cuda")
    Bm = torch.empty(big["b"], big["L"], big["G"], big["N"], dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ssd.SsdError) as err:
        ssd.ssd_fwd_noalloc(x, dt, A, Bm, Bm, chunk=big["Q"])
    assert err.value.status == ssd.SSD_ERR_UNSUPPORTED and "scratch" in str(err.value)
    # a size the fused kernel does not handle (fp32)
    c32 = to_cuda(make_inputs(1, 64, 2, 64, 64, 1, "f32", seed=34))
    with pytest.raises(ssd.SsdError) as err:
        ssd.ssd_fwd_noalloc(c32["x"], c32["dt"], c32["A"], c32["B"], c32["C"], chunk=64)
    assert err.value.status == ssd.SSD_ERR_UNSUPPORTED
    # the library still works after the rejections
    y, _ = _noalloc(c, 64)
    y_ref, _ = _regular(c, 64)
    assert_close(y.float().cpu().numpy(), y_ref.float().cpu().numpy(), TOL[torch.bfloat16], "y after rejections",
                 2 * STORAGE_U[torch.bfloat16])
