"""Parity of the CUDA backward (ssd_bwd) with the fp64 oracle's backward.

Both sides get the same seeded inputs and incoming gradients (dy in the dtype
of x, its exact values widened for the oracle; dfinal fp32).  Every gradient is
fp32 on the GPU and all its arithmetic is fp32, so the bound is the fp32 one for
both input dtypes: max |g_gpu - g_ref| <= 1e-4 x RMS(g_ref), per gradient.
Cases span several 64-token chunks with a ragged tail, one and several heads
per group (the per-head partial sums and their reduction), headdim and dstate
that are not multiples of the kernels' tiles, a one-token sequence, absent
optional inputs, and the 2.7B-shaped layer at full size.
"""
import numpy as np
import pytest
import torch

import oracle
import structured_state_space_03_b300 as ssd
from structured_state_space_03_b300.workloads import HEADLINE, make_cotangents, make_inputs
from parity import rel_err, to_cuda

pytestmark = pytest.mark.gpu

TOL = 1e-4
GRADS = ("dx", "ddt", "dA", "dB", "dC", "dD", "dinit")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    ssd.lib()


def _gpu(inp, dy, dfinal, **kw):
    c = to_cuda(inp)
    out = ssd.ssd_bwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init_state"], dy=dy.cuda(),
                      dfinal_state=None if dfinal is None else dfinal.cuda(), **kw)
    ssd.ssd_check_device_status()
    out["dinit"] = out.pop("dinit_state")
    return {k: (None if v is None else v.cpu().double().numpy()) for k, v in out.items()}


def _ref(inp, dy, dfinal):
    return oracle.backward(**inp, dy=dy.double().numpy(), dfinal=None if dfinal is None else dfinal.double().numpy())


def _compare(got, want, what, record=None):
    errs = {}
    for k in GRADS:
        if got.get(k) is None:
            continue
        errs[k] = rel_err(got[k], want[k])
    if record is not None:
        record.update(errs)
    bad = {k: e for k, e in errs.items() if e > TOL}
    assert not bad, f"{what}: gradients beyond {TOL:.0e} x RMS: " + ", ".join(f"{k} {e:.2e}" for k, e in bad.items())
    return errs


# (b, L, H, P, N, G, dtype, with_init, with_dfinal, with_D)
CASES = [
    (1, 256, 4, 16, 16, 1, "f32", False, False, True),     # the tiny fp32 workload
    (2, 300, 8, 64, 128, 2, "bf16", True, True, True),     # ragged tail, 4 heads per group
    (2, 130, 6, 40, 24, 3, "f32", True, True, True),       # headdim / dstate off the tiles
    (1, 200, 4, 128, 64, 4, "bf16", True, True, False),    # headdim 128, one head per group, no D
    (1, 100, 2, 64, 256, 1, "bf16", False, True, True),    # dstate 256
    (3, 64, 2, 16, 16, 1, "f32", True, True, True),        # exactly one chunk
    (2, 1, 2, 16, 16, 2, "f32", True, True, True),         # one token
    # the tensor-core in-chunk kernel (bf16, headdim 64, dstate 64, 128-token chunks)
    (2, 300, 8, 64, 64, 2, "bf16", True, True, True),      # ragged tail, 4 heads per group
    (1, 128, 4, 64, 64, 4, "bf16", True, True, False),     # exactly one chunk, one head per group, no D
    (2, 1, 2, 64, 64, 1, "bf16", True, True, True),        # one token
    (1, 1000, 2, 64, 64, 1, "bf16", False, False, True),   # eight chunks, no initial state, no dfinal
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}_L{}_H{}_P{}_N{}_G{}_{}".format(*c[:7]))
def test_backward_matches_oracle(case):
    b, L, H, P, N, G, dt, with_init, with_dfinal, with_D = case
    inp = make_inputs(b, L, H, P, N, G, dt, seed=500 + L, with_init=with_init, with_D=with_D)
    dy, dfinal = make_cotangents(b, L, H, P, N, dt, seed=500 + L, with_dfinal=with_dfinal)
    _compare(_gpu(inp, dy, dfinal), _ref(inp, dy, dfinal), str(case))


@pytest.mark.parametrize("case", [(2, 300, 8, 64, 64, 2, "bf16"), (1, 260, 4, 128, 64, 2, "bf16"), (1, 200, 4, 32, 48, 2, "f32")],
                         ids=["tensor_core", "simt_bf16", "simt_f32"])
def test_backward_with_large_steps(case):
    # steps of 0.5 .. 2 with |A| up to 16: the decay inside a chunk spans hundreds of e-folds;
    # every factor the kernels form is exp of a difference of segment sums in the decaying
    # direction, so none can overflow
    b, L, H, P, N, G, dt = case
    inp = make_inputs(b, L, H, P, N, G, dt, seed=600 + L, dt_range=(0.5, 2.0), with_init=True)
    dy, dfinal = make_cotangents(b, L, H, P, N, dt, seed=600 + L)
    _compare(_gpu(inp, dy, dfinal), _ref(inp, dy, dfinal), f"large steps {case}")


def test_optional_outputs_and_determinism():
    b, L, H, P, N, G = 2, 150, 4, 64, 64, 2
    inp = make_inputs(b, L, H, P, N, G, "bf16", seed=77, with_init=True)
    dy, dfinal = make_cotangents(b, L, H, P, N, "bf16", seed=77)
    full = _gpu(inp, dy, dfinal)
    again = _gpu(inp, dy, dfinal)
    for k in GRADS:
        assert np.array_equal(full[k], again[k]), f"{k} differs between two identical calls"
    part = _gpu(inp, dy, dfinal, want_dD=False, want_dinit=False)
    assert part["dD"] is None and part["dinit"] is None
    for k in ("dx", "ddt", "dA", "dB", "dC"):
        assert np.array_equal(full[k], part[k]), k


def test_headline_layer_full_size():
    # the 2.7B-shaped layer, every gradient element against the oracle
    w = HEADLINE
    inp = make_inputs(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.dtype, seed=w.seed,
                      dt_range=w.dt_range, with_init=True)
    dy, dfinal = make_cotangents(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.dtype, seed=w.seed)
    _compare(_gpu(inp, dy, dfinal), _ref(inp, dy, dfinal), w.name)



def test_per_kernel_timing_hook_outside_capture():
    # the timing hook records plain events around each backward kernel when no graph is being captured
    b, L, H, P, N, G = 1, 512, 8, 64, 64, 2
    inp = to_cuda(make_inputs(b, L, H, P, N, G, "bf16", seed=90))
    dy, dfinal = make_cotangents(b, L, H, P, N, "bf16", seed=90)
    names = ssd.ssd_bwd_kernels(b, L, H, P, G, N, torch.bfloat16)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * len(names))]
    for e in evs:
        e.record()  # torch creates the underlying CUDA event on first record
    torch.cuda.synchronize()
    ssd.ssd_profile_events(evs)
    try:
        ssd.ssd_bwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], None, dy=dy.cuda(),
                    dfinal_state=dfinal.cuda())
    finally:
        ssd.ssd_profile_events(None)
    ssd.ssd_check_device_status()
    times = [evs[2 * k].elapsed_time(evs[2 * k + 1]) for k in range(len(names))]
    assert all(t > 0 for t in times), dict(zip(names, times))


def test_tensor_core_kernel_is_the_one_that_runs():
    assert "bwd_chunk_tc" in ssd.ssd_bwd_kernels(2, 300, 8, 64, 2, 64, torch.bfloat16)
    assert ssd.ssd_bwd_kernels(2, 2048, 80, 64, 1, 64, torch.bfloat16) == [
        "chunk_state_tc", "chunk_state_tc", "bwd_state_pass", "bwd_chunk_tc", "bwd_reduce_groups", "bwd_reduce_heads"]
    # one head per group: the head pairs of the forward's chunk-state kernel straddle groups
    assert ssd.ssd_bwd_kernels(1, 128, 4, 64, 4, 64, torch.bfloat16) == [
        "bwd_chunk_states", "bwd_state_pass", "bwd_chunk_tc", "bwd_reduce_heads"]
    assert "bwd_chunk" in ssd.ssd_bwd_kernels(2, 300, 8, 64, 2, 128, torch.bfloat16)
    assert "bwd_chunk" in ssd.ssd_bwd_kernels(2, 300, 8, 64, 2, 64, torch.float32)
