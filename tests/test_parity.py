"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import structured_state_space_03_b300 as ssd
from structured_state_space_03_b300.workloads import WORKLOADS, make_inputs, sample_rows, workload_inputs
from parity import STORAGE_U, TOL, assert_close, check_all_rows, check_full, check_rows, run_gpu, to_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    ssd.lib()


# -- the five workloads ---------------------------------------------------------

def test_tiny_f32_full():
    w = WORKLOADS[0]
    inp = workload_inputs(w)
    check_full(inp, w.chunk)


@pytest.mark.parametrize("w", WORKLOADS[1:], ids=[w.name for w in WORKLOADS[1:]])
def test_workload_all_rows(w):
    """Each large workload at full size, in the launch configuration the
    benchmark times, compared with the oracle on every element of y and of the
    final state.  The storage-adjusted and the raw max-abs errors (x RMS) are
    printed, and appended as a JSON line to $SSD_PARITY_LOG when it is set."""
    assert ssd.ssd_fwd_path(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.chunk,
                            ssd.SSD_DTYPE_BF16) in ("tcgen05", "tcgen05_fused")
    inp = workload_inputs(w)
    rec = {}
    try:
        check_all_rows(inp, w.chunk, record=rec)
    finally:
        if rec:
            line = {"workload": w.name, "path": ssd.ssd_fwd_path(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups,
                                                                  w.dstate, w.chunk, ssd.SSD_DTYPE_BF16), **rec}
            print(json.dumps(line))
            if os.environ.get("SSD_PARITY_LOG"):
                with open(os.environ["SSD_PARITY_LOG"], "a") as fh:
                    fh.write(json.dumps(line) + "\n")


# -- mid-size cases compared element by element (several chunks, ragged tail) ---

MID = [
    # b, L, H, P, N, G, Q, dtype
    (2, 1000, 8, 64, 64, 2, 128, "bf16"),
    (3, 777, 4, 64, 64, 1, 128, "bf16"),      # one group of four heads, ragged tail
    (2, 1000, 8, 64, 64, 2, 64, "bf16"),      # chunk 64
    (1, 8000, 2, 64, 64, 1, 64, "bf16"),      # 125 chained chunks of one head pair: deep look-back
    (3, 700, 4, 128, 128, 2, 100, "bf16"),
    (1, 1000, 4, 64, 256, 1, 128, "bf16"),
    (1, 777, 4, 64, 128, 1, 256, "bf16"),
    (1, 600, 4, 64, 256, 1, 256, "bf16"),
    (2, 513, 8, 128, 128, 2, 128, "bf16"),
    (1, 300, 4, 64, 64, 4, 64, "bf16"),
    (2, 600, 4, 128, 64, 2, 128, "bf16"),     # persistent kernel, one head per unit, ragged tail
    (1, 700, 6, 64, 64, 3, 96, "bf16"),       # persistent kernel, nheads % 4 != 0 (dt without TMA), chunk 96
    (1, 700, 80, 64, 64, 1, 128, "bf16"),     # 40 sequences: the persistent look-back kernel, ragged tail
    (3, 300, 24, 64, 64, 2, 64, "bf16"),      # 36 sequences, chunk 64: the persistent look-back kernel
    (2, 333, 6, 32, 48, 3, 100, "f32"),
    (1, 1000, 4, 16, 16, 1, 64, "f32"),
]


@pytest.mark.parametrize("case", MID, ids=[f"b{c[0]}L{c[1]}H{c[2]}P{c[3]}N{c[4]}G{c[5]}Q{c[6]}{c[7]}" for c in MID])
@pytest.mark.parametrize("with_init", [False, True])
def test_mid_full(case, with_init):
    b, L, H, P, N, G, Q, dt = case
    inp = make_inputs(b, L, H, P, N, G, dt, seed=L + P + N, with_init=with_init)
    check_full(inp, Q)


def test_mid_cases_cover_both_dstate64_kernels():
    """dstate 64 runs on two fused kernels chosen by the number of (batch, head
    block) sequences; the element-by-element cases above exercise both."""
    names = {tuple(ssd.ssd_fwd_kernels(b, L, H, P, G, N, Q, torch.bfloat16))
             for b, L, H, P, N, G, Q, dt in MID if dt == "bf16" and N == 64}
    assert ("ssd_seq_pipe_tc",) in names and ("ssd_fused_pipe_tc",) in names, names


# -- edge cases ---------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("L", [1, 5, 63, 64, 65, 127, 129])
def test_short_and_ragged_sequences(dtype, L):
    inp = make_inputs(2, L, 4, 64, 64, 1, dtype, seed=100 + L, with_init=True)
    check_full(inp, 64)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_optional_tensors_absent(dtype):
    inp = make_inputs(1, 200, 4, 64, 64, 1, dtype, seed=5, with_init=False, with_D=False)
    check_full(inp, 64)
    yg, fg = run_gpu(to_cuda(inp), 64, return_final=False)
    assert fg is None
    yr, _ = oracle.recurrence(**inp)
    assert_close(yg.float().cpu().numpy(), yr, TOL[inp["x"].dtype], "y without final_state",
                 STORAGE_U[yg.dtype])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_A_zero_and_dt_zero(dtype):
    inp = make_inputs(1, 300, 4, 64, 64, 1, dtype, seed=6, with_init=True)
    inp["A"].zero_()
    check_full(inp, 128)
    inp = make_inputs(1, 300, 4, 64, 64, 1, dtype, seed=7, with_init=True)
    inp["dt"].zero_()
    check_full(inp, 128)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_in_place_state_carry(dtype):
    """init_state and final_state may be the same buffer."""
    inp = make_inputs(2, 300, 4, 64, 64, 1, dtype, seed=8, with_init=True)
    c = to_cuda(inp)
    state = c["init_state"].clone()
    y, f = ssd.ssd_fwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], state, chunk=128, final_state=state)
    ssd.ssd_check_device_status()
    yr, fr = oracle.recurrence(**inp)
    tol = TOL[inp["x"].dtype]
    assert_close(y.float().cpu().numpy(), yr, tol, "y", STORAGE_U[y.dtype])
    assert_close(state.cpu().numpy(), fr, tol, "in-place final state")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_state_split_on_gpu(dtype):
    """Two calls carrying the state match one call over the whole sequence."""
    inp = make_inputs(1, 700, 4, 64, 64, 1, dtype, seed=9, with_init=True)
    c = to_cuda(inp)
    y, f = run_gpu(c, 128)
    L1 = 300
    first = {k: (v[:, :L1].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in c.items()}
    second = {k: (v[:, L1:].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in c.items()}
    y1, f1 = run_gpu(first, 128)
    second["init_state"] = f1
    y2, f2 = run_gpu(second, 128)
    tol = TOL[inp["x"].dtype]
    yr, fr = oracle.recurrence(**inp)
    assert_close(torch.cat([y1, y2], 1).float().cpu().numpy(), yr, tol, "split y", STORAGE_U[y.dtype])
    assert_close(f2.cpu().numpy(), fr, tol, "split final state")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunk_size_invariance(dtype):
    inp = make_inputs(1, 1000, 4, 64, 64, 1, dtype, seed=10, with_init=True)
    c = to_cuda(inp)
    yr, fr = oracle.recurrence(**inp)
    tol = TOL[inp["x"].dtype]
    for Q in (64, 128, 256):
        y, f = run_gpu(c, Q)
        assert_close(y.float().cpu().numpy(), yr, tol, f"y chunk {Q}", STORAGE_U[y.dtype])
        assert_close(f.cpu().numpy(), fr, tol, f"final chunk {Q}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_groups_match_replicated_heads(dtype):
    inp = make_inputs(2, 400, 8, 64, 64, 2, dtype, seed=11, with_init=True)
    c = to_cuda(inp)
    y, f = run_gpu(c, 128)
    rep = dict(c)
    rep["B"] = c["B"].repeat_interleave(4, dim=2).contiguous()
    rep["C"] = c["C"].repeat_interleave(4, dim=2).contiguous()
    yr, fr = run_gpu(rep, 128)
    tol = TOL[inp["x"].dtype]
    assert_close(y.float().cpu().numpy(), yr.float().cpu().numpy(), tol, "grouped vs replicated",
                 2 * STORAGE_U[y.dtype])
    assert_close(f.cpu().numpy(), fr.cpu().numpy(), tol, "grouped vs replicated final")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_causality_and_determinism(dtype):
    inp = make_inputs(1, 500, 4, 64, 64, 1, dtype, seed=12)
    c = to_cuda(inp)
    y1, f1 = run_gpu(c, 128)
    y2, f2 = run_gpu(c, 128)
    assert torch.equal(y1, y2) and torch.equal(f1, f2), "two identical calls differ"
    t = 301
    c2 = dict(c)
    c2["x"] = c["x"].clone()
    c2["x"][:, t] += 1.0
    y3, _ = run_gpu(c2, 128)
    assert torch.equal(y3[:, :t], y1[:, :t]), "a later input changed an earlier output"
    assert not torch.equal(y3[:, t:], y1[:, t:])


def test_linearity_in_x_f32():
    inp = make_inputs(1, 300, 4, 32, 32, 1, "f32", seed=13, with_D=True)
    c = to_cuda(inp)
    y1, _ = run_gpu(c, 64)
    c2 = dict(c)
    c2["x"] = c["x"] * 2.0
    y2, _ = run_gpu(c2, 64)
    assert_close(y2.cpu().numpy(), 2.0 * y1.cpu().numpy(), 1e-5, "y(2x) vs 2y(x)")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_host_buffer_entry_matches_device_entry(dtype):
    inp = make_inputs(2, 300, 4, 64, 64, 1, dtype, seed=14, with_init=True)
    yd, fd = run_gpu(to_cuda(inp), 128)
    pinned = {k: (None if v is None else v.pin_memory()) for k, v in inp.items()}
    yh, fh = ssd.ssd_fwd_host(pinned["x"], pinned["dt"], pinned["A"], pinned["B"], pinned["C"], pinned["D"],
                              pinned["init_state"], chunk=128)
    # The host entry runs the problem in parts (token ranges with the state
    # carried between them), so its fp32 states round differently from one
    # call's; y may differ by one unit of its own rounding where that moves a
    # value across a rounding boundary.
    tol = TOL[yd.dtype] / 100
    assert_close(yh.float().numpy(), yd.float().cpu().numpy(), tol, "y, host vs device entry", 2 * STORAGE_U[yd.dtype])
    assert_close(fh.numpy(), fd.cpu().numpy(), tol, "final state, host vs device entry")
    yr, fr = oracle.recurrence(**inp)
    assert_close(yh.float().numpy(), yr, TOL[yd.dtype], "y, host entry vs oracle", STORAGE_U[yd.dtype])
    assert_close(fh.numpy(), fr, TOL[yd.dtype], "final state, host entry vs oracle")


# The largest sizes the library accepts: headdim, dstate and chunk at 256 together
# (fp32 kernels for headdim 256, the three-kernel tensor-core path at headdim 128),
# and many heads and batch elements (grid dimensions).
MAX_CASES = [(1, 600, 2, 256, 256, 1, 256, "bf16", "simt"), (1, 520, 2, 256, 256, 2, 256, "f32", "simt"),
             (1, 700, 4, 128, 256, 2, 256, "bf16", "tcgen05"), (2, 130, 1024, 16, 16, 8, 64, "f32", "simt"),
             (300, 40, 2, 64, 64, 1, 32, "bf16", "tcgen05_fused")]


@pytest.mark.parametrize("case", MAX_CASES, ids=[f"b{c[0]}L{c[1]}H{c[2]}P{c[3]}N{c[4]}Q{c[6]}{c[7]}" for c in MAX_CASES])
def test_maximum_sizes(case):
    b, L, H, P, N, G, Q, dtype, path = case
    assert ssd.ssd_fwd_path(b, L, H, P, G, N, Q, torch.float32 if dtype == "f32" else torch.bfloat16) == path
    inp = make_inputs(b, L, H, P, N, G, dtype, seed=17 + P + H, with_init=True)
    check_full(inp, Q)


# The host entry overlaps copies and compute over parts: batch groups (batch >= 4)
# or whole-chunk token ranges with the state carried between them (batch < 4);
# shapes whose token rows are not 16-byte multiples run as one part.
HOST_CASES = [(1, 700, 4, 64, 64, 1, 128, "bf16"), (5, 300, 4, 64, 64, 2, 128, "bf16"),
              (3, 450, 2, 128, 128, 1, 64, "bf16"), (1, 500, 4, 16, 6, 1, 64, "f32"),
              (2, 900, 4, 64, 256, 1, 256, "bf16")]


@pytest.mark.parametrize("case", HOST_CASES, ids=[f"b{c[0]}L{c[1]}N{c[4]}Q{c[6]}{c[7]}" for c in HOST_CASES])
def test_host_entry_parts_match_device_entry(case):
    b, L, H, P, N, G, Q, dtype = case
    inp = make_inputs(b, L, H, P, N, G, dtype, seed=15 + b, with_init=True)
    yd, fd = run_gpu(to_cuda(inp), Q)
    pinned = {k: (None if v is None else v.pin_memory()) for k, v in inp.items()}
    yh, fh = ssd.ssd_fwd_host(pinned["x"], pinned["dt"], pinned["A"], pinned["B"], pinned["C"], pinned["D"],
                              pinned["init_state"], chunk=Q)
    el = inp["x"].dtype
    assert_close(yh.float().numpy(), yd.float().cpu().numpy(), TOL[el] / 4, "y, host vs device entry", STORAGE_U[el])
    assert_close(fh.numpy(), fd.cpu().numpy(), TOL[el] / 4, "final state, host vs device entry")
    yr, fr = oracle.recurrence(**inp)
    assert_close(yh.float().numpy(), yr, TOL[el], "y, host entry vs oracle", STORAGE_U[el])
    assert_close(fh.numpy(), fr, TOL[el], "final state, host entry vs oracle")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_caller_workspace_matches(dtype):
    inp = make_inputs(2, 300, 4, 64, 64, 1, dtype, seed=15, with_init=True)
    c = to_cuda(inp)
    y, f = run_gpu(c, 128)
    n = ssd.ssd_fwd_workspace_size(2, 300, 4, 64, 1, 64, 128, c["x"].dtype)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    yw, fw = ssd.ssd_fwd_ws(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init_state"], chunk=128,
                            workspace=ws)
    ssd.ssd_check_device_status()
    assert torch.equal(y, yw) and torch.equal(f, fw)


def test_raw_c_abi_call_with_status_checks():
    # ssd_fwd through plain ctypes pointers (no binding wrapper): the status of every
    # call is checked on the host, then the result against the oracle
    import ctypes
    lib = ctypes.CDLL(ssd.LIB_PATH)
    b, L, H, P, N, G, Q = 2, 300, 4, 64, 64, 2, 128
    inp = make_inputs(b, L, H, P, N, G, "bf16", seed=18, with_init=True)
    c = to_cuda(inp)
    y = torch.empty_like(c["x"])
    fin = torch.empty(b, H, P, N, dtype=torch.float32, device="cuda")
    vp = lambda t: ctypes.c_void_p(t.data_ptr())
    lib.ssd_fwd.restype = ctypes.c_int
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = [vp(c["x"]), vp(c["dt"]), vp(c["A"]), vp(c["B"]), vp(c["C"]), vp(c["D"]), vp(c["init_state"]), vp(y),
            vp(fin)]
    st = lib.ssd_fwd(*args, b, L, H, P, G, N, Q, ssd.SSD_DTYPE_BF16, stream)
    assert st == ssd.SSD_OK, ssd.ssd_last_error_detail()
    lib.ssd_check_device_status.restype = ctypes.c_int
    assert lib.ssd_check_device_status(stream) == ssd.SSD_OK
    # a rejected call enqueues nothing and leaves the outputs alone
    y2 = y.clone()
    assert lib.ssd_fwd(*args, b, L, H, P, 3, N, Q, ssd.SSD_DTYPE_BF16, stream) == ssd.SSD_ERR_INVALID_ARG
    assert lib.ssd_check_device_status(stream) == ssd.SSD_OK and torch.equal(y, y2)
    yr, fr = oracle.recurrence(**inp)
    assert_close(y.float().cpu().numpy(), yr, TOL[torch.bfloat16], "y", STORAGE_U[torch.bfloat16])
    assert_close(fin.cpu().numpy(), fr, TOL[torch.bfloat16], "final state")


def test_runs_on_a_side_stream():
    inp = make_inputs(1, 400, 4, 64, 64, 1, "bf16", seed=16, with_init=True)
    c = to_cuda(inp)
    y0, f0 = run_gpu(c, 128)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y1, f1 = ssd.ssd_fwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init_state"], chunk=128,
                             stream=s)
    ssd.ssd_check_device_status(s)
    assert torch.equal(y0, y1) and torch.equal(f0, f1)


@pytest.mark.parametrize("case", [(1, 300, 4, 64, 64, 1, 128), (2, 256, 2, 128, 64, 1, 128), (1, 200, 2, 64, 128, 1, 64)],
                         ids=["P64N64", "P128N64", "P64N128Q64"])
def test_extreme_in_chunk_decay(case):
    """dt up to 2 with |A| up to 16: the decay inside one chunk spans far more
    than the factored (rank-one) path allows; those chunks are finished by the
    direct fp32 evaluation."""
    b, L, H, P, N, G, Q = case
    inp = make_inputs(b, L, H, P, N, G, "bf16", seed=77, dt_range=(0.5, 2.0), with_init=True)
    check_full(inp, Q)


def test_mixed_fast_and_queued_chunks():
    inp = make_inputs(1, 512, 8, 64, 64, 1, "bf16", seed=78, with_init=True)
    inp["dt"][:, :, 4:] *= 20.0  # head blocks 2 and 3: spans beyond the factored path in every chunk
    check_full(inp, 128)


# Wide in-chunk decay on each fused kernel: (b, L, H, P, N, G, Q, kernel).  Every
# chunk's cs range is far beyond the factored form's, so every unit takes the
# masked decayed matrix on the tensor cores.
WIDE = [
    (1, 700, 80, 64, 64, 1, 128, "ssd_fused_pipe_tc"),    # 40 sequences: the look-back kernel, ragged tail
    (2, 600, 36, 128, 64, 2, 128, "ssd_fused_pipe_tc"),   # one head per unit
    (1, 700, 66, 64, 64, 3, 96, "ssd_fused_pipe_tc"),     # chunk 96 (rows stored one by one), dt without TMA
    (2, 513, 8, 128, 128, 2, 128, "ssd_fused_tc"),        # dstate 128, one head per unit
    (1, 300, 4, 64, 128, 1, 128, "ssd_fused_tc"),         # dstate 128, two heads per unit
    (3, 700, 4, 128, 128, 2, 100, "ssd_fused_tc"),        # chunk 100
    (1, 3000, 16, 64, 64, 1, 128, "ssd_seq_pipe_tc"),     # 8 sequences: the sequence-pipelined kernel
    (2, 1500, 8, 128, 64, 2, 128, "ssd_seq_pipe_tc"),
]


@pytest.mark.parametrize("case", WIDE, ids=[f"{c[7]}_b{c[0]}L{c[1]}H{c[2]}P{c[3]}N{c[4]}Q{c[6]}" for c in WIDE])
def test_wide_decay_on_each_fused_kernel(case):
    b, L, H, P, N, G, Q, kern = case
    assert ssd.ssd_fwd_kernels(b, L, H, P, G, N, Q, ssd.SSD_DTYPE_BF16) == [kern]
    inp = make_inputs(b, L, H, P, N, G, "bf16", seed=79 + L, dt_range=(0.5, 2.0), with_init=True)
    ey, ef = check_full(inp, Q)
    print(f"{kern} wide: y error {ey:.2e} x RMS, final state {ef:.2e} x RMS")


@pytest.mark.parametrize("dims,Q", [((1, 700, 4, 64, 256, 1), 256), ((2, 600, 4, 128, 256, 2), 256),
                                    ((1, 520, 6, 64, 256, 3), 128)],
                         ids=["P64Q256", "P128Q256", "P64Q128"])
@pytest.mark.parametrize("mix", ["wide", "mixed"])
def test_wide_decay_on_the_three_kernel_path(dims, Q, mix):
    """dstate 256 (the three-kernel tcgen05 path): chunks whose in-chunk decay range
    is beyond the rank-one form of chunk_out_tc take the exp per element; with
    "mixed", only half the heads (and so some head blocks) do."""
    b, L, H, P, N, G = dims
    assert ssd.ssd_fwd_path(b, L, H, P, G, N, Q, ssd.SSD_DTYPE_BF16) == "tcgen05"
    if mix == "wide":
        inp = make_inputs(b, L, H, P, N, G, "bf16", seed=81 + L, dt_range=(0.5, 2.0), with_init=True)
    else:
        inp = make_inputs(b, L, H, P, N, G, "bf16", seed=82 + L, with_init=True)
        inp["dt"][:, :, H // 2:] *= 40.0
    ey, ef = check_full(inp, Q)
    print(f"three-kernel {mix}: y error {ey:.2e} x RMS, final state {ef:.2e} x RMS")


@pytest.mark.parametrize("kern,dims", [("ssd_fused_pipe_tc", (2, 512, 40, 64, 64, 1)),
                                       ("ssd_fused_tc", (2, 512, 8, 64, 128, 2)),
                                       ("ssd_seq_pipe_tc", (1, 3000, 16, 64, 64, 1))])
def test_wide_and_factored_units_interleaved(kern, dims):
    """Half the heads with steps ~20x larger: wide and factored units share the
    CTAs, the look-back chain and (in the persistent kernels) the two TMEM slots."""
    b, L, H, P, N, G = dims
    assert ssd.ssd_fwd_kernels(b, L, H, P, G, N, 128, ssd.SSD_DTYPE_BF16) == [kern]
    inp = make_inputs(b, L, H, P, N, G, "bf16", seed=80 + H, with_init=True)
    inp["dt"][:, :, H // 2:] *= 20.0
    inp["dt"][:, 300:, :4] *= 20.0  # and the first head block turns wide after token 300
    ey, ef = check_full(inp, 128)
    print(f"{kern} mixed: y error {ey:.2e} x RMS, final state {ef:.2e} x RMS")
