"""Packed variable-length sequences (ssd_fwd_varlen) against the oracle.

Each packed sequence is its own recurrence ("Mamba-2架构深度解析" §5, dynamic
sequence packing; the reading is pinned in test_oracle_varlen.py).  The cases
mix sequences shorter than one chunk, exactly one chunk, one token, empty
ones and long ones, so that chunks end inside the tile (rows of the next
sequence follow them in memory), every sequence restarts its state, and the
chunk-major unit order interleaves sequences of different lengths.
"""
import numpy as np
import pytest
import torch

import oracle
import structured_state_space_03_b300 as ssd
from structured_state_space_03_b300.workloads import make_varlen_inputs, varlen_lengths
from parity import STORAGE_U, TOL, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    ssd.lib()


def _cuda_inputs(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _run(d, chunk, **kw):
    c = _cuda_inputs(d)
    y, f = ssd.ssd_fwd_varlen(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init_state"],
                              cu_seqlens=d["cu_seqlens"], chunk=chunk, **kw)
    ssd.ssd_check_device_status()
    return y, f


def _check(d, chunk):
    y, f = _run(d, chunk)
    yr, fr = oracle.recurrence_varlen(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"],
                                      d["cu_seqlens"])
    el = d["x"].dtype
    assert_close(y.float().cpu().numpy(), yr, TOL[el], "y (packed)", STORAGE_U[el])
    assert_close(f.cpu().numpy(), fr, TOL[el], "final_state (packed)")


CASES = [
    # lengths, H, P, N, G, chunk
    ([700, 1, 128, 0, 255, 129, 64, 3], 8, 64, 64, 2, 128),
    ([300, 77, 0, 128, 1, 500], 4, 128, 64, 2, 100),
    ([17, 200, 33, 64, 65, 0, 0, 190], 6, 64, 64, 3, 64),
    ([400, 0, 1, 127, 129, 60], 4, 64, 128, 1, 128),    # dstate 128: the one-unit fused kernel
    ([250, 3, 128, 0, 77], 4, 128, 128, 2, 96),
]


@pytest.mark.parametrize("case", CASES, ids=[f"n{len(c[0])}H{c[1]}P{c[2]}Q{c[5]}" for c in CASES])
@pytest.mark.parametrize("with_init", [False, True])
def test_packed_sequences_match_oracle(case, with_init):
    lengths, H, P, N, G, Q = case
    d = make_varlen_inputs(lengths, H, P, N, G, "bf16", seed=sum(lengths) + Q, with_init=with_init)
    _check(d, Q)


# the multi-kernel paths, and long chunks: (lengths, H, P, N, G, chunk, dtype, path)
MULTI = [
    ([700, 1, 256, 0, 255, 257, 64, 3], 4, 64, 256, 1, 128, "bf16", "tcgen05"),   # dstate 256
    ([600, 0, 1, 256, 255, 300], 4, 64, 256, 1, 256, "bf16", "tcgen05"),          # chunk 256: two tiles per chunk
    ([600, 0, 1, 256, 255, 300], 4, 64, 128, 2, 256, "bf16", "tcgen05"),          # dstate 128 at chunk 256: three kernels
    ([300, 77, 0, 128, 1, 200], 4, 128, 64, 2, 256, "bf16", "tcgen05_fused"),     # headdim 128, chunk 256 as 2 x 128
    ([333, 17, 0, 64, 65, 1, 190], 6, 32, 48, 3, 100, "f32", "simt"),
    ([250, 3, 128, 0, 77], 4, 32, 64, 2, 64, "bf16", "simt"),                     # headdim 32: fp32 FMA path
]


@pytest.mark.parametrize("case", MULTI, ids=[f"{c[7]}_n{len(c[0])}P{c[2]}N{c[3]}Q{c[5]}{c[6]}" for c in MULTI])
@pytest.mark.parametrize("with_init", [False, True])
def test_packed_sequences_on_the_multi_kernel_paths(case, with_init):
    lengths, H, P, N, G, Q, dt, path = case
    el = torch.float32 if dt == "f32" else torch.bfloat16
    assert ssd.ssd_fwd_path(1, sum(lengths), H, P, G, N, Q, el) == path
    d = make_varlen_inputs(lengths, H, P, N, G, dt, seed=sum(lengths) + Q + 1, with_init=with_init)
    _check(d, Q)


def test_packed_multi_kernel_in_place_state_carry():
    # init_state == final_state on the three-kernel path: each sequence reads its own state before overwriting it
    lengths = [300, 0, 129, 5]
    d = make_varlen_inputs(lengths, 4, 64, 256, 1, "bf16", seed=41, with_init=True)
    yr, fr = oracle.recurrence_varlen(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"],
                                      d["cu_seqlens"])
    c = _cuda_inputs(d)
    st = c["init_state"].clone()
    y, f = ssd.ssd_fwd_varlen(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], st, cu_seqlens=d["cu_seqlens"],
                              chunk=128, final_state=st)
    ssd.ssd_check_device_status()
    assert f.data_ptr() == st.data_ptr()
    assert_close(y.float().cpu().numpy(), yr, TOL[torch.bfloat16], "y (packed, in place)", STORAGE_U[torch.bfloat16])
    assert_close(st.cpu().numpy(), fr, TOL[torch.bfloat16], "final_state (packed, in place)")


@pytest.mark.parametrize("N", [64, 128])
def test_packed_wide_decay(N):
    # steps of 0.5 .. 2 with |A| up to 16: every chunk is beyond the factored form's range
    lengths = [700, 1, 128, 0, 255, 129, 64, 3]
    d = make_varlen_inputs(lengths, 8, 64, N, 2, "bf16", seed=51 + N, dt_range=(0.5, 2.0), with_init=True)
    _check(d, 128)


def test_many_short_sequences():
    g = torch.Generator().manual_seed(11)
    lengths = [int(v) for v in torch.randint(0, 41, (300,), generator=g)]
    d = make_varlen_inputs(lengths, 4, 64, 64, 1, "bf16", seed=12, with_init=True)
    _check(d, 64)


def test_mixed_lengths_at_the_headline_shape():
    lengths = varlen_lengths(4096, 12, seed=5)
    d = make_varlen_inputs(lengths, 80, 64, 64, 1, "bf16", seed=13, with_init=False)
    rows = list(range(0, 80 * 64, 97))  # every 97th (h, p) row, compared over all tokens
    y, f = _run(d, 128)
    cu = d["cu_seqlens"]
    for s in range(len(lengths)):
        a, e = cu[s], cu[s + 1]
        xs = {k: d[k][a:e][None] for k in ("x", "dt", "B", "C")}
        yr, fr = oracle.recurrence(xs["x"], xs["dt"], d["A"], xs["B"], xs["C"], d["D"], None, rows=rows)
        yg = y[a:e].reshape(e - a, 80 * 64)[:, rows].T.float().cpu().numpy()
        assert_close(yg, yr, TOL[torch.bfloat16], f"y (sequence {s})", STORAGE_U[torch.bfloat16])
        assert_close(f[s].reshape(80 * 64, 64)[rows].cpu().numpy(), fr, TOL[torch.bfloat16], f"final (sequence {s})")


def test_equal_lengths_equal_the_batch_layout():
    b, L, H, P, N, G, Q = 3, 300, 4, 64, 64, 1, 128
    d = make_varlen_inputs([L] * b, H, P, N, G, "bf16", seed=21, with_init=True)
    y, f = _run(d, Q)
    c = _cuda_inputs(d)
    yb, fb = ssd.ssd_fwd(c["x"].reshape(b, L, H, P), c["dt"].reshape(b, L, H), c["A"], c["B"].reshape(b, L, G, N),
                         c["C"].reshape(b, L, G, N), c["D"], c["init_state"], chunk=Q)
    ssd.ssd_check_device_status()
    # the packed layout runs its own kernel instance (and, at dstate 64, another
    # kernel than the batch layout): the same values up to rounding, y within one
    # unit of its own bf16 rounding
    assert_close(y.reshape(b, L, H, P).float().cpu().numpy(), yb.float().cpu().numpy(), TOL[torch.bfloat16] / 100,
                 "y, packed vs batch layout", 2 * STORAGE_U[torch.bfloat16])
    assert_close(f.cpu().numpy(), fb.cpu().numpy(), TOL[torch.bfloat16] / 100, "final state, packed vs batch layout")


def test_state_carried_in_place_and_empty_sequences():
    d = make_varlen_inputs([0, 130, 0, 5], 4, 64, 64, 2, "bf16", seed=31, with_init=True)
    c = _cuda_inputs(d)
    st = c["init_state"].clone()
    y, f = ssd.ssd_fwd_varlen(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], st, cu_seqlens=d["cu_seqlens"],
                              chunk=128, final_state=st)
    ssd.ssd_check_device_status()
    assert f.data_ptr() == st.data_ptr()
    yr, fr = oracle.recurrence_varlen(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"],
                                      d["cu_seqlens"])
    assert_close(y.float().cpu().numpy(), yr, TOL[torch.bfloat16], "y (in place)", STORAGE_U[torch.bfloat16])
    assert_close(st.cpu().numpy(), fr, TOL[torch.bfloat16], "final (in place)")
    # only empty sequences: the final states are the initial states (or zero)
    e = make_varlen_inputs([0, 0], 4, 64, 64, 2, "bf16", seed=32, with_init=True)
    ce = _cuda_inputs(e)
    _, f2 = ssd.ssd_fwd_varlen(ce["x"], ce["dt"], ce["A"], ce["B"], ce["C"], ce["D"], ce["init_state"],
                               cu_seqlens=[0, 0, 0], chunk=128)
    torch.cuda.synchronize()
    assert torch.equal(f2, ce["init_state"])
    _, f3 = ssd.ssd_fwd_varlen(ce["x"], ce["dt"], ce["A"], ce["B"], ce["C"], ce["D"], None, cu_seqlens=[0, 0, 0],
                               chunk=128)
    torch.cuda.synchronize()
    assert torch.count_nonzero(f3) == 0


def test_sizes_outside_the_build_are_rejected():
    # every kernel family takes packed sequences; what ssd_fwd refuses, the packed entry refuses too
    d = _cuda_inputs(make_varlen_inputs([10, 20], 4, 64, 64, 1, "bf16", seed=41))
    with pytest.raises(ssd.SsdError) as err:
        ssd.ssd_fwd_varlen(d["x"], d["dt"], d["A"], d["B"], d["C"], cu_seqlens=[0, 10, 30], chunk=512)
    assert err.value.status == ssd.SSD_ERR_UNSUPPORTED
    d = _cuda_inputs(make_varlen_inputs([10, 20], 4, 64, 300, 1, "bf16", seed=42))
    with pytest.raises(ssd.SsdError) as err:
        ssd.ssd_fwd_varlen(d["x"], d["dt"], d["A"], d["B"], d["C"], cu_seqlens=[0, 10, 30], chunk=64)
    assert err.value.status == ssd.SSD_ERR_UNSUPPORTED
