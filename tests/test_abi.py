"""The C-ABI library loads, exports every declared symbol and rejects bad
arguments before touching the GPU (runs without a GPU)."""
import ctypes
import glob
import os
import re

import pytest

import structured_state_space_03_b300 as ssd
from structured_state_space_03_b300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(hdr).read()
        names |= set(re.findall(r"^SSD_API\s+[^;(]*?\b(\w+)\s*\(", text, flags=re.M))
    return names


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ssd.lib()


def test_header_declares_the_binding_surface():
    names = declared_symbols()
    assert "ssd_fwd" in names and "ssd_fwd_ws" in names
    assert names == set(ssd.SIGNATURES), names ^ set(ssd.SIGNATURES)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    # nothing internal leaks out of the library
    raw = ctypes.CDLL(ssd.LIB_PATH)
    with pytest.raises(AttributeError):
        raw.launch_state_pass  # noqa: B018


def test_version_and_status_strings(lib):
    assert "sm_103a" in ssd.ssd_version()
    for st in range(6):
        assert ssd.ssd_status_string(st).startswith("SSD_")
    assert "unknown" in ssd.ssd_status_string(99)


DIMS = dict(batch=2, seqlen=300, nheads=8, headdim=64, ngroups=2, dstate=64, chunk=128)


def _fwd(lib, x=1, dt=1, A=1, B=1, C=1, y=1, **over):
    d = dict(DIMS, dtype=ssd.SSD_DTYPE_BF16)
    d.update(over)
    p = lambda v: ctypes.c_void_p(v * 4096) if v else None
    return lib.ssd_fwd(p(x), p(dt), p(A), p(B), p(C), None, None, p(y), None, d["batch"], d["seqlen"],
                       d["nheads"], d["headdim"], d["ngroups"], d["dstate"], d["chunk"], d["dtype"], None)


@pytest.mark.parametrize("missing", ["x", "dt", "A", "B", "C", "y"])
def test_null_required_pointer_is_invalid(lib, missing):
    assert _fwd(lib, **{missing: 0}) == ssd.SSD_ERR_INVALID_ARG
    assert missing in ssd.ssd_last_error_detail()


@pytest.mark.parametrize("field", ["batch", "seqlen", "nheads", "headdim", "ngroups", "dstate", "chunk"])
@pytest.mark.parametrize("value", [0, -3])
def test_nonpositive_dimension_is_invalid(lib, field, value):
    assert _fwd(lib, **{field: value}) == ssd.SSD_ERR_INVALID_ARG


def test_group_divisibility_and_dtype(lib):
    assert _fwd(lib, ngroups=3) == ssd.SSD_ERR_INVALID_ARG
    assert _fwd(lib, dtype=7) == ssd.SSD_ERR_INVALID_ARG


def test_misaligned_bf16_pointer_is_invalid(lib):
    d = dict(DIMS)
    st = lib.ssd_fwd(ctypes.c_void_p(4096 + 2), ctypes.c_void_p(4096), ctypes.c_void_p(4096),
                     ctypes.c_void_p(4096), ctypes.c_void_p(4096), None, None, ctypes.c_void_p(8192), None,
                     *[d[k] for k in ("batch", "seqlen", "nheads", "headdim", "ngroups", "dstate", "chunk")],
                     ssd.SSD_DTYPE_BF16, None)
    assert st == ssd.SSD_ERR_INVALID_ARG and "aligned" in ssd.ssd_last_error_detail()


@pytest.mark.parametrize("field,value", [("chunk", 512), ("headdim", 512), ("dstate", 300)])
def test_outside_build_is_unsupported(lib, field, value):
    assert _fwd(lib, **{field: value}) == ssd.SSD_ERR_UNSUPPORTED


def test_workspace_size_and_checks(lib):
    nc = -(-DIMS["seqlen"] // DIMS["chunk"])
    units = DIMS["batch"] * DIMS["nheads"] * nc
    states = units * DIMS["headdim"] * DIMS["dstate"] * 4
    # multi-kernel paths: one fp32 state per (batch, head, chunk) plus the chunk decays
    got = ssd.ssd_fwd_workspace_size(*DIMS.values(), ssd.SSD_DTYPE_F32)
    assert states <= got <= states + units * 4 + 512
    # fused path: published aggregate and inclusive states, decays and flags
    assert ssd.ssd_fwd_path(*DIMS.values(), ssd.SSD_DTYPE_BF16) == "tcgen05_fused"
    got = ssd.ssd_fwd_workspace_size(*DIMS.values(), ssd.SSD_DTYPE_BF16)
    assert 2 * states <= got <= 2 * states + units * 8 + 1024
    out = ctypes.c_size_t(0)
    assert lib.ssd_fwd_workspace_size(0, 1, 1, 1, 1, 1, 1, 1, ctypes.byref(out)) == ssd.SSD_ERR_INVALID_ARG
    assert lib.ssd_fwd_workspace_size(1, 1, 1, 1, 1, 1, 1, 1, None) == ssd.SSD_ERR_INVALID_ARG


def test_too_small_workspace_is_invalid(lib):
    d = dict(DIMS)
    need = ssd.ssd_fwd_workspace_size(*d.values(), ssd.SSD_DTYPE_BF16)
    p = ctypes.c_void_p(1 << 20)
    st = lib.ssd_fwd_ws(p, p, p, p, p, None, None, ctypes.c_void_p(2 << 20), None,
                        *d.values(), ssd.SSD_DTYPE_BF16, ctypes.c_void_p(3 << 20), need - 1, None)
    assert st == ssd.SSD_ERR_INVALID_ARG and "too small" in ssd.ssd_last_error_detail()
    st = lib.ssd_fwd_ws(p, p, p, p, p, None, None, ctypes.c_void_p(2 << 20), None,
                        *d.values(), ssd.SSD_DTYPE_BF16, ctypes.c_void_p((3 << 20) + 16), need, None)
    assert st == ssd.SSD_ERR_INVALID_ARG and "aligned" in ssd.ssd_last_error_detail()


def test_path_selection_is_a_pure_host_query(lib):
    assert ssd.ssd_fwd_path(1, 256, 4, 16, 1, 16, 64, ssd.SSD_DTYPE_F32) == "simt"
    assert ssd.ssd_fwd_path(1, 256, 4, 16, 1, 16, 999, ssd.SSD_DTYPE_F32) == "none"
    assert ssd.ssd_fwd_path(1, 256, 4, 16, 3, 16, 64, ssd.SSD_DTYPE_F32) == "none"
    # bf16 with headdim 64/128 and dstate 64/128: one fused tcgen05 kernel (a chunk longer
    # than 128 evaluated as equal blocks of at most 128); dstate 256: the three-kernel path
    assert ssd.ssd_fwd_path(2, 2048, 80, 64, 1, 64, 128, ssd.SSD_DTYPE_BF16) == "tcgen05_fused"
    assert ssd.ssd_fwd_path(16, 4096, 32, 128, 8, 128, 128, ssd.SSD_DTYPE_BF16) == "tcgen05_fused"
    assert ssd.ssd_fwd_path(1, 8192, 80, 64, 1, 128, 256, ssd.SSD_DTYPE_BF16) == "tcgen05"
    assert ssd.ssd_fwd_path(1, 8192, 80, 64, 1, 128, 128, ssd.SSD_DTYPE_BF16) == "tcgen05_fused"
    assert ssd.ssd_fwd_path(1, 131072, 24, 64, 1, 256, 256, ssd.SSD_DTYPE_BF16) == "tcgen05"
    assert ssd.ssd_fwd_path(1, 1000, 4, 64, 1, 256, 128, ssd.SSD_DTYPE_BF16) == "tcgen05"
    assert ssd.ssd_fwd_path(2, 333, 6, 32, 3, 48, 100, ssd.SSD_DTYPE_BF16) == "simt"
    assert ssd.ssd_fwd_path(2, 2048, 80, 64, 1, 64, 128, ssd.SSD_DTYPE_F32) == "simt"
    assert ssd.ssd_fwd_kernels(2, 2048, 80, 64, 1, 64, 128, ssd.SSD_DTYPE_BF16) == ["ssd_fused_pipe_tc"]
    assert ssd.ssd_fwd_kernels(1, 65536, 8, 64, 1, 64, 128, ssd.SSD_DTYPE_BF16) == ["ssd_seq_pipe_tc"]
    assert ssd.ssd_fwd_kernels(16, 4096, 32, 128, 8, 128, 128, ssd.SSD_DTYPE_BF16) == ["ssd_fused_tc"]
    assert ssd.ssd_fwd_kernels(1, 8192, 80, 64, 1, 128, 256, ssd.SSD_DTYPE_BF16) == [
        "chunk_state_tc", "state_pass_hilo", "chunk_out_tc"]
    assert ssd.ssd_fwd_kernels(1, 131072, 24, 64, 1, 256, 256, ssd.SSD_DTYPE_BF16) == [
        "chunk_state_tc", "state_pass_hilo", "chunk_out_tc"]


def test_block_length_of_long_chunks(lib):
    # the evaluated chunk length: at most 128 on the fused paths, the requested one elsewhere;
    # blocks of a longer chunk at dstate 64 (dstate 128 keeps it on the three-kernel path)
    B = ssd.SSD_DTYPE_BF16
    assert ssd.ssd_fwd_block(1, 8192, 80, 64, 1, 128, 256, B) == 256    # dstate 128: three-kernel path
    assert ssd.ssd_fwd_block(2, 2048, 80, 64, 1, 64, 200, B) == 100
    assert ssd.ssd_fwd_block(2, 2048, 80, 64, 1, 64, 129, B) == 65
    assert ssd.ssd_fwd_block(2, 2048, 80, 64, 1, 64, 96, B) == 96
    assert ssd.ssd_fwd_block(1, 131072, 24, 64, 1, 256, 256, B) == 256   # dstate 256: three-kernel path
    assert ssd.ssd_fwd_block(1, 1000, 4, 32, 1, 64, 256, B) == 256       # headdim 32: SIMT path
    assert ssd.ssd_fwd_block(1, 1000, 4, 64, 1, 64, 256, ssd.SSD_DTYPE_F32) == 256
    assert ssd.ssd_fwd_block(1, 1000, 4, 64, 1, 64, 999, B) == -1
    # the workspace follows the evaluated length
    n256, n128 = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.ssd_fwd_workspace_size(2, 2048, 80, 64, 1, 64, 256, B, ctypes.byref(n256)) == ssd.SSD_OK
    assert lib.ssd_fwd_workspace_size(2, 2048, 80, 64, 1, 64, 128, B, ctypes.byref(n128)) == ssd.SSD_OK
    assert n256.value == n128.value


def _step(lib, x=1, dt=1, A=1, B=1, C=1, state=1, y=1, **over):
    d = dict(batch=2, nheads=8, headdim=64, ngroups=2, dstate=64, dtype=ssd.SSD_DTYPE_BF16)
    d.update(over)
    p = lambda v: ctypes.c_void_p(v * 4096) if v else None
    return lib.ssd_step(p(x), p(dt), p(A), p(B), p(C), None, p(state), p(y), d["batch"], d["nheads"], d["headdim"],
                        d["ngroups"], d["dstate"], d["dtype"], None)


@pytest.mark.parametrize("missing", ["x", "dt", "A", "B", "C", "state", "y"])
def test_step_null_pointer_is_invalid(lib, missing):
    assert _step(lib, **{missing: 0}) == ssd.SSD_ERR_INVALID_ARG
    assert "non-NULL" in ssd.ssd_last_error_detail()


@pytest.mark.parametrize("field", ["batch", "nheads", "headdim", "ngroups", "dstate"])
def test_step_nonpositive_dimension_is_invalid(lib, field):
    assert _step(lib, **{field: 0}) == ssd.SSD_ERR_INVALID_ARG


def test_step_groups_dtype_and_alignment(lib):
    assert _step(lib, ngroups=3) == ssd.SSD_ERR_INVALID_ARG
    assert _step(lib, dtype=9) == ssd.SSD_ERR_INVALID_ARG
    st = lib.ssd_step(ctypes.c_void_p(4097), ctypes.c_void_p(4096), ctypes.c_void_p(4096), ctypes.c_void_p(4096),
                      ctypes.c_void_p(4096), None, ctypes.c_void_p(4096), ctypes.c_void_p(8192), 1, 2, 4, 1, 8,
                      ssd.SSD_DTYPE_BF16, None)
    assert st == ssd.SSD_ERR_INVALID_ARG and "aligned" in ssd.ssd_last_error_detail()


def test_pre_flags_and_bias_alignment(lib):
    d = dict(DIMS)
    p = ctypes.c_void_p(4096)
    args = lambda flags, bias: (p, p, bias, flags, p, p, p, None, None, ctypes.c_void_p(8192), None,
                                *[d[k] for k in ("batch", "seqlen", "nheads", "headdim", "ngroups", "dstate", "chunk")],
                                ssd.SSD_DTYPE_BF16, None)
    assert lib.ssd_fwd_pre(*args(4, None)) == ssd.SSD_ERR_INVALID_ARG
    assert "pre_flags" in ssd.ssd_last_error_detail()
    assert lib.ssd_fwd_pre(*args(ssd.SSD_PRE_ZOH, ctypes.c_void_p(4098))) == ssd.SSD_ERR_INVALID_ARG
    assert "dt_bias" in ssd.ssd_last_error_detail()
    # the shared checks of ssd_fwd still apply
    d["ngroups"] = 3
    assert lib.ssd_fwd_pre(*args(0, None)) == ssd.SSD_ERR_INVALID_ARG


def _varlen(lib, cu, nseq=None, dstate=64, dtype=ssd.SSD_DTYPE_BF16, headdim=64):
    p = ctypes.c_void_p(1 << 20)
    offs = None if cu is None else (ctypes.c_int * len(cu))(*cu)
    n = (len(cu) - 1) if nseq is None else nseq
    return lib.ssd_fwd_varlen(p, p, p, p, p, None, offs, n, None, ctypes.c_void_p(2 << 20), None,
                              8, headdim, 2, dstate, 128, dtype, None)


def test_varlen_offsets_are_checked_before_any_launch(lib):
    assert _varlen(lib, None, nseq=2) == ssd.SSD_ERR_INVALID_ARG
    assert _varlen(lib, [0, 5], nseq=0) == ssd.SSD_ERR_INVALID_ARG
    assert _varlen(lib, [1, 5]) == ssd.SSD_ERR_INVALID_ARG
    assert "cu_seqlens[0]" in ssd.ssd_last_error_detail()
    assert _varlen(lib, [0, 5, 4]) == ssd.SSD_ERR_INVALID_ARG
    assert "decreases" in ssd.ssd_last_error_detail()


def test_varlen_rejects_what_the_forward_rejects(lib):
    # every kernel family takes packed sequences; sizes outside the build are refused up front
    assert _varlen(lib, [0, 5, 9], dstate=300) == ssd.SSD_ERR_UNSUPPORTED
    assert _varlen(lib, [0, 5, 9], headdim=512) == ssd.SSD_ERR_UNSUPPORTED
    assert _varlen(lib, [0, 5, 9], dtype=9) == ssd.SSD_ERR_INVALID_ARG


def test_fault_hook_argument_checks(lib):
    assert lib.ssd_test_set_fault(0, -2) == ssd.SSD_ERR_INVALID_ARG
    assert lib.ssd_test_set_fault(1000, 3) == ssd.SSD_OK
    assert lib.ssd_test_set_fault(0, -1) == ssd.SSD_OK


def _bwd(lib, headdim=64, dstate=64, ngroups=2, dtype=None, **ptrs):
    names = ("x", "dt", "A", "B", "C", "D", "init", "dy", "dfinal", "dx", "ddt", "dA", "dB", "dC", "dD", "dinit")
    required = {"x", "dt", "A", "B", "C", "dy", "dx", "ddt", "dA", "dB", "dC"}
    vals = {n: (ptrs.get(n, 1 if n in required else 0)) for n in names}
    p = lambda v: ctypes.c_void_p(v * 4096) if v else None
    return lib.ssd_bwd(*[p(vals[n]) for n in names], 2, 300, 8, headdim, ngroups, dstate,
                       ssd.SSD_DTYPE_BF16 if dtype is None else dtype, None)


@pytest.mark.parametrize("missing", ["x", "dt", "A", "B", "C", "dy", "dx", "ddt", "dA", "dB", "dC"])
def test_backward_null_required_pointer_is_invalid(lib, missing):
    assert _bwd(lib, **{missing: 0}) == ssd.SSD_ERR_INVALID_ARG
    assert missing in ssd.ssd_last_error_detail()


def test_backward_size_and_type_checks(lib):
    assert _bwd(lib, headdim=256) == ssd.SSD_ERR_UNSUPPORTED
    assert _bwd(lib, dstate=300) == ssd.SSD_ERR_UNSUPPORTED
    assert _bwd(lib, ngroups=3) == ssd.SSD_ERR_INVALID_ARG
    assert _bwd(lib, dtype=5) == ssd.SSD_ERR_INVALID_ARG
    st = lib.ssd_bwd(*[ctypes.c_void_p(4096 + 1)] + [ctypes.c_void_p(4096)] * 15, 2, 300, 8, 64, 2, 64,
                     ssd.SSD_DTYPE_BF16, None)
    assert st == ssd.SSD_ERR_INVALID_ARG and "aligned" in ssd.ssd_last_error_detail()


def test_backward_kernel_list_and_workspace(lib):
    assert ssd.ssd_bwd_kernels(2, 300, 8, 64, 2, 128, ssd.SSD_DTYPE_BF16) == [
        "bwd_chunk_states", "bwd_state_pass", "bwd_chunk", "bwd_reduce_groups", "bwd_reduce_heads"]
    # one head per group: dB and dC are written directly, no reduction over heads
    assert ssd.ssd_bwd_kernels(2, 300, 8, 64, 8, 128, ssd.SSD_DTYPE_BF16) == [
        "bwd_chunk_states", "bwd_state_pass", "bwd_chunk", "bwd_reduce_heads"]
    nc = -(-300 // 64)
    states = 2 * (2 * 8 * nc * 64 * 128 * 4)
    parts = 2 * (2 * 300 * 8 * 128 * 4)
    grouped = ssd.ssd_bwd_workspace_size(2, 300, 8, 64, 2, 128, ssd.SSD_DTYPE_BF16)
    per_head = ssd.ssd_bwd_workspace_size(2, 300, 8, 64, 8, 128, ssd.SSD_DTYPE_BF16)
    assert states <= per_head <= states + 4096
    assert grouped - per_head >= parts
