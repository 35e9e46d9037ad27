"""The C ABI library builds, loads and exports every entry point that
include/ep.h declares; host-side argument checks reject bad calls before
anything reaches CUDA.  No test here launches a kernel (no GPU needed)."""
from __future__ import annotations

import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ep.h")

EP_ERR_INVALID_ARG = 1
EP_ERR_CAPACITY = 2


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ep_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def eplib():
    from combine_get_dispatch_04_gb300 import build
    build.build()
    import combine_get_dispatch_04_gb300 as ep
    return ep.load()


def test_header_declares_the_entry_points():
    import combine_get_dispatch_04_gb300 as ep
    assert declared_functions() == sorted(ep.EXPORTED)


def test_library_exports_every_declared_symbol(eplib):
    for name in declared_functions():
        assert hasattr(eplib, name), name


def test_status_strings(eplib):
    for code in range(5):
        s = eplib.ep_status_string(code).decode()
        assert s.startswith("EP_")
    assert eplib.ep_status_string(99).decode() == "unknown ep_status_t"


def test_workspace_bytes(eplib):
    wb = eplib.ep_workspace_bytes
    assert wb(0, 4, 16) == 0  # an empty batch needs no scratch
    assert wb(131072, 16, 64) >= 131072 * 8  # one 64-bit rank mask per token
    assert wb(512, 4, 16) <= wb(1024, 4, 16)
    assert wb(10, 4, 16) == 0   # T % R != 0
    assert wb(512, 3, 16) == 0  # E % R != 0
    assert wb(512, 65, 65) == 0  # R above the maximum
    assert wb(512, 4, 4100) == 0  # E above the maximum
    assert wb(-4, 4, 16) == 0


def _expected_workspace(T, R, E):
    """One 8-byte rank mask per token, then per 512-token block (blocks never
    straddle two source ranks) R counts, R offsets and E expert counts, each
    array padded to 256 bytes."""
    pad = lambda n: (n + 255) // 256 * 256  # noqa: E731
    nb = R * ((T // R + 511) // 512)
    return pad(8 * T) + 2 * pad(4 * R * nb) + pad(4 * nb * E)


@pytest.mark.parametrize("T,R,E", [(512, 4, 16), (4096, 32, 256), (131072, 16, 64),
                                   (1000, 1, 3), (4096, 64, 128)])
def test_workspace_bytes_exact(eplib, T, R, E):
    assert eplib.ep_workspace_bytes(T, R, E) == _expected_workspace(T, R, E)


def _layout_call(eplib, T=8, K=2, E=8, R=2, ptrs=True, ws_bytes=1 << 20):
    p = C.c_void_p(16) if ptrs else None  # never dereferenced: the checks fail first
    return eplib.ep_get_dispatch_layout(p, T, K, E, R, p, p, p, p, p, None, p, ws_bytes, None)


def _layout_path_call(eplib, path, T=8, K=2, E=8, R=2):
    p = C.c_void_p(16)  # never dereferenced: the checks fail first
    return eplib.ep_get_dispatch_layout_path(p, T, K, E, R, p, p, p, p, p, None, p, 1 << 20,
                                             path, None)


def test_layout_rejects_bad_arguments(eplib):
    assert _layout_call(eplib, E=7) == EP_ERR_INVALID_ARG        # E % R
    assert _layout_call(eplib, T=9) == EP_ERR_INVALID_ARG        # T % R
    assert _layout_call(eplib, K=0) == EP_ERR_INVALID_ARG
    assert _layout_call(eplib, K=33) == EP_ERR_INVALID_ARG       # above EP_MAX_TOPK
    assert _layout_call(eplib, R=65, E=65 * 2, T=130) == EP_ERR_INVALID_ARG
    assert _layout_call(eplib, ptrs=False) == EP_ERR_INVALID_ARG
    # workspace too small (a batch too large for the single-launch form, which needs none)
    assert not eplib.ep_layout_single_launch_fits(40000, 2, 8)
    assert _layout_call(eplib, T=40000, ws_bytes=8) == EP_ERR_CAPACITY


def test_single_launch_layout_limits(eplib):
    fits = eplib.ep_layout_single_launch_fits
    assert fits(4096, 32, 256) == 1       # decode: 32 ranks x 128 tokens, 256 experts
    assert fits(16384, 8, 256) == 1       # 8 CTAs x 8 chunks x 256 tokens
    assert fits(512, 4, 16) == 1
    assert fits(16386, 2, 8) == 0         # more tokens than one cluster holds
    assert fits(32768, 8, 256) == 0
    assert fits(131072, 16, 64) == 0
    assert fits(512, 64, 512) == 0        # R * E above the shared-memory histogram
    assert fits(0, 4, 16) == 0            # T = 0 takes the multi-launch form
    assert fits(10, 4, 16) == 0           # invalid sizes
    auto = eplib.ep_layout_auto_single_launch
    assert auto(4096, 32, 256) == 1 and auto(8192, 8, 256) == 1
    assert auto(16384, 8, 256) == 0       # fits, but the multi-launch form is faster there
    assert auto(512, 64, 512) == 0


def test_ll_single_launch_layout_limits(eplib):
    fits = eplib.ep_ll_layout_single_launch_fits
    auto = eplib.ep_ll_layout_auto_single_launch
    assert fits(4096, 8, 32, 256) == 1      # decode: 2 warps of 64 tokens per source at 8 CTAs
    assert fits(512, 4, 4, 16) == 1
    assert fits(8192, 16, 1, 16) == 1       # one source: 64 warps of 128 tokens x 16 slots
    assert fits(8192 + 1, 16, 1, 16) == 0   # a warp would walk more than 2048 slots
    assert fits(4096, 8, 32, 2048) == 0     # more experts than the per-warp counters hold
    assert fits(0, 8, 32, 256) == 0
    assert fits(10, 8, 4, 16) == 0          # invalid sizes
    assert auto(4096, 8, 32, 256) == 1
    assert fits(16384, 8, 8, 256) == 1      # 8 warps of 256 tokens per source at 8 CTAs
    assert auto(16384, 8, 8, 256) == 1      # the single launch wins wherever it fits
    assert auto(32768, 8, 8, 256) == 0
    assert fits(32768, 8, 8, 256) == 0      # 4096 slots per warp at 8 CTAs


def _ll_path_call(eplib, path, T=8, K=2, E=8, R=2, cap=8):
    p = C.c_void_p(16)  # never dereferenced: the checks fail first
    return eplib.ep_ll_get_dispatch_layout_path(p, T, K, E, R, cap, p, p, p, None, p, 1 << 20,
                                                path, None)


def test_ll_layout_path_rejects_bad_arguments(eplib):
    SINGLE = 2
    assert _ll_path_call(eplib, 3) == EP_ERR_INVALID_ARG
    assert _ll_path_call(eplib, SINGLE, T=0) == EP_ERR_INVALID_ARG
    assert _ll_path_call(eplib, SINGLE, E=2048, R=2) == EP_ERR_INVALID_ARG  # E above 1024
    assert _ll_path_call(eplib, SINGLE, cap=-1) == EP_ERR_INVALID_ARG
    assert _ll_path_call(eplib, 1, T=9) == EP_ERR_INVALID_ARG


def test_layout_path_rejects_bad_arguments(eplib):
    AUTO, MULTI, SINGLE = 0, 1, 2
    assert _layout_path_call(eplib, 3) == EP_ERR_INVALID_ARG     # unknown path
    assert _layout_path_call(eplib, -1) == EP_ERR_INVALID_ARG
    assert _layout_path_call(eplib, SINGLE, T=40000) == EP_ERR_INVALID_ARG  # does not fit
    assert _layout_path_call(eplib, SINGLE, T=0) == EP_ERR_INVALID_ARG
    assert _layout_path_call(eplib, MULTI, E=7) == EP_ERR_INVALID_ARG
    assert _layout_path_call(eplib, AUTO, T=9) == EP_ERR_INVALID_ARG


def test_dispatch_rejects_bad_arguments(eplib):
    p = C.c_void_p(16)
    base = dict(x=p, H=256, idx=p, w=p, T=8, K=2, E=8, R=2, slot=p, ntpe=None, cap=16,
                fp8=0, rx=p, rs=None)

    def call(**kw):
        a = dict(base, **kw)
        return eplib.ep_dispatch(a["x"], a["H"], a["idx"], a["w"], a["T"], a["K"], a["E"],
                                 a["R"], a["slot"], a["ntpe"], a["cap"], a["fp8"], a["rx"],
                                 a["rs"], None, None, None, None, None, None)
    assert call(H=12) == EP_ERR_INVALID_ARG                 # H % 8
    assert call(H=264, fp8=1, rs=p) == EP_ERR_INVALID_ARG   # FP8 needs H % 128
    assert call(fp8=1) == EP_ERR_INVALID_ARG                # FP8 needs scales
    assert call(cap=-1) == EP_ERR_INVALID_ARG
    assert call(x=C.c_void_p(24)) == EP_ERR_INVALID_ARG    # misaligned payload
    assert call(rx=None) == EP_ERR_INVALID_ARG
    assert call(E=7) == EP_ERR_INVALID_ARG                  # E % R


def test_combine_rejects_bad_arguments_and_accepts_empty(eplib):
    p = C.c_void_p(16)
    assert eplib.ep_combine(p, 12, p, p, 8, 2, 8, 2, p, p, None, None) == EP_ERR_INVALID_ARG
    assert eplib.ep_combine(p, 256, None, p, 8, 2, 8, 2, p, p, None, None) == EP_ERR_INVALID_ARG
    assert eplib.ep_combine(C.c_void_p(8), 256, p, p, 8, 2, 8, 2, p, p, None, None) == EP_ERR_INVALID_ARG
    # no tokens: nothing to do, nothing enqueued
    assert eplib.ep_combine(None, 256, None, None, 0, 2, 8, 2, None, None, None, None) == 0


def test_sched_combines_reject_bad_arguments_and_accept_empty(eplib):
    p = C.c_void_p(4096)
    ok_sched, bad_sched = C.c_void_p(8192), C.c_void_p(8196)  # the counters need 8-byte alignment
    f = eplib.ep_combine_sched
    assert f(p, 12, p, p, 8, 2, 8, 2, p, p, ok_sched, None, None) == EP_ERR_INVALID_ARG
    assert f(p, 256, None, p, 8, 2, 8, 2, p, p, ok_sched, None, None) == EP_ERR_INVALID_ARG
    assert f(p, 256, p, p, 8, 2, 8, 2, p, p, bad_sched, None, None) == EP_ERR_INVALID_ARG
    assert f(None, 256, None, None, 0, 2, 8, 2, None, None, bad_sched, None, None) == 0
    g = eplib.ep_ll_combine_sched
    assert g(p, 12, p, 8, 2, p, p, ok_sched, None, None) == EP_ERR_INVALID_ARG
    assert g(p, 256, p, 8, 2, None, p, ok_sched, None, None) == EP_ERR_INVALID_ARG
    assert g(p, 256, p, 8, 2, p, p, bad_sched, None, None) == EP_ERR_INVALID_ARG
    assert g(None, 256, None, 0, 2, None, None, None, None, None) == 0


def test_binding_fails_loudly_without_the_library(tmp_path):
    import combine_get_dispatch_04_gb300 as ep
    saved = ep._lib
    ep._lib = None
    try:
        with pytest.raises(ep.EPError):
            ep.load(str(tmp_path / "missing.so"))
    finally:
        ep._lib = saved


def test_error_word_description():
    import combine_get_dispatch_04_gb300 as ep
    assert ep.describe_error_word(0) == "no error"
    assert "expert id" in ep.describe_error_word(ep.EP_ERRBIT_BAD_EXPERT)
    both = ep.describe_error_word(ep.EP_ERRBIT_CAPACITY | ep.EP_ERRBIT_TIMEOUT)
    assert "capacity" in both and "wait" in both


def test_fused_fits_and_rejects_bad_arguments(eplib):
    fits = eplib.ep_layout_dispatch_fused_fits
    assert fits(4096, 32, 256) == 1          # the decode workload
    assert fits(512, 4, 16) == 1
    assert fits(16384, 8, 256) == 1           # 8 * 8 * 64 = 4096 ballots
    assert fits(16384 + 8, 8, 256) == 0       # above the token limit
    assert fits(0, 4, 16) == 0                # empty batches take the separate calls
    assert fits(8192, 32, 256) == 1           # 32 * 32 * 8 = 8192 ballots
    assert fits(8192 + 32 * 32, 32, 256) == 0  # 32 * 32 * 9 ballots
    assert fits(4096, 64, 128) == 1           # 64 * 64 * 2 ballots
    assert fits(10, 4, 16) == 0               # T % R
    f = eplib.ep_layout_dispatch_fused
    p = C.c_void_p(4096)  # never dereferenced: the checks fail first
    bad_sync = C.c_void_p(4100)

    def call(T=512, K=4, E=16, R=4, H=256, fp8=0, sync=p, ws_bytes=1 << 20):
        return f(p, H, p, p, T, K, E, R, p, p, p, p, p, T * 4, fp8, p, p, None, None, None, None,
                 p, ws_bytes, sync, None, None)

    assert call(T=16392, R=8, E=256) == EP_ERR_INVALID_ARG
    assert call(H=12) == EP_ERR_INVALID_ARG
    assert call(H=256 + 8, fp8=1) == EP_ERR_INVALID_ARG   # FP8 needs H % 128
    assert call(sync=None) == EP_ERR_INVALID_ARG
    assert call(sync=bad_sync) == EP_ERR_INVALID_ARG      # 8-byte alignment
    need = eplib.ep_layout_dispatch_fused_workspace_bytes(512, 4, 16)
    # ballots then offsets, R * R * ceil(T_r / 32) of each, the ballots padded to 256 bytes
    assert need == 256 + 4 * 4 * 4 * 4
    assert eplib.ep_layout_dispatch_fused_workspace_bytes(16392, 8, 256) == 0
    assert call(ws_bytes=need - 1) == EP_ERR_CAPACITY
