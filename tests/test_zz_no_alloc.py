"""The layout entry point that allocates nothing (ep_get_dispatch_layout_noalloc).

Some callers cannot allocate device memory when they call the library: a
plugin or custom-op host that passes in only the tensors it owns, a C caller
with no device allocator, or a serving loop whose device-memory budget is
fixed at start-up.  For them the layout takes its scratch from a fixed array
inside the library instead of a caller-provided workspace.  These tests call
that entry point through the C ABI, twice in a row on different routing (the
second call reuses the scratch the first one left behind), and require the
CPU oracle's layout, and the same results as ep_get_dispatch_layout with a
workspace.  The layout is integer work, so both comparisons are bit-exact,
as in the other layout tests.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from workloads import CONFIGS, make_case

pytestmark = pytest.mark.gpu

EP_ERR_CAPACITY = 2
NOALLOC_LIMIT = 8 << 20  # EP_NOALLOC_SCRATCH_BYTES in include/ep.h


def _noalloc_fn(ep):
    f = ep.lib().ep_get_dispatch_layout_noalloc
    P, i32, i64 = C.c_void_p, C.c_int, C.c_int64
    f.argtypes = [P, i64, i32, i32, i32, P, P, P, P, P, P, P]
    f.restype = i32
    return f


def _call_noalloc(ep, topk_idx, num_experts, num_ranks):
    T, K = topk_idx.shape
    R, E, dev = num_ranks, num_experts, topk_idx.device
    i32 = dict(dtype=torch.int32, device=dev)
    L = ep.Layout(torch.empty((R, R), **i32), torch.empty((R, E), **i32),
                  torch.empty((T, R), dtype=torch.bool, device=dev),
                  torch.empty((T, R), **i32), torch.empty(R + 1, **i32), E, R, None)
    # poison every output so an unwritten element cannot pass
    L.num_tokens_per_rank.fill_(-7)
    L.num_tokens_per_expert.fill_(-7)
    L.slot.fill_(-7)
    L.recv_base.fill_(-7)
    L.is_token_in_rank.view(torch.uint8).fill_(0xAB)
    err = torch.zeros(1, dtype=torch.int32, device=topk_idx.device)
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: t.data_ptr()  # noqa: E731
    status = _noalloc_fn(ep)(p(topk_idx), T, K, num_experts, num_ranks,
                             p(L.num_tokens_per_rank), p(L.num_tokens_per_expert),
                             p(L.is_token_in_rank), p(L.slot), p(L.recv_base), p(err), stream)
    assert status == 0, ep.lib().ep_status_string(status).decode()
    return L, err


def _assert_same_layout(a, b):
    for name in ("num_tokens_per_rank", "num_tokens_per_expert", "slot", "recv_base"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert torch.equal(a.is_token_in_rank.view(torch.uint8), b.is_token_in_rank.view(torch.uint8))


def _assert_oracle_layout(got, want):
    for name in ("num_tokens_per_rank", "num_tokens_per_expert", "slot", "recv_base"):
        assert np.array_equal(getattr(got, name).cpu().numpy(), getattr(want, name)), name
    assert np.array_equal(got.is_token_in_rank.view(torch.uint8).cpu().numpy(),
                          want.is_token_in_rank)


def test_noalloc_layout_matches_oracle_on_two_calls_in_a_row(ep):
    big = CONFIGS["skewed"].scaled(2048)   # 32768 tokens, Zipf routing, masked slots
    small = CONFIGS["tiny"]                # 512 tokens, uniform routing
    cases = [make_case(big, with_hidden=False), make_case(small, with_hidden=False)]
    inputs = [torch.from_numpy(c.topk_idx).cuda() for c in cases]
    got = [_call_noalloc(ep, idx, c.cfg.num_experts, c.cfg.num_ranks)
           for idx, c in zip(inputs, cases)]  # two calls in a row, no sync between
    torch.cuda.synchronize()
    for (L, err), idx, c in zip(got, inputs, cases):
        assert int(err.item()) == 0
        _assert_oracle_layout(L, oracle.layout(c.topk_idx, c.cfg.num_experts, c.cfg.num_ranks))
        # and the entry point with a caller workspace, on the kernels it picks
        want_err = torch.zeros(1, dtype=torch.int32, device="cuda")
        want = ep.get_dispatch_layout(idx, c.cfg.num_experts, c.cfg.num_ranks, err=want_err)
        torch.cuda.synchronize()
        _assert_same_layout(L, want)
        assert int(want_err.item()) == 0


def test_noalloc_layout_rejects_problems_beyond_its_scratch(ep):
    T, R, E = 1 << 20, 8, 256
    need = int(ep.lib().ep_workspace_bytes(T, R, E))
    assert need > NOALLOC_LIMIT
    dummy = C.c_void_p(256)  # never dereferenced: the size check fails first
    status = _noalloc_fn(ep)(dummy, T, 8, E, R, dummy, dummy, dummy, dummy, dummy, None, None)
    assert status == EP_ERR_CAPACITY
    # 786432 tokens at 8 ranks and 256 experts still fit
    assert int(ep.lib().ep_workspace_bytes(786432, R, E)) <= NOALLOC_LIMIT


def test_noalloc_layout_empty(ep):
    idx = torch.empty((0, 4), dtype=torch.int64, device="cuda")
    L, err = _call_noalloc(ep, idx, 16, 4)
    torch.cuda.synchronize()
    assert not L.num_tokens_per_rank.any() and not L.num_tokens_per_expert.any()
    assert not L.recv_base.any() and int(err.item()) == 0
