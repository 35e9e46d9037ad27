"""The dynamically scheduled combine (ep_combine_sched / ep_ll_combine_sched,
used by the binding through each layout's counters) gives exactly the
static schedule's output (ep_combine with no counters): every token is
summed in the same order whichever block claims it.  The counters are zero
after every launch, so one state serves back-to-back launches on a stream.
Shapes cover one-token batches (768 tokens over 456 or 608 blocks),
multi-token batches (many small rows), fewer tokens than blocks, and the
unweighted rank sum; and two streams combining through one layout at once
(the binding gives each stream its own counters).  A launch whose counters
were not zero, or that shares them with a launch on another stream, reports
EP_ERRBIT_SCHED."""
from __future__ import annotations

import ctypes as C
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from ep_testlib import assert_combine_close, bits_of, combine_bound, device_inputs
from workloads import Config, make_case

pytestmark = pytest.mark.gpu

SHAPES = [
    Config("sched_decode_like", 32, 24, 1024, 256, 8, seed=1201),
    Config("sched_small_rows", 16, 2048, 256, 64, 6, routing="zipf", zipf_s=1.2, mask_prob=0.05,
           seed=1202),
    Config("sched_few_tokens", 4, 16, 1024, 16, 4, seed=1203),
    Config("sched_two_experts", 8, 1024, 512, 8, 2, seed=1204),
]


def _recv_rows(L):
    return int(L.recv_base[-1].item())


@pytest.mark.parametrize("cfg", SHAPES, ids=lambda c: c.name)
@pytest.mark.parametrize("weighted", [True, False])
def test_scheduled_combine_equals_static(ep, cfg, weighted):
    c = make_case(cfg)
    idx, w, x = device_inputs(c)
    E, R = cfg.num_experts, cfg.num_ranks
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = ep.get_dispatch_layout(idx, E, R, err=err)
    d = ep.dispatch(x, idx, w, L, err=err)
    wt = w if weighted else None
    assert L.sched is not None
    dyn = ep.combine(d.recv_x, idx, wt, L, err=err)
    static = ep.combine(d.recv_x, idx, wt, replace(L, sched=None), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    np.testing.assert_array_equal(bits_of(dyn), bits_of(static))
    assert L.sched.tolist() == [0, 0]
    if weighted:
        P = _recv_rows(L)
        slot = L.slot.cpu().numpy()
        y = bits_of(d.recv_x[:P])
        want = oracle.combine(y, c.topk_idx, c.topk_weights, E, R, slot)
        bound = combine_bound(oracle.bf16_to_double(y), c.topk_idx, c.topk_weights, slot, E // R,
                              np.arange(cfg.num_tokens))
        assert_combine_close(bits_of(dyn), want, bound)


def test_one_state_serves_back_to_back_launches(ep):
    cfg = SHAPES[1]
    c = make_case(cfg)
    idx, w, x = device_inputs(c)
    E, R = cfg.num_experts, cfg.num_ranks
    L = ep.get_dispatch_layout(idx, E, R)
    d = ep.dispatch(x, idx, w, L)
    outs = [ep.combine(d.recv_x, idx, w, L) for _ in range(6)]  # no host sync in between
    torch.cuda.synchronize()
    first = bits_of(outs[0])
    for o in outs[1:]:
        np.testing.assert_array_equal(bits_of(o), first)
    assert L.sched.tolist() == [0, 0]


@pytest.mark.parametrize("cfg", SHAPES[:2], ids=lambda c: c.name)
def test_expert_major_scheduled_combine_equals_static(ep, cfg):
    c = make_case(cfg)
    idx, w, x = device_inputs(c)
    E, R, T = cfg.num_experts, cfg.num_ranks, cfg.num_tokens
    cap = max(1, int(oracle.ll_layout(c.topk_idx, E, R, T).ll_count.max()))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    LL = ep.ll_get_dispatch_layout(idx, E, R, cap, err=err)
    y = torch.randn((LL.num_rows, cfg.hidden), device="cuda").to(torch.bfloat16)
    dyn = ep.ll_combine(y, w, LL, err=err)
    static = ep.ll_combine(y, w, replace(LL, sched=None), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    np.testing.assert_array_equal(bits_of(dyn), bits_of(static))
    assert LL.sched.tolist() == [0, 0]


def _two_outputs(ep, cfg, seed=77):
    c = make_case(cfg)
    idx, w, _ = device_inputs(c)
    L = ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks)
    rows = ep.worst_case_rows(cfg.num_tokens, cfg.num_topk, cfg.num_ranks)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    ys = [torch.randn((rows, cfg.hidden), device="cuda", generator=g).to(torch.bfloat16)
          for _ in range(2)]
    return idx, w, L, ys


def test_overlapping_combines_through_one_layout_get_their_own_counters(ep):
    """Two streams combine different expert outputs through one layout at the
    same time; the binding hands each stream its own counters, so each gets
    exactly its result alone."""
    cfg = SHAPES[1]
    idx, w, L, ys = _two_outputs(ep, cfg)
    alone = [ep.combine(ys[0], idx, w, L), ep.combine(ys[1], idx, w, L)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    outs = [[], []]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):
        for i in (0, 1):  # interleave the two streams' launches
            with torch.cuda.stream(streams[i]):
                outs[i].append(ep.combine(ys[i], idx, w, L, err=err))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for i in (0, 1):
        for o in outs[i]:
            np.testing.assert_array_equal(bits_of(o), bits_of(alone[i]))
    used = [ep.sched_for(L, idx.device)]
    for s in streams:
        with torch.cuda.stream(s):
            used.append(ep.sched_for(L, idx.device))
    assert len({t.data_ptr() for t in used}) == 3  # the home stream's and one per side stream
    assert all(t.tolist() == [0, 0] for t in used)


def test_counters_not_zero_at_launch_are_reported(ep):
    """A claim counter left non-zero (as if another launch had claimed from
    it) shifts the batches: the launch reports EP_ERRBIT_SCHED, still leaves
    the counters at zero, and the next launch is exact again."""
    cfg = SHAPES[1]
    idx, w, L, ys = _two_outputs(ep, cfg)
    alone = ep.combine(ys[0], idx, w, L)
    torch.cuda.synchronize()
    L.sched[0] = 1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.combine(ys[0], idx, w, L, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == ep.EP_ERRBIT_SCHED
    assert L.sched.tolist() == [0, 0]
    err.zero_()
    again = ep.combine(ys[0], idx, w, L, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    np.testing.assert_array_equal(bits_of(again), bits_of(alone))


def test_shared_counters_on_two_streams_never_go_unreported(ep):
    """Through the C ABI, two launches on two streams share one counter state
    (the misuse the binding prevents).  Whenever either output differs from
    its result alone, the shared error word carries EP_ERRBIT_SCHED.  The
    persistent grid fills the GPU, so the second launch's blocks start only
    as the first one's leave, and often after its last block has reset the
    counters: then both outputs are whole and nothing is reported.  The
    deterministic case is test_counters_not_zero_at_launch_are_reported."""
    cfg = Config("sched_overlap", 16, 2048, 4096, 64, 6, routing="zipf", zipf_s=1.2,
                 mask_prob=0.05, seed=1205)
    idx, w, L, ys = _two_outputs(ep, cfg)
    alone = [bits_of(ep.combine(ys[i], idx, w, L)) for i in (0, 1)]
    lib = ep.lib()
    sched = ep.alloc_combine_sched(idx.device)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    T, K = idx.shape
    caught = 0
    for _ in range(4):
        sched.zero_()
        err.zero_()
        outs = [torch.zeros_like(x[:T]) for x in (ys[0], ys[1])]
        torch.cuda.synchronize()
        for i in (0, 1):
            st = C.c_void_p(streams[i].cuda_stream)
            status = lib.ep_combine_sched(ys[i].data_ptr(), cfg.hidden, idx.data_ptr(),
                                          w.data_ptr(), T, K, cfg.num_experts, cfg.num_ranks,
                                          L.slot.data_ptr(), outs[i].data_ptr(),
                                          sched.data_ptr(), err.data_ptr(), st)
            assert status == 0
        torch.cuda.synchronize()
        wrong = any(not np.array_equal(bits_of(outs[i]), alone[i]) for i in (0, 1))
        flagged = bool(int(err.item()) & ep.EP_ERRBIT_SCHED)
        assert flagged or not wrong, "an incomplete combine went unreported"
        caught += wrong
    print(f"{caught} of 4 overlapping pairs lost tokens, all reported")
