"""Independent steps on two streams at once: each stream runs layout ->
dispatch -> combine on its own routing and buffers, launches interleaved,
and must get exactly what it gets alone.  The library keeps no per-call
state outside the caller's buffers (the no-alloc layout excepted, which is
documented to race), so overlapping calls must not interfere."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from ep_testlib import bits_of, device_inputs
from workloads import Config, make_case

pytestmark = pytest.mark.gpu


def _step(ep, idx, w, x, E, R, path, fp8):
    L = ep.get_dispatch_layout(idx, E, R, path=path)
    d = ep.dispatch(x, idx, w, L, use_fp8=fp8)
    y = d.recv_x if not fp8 else torch.ones((d.recv_x.shape[0], x.shape[1]),
                                               dtype=torch.bfloat16, device=x.device)
    out = ep.combine(y, idx, w, L)
    LL = ep.ll_get_dispatch_layout(idx, E, R, path=path)
    dl = ep.ll_dispatch(x, LL, use_fp8=fp8)
    return L, d, out, LL, dl


@pytest.mark.parametrize("path", ["single", "multi"])
def test_two_streams_do_not_interfere(ep, path):
    cfgs = [Config("s0", 8, 300, 512, 64, 6, routing="zipf", zipf_s=1.2, mask_prob=0.05, seed=31),
            Config("s1", 8, 300, 512, 64, 6, mask_prob=0.1, seed=32)]
    cases = [make_case(c) for c in cfgs]
    ins = [device_inputs(c) for c in cases]
    E, R = cfgs[0].num_experts, cfgs[0].num_ranks
    alone = []
    for (idx, w, x) in ins:
        alone.append(_step(ep, idx, w, x, E, R, path, False))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    results = [None, None]
    for rep in range(3):
        for i in (0, 1):  # interleave the two steps' launches
            with torch.cuda.stream(streams[i]):
                idx, w, x = ins[i]
                results[i] = _step(ep, idx, w, x, E, R, path, False)
        torch.cuda.synchronize()
        for i in (0, 1):
            La, da, oa, LLa, dla = alone[i]
            Lb, db, ob, LLb, dlb = results[i]
            assert torch.equal(La.slot, Lb.slot) and torch.equal(La.recv_base, Lb.recv_base)
            P = int(La.recv_base[-1].item())
            np.testing.assert_array_equal(bits_of(da.recv_x[:P]), bits_of(db.recv_x[:P]))
            np.testing.assert_array_equal(bits_of(oa), bits_of(ob))
            assert torch.equal(LLa.ll_slot, LLb.ll_slot) and torch.equal(LLa.ll_count, LLb.ll_count)
            live = LLa.ll_slot[LLa.ll_slot >= 0].long()
            np.testing.assert_array_equal(bits_of(dla.recv_x[live]), bits_of(dlb.recv_x[live]))


def test_two_host_threads_on_their_own_streams(ep):
    """The library's per-device caches are shared by host threads (and filled
    under a lock); two threads, each with its own stream and buffers, calling
    at the same time get the same results as one thread alone."""
    import threading
    cfgs = [Config("h0", 4, 500, 256, 32, 4, routing="zipf", zipf_s=1.2, seed=41),
            Config("h1", 4, 500, 256, 32, 4, mask_prob=0.2, seed=42)]
    cases = [make_case(c) for c in cfgs]
    ins = [device_inputs(c) for c in cases]
    E, R = cfgs[0].num_experts, cfgs[0].num_ranks
    want = [bits_of(_step(ep, *ins[i], E, R, "auto", False)[2]) for i in (0, 1)]
    got = [[], []]
    errors = []

    def worker(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(10):
                    out = _step(ep, *ins[i], E, R, "auto", False)[2]
                    s.synchronize()
                    got[i].append(bits_of(out))
        except Exception as e:  # reported below, in the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in (0, 1)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for i in (0, 1):
        assert len(got[i]) == 10
        for g in got[i]:
            np.testing.assert_array_equal(g, want[i])
