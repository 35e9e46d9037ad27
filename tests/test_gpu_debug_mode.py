"""The binding's debug mode: with it on, a call whose kernels set a bit of the
device error word raises at once, naming the call and the problem; with it
off (the default) the same calls return and leave the bits to the caller."""
from __future__ import annotations

import pytest
import torch

from ep_testlib import device_inputs
from workloads import CONFIGS, make_case

pytestmark = pytest.mark.gpu


def test_debug_mode_raises_on_the_failing_call(ep):
    cfg = CONFIGS["tiny"]
    c = make_case(cfg)
    idx, w, x = device_inputs(c)
    E, R = cfg.num_experts, cfg.num_ranks
    bad = idx.clone()
    bad[3, 1] = E + 5
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.set_debug(True)
    try:
        with pytest.raises(ep.EPError, match="get_dispatch_layout.*expert id"):
            ep.get_dispatch_layout(bad, E, R, err=err)
        err.zero_()
        L = ep.get_dispatch_layout(idx, E, R, err=err)  # clean routing passes
        with pytest.raises(ep.EPError, match="dispatch.*receive capacity"):
            ep.dispatch(x, idx, w, L, capacity=2, err=err)
        err.zero_()
        ep.dispatch(x, idx, w, L, err=err)
    finally:
        ep.set_debug(False)
    # off again: the same overflow only sets the bit
    err.zero_()
    ep.dispatch(x, idx, w, L, capacity=2, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ep.EP_ERRBIT_CAPACITY
