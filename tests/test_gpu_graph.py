"""The shuffle is stream-ordered and, once its buffers exist, needs no host
synchronisation or allocation, so a whole step (layout -> dispatch ->
combine) can be captured in a CUDA graph and replayed.  Each replay must
give the oracle's layout and the eager step's output, also after new routing
and new hidden states are written in place between replays."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from ep_testlib import bits_of
from workloads import Config, make_case

pytestmark = pytest.mark.gpu


def _cases():
    base = Config("graph_r8", 8, 96, 512, 32, 4, routing="zipf", zipf_s=1.2, mask_prob=0.05,
                  seed=990)
    other = Config("graph_r8", 8, 96, 512, 32, 4, mask_prob=0.1, seed=991)
    return make_case(base), make_case(other)


def _to_device(c, idx, w, x):
    idx.copy_(torch.from_numpy(c.topk_idx))
    w.copy_(torch.from_numpy(c.topk_weights))
    x.copy_(torch.from_numpy(c.x_bits.view(np.int16)).view(torch.bfloat16))


@pytest.mark.parametrize("path", ["single", "multi", "fused"])
def test_rank_major_step_in_a_cuda_graph(ep, path):
    """path: the layout's kernels, or "fused" for layout and dispatch in one
    launch (whose counters must be back at zero for every replay)."""
    c0, c1 = _cases()
    cfg = c0.cfg
    T, H, K, E, R = cfg.num_tokens, cfg.hidden, cfg.num_topk, cfg.num_experts, cfg.num_ranks
    dev = torch.device("cuda")
    idx = torch.empty((T, K), dtype=torch.int64, device=dev)
    w = torch.empty((T, K), dtype=torch.float32, device=dev)
    x = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    L = ep.alloc_layout(T, E, R, dev)
    D = ep.alloc_dispatched(ep.worst_case_rows(T, K, R), H, K, E, R, False, dev)

    def step():
        if path == "fused":
            ep.layout_dispatch(x, idx, w, E, R, err=err, layout=L, out=D)
        else:
            ep.get_dispatch_layout(idx, E, R, err=err, out=L, path=path)
            ep.dispatch(x, idx, w, L, err=err, out=D)
        ep.combine(D.recv_x, idx, w, L, err=err, out=out)

    _to_device(c0, idx, w, x)
    step()  # eager, also does every one-time set-up
    torch.cuda.synchronize()
    eager = bits_of(out)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits_of(out), eager)

    for c in (c1, c0):  # new routing and hidden states, written in place
        _to_device(c, idx, w, x)
        g.replay()
        torch.cuda.synchronize()
        want = oracle.layout(c.topk_idx, E, R)
        np.testing.assert_array_equal(L.slot.cpu().numpy(), want.slot)
        np.testing.assert_array_equal(L.recv_base.cpu().numpy(), want.recv_base)
        wd = oracle.dispatch(c.x_bits, c.topk_idx, c.topk_weights, E, R, want.slot,
                             want.num_rows)
        np.testing.assert_array_equal(bits_of(D.recv_x[:want.num_rows]), wd.recv_x)
    np.testing.assert_array_equal(bits_of(out), eager)  # back on the first inputs
    assert int(err.item()) == 0


def test_expert_major_step_in_a_cuda_graph(ep):
    c0, c1 = _cases()
    cfg = c0.cfg
    T, H, K, E, R = cfg.num_tokens, cfg.hidden, cfg.num_topk, cfg.num_experts, cfg.num_ranks
    dev = torch.device("cuda")
    idx = torch.empty((T, K), dtype=torch.int64, device=dev)
    w = torch.empty((T, K), dtype=torch.float32, device=dev)
    x = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    LL = ep.alloc_ll_layout(T, K, E, R, T, dev)
    _to_device(c0, idx, w, x)
    ep.ll_get_dispatch_layout(idx, E, R, err=err, out=LL)
    DL = ep.ll_dispatch(x, LL, use_fp8=True, err=err)

    # the expert-major combine reads bf16 expert outputs in the slot rows:
    # a fixed random buffer stands in for them
    y = torch.randn((E * T, H), device=dev).to(torch.bfloat16)

    def step():
        ep.ll_get_dispatch_layout(idx, E, R, err=err, out=LL)
        ep.ll_dispatch(x, LL, use_fp8=True, err=err, out=DL)
        ep.ll_combine(y, w, LL, err=err, out=out)

    step()
    torch.cuda.synchronize()
    eager = bits_of(out)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for c in (c1, c0):
        _to_device(c, idx, w, x)
        g.replay()
        torch.cuda.synchronize()
        want = oracle.ll_layout(c.topk_idx, E, R, T)
        np.testing.assert_array_equal(LL.ll_slot.cpu().numpy(), want.ll_slot)
        np.testing.assert_array_equal(LL.ll_count.cpu().numpy(), want.ll_count)
    np.testing.assert_array_equal(bits_of(out), eager)
    assert int(err.item()) == 0
