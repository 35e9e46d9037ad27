"""GPU parity: ep_get_dispatch_layout against the CPU oracle, bit-exact on
every output (counts, is_token_in_rank, slot, recv_base), on small and ragged
cases, the extremes, and all five workloads at full size."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from ep_testlib import device_inputs, full_case, small_configs
from workloads import CONFIGS, make_case

pytestmark = pytest.mark.gpu


def compare_layout(L, want):
    np.testing.assert_array_equal(L.num_tokens_per_rank.cpu().numpy(), want.num_tokens_per_rank)
    np.testing.assert_array_equal(L.num_tokens_per_expert.cpu().numpy(), want.num_tokens_per_expert)
    np.testing.assert_array_equal(L.is_token_in_rank.cpu().numpy().astype(np.uint8),
                                  want.is_token_in_rank)
    np.testing.assert_array_equal(L.slot.cpu().numpy(), want.slot)
    np.testing.assert_array_equal(L.recv_base.cpu().numpy(), want.recv_base)


def poison_layout(L):
    L.num_tokens_per_rank.fill_(-7)
    L.num_tokens_per_expert.fill_(-7)
    L.slot.fill_(-7)
    L.recv_base.fill_(-7)
    L.is_token_in_rank.view(torch.uint8).fill_(0xAB)
    if L.workspace is not None:
        L.workspace.fill_(0xCD)


@pytest.mark.parametrize("cfg", small_configs(), ids=lambda c: c.name)
def test_layout_small(ep, cfg):
    c = make_case(cfg, with_hidden=False)
    idx, _, _ = device_inputs(c)
    L = ep.alloc_layout(cfg.num_tokens, cfg.num_experts, cfg.num_ranks, idx.device)
    poison_layout(L)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks, err=err, out=L)
    want = oracle.layout(c.topk_idx, cfg.num_experts, cfg.num_ranks)
    compare_layout(L, want)
    assert int(err.item()) == 0
    assert ep.total_rows(L) == want.num_rows


@pytest.mark.parametrize("name", list(CONFIGS))
def test_layout_full_size(ep, name):
    cfg = CONFIGS[name]
    c, want = full_case(name)
    idx, _, _ = device_inputs(type(c)(c.cfg, c.topk_idx, c.topk_weights, None))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks, err=err)
    compare_layout(L, want)
    assert int(err.item()) == 0


def test_layout_repeated_calls_reuse_buffers(ep):
    # The workspace needs no clearing between calls: a second call on other
    # routing with the same buffers gives that routing's layout.
    cfg = CONFIGS["tiny"]
    L = ep.alloc_layout(cfg.num_tokens, cfg.num_experts, cfg.num_ranks, torch.device("cuda"))
    for seed in (1, 2):
        c = make_case(type(cfg)(**{**cfg.__dict__, "seed": seed}), with_hidden=False)
        idx, _, _ = device_inputs(c)
        ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks, out=L)
        compare_layout(L, oracle.layout(c.topk_idx, cfg.num_experts, cfg.num_ranks))


def test_layout_out_of_range_ids_are_flagged_and_masked(ep):
    cfg = CONFIGS["tiny"]
    c = make_case(cfg, with_hidden=False)
    idx_np = c.topk_idx.copy()
    idx_np[3, 1] = cfg.num_experts
    idx_np[100, 0] = -5
    idx_np[511, 3] = 1 << 40
    idx = torch.from_numpy(idx_np).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks, err=err)
    want = oracle.layout(idx_np, cfg.num_experts, cfg.num_ranks)
    assert want.err_bits == 1
    compare_layout(L, want)
    assert int(err.item()) & ep.EP_ERRBIT_BAD_EXPERT


def test_layout_empty(ep):
    idx = torch.empty((0, 4), dtype=torch.int64, device="cuda")
    L = ep.alloc_layout(0, 16, 4, idx.device)
    poison_layout(L)
    ep.get_dispatch_layout(idx, 16, 4, out=L)
    assert not L.num_tokens_per_rank.any() and not L.num_tokens_per_expert.any()
    assert not L.recv_base.any() and ep.total_rows(L) == 0


def test_layout_on_a_side_stream(ep):
    cfg = CONFIGS["tiny"]
    c = make_case(cfg, with_hidden=False)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        idx = torch.from_numpy(c.topk_idx).cuda(non_blocking=False)
        L = ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks)
    s.synchronize()
    compare_layout(L, oracle.layout(c.topk_idx, cfg.num_experts, cfg.num_ranks))


def test_layout_unfolded_scan_path(ep):
    """64 ranks x 2048 tokens per rank give 64 * 256 blocks > 8192, so the
    layout runs the separate scan kernel between count and assign."""
    from workloads import Config
    cfg = Config("r64_unfolded", 64, 2048, 8, 128, 4, routing="zipf", zipf_s=1.2,
                 mask_prob=0.05, seed=901)
    c = make_case(cfg, with_hidden=False)
    idx, _, _ = device_inputs(c)
    L = ep.alloc_layout(cfg.num_tokens, cfg.num_experts, cfg.num_ranks, idx.device)
    poison_layout(L)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks, err=err, out=L)
    compare_layout(L, oracle.layout(c.topk_idx, cfg.num_experts, cfg.num_ranks))
    assert int(err.item()) == 0
