"""GPU parity: ep_get_dispatch_layout against the CPU oracle, bit-exact on
every output (counts, is_token_in_rank, slot, recv_base), on small and ragged
cases, the extremes, and all five workloads at full size.  Both kernel paths
are checked: the multi-launch form and the single-launch (one thread-block
cluster) form for the batches it takes."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from ep_testlib import device_inputs, full_case, small_configs
from workloads import CONFIGS, Config, make_case

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


PATHS = ["multi", "single"]


def layout_on(ep, idx, cfg, path, err=None):
    """The layout on the given path, poisoned first; None (after checking
    that the call is refused on the host) when the single-launch form does
    not take this batch."""
    L = ep.alloc_layout(cfg.num_tokens, cfg.num_experts, cfg.num_ranks, idx.device)
    poison_layout(L)
    if path == "single" and not ep.single_launch_fits(cfg.num_tokens, cfg.num_ranks,
                                                      cfg.num_experts):
        with pytest.raises(ep.EPError):
            ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks, out=L, path=path)
        return None
    ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks, err=err, out=L, path=path)
    return L


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("cfg", small_configs(), ids=lambda c: c.name)
def test_layout_small(ep, cfg, path):
    c = make_case(cfg, with_hidden=False)
    idx, _, _ = device_inputs(c)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = layout_on(ep, idx, cfg, path, err)
    if L is None:
        return
    want = oracle.layout(c.topk_idx, cfg.num_experts, cfg.num_ranks)
    compare_layout(L, want)
    assert int(err.item()) == 0
    assert ep.total_rows(L) == want.num_rows


def single_launch_configs():
    """Shapes that drive the single-launch form through several CTAs and
    chunks, ragged last CTAs and chunks, sources spread over several CTAs,
    warps holding many sources, and the largest histogram it takes."""
    specs = [  # name, R, T_r, E, K, routing, mask
        ("s_r3_ragged", 3, 5000, 12, 4, "zipf", 0.05),     # several chunks, last CTA ragged
        ("s_r7_16380", 7, 2340, 14, 2, "uniform", 0.0),    # four tokens short of the maximum
        ("s_r2_16384", 2, 8192, 8, 6, "zipf", 0.1),        # exactly the maximum
        ("s_r64_tr1", 64, 1, 128, 8, "uniform", 0.0),      # every lane its own source
        ("s_r64_e256", 64, 100, 256, 8, "zipf", 0.05),     # R * E = 16384
        ("s_r5_k32", 5, 1500, 40, 32, "uniform", 0.3),     # four batches of ids per token
        ("s_r16_1000", 16, 1000, 64, 6, "zipf", 0.05),     # sources straddle CTAs
        ("s_r3_tr5", 3, 5, 6, 2, "uniform", 0.0),          # one CTA, 15 tokens
    ]
    return [Config(n, R, Tr, 8, E, K, routing=rt, zipf_s=1.2 if rt == "zipf" else 0.0,
                   mask_prob=m, seed=950 + i)
            for i, (n, R, Tr, E, K, rt, m) in enumerate(specs)]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("cfg", single_launch_configs(), ids=lambda c: c.name)
def test_layout_single_launch_shapes(ep, cfg, path):
    assert ep.single_launch_fits(cfg.num_tokens, cfg.num_ranks, cfg.num_experts)
    c = make_case(cfg, with_hidden=False)
    idx, _, _ = device_inputs(c)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = layout_on(ep, idx, cfg, path, err)
    compare_layout(L, oracle.layout(c.topk_idx, cfg.num_experts, cfg.num_ranks))
    assert int(err.item()) == 0


@pytest.mark.parametrize("path", ["auto"] + PATHS)
@pytest.mark.parametrize("name", list(CONFIGS))
def test_layout_full_size(ep, name, path):
    cfg = CONFIGS[name]
    c, want = full_case(name)
    idx, _, _ = device_inputs(type(c)(c.cfg, c.topk_idx, c.topk_weights, None))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = layout_on(ep, idx, cfg, path, err)
    if L is None:
        return
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


@pytest.mark.parametrize("path", PATHS)
def test_layout_out_of_range_ids_are_flagged_and_masked(ep, path):
    cfg = CONFIGS["tiny"]
    c = make_case(cfg, with_hidden=False)
    idx_np = c.topk_idx.copy()
    idx_np[3, 1] = cfg.num_experts
    idx_np[100, 0] = -5
    idx_np[511, 3] = 1 << 40
    idx = torch.from_numpy(idx_np).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = layout_on(ep, idx, cfg, path, err)
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
