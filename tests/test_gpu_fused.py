"""GPU parity: the one-launch layout + dispatch (ep_layout_dispatch_fused)
against the CPU oracle, bit-exact on every layout output (counts,
is_token_in_rank, slots, recv_base) and every dispatched byte (bf16 rows, or
FP8 codes and scales) with the per-row metadata and the per-expert receive
counts.  Small, ragged and extreme shapes, the random sweep's shapes that
fit, the small and decode workloads at full size, bad ids, a tight
capacity, back-to-back launches on one state, and the bounded waits run out
on purpose through the test hook."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from ep_testlib import bits_of, device_inputs, fp8_small_configs, small_configs
from test_gpu_random import N_CASES, random_config
from test_gpu_adversarial import CASES as _ADV, _case as _adv_case
from workloads import CONFIGS, make_case

pytestmark = pytest.mark.gpu


def _poisoned(ep, T, H, K, E, R, cap, use_fp8, dev):
    L = ep.alloc_layout(T, E, R, dev)
    for t in (L.num_tokens_per_rank, L.num_tokens_per_expert, L.slot, L.recv_base):
        t.fill_(-7)
    L.is_token_in_rank.view(torch.uint8).fill_(0xAB)
    D = ep.alloc_dispatched(cap, H, K, E, R, use_fp8, dev)
    D.recv_x.view(torch.uint8).fill_(0xFF)
    if D.recv_scales is not None:
        D.recv_scales.fill_(float("nan"))
    D.recv_src_idx.fill_(-9)
    D.recv_topk_idx.fill_(-9)
    D.recv_topk_weights.fill_(float("nan"))
    D.num_recv_tokens_per_expert.fill_(-9)
    return L, D


def check_fused(ep, cfg, c, use_fp8, cap_extra=5):
    T, H, K, E, R = cfg.num_tokens, cfg.hidden, cfg.num_topk, cfg.num_experts, cfg.num_ranks
    idx, w, x = device_inputs(c)
    want = oracle.layout(c.topk_idx, E, R)
    P = want.num_rows
    L, D = _poisoned(ep, T, H, K, E, R, P + cap_extra, use_fp8, x.device)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.layout_dispatch(x, idx, w, E, R, use_fp8=use_fp8, err=err, layout=L, out=D)
    torch.cuda.synchronize()
    assert int(err.item()) == want.err_bits
    np.testing.assert_array_equal(L.slot.cpu().numpy(), want.slot)
    np.testing.assert_array_equal(L.num_tokens_per_rank.cpu().numpy(), want.num_tokens_per_rank)
    np.testing.assert_array_equal(L.num_tokens_per_expert.cpu().numpy(),
                                  want.num_tokens_per_expert)
    np.testing.assert_array_equal(L.recv_base.cpu().numpy(), want.recv_base)
    np.testing.assert_array_equal(L.is_token_in_rank.view(torch.uint8).cpu().numpy(),
                                  want.is_token_in_rank)
    wd = oracle.dispatch(c.x_bits, c.topk_idx, c.topk_weights, E, R, want.slot, P,
                         use_fp8=use_fp8)
    if use_fp8:
        np.testing.assert_array_equal(D.recv_x[:P].cpu().numpy(), wd.recv_x)
        np.testing.assert_array_equal(D.recv_scales[:P].cpu().numpy().view(np.uint32),
                                      wd.recv_scales.view(np.uint32))
        assert (D.recv_x[P:].cpu().numpy() == 0xFF).all()  # rows past P untouched
    else:
        np.testing.assert_array_equal(bits_of(D.recv_x[:P]), wd.recv_x)
        assert (bits_of(D.recv_x[P:]) == 0xFFFF).all()
    np.testing.assert_array_equal(D.recv_src_idx[:P].cpu().numpy(), wd.recv_src_idx)
    np.testing.assert_array_equal(D.recv_topk_idx[:P].cpu().numpy(), wd.recv_topk_idx)
    np.testing.assert_array_equal(D.recv_topk_weights[:P].cpu().numpy().view(np.uint32),
                                  wd.recv_topk_weights.view(np.uint32))
    np.testing.assert_array_equal(D.num_recv_tokens_per_expert.cpu().numpy(),
                                  oracle.num_recv_tokens_per_expert(want.num_tokens_per_expert, E, R))
    assert not L.fused_sync.any()
    return L, D


@pytest.mark.parametrize("cfg", [c for c in small_configs() if c.num_tokens > 0],
                         ids=lambda c: c.name)
def test_fused_small_bf16(ep, cfg):
    if not ep.fused_fits(cfg.num_tokens, cfg.num_ranks, cfg.num_experts):
        pytest.skip("outside the one-launch limits")
    check_fused(ep, cfg, make_case(cfg), use_fp8=False)


@pytest.mark.parametrize("cfg", fp8_small_configs(), ids=lambda c: c.name)
def test_fused_small_fp8(ep, cfg):
    check_fused(ep, cfg, make_case(cfg), use_fp8=True)


@pytest.mark.parametrize("i", range(N_CASES))
def test_fused_random_shape(ep, i):
    cfg = random_config(i)
    if not ep.fused_fits(cfg.num_tokens, cfg.num_ranks, cfg.num_experts):
        pytest.skip("outside the one-launch limits")
    c = make_case(cfg)
    check_fused(ep, cfg, c, use_fp8=False)
    if cfg.hidden % 128 == 0:
        check_fused(ep, cfg, c, use_fp8=True)


@pytest.mark.parametrize("name", ["tiny", "decode_fp8"])
def test_fused_full_workload(ep, name):
    cfg = CONFIGS[name]
    check_fused(ep, cfg, make_case(cfg), use_fp8=cfg.fp8)


def test_fused_bad_ids_and_tight_capacity(ep):
    cfg = CONFIGS["tiny"]
    c = make_case(cfg)
    c.topk_idx[7, 2] = 999
    c.topk_idx[40, 0] = -5
    T, H, K, E, R = cfg.num_tokens, cfg.hidden, cfg.num_topk, cfg.num_experts, cfg.num_ranks
    idx, w, x = device_inputs(c)
    want = oracle.layout(c.topk_idx, E, R)
    cap = want.num_rows - 3
    L, D = _poisoned(ep, T, H, K, E, R, cap, False, x.device)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.layout_dispatch(x, idx, w, E, R, err=err, layout=L, out=D)
    torch.cuda.synchronize()
    assert int(err.item()) == ep.EP_ERRBIT_BAD_EXPERT | ep.EP_ERRBIT_CAPACITY
    np.testing.assert_array_equal(L.slot.cpu().numpy(), want.slot)
    wd = oracle.dispatch(c.x_bits, c.topk_idx, c.topk_weights, E, R, want.slot, want.num_rows)
    np.testing.assert_array_equal(bits_of(D.recv_x), wd.recv_x[:cap])


def test_fused_back_to_back_on_one_state(ep):
    """Six launches on new routing each, no host sync between: the state
    returns to zero after each, and every launch matches the oracle."""
    dev = torch.device("cuda")
    base = CONFIGS["decode_fp8"]
    cases = [make_case(base.__class__(**{**base.__dict__, "seed": 90 + i}))
             for i in range(6)]
    cfg = base
    T, H, K, E, R = cfg.num_tokens, cfg.hidden, cfg.num_topk, cfg.num_experts, cfg.num_ranks
    L = ep.alloc_layout(T, E, R, dev)
    outs = []
    for c in cases:
        idx, w, x = device_inputs(c)
        Lc = ep.alloc_layout(T, E, R, dev)
        Lc.fused_sync = L.fused_sync  # one state for all six
        outs.append((c, ep.layout_dispatch(x, idx, w, E, R, use_fp8=True, layout=Lc)))
    torch.cuda.synchronize()
    assert not L.fused_sync.any()
    for c, (Lc, D) in outs:
        want = oracle.layout(c.topk_idx, E, R)
        np.testing.assert_array_equal(Lc.slot.cpu().numpy(), want.slot)
        P = want.num_rows
        wd = oracle.dispatch(c.x_bits, c.topk_idx, c.topk_weights, E, R, want.slot, P,
                             use_fp8=True)
        np.testing.assert_array_equal(D.recv_x[:P].cpu().numpy(), wd.recv_x)


def test_fused_wait_runs_out_then_recovers(ep):
    """The hook leaves one layout block's barrier arrival out: the launch
    reports EP_ERRBIT_TIMEOUT (after about 1 s per bounded wait, no fault),
    dispatches nothing, returns its state to zero, and the next launch on
    the same state is exact."""
    cfg = CONFIGS["tiny"]
    c = make_case(cfg)
    T, H, K, E, R = cfg.num_tokens, cfg.hidden, cfg.num_topk, cfg.num_experts, cfg.num_ranks
    idx, w, x = device_inputs(c)
    L, D = _poisoned(ep, T, H, K, E, R, T * 4, False, x.device)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.lib().ep_debug_set_fused_stall(1)
    ep.layout_dispatch(x, idx, w, E, R, err=err, layout=L, out=D)
    torch.cuda.synchronize()
    assert int(err.item()) & ep.EP_ERRBIT_TIMEOUT
    assert (bits_of(D.recv_x) == 0xFFFF).all()  # nothing dispatched
    assert not L.fused_sync.any()
    check_fused(ep, cfg, c, use_fp8=False)


@pytest.mark.parametrize("i", range(len(_ADV)), ids=lambda i: "{}-{}".format(_ADV[i][0], _ADV[i][1][0]))
def test_fused_adversarial_routing(ep, i):
    """The adversarial routings (duplicate experts, bad ids, one hot expert or
    rank, masked tokens) through the one-launch layout + dispatch."""
    kind, shape = _ADV[i]
    cfg, c = _adv_case(kind, shape, i)
    if not ep.fused_fits(cfg.num_tokens, cfg.num_ranks, cfg.num_experts):
        pytest.skip("outside the one-launch limits")
    check_fused(ep, cfg, c, use_fp8=False)
    if cfg.hidden % 128 == 0:
        check_fused(ep, cfg, c, use_fp8=True)
