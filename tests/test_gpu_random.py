"""Randomised parity sweep (256 cases; EP_RANDOM_CASES=n for more): many
small seeded shapes (ranks 1..64, ragged tokens per rank, 1..8 experts per
rank, top-1..12, hidden sizes from one 16-byte vector up, uniform or Zipf
routing, 0-50% masked slots), each run through every entry point and
compared with the CPU oracle: both layouts on both kernel paths (bit-exact),
both dispatches (bit-exact bf16 rows; E4M3 codes and scales where
H % 128 == 0), and the weighted and unweighted combines (the combine
tolerance)."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from ep_testlib import assert_combine_close, bf16_from_bits, bits_of, combine_bound, device_inputs
from workloads import Config, make_case

pytestmark = pytest.mark.gpu

N_CASES = int(os.environ.get("EP_RANDOM_CASES", "256"))


def random_config(i: int) -> Config:
    """Shapes kept to T * K * H <= 2^22, so the float64 tolerance bounds stay small."""
    rng = np.random.default_rng(7000 + i)
    R = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 13, 16, 32, 64]))
    Tr = int(rng.integers(1, min(200, max(2, 6000 // R))))
    El = int(rng.integers(1, 9))
    E = R * El
    K = int(rng.integers(1, min(E, 12) + 1))
    hs = [h for h in (8, 16, 72, 128, 264, 384, 1024) if R * Tr * K * h <= (1 << 22)] or [8]
    H = int(rng.choice(hs))
    routing = "zipf" if rng.random() < 0.4 else "uniform"
    mask = float(rng.choice([0.0, 0.1, 0.5]))
    return Config(f"rand{i}_r{R}_t{Tr}_e{E}_k{K}_h{H}", R, Tr, H, E, K, routing=routing,
                  zipf_s=1.2 if routing == "zipf" else 0.0, mask_prob=mask, seed=8000 + i)


def _paths(fits: bool):
    return ["multi", "single"] if fits else ["multi"]


@pytest.mark.parametrize("i", range(N_CASES))
def test_rank_major_random_shape(ep, i):
    cfg = random_config(i)
    check_rank_major(ep, cfg, make_case(cfg))


def check_rank_major(ep, cfg, c):
    """Every rank-major entry point on case c against the oracle: the layout
    on both kernel paths, both dispatches, the weighted and unweighted
    combines, and the error bits."""
    T, H, K, E, R = cfg.num_tokens, cfg.hidden, cfg.num_topk, cfg.num_experts, cfg.num_ranks
    idx, w, x = device_inputs(c)
    want = oracle.layout(c.topk_idx, E, R)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for path in _paths(ep.single_launch_fits(T, R, E)):
        L = ep.get_dispatch_layout(idx, E, R, err=err, path=path)
        np.testing.assert_array_equal(L.slot.cpu().numpy(), want.slot, err_msg=path)
        np.testing.assert_array_equal(L.num_tokens_per_rank.cpu().numpy(),
                                      want.num_tokens_per_rank, err_msg=path)
        np.testing.assert_array_equal(L.num_tokens_per_expert.cpu().numpy(),
                                      want.num_tokens_per_expert, err_msg=path)
        np.testing.assert_array_equal(L.recv_base.cpu().numpy(), want.recv_base, err_msg=path)
    P = want.num_rows
    d = ep.dispatch(x, idx, w, L, err=err)
    wd = oracle.dispatch(c.x_bits, c.topk_idx, c.topk_weights, E, R, want.slot, P)
    np.testing.assert_array_equal(bits_of(d.recv_x[:P]), wd.recv_x)
    if H % 128 == 0:
        d8 = ep.dispatch(x, idx, w, L, use_fp8=True, err=err)
        w8 = oracle.dispatch(c.x_bits, c.topk_idx, c.topk_weights, E, R, want.slot, P,
                             use_fp8=True)
        np.testing.assert_array_equal(d8.recv_x[:P].cpu().numpy(), w8.recv_x)
        np.testing.assert_array_equal(d8.recv_scales[:P].cpu().numpy().view(np.uint32),
                                      w8.recv_scales.view(np.uint32))
    y_bits = workloads.expert_outputs(max(P, 1), H, seed=cfg.seed + 11)
    y = bf16_from_bits(y_bits)
    out = ep.combine(y, idx, w, L, err=err)
    ref = oracle.combine(y_bits, c.topk_idx, c.topk_weights, E, R, want.slot)
    bound = combine_bound(oracle.bf16_to_double(y_bits), c.topk_idx, c.topk_weights, want.slot,
                          E // R, np.arange(T))
    assert_combine_close(bits_of(out), ref, bound)
    out_u = ep.combine(y, idx, None, L, err=err)
    ref_u = oracle.combine_ranksum(y_bits, want.slot)
    bound_u = np.zeros((T, H))
    for r in range(R):
        s = want.slot[:, r]
        bound_u[s >= 0] += np.abs(oracle.bf16_to_double(y_bits[s[s >= 0]]))
    assert_combine_close(bits_of(out_u), ref_u, bound_u)
    torch.cuda.synchronize()
    assert int(err.item()) == want.err_bits


@pytest.mark.parametrize("i", range(N_CASES))
def test_expert_major_random_shape(ep, i):
    cfg = random_config(i)
    check_expert_major(ep, cfg, make_case(cfg))


def check_expert_major(ep, cfg, c):
    """The expert-major layout, dispatch and combine on case c against the
    oracle, and the error bits."""
    T, H, K, E, R = cfg.num_tokens, cfg.hidden, cfg.num_topk, cfg.num_experts, cfg.num_ranks
    idx, w, x = device_inputs(c)
    # capacity: the largest count, so that the E * cap row buffers stay small
    cap = max(1, int(oracle.ll_layout(c.topk_idx, E, R, T).ll_count.max()))
    want = oracle.ll_layout(c.topk_idx, E, R, cap)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for path in _paths(ep.ll_single_launch_fits(T, K, R, E)):
        LL = ep.ll_get_dispatch_layout(idx, E, R, cap, err=err, path=path)
        np.testing.assert_array_equal(LL.ll_slot.cpu().numpy(), want.ll_slot, err_msg=path)
        np.testing.assert_array_equal(LL.ll_count.cpu().numpy(), want.ll_count, err_msg=path)
        np.testing.assert_array_equal(LL.ll_src_offset.cpu().numpy(), want.ll_src_offset,
                                      err_msg=path)
    slot = want.ll_slot
    live = slot >= 0
    d = ep.ll_dispatch(x, LL, err=err)
    if live.any():
        rows = torch.from_numpy(slot[live].astype(np.int64)).cuda()
        compact = np.full_like(slot, -1)
        compact[live] = np.arange(int(live.sum()), dtype=np.int32)
        wr, _, _ = oracle.ll_dispatch(c.x_bits, compact, int(live.sum()))
        np.testing.assert_array_equal(bits_of(d.recv_x[rows]), wr)
    y_bits = workloads.expert_outputs(E * cap, H, seed=cfg.seed + 13)
    out = ep.ll_combine(bf16_from_bits(y_bits), w, LL, err=err)
    ref = oracle.ll_combine(y_bits, c.topk_weights, slot)
    bound = np.zeros((T, H))
    for k in range(K):
        p = slot[:, k]
        ok = p >= 0
        bound[ok] += (np.abs(c.topk_weights[ok, k].astype(np.float64))[:, None]
                      * np.abs(oracle.bf16_to_double(y_bits[p[ok]])))
    assert_combine_close(bits_of(out), ref, bound)
    torch.cuda.synchronize()
    assert int(err.item()) == want.err_bits
