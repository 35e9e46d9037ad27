"""GPU parity: ep_combine against the CPU oracle.

Tolerance (floating point, bf16 output of a float32 accumulation): per
element |g - r| <= 1e-2 * (|r| + sum_k |w_k y_k|), i.e. 1e-2 relative with a
guard for cancellation; r is the oracle's float64 sum rounded once to bf16.
Exact cases (one-hot weights, identity experts with weights summing to one)
are compared bit for bit."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from ep_testlib import (assert_combine_close, bf16_from_bits, bits_of, combine_bound,
                        compact_slots, device_inputs, full_case, renormalised,
                        sample_token_ranges, small_configs)
from workloads import CONFIGS, make_case

pytestmark = pytest.mark.gpu


def layout_of(ep, cfg, idx):
    L = ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks)
    return L, ep.total_rows(L)


@pytest.mark.parametrize("cfg", small_configs(), ids=lambda c: c.name)
def test_combine_random_outputs(ep, cfg):
    c = make_case(cfg, with_hidden=False)
    idx, _, _ = device_inputs(c)
    L, P = layout_of(ep, cfg, idx)
    y_bits = workloads.expert_outputs(max(P, 1), cfg.hidden, seed=cfg.seed + 1)
    rng = np.random.default_rng(cfg.seed + 2)
    w_np = (rng.standard_normal(c.topk_idx.shape)).astype(np.float32)  # signed weights
    y = bf16_from_bits(y_bits)
    w = torch.from_numpy(w_np).cuda()
    out = torch.full((cfg.num_tokens, cfg.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.combine(y, idx, w, L, err=err, out=out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    slot = L.slot.cpu().numpy()
    want = oracle.combine(y_bits, c.topk_idx, w_np, cfg.num_experts, cfg.num_ranks, slot)
    bound = combine_bound(oracle.bf16_to_double(y_bits), c.topk_idx, w_np, slot,
                          cfg.num_experts // cfg.num_ranks, np.arange(cfg.num_tokens))
    assert_combine_close(bits_of(out), want, bound)


def test_combine_one_hot_weights_bit_exact(ep):
    cfg = small_configs()[7]
    c = make_case(cfg, with_hidden=False)
    idx, _, _ = device_inputs(c)
    L, P = layout_of(ep, cfg, idx)
    y_bits = workloads.expert_outputs(P, cfg.hidden, seed=77)
    w_np = np.zeros_like(c.topk_weights)
    w_np[:, 0] = 1.0
    out = ep.combine(bf16_from_bits(y_bits), idx, torch.from_numpy(w_np).cuda(), L)
    want = oracle.combine(y_bits, c.topk_idx, w_np, cfg.num_experts, cfg.num_ranks,
                          L.slot.cpu().numpy())
    np.testing.assert_array_equal(bits_of(out), want)


@pytest.mark.parametrize("cfg", small_configs(), ids=lambda c: c.name)
def test_round_trip_identity_experts_small(ep, cfg):
    """combine(dispatch(x)) == x with identity experts and weights renormalised
    to sum to one ("combine diff=0"), compared as values; all-masked tokens give 0."""
    c = make_case(cfg)
    idx, _, x = device_inputs(c)
    w_np = renormalised(c)
    w = torch.from_numpy(w_np).cuda()
    L = ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks)
    d = ep.dispatch(x, idx, w, L)
    out = ep.combine(d.recv_x, idx, w, L)
    got = bits_of(out)
    live = (c.topk_idx >= 0).any(axis=1)
    # equal as values (a -0.0 in x returns as +0.0); masked tokens give +0
    np.testing.assert_array_equal(oracle.bf16_to_double(got[live]),
                                  oracle.bf16_to_double(c.x_bits[live]))
    assert (got[~live] == 0).all()


def test_combine_empty(ep):
    idx = torch.empty((0, 4), dtype=torch.int64, device="cuda")
    L = ep.get_dispatch_layout(idx, 16, 4)
    y = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    out = ep.combine(y, idx, torch.empty((0, 4), device="cuda"), L)
    assert out.shape == (0, 256)


def test_combine_out_of_range_ids_are_skipped_and_flagged(ep):
    cfg = CONFIGS["tiny"]
    c = make_case(cfg)
    idx_np = c.topk_idx.copy()
    idx_np[7, 2] = 999
    idx = torch.from_numpy(idx_np).cuda()
    w_np = c.topk_weights
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks, err=err)
    P = ep.total_rows(L)
    y_bits = workloads.expert_outputs(P, cfg.hidden, seed=5)
    out = ep.combine(bf16_from_bits(y_bits), idx, torch.from_numpy(w_np).cuda(), L, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ep.EP_ERRBIT_BAD_EXPERT
    slot = L.slot.cpu().numpy()
    want = oracle.combine(y_bits, idx_np, w_np, cfg.num_experts, cfg.num_ranks, slot)
    bound = combine_bound(oracle.bf16_to_double(y_bits), idx_np, w_np, slot, 4,
                          np.arange(cfg.num_tokens))
    assert_combine_close(bits_of(out), want, bound)


@pytest.mark.parametrize("name", list(CONFIGS))
def test_combine_full_size(ep, name):
    """Full-size workloads in the benchmark's launch configuration: layout ->
    dispatch -> combine with the expert outputs taken as the dispatched rows
    (identity experts; for FP8 dispatch, random bf16 expert outputs, since
    combine is bf16 in / bf16 out).  Sampled token ranges are compared with
    the oracle within the tolerance; with weights renormalised over the live
    slots every token must come back exactly (as values; bf16 workloads)."""
    cfg = CONFIGS[name]
    c, want_layout = full_case(name)
    idx, w, x = device_inputs(c)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks, err=err)
    d = ep.dispatch(x, idx, w, L, use_fp8=cfg.fp8, err=err)
    slot = L.slot.cpu().numpy()
    P = want_layout.num_rows
    if cfg.fp8:
        y_bits = workloads.expert_outputs(P, cfg.hidden, seed=cfg.seed + 10)
        y = bf16_from_bits(y_bits)
    else:
        y = d.recv_x
    out = ep.combine(y, idx, w, L, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    T = cfg.num_tokens
    El = cfg.num_experts // cfg.num_ranks
    for (a, b) in sample_token_ranges(T):
        toks = np.arange(a, b)
        sub, orig, compact = compact_slots(slot, toks)
        ysub = np.empty((orig.size, cfg.hidden), np.uint16)
        ysub[compact] = bits_of(y[torch.from_numpy(orig.astype(np.int64)).cuda()])
        want = oracle.combine(ysub, c.topk_idx, c.topk_weights, cfg.num_experts, cfg.num_ranks,
                              sub, t_range=(a, b))[a:b]
        bound = combine_bound(oracle.bf16_to_double(ysub), c.topk_idx, c.topk_weights, sub, El, toks)
        assert_combine_close(bits_of(out[a:b]), want, bound)
    if not cfg.fp8:
        wn = torch.from_numpy(renormalised(c)).cuda()
        out2 = ep.combine(d.recv_x, idx, wn, L)
        live = torch.from_numpy((c.topk_idx >= 0).any(axis=1)).cuda()
        # values, not bits: a -0.0 in x comes back as +0.0 (0 + w * -0 = +0)
        diff = (out2.float() != x.float()).any(dim=1) & live
        if bool(diff.any()):
            bad = torch.nonzero(diff).flatten().cpu().numpy()
            t = int(bad[0])
            rows = [int(s) for s in slot[t] if s >= 0]
            same = [bool(torch.equal(d.recv_x[r].view(torch.int16), x[t].view(torch.int16)))
                    for r in rows]
            ndiff = int((out2[t].float() != x[t].float()).sum())
            raise AssertionError(f"{bad.size} tokens differ (first {bad[:8].tolist()}); token {t}: "
                                 f"rows {rows} equal x: {same}; {ndiff} channels differ")
        assert not out2[~live].view(torch.int16).any()


@pytest.mark.parametrize("name", ["tiny", "dsv3_prefill", "decode_fp8", "skewed", "mixtral"])
def test_combine_full_batch_weighted_vs_oracle(ep, name):
    """Every token of a full-size workload against the oracle, under the
    workload's own (softmax, partly masked) weights and random expert outputs,
    so that each destination rank's row differs: a wrong row, or a wrong
    merge of the weights of slots that share a rank, shows up.  The oracle
    runs once over the whole batch; the tolerance is checked on the device in
    token chunks."""
    cfg = CONFIGS[name]
    c, want_layout = full_case(name)
    idx, w, _ = device_inputs(c)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks, err=err)
    P = want_layout.num_rows
    y_bits = workloads.signed_unit_bf16_bits(P, cfg.hidden, seed=cfg.seed + 40)
    y = bf16_from_bits(y_bits)
    out = torch.full((cfg.num_tokens, cfg.hidden), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    ep.combine(y, idx, w, L, err=err, out=out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    np.testing.assert_array_equal(L.slot.cpu().numpy(), want_layout.slot)
    want = oracle.combine(y_bits, c.topk_idx, c.topk_weights, cfg.num_experts, cfg.num_ranks,
                          want_layout.slot)
    del y_bits
    El = cfg.num_experts // cfg.num_ranks
    slot = L.slot.long()
    T, K = c.topk_idx.shape
    n_same = 0
    for a in range(0, T, 8192):
        b = min(T, a + 8192)
        # sum_k |w_k y_k| per element, for the tolerance's cancellation guard
        bound = torch.zeros((b - a, cfg.hidden), dtype=torch.float64, device="cuda")
        ar = torch.arange(b - a, device="cuda")
        for k in range(K):
            e = idx[a:b, k]
            live = (e >= 0) & (e < cfg.num_experts)
            rows = slot[a:b][ar, torch.where(live, e // El, 0)]
            term = w[a:b, k].double().abs()[:, None] * y[rows.clamp(min=0)].double().abs()
            bound += torch.where(live[:, None], term, 0.0)
        g = out[a:b].double()
        r_bits = torch.from_numpy(want[a:b].view(np.int16)).cuda()
        r = r_bits.view(torch.bfloat16).double()
        assert bool(torch.isfinite(g).all())
        excess = (g - r).abs() - 1e-2 * (r.abs() + bound)
        assert not bool((excess > 0).any()), (
            f"tokens [{a}, {b}): {int((excess > 0).sum())} elements out of tolerance, "
            f"worst excess {float(excess.max()):.3e}")
        n_same += int((out[a:b].view(torch.int16) == r_bits).sum())
    # float32 FMA against a float64 sum: nearly every element rounds the same
    assert n_same >= 0.9 * T * cfg.hidden


@pytest.mark.parametrize("cfg", small_configs()[:9] + [CONFIGS["tiny"]], ids=lambda c: c.name)
def test_combine_unweighted_rank_sum(ep, cfg):
    """topk_weights=None: each destination rank's row once (the high-throughput
    combine's rank sum), against the oracle within the tolerance."""
    c = make_case(cfg, with_hidden=False)
    idx, _, _ = device_inputs(c)
    L, P = layout_of(ep, cfg, idx)
    y_bits = workloads.expert_outputs(max(P, 1), cfg.hidden, seed=cfg.seed + 3)
    out = ep.combine(bf16_from_bits(y_bits), idx, None, L)
    torch.cuda.synchronize()
    slot = L.slot.cpu().numpy()
    want = oracle.combine_ranksum(y_bits, slot)
    yv = np.abs(oracle.bf16_to_double(y_bits))
    bound = np.zeros((cfg.num_tokens, cfg.hidden))
    for r in range(cfg.num_ranks):
        p = slot[:, r]
        bound[p >= 0] += yv[p[p >= 0]]
    assert_combine_close(bits_of(out), want, bound)


def test_combine_unweighted_full_skewed(ep):
    """Rank sum at full size (skewed workload, dispatched rows as expert
    outputs): every token against the oracle, the tolerance checked on the
    device in token chunks."""
    cfg = CONFIGS["skewed"]
    c, want_layout = full_case("skewed")
    idx, w, x = device_inputs(c)
    L = ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks)
    d = ep.dispatch(x, idx, w, L)
    out = ep.combine(d.recv_x, idx, None, L)
    torch.cuda.synchronize()
    P = want_layout.num_rows
    want = oracle.combine_ranksum(bits_of(d.recv_x[:P]), want_layout.slot)
    slot = L.slot.long()
    T = cfg.num_tokens
    for a in range(0, T, 2048):
        b = min(T, a + 2048)
        s = slot[a:b]
        rows = d.recv_x[s.clamp(min=0)].double().abs()  # [tokens, R, H]: 1 GB
        bound = torch.where((s >= 0)[:, :, None], rows, 0.0).sum(dim=1)
        g = out[a:b].double()
        r = torch.from_numpy(want[a:b].view(np.int16)).cuda().view(torch.bfloat16).double()
        assert bool(torch.isfinite(g).all())
        excess = (g - r).abs() - 1e-2 * (r.abs() + bound)
        assert not bool((excess > 0).any()), (
            f"tokens [{a}, {b}): {int((excess > 0).sum())} elements out of tolerance")


def test_combine_bounded_wait_reports_timeout_and_recovers(ep):
    """A pipeline unit that is never armed (test hook) makes the combine's
    bounded waits run out: the launch ends by itself with EP_ERRBIT_TIMEOUT in
    the error word, and the next combine on the same context is correct."""
    import time
    cfg = CONFIGS["tiny"]
    c = make_case(cfg)
    idx, w, x = device_inputs(c)
    L = ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks)
    d = ep.dispatch(x, idx, w, L)
    torch.cuda.synchronize()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.lib().ep_debug_set_combine_stall(0)
    t0 = time.time()
    ep.combine(d.recv_x, idx, w, L, err=err)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert int(err.item()) & ep.EP_ERRBIT_TIMEOUT
    assert elapsed < 10, elapsed
    # the launch that timed out still returned its scheduling counters to zero
    assert L.sched is not None and L.sched.tolist() == [0, 0]
    # the context is intact: a normal combine matches the oracle
    err.zero_()
    out = ep.combine(d.recv_x, idx, w, L, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    slot = L.slot.cpu().numpy()
    P = ep.total_rows(L)
    want = oracle.combine(bits_of(d.recv_x[:P]), c.topk_idx, c.topk_weights, cfg.num_experts,
                          cfg.num_ranks, slot)
    bound = combine_bound(oracle.bf16_to_double(bits_of(d.recv_x[:P])), c.topk_idx,
                          c.topk_weights, slot, cfg.num_experts // cfg.num_ranks,
                          np.arange(cfg.num_tokens))
    assert_combine_close(bits_of(out), want, bound)
