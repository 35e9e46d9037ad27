"""GPU parity of the low-latency (expert-major) path against the CPU oracle:
ep_ll_get_dispatch_layout (bit-exact, on both kernel paths: multi-launch and
one thread-block cluster), ep_ll_dispatch (bit-exact bf16 rows, E4M3 codes
and scales) and ep_ll_combine (the combine tolerance; exact for the identity
round trip)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from ep_testlib import assert_combine_close, bf16_from_bits, bits_of, device_inputs, full_case
from workloads import CONFIGS, Config, make_case

pytestmark = pytest.mark.gpu


def ll_cases():
    return [CONFIGS["tiny"],
            Config("ll_r3_zipf", 3, 7, 136, 9, 3, routing="zipf", zipf_s=1.2, mask_prob=0.2, seed=801),
            Config("ll_r8_k8", 8, 33, 264, 64, 8, mask_prob=0.1, seed=802),
            Config("ll_r1", 1, 300, 40, 5, 2, routing="zipf", zipf_s=1.2, seed=803),
            Config("ll_r32", 32, 5, 128, 256, 8, seed=804),
            Config("ll_k32", 4, 9, 64, 64, 32, seed=805)]


def compare_ll_layout(L, want, check_offsets=True):
    np.testing.assert_array_equal(L.ll_slot.cpu().numpy(), want.ll_slot)
    np.testing.assert_array_equal(L.ll_count.cpu().numpy(), want.ll_count)
    if check_offsets:
        np.testing.assert_array_equal(L.ll_src_offset.cpu().numpy(), want.ll_src_offset)


PATHS = ["multi", "single"]


def ll_layout_on(ep, idx, E, R, path, cap=None, err=None):
    """The expert-major layout on the given path with poisoned outputs; None
    (after checking that the call is refused on the host) when the
    single-launch form does not take this batch."""
    T, K = idx.shape
    L = ep.alloc_ll_layout(T, K, E, R, T if cap is None else cap, idx.device)
    L.ll_slot.fill_(-7)
    L.ll_count.fill_(-7)
    L.ll_src_offset.fill_(-7)
    if path == "single" and not ep.ll_single_launch_fits(T, K, R, E):
        with pytest.raises(ep.EPError):
            ep.ll_get_dispatch_layout(idx, E, R, err=err, out=L, path=path)
        return None
    ep.ll_get_dispatch_layout(idx, E, R, err=err, out=L, path=path)
    return L


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("cfg", ll_cases(), ids=lambda c: c.name)
def test_ll_layout_small(ep, cfg, path):
    c = make_case(cfg, with_hidden=False)
    idx, _, _ = device_inputs(c)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = ll_layout_on(ep, idx, cfg.num_experts, cfg.num_ranks, path, err=err)
    if L is None:
        return
    compare_ll_layout(L, oracle.ll_layout(c.topk_idx, cfg.num_experts, cfg.num_ranks,
                                          cfg.num_tokens))
    assert int(err.item()) == 0


def ll_single_launch_cases():
    """Shapes aimed at the single-launch form: many warps per source, ragged
    last warps, one-token sources, 2048-slot warps, E = 1024, K = 32, a tight
    capacity."""
    specs = [  # name, R, T_r, E, K, routing, mask
        ("lls_r3_ragged", 3, 1000, 12, 4, "zipf", 0.05),
        ("lls_r64_tr1", 64, 1, 128, 8, "uniform", 0.0),
        ("lls_r1_2048slots", 1, 8192, 16, 16, "zipf", 0.1),
        ("lls_r8_e1024", 8, 300, 1024, 8, "uniform", 0.0),
        ("lls_r5_k32", 5, 77, 40, 32, "uniform", 0.3),
        ("lls_r32_decodeish", 32, 100, 256, 8, "zipf", 0.0),
    ]
    return [Config(n, R, Tr, 8, E, K, routing=rt, zipf_s=1.2 if rt == "zipf" else 0.0,
                   mask_prob=m, seed=970 + i)
            for i, (n, R, Tr, E, K, rt, m) in enumerate(specs)]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("cfg", ll_single_launch_cases(), ids=lambda c: c.name)
def test_ll_layout_single_launch_shapes(ep, cfg, path):
    T, K, R, E = cfg.num_tokens, cfg.num_topk, cfg.num_ranks, cfg.num_experts
    assert ep.ll_single_launch_fits(T, K, R, E)
    c = make_case(cfg, with_hidden=False)
    idx, _, _ = device_inputs(c)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = ll_layout_on(ep, idx, E, R, path, err=err)
    compare_ll_layout(L, oracle.ll_layout(c.topk_idx, E, R, T))
    assert int(err.item()) == 0
    # a capacity below the largest count drops rows and flags it, identically
    cnt = oracle.ll_layout(c.topk_idx, E, R, T).ll_count
    cap = max(1, int(cnt.max()) // 2)
    err.zero_()
    L = ll_layout_on(ep, idx, E, R, path, cap=cap, err=err)
    want = oracle.ll_layout(c.topk_idx, E, R, cap)
    compare_ll_layout(L, want)
    assert int(err.item()) == want.err_bits


@pytest.mark.parametrize("path", PATHS)
def test_ll_layout_duplicates_bad_ids_and_capacity(ep, path):
    idx_np = np.array([[2, 2, 0], [1, 2, -1], [2, 0, 2], [-1, -1, -1], [9, 1, -4], [2, 2, 2]],
                      np.int64)
    idx = torch.from_numpy(idx_np).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = ll_layout_on(ep, idx, 3, 1, path, cap=3, err=err)
    want = oracle.ll_layout(idx_np, 3, 1, 3)
    assert want.err_bits == 3
    compare_ll_layout(L, want)
    assert int(err.item()) & ep.EP_ERRBIT_BAD_EXPERT and int(err.item()) & ep.EP_ERRBIT_CAPACITY


@pytest.mark.parametrize("path", ["auto"] + PATHS)
@pytest.mark.parametrize("name", ["decode_fp8", "skewed"])
def test_ll_layout_full_size(ep, name, path):
    cfg = CONFIGS[name]
    c, _ = full_case(name)
    idx = torch.from_numpy(c.topk_idx).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = ll_layout_on(ep, idx, cfg.num_experts, cfg.num_ranks, path, err=err)
    if L is None:
        return
    compare_ll_layout(L, oracle.ll_layout(c.topk_idx, cfg.num_experts, cfg.num_ranks,
                                          cfg.num_tokens))
    assert int(err.item()) == 0


def _dispatch_and_check(ep, cfg, c, use_fp8, cap=None):
    idx, _, x = device_inputs(c)
    E, R, T = cfg.num_experts, cfg.num_ranks, cfg.num_tokens
    want_layout = oracle.ll_layout(c.topk_idx, E, R, T)
    cap = cap or max(1, int(want_layout.ll_count.max()))
    L = ep.ll_get_dispatch_layout(idx, E, R, cap)
    if use_fp8:  # poisoned buffers: 0xFF codes / NaN scales / -9 sources
        recv = torch.full((E * cap, cfg.hidden), 0xFF, dtype=torch.uint8, device="cuda")
        scales = torch.full((E * cap, cfg.hidden // 128), float("nan"), device="cuda")
    else:
        recv = torch.full((E * cap, cfg.hidden), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        scales = None
    out = ep.LLDispatched(recv, scales, torch.full((E * cap,), -9, dtype=torch.int32, device="cuda"),
                          use_fp8)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ll_dispatch(x, L, use_fp8=use_fp8, err=err, out=out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    slot = L.ll_slot.cpu().numpy()
    want_slot = oracle.ll_layout(c.topk_idx, E, R, cap).ll_slot
    np.testing.assert_array_equal(slot, want_slot)
    # the oracle on compactly renumbered rows
    live = slot >= 0
    rows = slot[live]
    compact = np.full_like(slot, -1)
    compact[live] = np.arange(rows.size, dtype=np.int32)
    recv, scales, src = oracle.ll_dispatch(c.x_bits, compact, rows.size, use_fp8=use_fp8)
    r = torch.from_numpy(rows.astype(np.int64)).cuda()
    if use_fp8:
        np.testing.assert_array_equal(out.recv_x[r].cpu().numpy(), recv)
        np.testing.assert_array_equal(out.recv_scales[r].cpu().numpy().view(np.uint32),
                                      scales.view(np.uint32))
    else:
        np.testing.assert_array_equal(bits_of(out.recv_x[r]), recv)
    np.testing.assert_array_equal(out.recv_src_idx[r].cpu().numpy(), src)
    # rows nobody names stay untouched
    untouched = torch.ones(E * cap, dtype=torch.bool, device="cuda")
    untouched[r] = False
    assert bool((out.recv_src_idx[untouched] == -9).all())
    return L, out


@pytest.mark.parametrize("cfg", ll_cases()[:5], ids=lambda c: c.name)
def test_ll_dispatch_bf16(ep, cfg):
    _dispatch_and_check(ep, cfg, make_case(cfg), use_fp8=False)


@pytest.mark.parametrize("cfg", [Config("llf_h128", 2, 9, 128, 4, 2, seed=811),
                                 Config("llf_h384", 3, 5, 384, 9, 3, mask_prob=0.2, seed=812),
                                 Config("llf_r32", 32, 3, 7168, 256, 8, seed=813)],
                         ids=lambda c: c.name)
def test_ll_dispatch_fp8(ep, cfg):
    _dispatch_and_check(ep, cfg, make_case(cfg), use_fp8=True)


def test_ll_dispatch_fp8_full_decode(ep):
    cfg = CONFIGS["decode_fp8"]
    c, _ = full_case("decode_fp8")
    _dispatch_and_check(ep, cfg, c, use_fp8=True)


def test_ll_dispatch_capacity_overflow(ep):
    cfg = ll_cases()[2]
    c = make_case(cfg)
    idx, _, x = device_inputs(c)
    E = cfg.num_experts
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = ep.ll_get_dispatch_layout(idx, E, cfg.num_ranks, 2, err=err)  # two rows per expert
    out = ep.ll_dispatch(x, L, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ep.EP_ERRBIT_CAPACITY
    want = oracle.ll_layout(c.topk_idx, E, cfg.num_ranks, 2)
    np.testing.assert_array_equal(L.ll_slot.cpu().numpy(), want.ll_slot)
    for t, k in zip(*np.nonzero(want.ll_slot >= 0)):
        assert np.array_equal(bits_of(out.recv_x[int(want.ll_slot[t, k])]), c.x_bits[t])


@pytest.mark.parametrize("cfg", ll_cases(), ids=lambda c: c.name)
@pytest.mark.parametrize("weighted", [True, False])
def test_ll_combine(ep, cfg, weighted):
    c = make_case(cfg, with_hidden=False)
    idx, w, _ = device_inputs(c)
    E, R, T = cfg.num_experts, cfg.num_ranks, cfg.num_tokens
    L = ep.ll_get_dispatch_layout(idx, E, R)
    y_bits = workloads.expert_outputs(E * T, cfg.hidden, seed=cfg.seed + 5)
    out = ep.ll_combine(bf16_from_bits(y_bits), w if weighted else None, L)
    torch.cuda.synchronize()
    slot = L.ll_slot.cpu().numpy()
    wn = c.topk_weights if weighted else None
    want = oracle.ll_combine(y_bits, wn, slot)
    yv = np.abs(oracle.bf16_to_double(y_bits))
    bound = np.zeros((T, cfg.hidden))
    for k in range(cfg.num_topk):
        p = slot[:, k]
        wk = np.abs(c.topk_weights[:, k]).astype(np.float64) if weighted else np.ones(T)
        bound[p >= 0] += wk[p >= 0, None] * yv[p[p >= 0]]
    assert_combine_close(bits_of(out), want, bound)


@pytest.mark.parametrize("name", ["decode_fp8", "tiny"])
def test_ll_round_trip_identity(ep, name):
    """ll_combine(ll_dispatch(x)) == x (as values) with weights summing to one."""
    cfg = CONFIGS[name]
    c, want_layout = full_case(name) if name == "decode_fp8" else (make_case(cfg), None)
    idx, _, x = device_inputs(c)
    w = c.topk_weights.astype(np.float64)
    w = np.where(c.topk_idx >= 0, w, 0.0)
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    E, R = cfg.num_experts, cfg.num_ranks
    cnt = oracle.ll_layout(c.topk_idx, E, R, cfg.num_tokens).ll_count
    L = ep.ll_get_dispatch_layout(idx, E, R, int(cnt.max()))
    d = ep.ll_dispatch(x, L)
    out = ep.ll_combine(d.recv_x, torch.from_numpy(w).cuda(), L)
    assert torch.equal(out.float(), x.float())
