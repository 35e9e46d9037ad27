"""GPU parity: ep_dispatch against the CPU oracle, bit-exact on the
dispatched bytes (bf16 rows, or FP8 E4M3 codes and float32 scales) and the
per-row metadata; rows beyond P stay untouched (poisoned buffers)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from ep_testlib import (POISON_BF16, POISON_U8, bits_of, device_inputs, fp8_small_configs,
                        full_case, small_configs)
from workloads import CONFIGS, make_case

pytestmark = pytest.mark.gpu


def run_dispatch(ep, cfg, c, use_fp8, capacity=None):
    idx, w, x = device_inputs(c)
    L = ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks)
    P = ep.total_rows(L)
    cap = capacity if capacity is not None else P + 5
    out = ep.alloc_dispatched(cap + 3, cfg.hidden, cfg.num_topk, cfg.num_experts, cfg.num_ranks,
                              use_fp8, x.device)
    out.recv_x.view(torch.uint8).fill_(0xFF)
    if out.recv_scales is not None:
        out.recv_scales.fill_(float("nan"))
    out.recv_src_idx.fill_(-9)
    out.recv_topk_idx.fill_(-9)
    out.recv_topk_weights.fill_(float("nan"))
    out.num_recv_tokens_per_expert.fill_(-9)
    # pass a capacity smaller than the allocation to check nothing is written past it
    full = out
    view = ep.Dispatched(full.recv_x[:cap], None if full.recv_scales is None else full.recv_scales[:cap],
                         full.recv_src_idx[:cap], full.recv_topk_idx[:cap],
                         full.recv_topk_weights[:cap], full.num_recv_tokens_per_expert, use_fp8)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.dispatch(x, idx, w, L, use_fp8=use_fp8, err=err, out=view)
    torch.cuda.synchronize()
    return L, P, full, int(err.item())


def check_against_oracle(cfg, c, L, P, got, use_fp8, t_range=None, poison_tail=True):
    slot = L.slot.cpu().numpy()
    want_layout = oracle.layout(c.topk_idx, cfg.num_experts, cfg.num_ranks)
    np.testing.assert_array_equal(slot, want_layout.slot)
    want = oracle.dispatch(c.x_bits, c.topk_idx, c.topk_weights, cfg.num_experts, cfg.num_ranks,
                           slot, P, use_fp8=use_fp8)
    if use_fp8:
        np.testing.assert_array_equal(got.recv_x[:P].cpu().numpy(), want.recv_x)
        np.testing.assert_array_equal(got.recv_scales[:P].cpu().numpy().view(np.uint32),
                                      want.recv_scales.view(np.uint32))
    else:
        np.testing.assert_array_equal(bits_of(got.recv_x[:P]), want.recv_x)
    np.testing.assert_array_equal(got.recv_src_idx[:P].cpu().numpy(), want.recv_src_idx)
    np.testing.assert_array_equal(got.recv_topk_idx[:P].cpu().numpy(), want.recv_topk_idx)
    np.testing.assert_array_equal(got.recv_topk_weights[:P].cpu().numpy().view(np.uint32),
                                  want.recv_topk_weights.view(np.uint32))
    np.testing.assert_array_equal(
        got.num_recv_tokens_per_expert.cpu().numpy(),
        oracle.num_recv_tokens_per_expert(want_layout.num_tokens_per_expert, cfg.num_experts,
                                          cfg.num_ranks))
    if poison_tail:
        tail = got.recv_x[P:].contiguous().view(torch.uint8)
        assert bool((tail == 0xFF).all()), "rows past P were written"
        assert bool((got.recv_src_idx[P:] == -9).all())


@pytest.mark.parametrize("cfg", small_configs(), ids=lambda c: c.name)
def test_dispatch_bf16_small(ep, cfg):
    c = make_case(cfg)
    L, P, got, err = run_dispatch(ep, cfg, c, use_fp8=False)
    assert err == 0
    check_against_oracle(cfg, c, L, P, got, use_fp8=False)


@pytest.mark.parametrize("cfg", fp8_small_configs(), ids=lambda c: c.name)
def test_dispatch_fp8_small(ep, cfg):
    c = make_case(cfg)
    L, P, got, err = run_dispatch(ep, cfg, c, use_fp8=True)
    assert err == 0
    check_against_oracle(cfg, c, L, P, got, use_fp8=True)


def test_dispatch_fp8_block_extremes(ep):
    """Blocks whose amax sits below the 1e-4 floor, all-zero and negative-zero
    blocks, ties at E4M3 midpoints, and the largest bf16 magnitudes."""
    cfg = fp8_small_configs()[1]
    c = make_case(cfg)
    x = c.x_bits.copy()
    x[0, :128] = 0                              # all zero
    x[1, :128] = 0x8000                         # all negative zero
    x[2, 128:256] = 0x3800 | (np.arange(128) & 0x7F)  # ~1e-5 magnitudes: below the floor
    x[3, :128] = 0x7F7F                         # largest finite bf16
    x[3, 5] = 0xFF7F
    x[4, 256:384] = (np.arange(128, dtype=np.uint16) * 37) & 0x7FFF  # every exponent
    x[5, :] = 0x3F80                            # ones: exact codes
    c.x_bits = x
    L, P, got, err = run_dispatch(ep, cfg, c, use_fp8=True)
    assert err == 0
    check_against_oracle(cfg, c, L, P, got, use_fp8=True)


def test_dispatch_fp8_full_decode(ep):
    """The 32-rank x 128-token FP8 decode workload, every row compared."""
    cfg = CONFIGS["decode_fp8"]
    c, _ = full_case("decode_fp8")
    L, P, got, err = run_dispatch(ep, cfg, c, use_fp8=True)
    assert err == 0
    check_against_oracle(cfg, c, L, P, got, use_fp8=True)


def test_dispatch_capacity_overflow(ep):
    cfg = small_configs()[6]
    c = make_case(cfg)
    idx, w, x = device_inputs(c)
    L = ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks)
    P = ep.total_rows(L)
    cap = P // 2
    buf = torch.full((P, cfg.hidden), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    src = torch.full((P,), -9, dtype=torch.int32, device="cuda")
    out = ep.Dispatched(buf[:cap], None, src[:cap], torch.empty((cap, cfg.num_topk), dtype=torch.int64, device="cuda"),
                        torch.empty((cap, cfg.num_topk), device="cuda"),
                        torch.empty((cfg.num_ranks, cfg.num_experts // cfg.num_ranks), dtype=torch.int32, device="cuda"), False)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.dispatch(x, idx, w, L, err=err, out=out)
    torch.cuda.synchronize()
    assert int(err.item()) & ep.EP_ERRBIT_CAPACITY
    want = oracle.dispatch(c.x_bits, c.topk_idx, c.topk_weights, cfg.num_experts, cfg.num_ranks,
                           L.slot.cpu().numpy(), P)
    np.testing.assert_array_equal(bits_of(buf[:cap]), want.recv_x[:cap])
    assert bool((buf[cap:].view(torch.int16) == -1).all())
    assert bool((src[cap:] == -9).all())


def test_dispatch_empty(ep):
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((0, 4), dtype=torch.int64, device="cuda")
    w = torch.empty((0, 4), dtype=torch.float32, device="cuda")
    L = ep.get_dispatch_layout(idx, 16, 4)
    out = ep.dispatch(x, idx, w, L, capacity=0)
    torch.cuda.synchronize()
    assert not out.num_recv_tokens_per_expert.any()


def test_dispatch_with_no_receive_rows(ep):
    """Tokens whose slots are all masked, into buffers of no rows (NULL
    pointers): every dispatch entry point writes nothing and reports nothing
    (a shard whose tokens all go nowhere has such an empty send buffer); one
    live slot with no rows to hold it sets the capacity bit."""
    T, H, K, E, R = 64, 256, 2, 8, 4
    idx = torch.full((T, K), -1, dtype=torch.int64, device="cuda")
    w = torch.rand((T, K), device="cuda")
    x = torch.randn((T, H), device="cuda").to(torch.bfloat16)
    for fp8 in (False, True):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        L = ep.get_dispatch_layout(idx, E, R)
        d = ep.dispatch(x, idx, w, L, use_fp8=fp8, capacity=0, err=err)
        assert d.recv_x.data_ptr() == 0
        L2, d2 = ep.layout_dispatch(x, idx, w, E, R, use_fp8=fp8, capacity=0, err=err)
        LL = ep.ll_get_dispatch_layout(idx, E, R, 0, err=err)
        dl = ep.ll_dispatch(x, LL, use_fp8=fp8, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, fp8
        assert dl.recv_x.shape[0] == 0 and d2.recv_x.shape[0] == 0
        assert not d.num_recv_tokens_per_expert.any() and not d2.num_recv_tokens_per_expert.any()
        assert not L2.num_tokens_per_rank.any()
    idx[5, 0] = 3
    L = ep.get_dispatch_layout(idx, E, R)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.dispatch(x, idx, w, L, capacity=0, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == ep.EP_ERRBIT_CAPACITY


@pytest.mark.parametrize("name", ["tiny", "dsv3_prefill", "skewed", "mixtral"])
def test_dispatch_bf16_full_size(ep, name):
    """Full-size bf16 workloads in the benchmark's launch configuration
    (worst-case capacity T*min(K,R), no synchronisation between the calls):
    every (token, rank) row is checked against the token on the device, and
    the whole receive buffer and its metadata against the oracle."""
    cfg = CONFIGS[name]
    c, want_layout = full_case(name)
    idx, w, x = device_inputs(c)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = ep.get_dispatch_layout(idx, cfg.num_experts, cfg.num_ranks, err=err)
    out = ep.dispatch(x, idx, w, L, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    slot = L.slot.cpu().numpy()
    np.testing.assert_array_equal(slot, want_layout.slot)
    P = want_layout.num_rows
    # property over every pair, on the device, in chunks
    slot_d = L.slot
    T, R = slot_d.shape
    step = max(1, (1 << 28) // (cfg.hidden * 2 * R))
    for t0 in range(0, T, step):
        s = slot_d[t0:t0 + step]
        tok, r = torch.nonzero(s >= 0, as_tuple=True)
        rows = s[tok, r].long()
        assert torch.equal(out.recv_x[rows].view(torch.int16), x[t0 + tok].view(torch.int16))
        assert torch.equal(out.recv_src_idx[rows], (t0 + tok).int())
    # the whole batch against the oracle
    assert P <= out.recv_x.shape[0]
    want = oracle.dispatch(c.x_bits, c.topk_idx, c.topk_weights, cfg.num_experts,
                           cfg.num_ranks, slot, P)
    assert np.array_equal(bits_of(out.recv_x[:P]), want.recv_x)
    assert np.array_equal(out.recv_src_idx[:P].cpu().numpy(), want.recv_src_idx)
    assert np.array_equal(out.recv_topk_idx[:P].cpu().numpy(), want.recv_topk_idx)
    assert np.array_equal(out.recv_topk_weights[:P].cpu().numpy().view(np.uint32),
                          want.recv_topk_weights.view(np.uint32))


def test_dispatch_fp8_every_bf16_value(ep):
    """Every finite bf16 value with |x| <= 448 quantised by the device: each
    128-channel block holds +448 (so amax = 448 and the multiplier 448/a is
    exactly 1) and 127 of the values.  The device's E4M3 codes must equal the
    oracle's for all of them, ties at E4M3 midpoints, zeros and subnormals
    included."""
    from workloads import Config
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_to_double(codes)
    keep = np.isfinite(vals) & (np.abs(vals) <= 448.0)
    pats = codes[keep]
    per_block = 127
    nblk = -(-pats.size // per_block)
    blocks = np.zeros((nblk, 128), np.uint16)
    blocks[:, 0] = 0x43E0  # +448.0
    flat = np.full(nblk * per_block, 0x3F80, np.uint16)  # pad with 1.0
    flat[:pats.size] = pats
    blocks[:, 1:] = flat.reshape(nblk, per_block)
    H = 1024
    T = -(-nblk * 128 // H)
    x_bits = np.full(T * H, 0x3F80, np.uint16)
    x_bits[:blocks.size] = blocks.ravel()
    x_bits = x_bits.reshape(T, H)
    # route every token to expert 0 of a single rank
    cfg = Config("fp8_all_bf16", 1, T, H, 1, 1, fp8=True, seed=0)
    c = make_case(cfg)
    c.x_bits = x_bits
    c.topk_idx[:] = 0
    L, P, got, err = run_dispatch(ep, cfg, c, use_fp8=True)
    assert err == 0 and P == T
    check_against_oracle(cfg, c, L, P, got, use_fp8=True)
    # and the blocks with amax 448 have scale exactly 1
    assert bool((got.recv_scales[:P].reshape(-1)[:nblk] == 1.0).all())
