"""The largest batch the rank-major entry points take: 64 ranks and
T = 2^25 - 64 tokens, so that T * R sits just below the 2^31 limit of the
slot matrix (about 63 million receive rows).  Every offset past 2^31 bytes
or elements must be 64-bit; this run compares the whole layout and the whole
dispatch with the oracle, the unweighted combine over every token, and the
weighted combine on the first, middle and last 65536 tokens.  Rows are one
16-byte vector (H = 8) to keep the buffers to about 15 GB on the device."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from ep_testlib import assert_combine_close, bits_of, combine_bound

pytestmark = pytest.mark.gpu


def test_largest_batch_the_api_takes(ep):
    R, E, K, H = 64, 64, 2, 8
    T = (1 << 25) - 64  # T * R < 2^31, T % R == 0
    assert T * R < (1 << 31) and T % R == 0
    rng = np.random.default_rng(31)
    idx_h = rng.integers(0, E, (T, K), dtype=np.int64)
    idx_h[rng.random((T, K)) < 0.05] = -1
    w_h = rng.random((T, K), dtype=np.float32)
    x_bits = rng.integers(0, 1 << 16, (T, H), dtype=np.uint16) & np.uint16(0xBFFF)  # finite
    idx = torch.from_numpy(idx_h).cuda()
    w = torch.from_numpy(w_h).cuda()
    x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    want = oracle.layout(idx_h, E, R)
    P = want.num_rows
    L = ep.get_dispatch_layout(idx, E, R, err=err)
    assert ep.total_rows(L) == P
    assert np.array_equal(L.num_tokens_per_rank.cpu().numpy(), want.num_tokens_per_rank)
    assert np.array_equal(L.num_tokens_per_expert.cpu().numpy(), want.num_tokens_per_expert)
    assert np.array_equal(L.recv_base.cpu().numpy(), want.recv_base)
    assert np.array_equal(L.slot.cpu().numpy(), want.slot)
    assert np.array_equal(L.is_token_in_rank.view(torch.uint8).cpu().numpy(),
                          want.is_token_in_rank)
    slot = want.slot
    del want

    d = ep.dispatch(x, idx, w, L, capacity=P, err=err)
    wd = oracle.dispatch(x_bits, idx_h, w_h, E, R, slot, P)
    assert np.array_equal(bits_of(d.recv_x), wd.recv_x)
    assert np.array_equal(d.recv_src_idx.cpu().numpy(), wd.recv_src_idx)
    assert np.array_equal(d.recv_topk_idx.cpu().numpy(), wd.recv_topk_idx)
    assert np.array_equal(d.recv_topk_weights.cpu().numpy().view(np.uint32),
                          wd.recv_topk_weights.view(np.uint32))
    del wd

    y = d.recv_x  # identity experts
    out_u = ep.combine(y, idx, None, L, err=err)
    y_bits = bits_of(y)
    assert np.array_equal(bits_of(out_u), oracle.combine_ranksum(y_bits, slot))
    out = bits_of(ep.combine(y, idx, w, L, err=err))
    for a in (0, T // 2, T - 65536):
        b = a + 65536
        ref = oracle.combine(y_bits, idx_h, w_h, E, R, slot, t_range=(a, b))[a:b]
        # the tolerance's sum_k |w_k y_k| over the window's own rows only
        win = slot[a:b]
        rows = np.unique(win[win >= 0])
        local = np.full_like(win, -1)
        local[win >= 0] = np.searchsorted(rows, win[win >= 0])
        y_f64 = oracle.bf16_to_double(y_bits[rows])
        bound = combine_bound(y_f64, idx_h[a:b], w_h[a:b], local, E // R, np.arange(b - a))
        assert_combine_close(out[a:b], ref, bound)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


@pytest.mark.parametrize("H", [16384, 65528, 131072])
def test_wide_rows(ep, H):
    """Rows far wider than any workload's (up to 256 KB of bf16): many
    chunks per row in the combine, many rounds per warp in the dispatch; FP8
    where H % 128 == 0."""
    from test_gpu_random import check_expert_major, check_rank_major
    from workloads import Config, make_case
    cfg = Config(f"wide_h{H}", 4, 16, H, 8, 3, routing="zipf", zipf_s=1.2, mask_prob=0.1,
                 seed=9700 + H % 97)
    c = make_case(cfg)
    check_rank_major(ep, cfg, c)
    check_expert_major(ep, cfg, c)
