"""FP8 round trip at the full decode workload (32 ranks x 128 tokens, H 7168,
top-8): dispatch quantises to E4M3 with per-128-channel scales, identity
experts dequantise (code x scale, rounded to bf16), and combine with weights
summing to one must give back x within the format's error bound.  Per
element: half an E4M3 ulp of x for normal codes (2^-4 relative), half the
subnormal step times the block scale (2^-10 x scale) below the normal range,
plus the two bf16 roundings (2^-9 relative each) on the way back; the test
allows 2^-4 + 2^-7 relative and 2^-9 x scale, which a wrong code, scale or
row (errors of the order of |x|) cannot meet."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from ep_testlib import device_inputs, full_case, renormalised
from workloads import CONFIGS

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("layout", ["ht", "ll"])
def test_fp8_round_trip_full_decode(ep, layout):
    cfg = CONFIGS["decode_fp8"]
    c, want = full_case("decode_fp8")
    T, H, E, R = cfg.num_tokens, cfg.hidden, cfg.num_experts, cfg.num_ranks
    idx, _, x = device_inputs(c)
    w = torch.from_numpy(renormalised(c)).cuda()
    nb = H // 128
    if layout == "ht":
        L = ep.get_dispatch_layout(idx, E, R)
        d = ep.dispatch(x, idx, w, L, use_fp8=True)
        rows = want.num_rows
    else:
        cap = int(np.bincount(c.topk_idx[c.topk_idx >= 0], minlength=E).max())
        L = ep.ll_get_dispatch_layout(idx, E, R, cap)
        d = ep.ll_dispatch(x, L, use_fp8=True)
        rows = L.num_rows
    codes = d.recv_x[:rows].view(torch.float8_e4m3fn).float().view(rows, nb, 128)
    scales = d.recv_scales[:rows]
    y = (codes * scales[:, :, None]).view(rows, H).to(torch.bfloat16)  # identity experts
    out = ep.ll_combine(y, w, L) if layout == "ll" else ep.combine(y, idx, w, L)
    torch.cuda.synchronize()
    # the block scales of each token (every destination row of a token holds
    # the same codes and scales): take them from the token's first row
    if layout == "ht":
        slot = L.slot.cpu().numpy()
    else:
        slot = L.ll_slot.cpu().numpy()
    first = np.array([s[s >= 0][0] for s in slot])  # decode has no masked slots
    tok_scale = scales[torch.from_numpy(first).cuda()]                   # [T, nb]
    xs = x.float().view(T, nb, 128)
    bound = (2.0 ** -4 + 2.0 ** -7) * xs.abs() + (2.0 ** -9) * tok_scale[:, :, None] + 1e-30
    diff = (out.float().view(T, nb, 128) - xs).abs()
    assert bool((diff <= bound).all()), float((diff - bound).max())
    # and the error is not trivially zero: E4M3 keeps 3 mantissa bits
    assert float(diff.max()) > 0
