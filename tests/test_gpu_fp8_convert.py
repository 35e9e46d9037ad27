"""The FP8 dispatch's E4M3 conversion against the oracle's encoder on every
float32 bit pattern: 2^32 inputs, NaNs excluded (the format's handling of
NaN inputs is left open), infinities included.  The device side is the
dispatch's own conversion (round to nearest even, saturating to +-448),
reached through the library's ep_debug_e4m3_range hook; the oracle side is
the encoder written from the OCP E4M3 definition."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28  # bit patterns per launch (256 MB of codes)


def test_e4m3_conversion_on_every_float32(ep):
    out = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    n_checked = 0
    for first in range(0, 1 << 32, CHUNK):
        ep.debug_e4m3_range(first, out)
        got = out.cpu().numpy()
        bits = np.arange(CHUNK, dtype=np.uint32) + np.uint32(first)  # no wrap: first + CHUNK <= 2^32
        x = bits.view(np.float32)
        want = oracle.e4m3_from_float(x)
        ok = ~np.isnan(x)
        bad = np.flatnonzero((got != want) & ok)
        assert bad.size == 0, (
            f"{bad.size} mismatches from bit pattern {int(bits[bad[0]]):#010x}: "
            f"device {int(got[bad[0]]):#04x}, oracle {int(want[bad[0]]):#04x}")
        n_checked += int(ok.sum())
    assert n_checked == (1 << 32) - 2 * ((1 << 23) - 1)  # every non-NaN float32


def test_e4m3_range_hook_rejects_bad_ranges(ep):
    out = torch.empty(8, dtype=torch.uint8, device="cuda")
    with pytest.raises(ep.EPError):
        ep.debug_e4m3_range((1 << 32) - 4, out)  # would run past 2^32
    with pytest.raises(ep.EPError):
        ep.debug_e4m3_range(0, out[:6])  # not a multiple of 4
