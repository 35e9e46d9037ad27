"""Helpers shared by the GPU parity tests: moving seeded cases to the device,
bf16 bit views, cached full-size workloads and their oracle layouts, and the
combine tolerance."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from workloads import CONFIGS, Config, make_case

POISON_BF16 = 0xFFFF  # a NaN pattern that no dispatched bf16 row contains
POISON_U8 = 0xFF      # E4M3 NaN (never produced by the saturating cast)


def bf16_from_bits(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def device_inputs(case, device="cuda"):
    idx = torch.from_numpy(case.topk_idx).to(device)
    w = torch.from_numpy(case.topk_weights).to(device)
    x = bf16_from_bits(case.x_bits, device) if case.x_bits is not None else None
    return idx, w, x


@functools.lru_cache(maxsize=2)
def full_case(name: str):
    """A full-size workload and its oracle layout (cached: inputs are large)."""
    cfg = CONFIGS[name]
    c = make_case(cfg)
    L = oracle.layout(c.topk_idx, cfg.num_experts, cfg.num_ranks)
    return c, L


def sample_token_ranges(T: int, n: int = 64):
    """Start, middle (unaligned) and ragged end of the token range."""
    if T <= 3 * n:
        return [(0, T)]
    mid = T // 2 + 17
    return [(0, n), (mid, mid + n), (T - n + 5, T)]


def compact_slots(slot: np.ndarray, tokens: np.ndarray):
    """Renumber the rows of the sampled tokens 0..m-1 (same order as their
    original slots), -1 elsewhere.  Returns (slot_sub, orig_rows, compact_rows)."""
    sub = np.full_like(slot, -1)
    rows = slot[tokens]
    mask = rows >= 0
    orig = rows[mask]
    order = np.argsort(orig, kind="stable")
    compact = np.empty_like(orig)
    compact[order] = np.arange(orig.size, dtype=slot.dtype)
    tmp = np.full(rows.shape, -1, slot.dtype)
    tmp[mask] = compact
    sub[tokens] = tmp
    return sub, orig, compact


def combine_bound(y_f64: np.ndarray, topk_idx: np.ndarray, w: np.ndarray, slot: np.ndarray,
                  El: int, tokens: np.ndarray) -> np.ndarray:
    """sum_k |w_k * y_k| per (token, channel), for the combine tolerance."""
    H = y_f64.shape[1]
    out = np.zeros((tokens.size, H))
    for k in range(topk_idx.shape[1]):
        e = topk_idx[tokens, k]
        ok = (e >= 0) & (e < El * slot.shape[1])
        rows = slot[tokens[ok], e[ok] // El]
        out[ok] += np.abs(w[tokens[ok], k].astype(np.float64))[:, None] * np.abs(y_f64[rows])
    return out


def assert_combine_close(got_bits: np.ndarray, want_bits: np.ndarray, bound: np.ndarray,
                         rtol: float = 1e-2):
    """|g - r| <= rtol * (|r| + sum_k |w_k y_k|): 1e-2 relative, guarded
    against cancellation.  Returns (max relative error over |r| > 1e-3, fraction
    of bit-identical elements)."""
    g = oracle.bf16_to_double(got_bits)
    r = oracle.bf16_to_double(want_bits)
    assert np.isfinite(g).all()
    err = np.abs(g - r)
    lim = rtol * (np.abs(r) + bound)
    bad = err > lim
    assert not bad.any(), (f"{bad.sum()} elements out of tolerance; worst "
                           f"{(err - lim).max():.3e} at {np.unravel_index(np.argmax(err - lim), err.shape)}")
    big = np.abs(r) > 1e-3
    rel = float((err[big] / np.abs(r[big])).max()) if big.any() else 0.0
    return rel, float((got_bits == want_bits).mean())


def renormalised(case) -> np.ndarray:
    """Weights renormalised over the unmasked slots (sum to 1 where any slot is live)."""
    w = np.where(case.topk_idx >= 0, case.topk_weights.astype(np.float64), 0.0)
    s = w.sum(axis=1, keepdims=True)
    return np.where(s > 0, w / np.where(s > 0, s, 1.0), 0.0).astype(np.float32)


def small_configs():
    """Small, ragged and extreme shapes (the oracle finishes them in well under a second)."""
    specs = [  # name, R, T_r, H, E, K, routing, mask
        ("r1_k1", 1, 1000, 40, 3, 1, "uniform", 0.0),
        ("r2_tr1", 2, 1, 264, 4, 4, "uniform", 0.0),
        ("r3_zipf", 3, 7, 136, 6, 2, "zipf", 0.2),
        ("r5_mask", 5, 3, 8, 10, 3, "uniform", 0.3),
        ("r7_513", 7, 513, 72, 14, 3, "zipf", 0.05),
        ("r8_k8", 8, 33, 2056, 64, 8, "uniform", 0.1),
        ("r16_h4200", 16, 20, 4200, 64, 6, "zipf", 0.05),
        ("r32_dsv3ish", 32, 9, 7168, 256, 8, "uniform", 0.0),
        ("max_r64_k32", 64, 3, 128, 4096, 32, "uniform", 0.0),
        ("all_masked", 4, 5, 64, 8, 2, "uniform", 1.0),
    ]
    cfgs = [CONFIGS["tiny"]]
    for i, (name, R, Tr, H, E, K, routing, m) in enumerate(specs):
        cfgs.append(Config(name, R, Tr, H, E, K, routing=routing,
                           zipf_s=1.2 if routing == "zipf" else 0.0, mask_prob=m, seed=500 + i))
    return cfgs


def fp8_small_configs():
    specs = [("fp8_h128", 2, 5, 128, 4, 2), ("fp8_h384_r3", 3, 11, 384, 9, 3),
             ("fp8_h640_r32", 32, 2, 640, 256, 8), ("fp8_h7168_r4", 4, 40, 7168, 16, 4)]
    return [Config(n, R, Tr, H, E, K, fp8=True, seed=700 + i)
            for i, (n, R, Tr, H, E, K) in enumerate(specs)]
