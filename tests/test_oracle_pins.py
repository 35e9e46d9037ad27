"""Pins for the CPU oracle: each check compares it against something other than
itself (brute force written differently, a library routine, a closed form, an
invariant, or values fixed by a number format's definition).

Sources: "[Not ready] MSCCLPP EP implementation" (mscclpp pull request 852):
section "Scope" (get_dispatch_layout / intranode_dispatch / intranode_combine
ported from DeepEP), the intranode validation commit (every rank recovers its
tokens, "combine diff=0"), the internode-combine commit (receiver-side prefix
matrices), and the low-latency port (dispatch<kUseFP8,...>).
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import Config, CONFIGS, make_case


# --------------------------------------------------------------------------
# brute-force layout: builds each destination's receive list directly, by
# walking destinations, then source ranks, then tokens, and handing out rows
# in that order (a different route to the same definition).
# --------------------------------------------------------------------------
def brute_layout(topk_idx, E, R):
    T, K = topk_idx.shape
    El, Tr = E // R, T // R
    members = [set() for _ in range(T)]
    per_expert = [[0] * E for _ in range(R)]
    bad = 0
    for t in range(T):
        for k in range(K):
            e = int(topk_idx[t, k])
            if e == -1:
                continue
            if not (0 <= e < E):
                bad = 1
                continue
            members[t].add(e // El)
            per_expert[t // Tr][e] += 1
    slot = [[-1] * R for _ in range(T)]
    row = 0
    base = [0]
    for r in range(R):
        for s in range(R):
            for t in range(s * Tr, (s + 1) * Tr):
                if r in members[t]:
                    slot[t][r] = row
                    row += 1
        base.append(row)
    per_rank = [[sum(1 for t in range(s * Tr, (s + 1) * Tr) if r in members[t])
                 for r in range(R)] for s in range(R)]
    itr = [[1 if r in members[t] else 0 for r in range(R)] for t in range(T)]
    return dict(slot=np.array(slot, np.int32).reshape(T, R),
                itr=np.array(itr, np.uint8).reshape(T, R),
                per_rank=np.array(per_rank, np.int32).reshape(R, R),
                per_expert=np.array(per_expert, np.int32).reshape(R, E),
                base=np.array(base, np.int32), bad=bad)


def small_cases():
    cases = [CONFIGS["tiny"]]
    specs = [  # (R, T_r, E, K, routing, mask)
        (1, 5, 3, 2, "uniform", 0.0), (2, 1, 4, 4, "uniform", 0.0),
        (3, 7, 6, 2, "zipf", 0.2), (5, 3, 10, 3, "uniform", 0.3),
        (4, 9, 8, 1, "zipf", 0.0), (8, 4, 64, 8, "uniform", 0.1),
        (2, 33, 2, 2, "uniform", 0.5), (6, 2, 12, 5, "zipf", 1.0),
    ]
    for i, (R, Tr, E, K, routing, m) in enumerate(specs):
        cases.append(Config(f"small{i}", R, Tr, 16, E, K, routing=routing,
                            zipf_s=1.2 if routing == "zipf" else 0.0, mask_prob=m,
                            seed=100 + i))
    return cases


@pytest.mark.parametrize("cfg", small_cases(), ids=lambda c: c.name)
def test_layout_matches_brute_force(cfg):
    c = make_case(cfg, with_hidden=False)
    E, R = cfg.num_experts, cfg.num_ranks
    got = oracle.layout(c.topk_idx, E, R)
    want = brute_layout(c.topk_idx, E, R)
    np.testing.assert_array_equal(got.slot, want["slot"])
    np.testing.assert_array_equal(got.is_token_in_rank, want["itr"])
    np.testing.assert_array_equal(got.num_tokens_per_rank, want["per_rank"])
    np.testing.assert_array_equal(got.num_tokens_per_expert, want["per_expert"])
    np.testing.assert_array_equal(got.recv_base, want["base"])
    assert got.err_bits == want["bad"] == 0


def test_layout_bad_ids_and_duplicates():
    # Out-of-range ids are ignored and flagged; a duplicated expert counts
    # twice per expert but once for membership.
    idx = np.array([[0, 0, -1], [5, 1, 9], [-7, 2, 3], [3, 3, 3]], np.int64)
    got = oracle.layout(idx, 4, 2)
    want = brute_layout(idx, 4, 2)
    np.testing.assert_array_equal(got.slot, want["slot"])
    np.testing.assert_array_equal(got.num_tokens_per_expert, want["per_expert"])
    assert got.err_bits == 1 and want["bad"] == 1
    assert got.num_tokens_per_expert[0, 0] == 2 and got.num_tokens_per_expert[1, 3] == 4


def test_layout_empty():
    got = oracle.layout(np.zeros((0, 3), np.int64), 8, 4)
    assert got.num_rows == 0 and got.slot.shape == (0, 4)
    assert not got.num_tokens_per_rank.any() and not got.num_tokens_per_expert.any()


def _layout_invariants(cfg, c, L):
    T, R, E, K = cfg.num_tokens, cfg.num_ranks, cfg.num_experts, cfg.num_topk
    El, Tr = E // R, T // R
    idx = c.topk_idx
    valid = idx >= 0
    ranks = np.where(valid, idx // El, -1)
    member = np.zeros((T, R), bool)
    for k in range(K):
        ok = ranks[:, k] >= 0
        member[np.nonzero(ok)[0], ranks[ok, k]] = True
    # per-rank counts sum to the number of unique (token, rank) pairs of each source
    pairs_per_src = member.reshape(R, Tr, R).sum(axis=(1, 2))
    assert (L.num_tokens_per_rank.sum(axis=1) == pairs_per_src).all()
    # per-expert counts sum to the number of unmasked top-k slots
    assert L.num_tokens_per_expert.sum() == valid.sum()
    assert (L.num_tokens_per_expert.sum(axis=1) == valid.reshape(R, Tr * K).sum(axis=1)).all()
    # slot is a bijection from in-rank pairs onto [0, P)
    P = L.num_rows
    s = L.slot[L.slot >= 0]
    assert P == member.sum() == s.size
    assert np.array_equal(np.sort(s), np.arange(P, dtype=np.int32))
    assert np.array_equal(L.slot >= 0, member)
    # within each destination, slots increase with the token index, starting at recv_base[r]
    for r in range(R):
        col = L.slot[:, r]
        col = col[col >= 0]
        assert (np.diff(col) == 1).all()
        if col.size:
            assert col[0] == L.recv_base[r] and col[-1] == L.recv_base[r + 1] - 1
    # receiver-side per-expert counts: column sums of the per-source matrix
    nr = oracle.num_recv_tokens_per_expert(L.num_tokens_per_expert, E, R)
    for r in range(R):
        for j in range(El):
            assert nr[r, j] == (idx == r * El + j).sum()
        assert nr[r].sum() == L.num_tokens_per_expert[:, r * El:(r + 1) * El].sum()


@pytest.mark.parametrize("name", list(CONFIGS))
def test_layout_invariants_full_configs(name):
    cfg = CONFIGS[name]
    c = make_case(cfg, with_hidden=False)
    L = oracle.layout(c.topk_idx, cfg.num_experts, cfg.num_ranks)
    assert L.err_bits == 0
    _layout_invariants(cfg, c, L)
    T, R, E, K = cfg.num_tokens, cfg.num_ranks, cfg.num_experts, cfg.num_topk
    if name == "mixtral":
        # one expert per rank and two distinct experts per token: exactly 2T rows
        assert L.num_rows == 2 * T
    if cfg.routing == "uniform" and cfg.mask_prob == 0:
        # E[pairs per token] = R * (1 - C(E - E_l, K) / C(E, K)) for K distinct
        # uniformly drawn experts; the count per token is bounded by min(K, R).
        El = E // R
        p_miss = math.comb(E - El, K) / math.comb(E, K)
        mean = R * (1 - p_miss)
        per_tok = L.is_token_in_rank.sum(axis=1)
        se = per_tok.std() / math.sqrt(T)
        assert abs(per_tok.mean() - mean) < 6 * se + 1e-9, (per_tok.mean(), mean, se)
        assert per_tok.max() <= min(K, R)


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------
def _torch_bf16_bits(x32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_decode_exhaustive_vs_torch():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_to_double(codes)
    want = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_bf16_encode_vs_torch_round_to_nearest_even():
    rng = np.random.default_rng(7)
    # random bit patterns (all magnitudes, subnormals included) plus ties:
    # patterns whose low 16 bits are exactly the half-way point 0x8000
    bits = rng.integers(0, 2**32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 2**16, size=1 << 16, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    near = np.concatenate([ties - 1, ties + 1])
    x32 = np.concatenate([bits, ties, near]).view(np.float32)
    x32 = x32[~np.isnan(x32)]
    got = oracle.bf16_from_double(x32.astype(np.float64))
    want = _torch_bf16_bits(x32)
    assert np.array_equal(got, want)


def test_bf16_encode_single_rounding_from_double():
    # A double just above a bf16 midpoint must round up: rounding through
    # float32 first would land on the midpoint and then round to even.
    one_plus_half_ulp = 1.0 + 2.0 ** -8
    x = np.array([one_plus_half_ulp + 2.0 ** -40, one_plus_half_ulp,
                  1.0 + 3 * 2.0 ** -8, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -134,
                  -0.0, 2.0 ** 128, 3.3895313892515355e38], np.float64)
    got = oracle.bf16_from_double(x)
    assert list(got) == [0x3F81, 0x3F80, 0x3F82, 0x0001, 0x0000, 0x0002,
                         0x8000, 0x7F80, 0x7F7F]


def _golden_e4m3():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "e4m3_codes.txt")
    rows = []
    with open(path) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                v, code = line.split()
                rows.append((float.fromhex(v) if "0x" in v else float(v), int(code, 16)))
    return rows


def test_e4m3_golden_codes():
    rows = _golden_e4m3()
    vals = np.array([v for v, _ in rows], np.float32)
    codes = np.array([c for _, c in rows], np.uint8)
    assert np.array_equal(oracle.e4m3_from_float(vals), codes)


def test_e4m3_decode_exhaustive_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_to_double(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], want[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_e4m3_encode_vs_torch_in_range():
    # torch's float8_e4m3fn conversion rounds to nearest even and only
    # differs from a saturating conversion above 464 (where it returns NaN),
    # so inside (-464, 464) it is an independent library reference.
    rng = np.random.default_rng(11)
    finite = np.array([v for v in oracle.e4m3_to_double(np.arange(256, dtype=np.uint8))
                       if np.isfinite(v) and v >= 0])
    finite = np.unique(finite)
    mids = (finite[:-1] + finite[1:]) / 2
    m32 = mids.astype(np.float32)
    assert np.array_equal(m32.astype(np.float64), mids)  # ties are exact in float32
    around = np.concatenate([m32, np.nextafter(m32, np.float32(0)),
                             np.nextafter(m32, np.float32(1000)), finite.astype(np.float32)])
    # every float32 whose top 16 bits vary, low bits from a fixed set
    top = (np.arange(0, 0x43E8, dtype=np.uint32) << 16)
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint32)
    sweep = (top[:, None] | lows[None, :]).ravel().view(np.float32)
    rand = (rng.random(1 << 20) * 470).astype(np.float32)
    x = np.concatenate([around, sweep, rand])
    x = x[np.abs(x) < 464]
    x = np.concatenate([x, -x])
    got = oracle.e4m3_from_float(x)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


def test_e4m3_saturates():
    x = np.array([448.0, 448.1, 463.9, 464.0, 479.0, 1e30, np.inf, -500.0, -np.inf], np.float32)
    got = oracle.e4m3_from_float(x)
    assert list(got) == [0x7E] * 7 + [0xFE, 0xFE]


# --------------------------------------------------------------------------
# FP8 block quantiser (kUseFP8 dispatch)
# --------------------------------------------------------------------------
def torch_quantize_block(x_bits):
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).to(torch.float32)
    amax = x.abs().max()
    a = torch.maximum(amax, torch.tensor(1e-4, dtype=torch.float32))
    scale = a / torch.tensor(448.0, dtype=torch.float32)
    inv = torch.tensor(448.0, dtype=torch.float32) / a
    q = (x * inv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return q, float(scale)


def test_quantize_block_vs_torch_reference():
    rng = np.random.default_rng(5)
    for i in range(300):
        mag = 10.0 ** rng.uniform(-8, 4)
        x = workloads._bf16_bits_from_f32((rng.standard_normal(128) * mag).astype(np.float32))
        if i % 7 == 0:
            x[rng.integers(0, 128, 40)] = 0
        q, s = oracle.quantize_block_e4m3(x)
        qt, st = torch_quantize_block(x)
        assert np.array_equal(q, qt), i
        assert np.float32(s) == np.float32(st), i


def test_quantize_block_closed_forms():
    rng = np.random.default_rng(6)
    x = workloads._bf16_bits_from_f32(rng.standard_normal(128).astype(np.float32))
    q, s = oracle.quantize_block_e4m3(x)
    xv = oracle.bf16_to_double(x)
    i = int(np.argmax(np.abs(xv)))
    # the amax element maps to +-448
    assert q[i] == (0x7E if xv[i] > 0 else 0xFE)
    assert np.float32(s) == np.float32(np.float32(np.abs(xv).max()) / np.float32(448.0))
    # dequantisation error: half an E4M3 ulp (relative 2^-4 for normals,
    # absolute 2^-10 in scaled units for subnormals), plus float32 rounding
    deq = oracle.e4m3_to_double(q) * s
    scaled = np.abs(xv) / s
    bound = np.where(scaled >= 2.0 ** -6, 2.0 ** -4 * np.abs(xv), 2.0 ** -10 * s) * (1 + 1e-6) + 1e-30
    assert (np.abs(deq - xv) <= bound).all()
    # an all-zero block: codes 0 and the floor scale 1e-4/448
    z = np.zeros(128, np.uint16)
    qz, sz = oracle.quantize_block_e4m3(z)
    assert not qz.any() and np.float32(sz) == np.float32(np.float32(1e-4) / np.float32(448.0))
    # negative zero keeps its sign bit
    qn, _ = oracle.quantize_block_e4m3(np.full(128, 0x8000, np.uint16))
    assert (qn == 0x80).all()


# --------------------------------------------------------------------------
# dispatch and combine
# --------------------------------------------------------------------------
@pytest.mark.parametrize("cfg", small_cases()[:5], ids=lambda c: c.name)
def test_dispatch_brute_force(cfg):
    c = make_case(cfg)
    E, R, K = cfg.num_experts, cfg.num_ranks, cfg.num_topk
    El = E // R
    want = brute_layout(c.topk_idx, E, R)
    P = int(want["base"][-1])
    d = oracle.dispatch(c.x_bits, c.topk_idx, c.topk_weights, E, R, want["slot"], P)
    seen = np.zeros(P, bool)
    for t in range(cfg.num_tokens):
        for r in range(R):
            p = want["slot"][t, r]
            if p < 0:
                continue
            seen[p] = True
            assert np.array_equal(d.recv_x[p], c.x_bits[t])
            assert d.recv_src_idx[p] == t
            for k in range(K):
                e = c.topk_idx[t, k]
                if e >= 0 and e // El == r:
                    assert d.recv_topk_idx[p, k] == e - r * El
                    assert d.recv_topk_weights[p, k] == c.topk_weights[t, k]
                else:
                    assert d.recv_topk_idx[p, k] == -1 and d.recv_topk_weights[p, k] == 0
    assert seen.all()


def test_dispatch_fp8_rows_are_the_block_quantiser():
    cfg = Config("fp8small", 2, 3, 256, 4, 2, seed=9)
    c = make_case(cfg)
    L = oracle.layout(c.topk_idx, 4, 2)
    d = oracle.dispatch(c.x_bits, c.topk_idx, c.topk_weights, 4, 2, L.slot, L.num_rows, use_fp8=True)
    for t in range(cfg.num_tokens):
        for r in range(2):
            p = L.slot[t, r]
            if p < 0:
                continue
            for b in range(2):
                qt, st = torch_quantize_block(c.x_bits[t, b * 128:(b + 1) * 128])
                assert np.array_equal(d.recv_x[p, b * 128:(b + 1) * 128], qt)
                assert d.recv_scales[p, b] == np.float32(st)


def _bf16_value(bits: int) -> Fraction:
    v = torch.tensor([bits], dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    return Fraction(float(v.to(torch.float64)[0]))


def _exact_bf16_check(out_bits, terms):
    """out must be the bfloat16 nearest to the exact sum, ties to even mantissa."""
    exact = sum((Fraction(w) * Fraction(y) for w, y in terms), Fraction(0))
    b = int(out_bits)
    sign, mag = b & 0x8000, b & 0x7FFF
    if mag == 0:
        neighbours = [0x0001, 0x8001]
    else:
        neighbours = [sign | (mag - 1)] + ([sign | (mag + 1)] if mag + 1 < 0x7F80 else [])
    err = abs(_bf16_value(b) - exact)
    for n in neighbours:
        en = abs(_bf16_value(n) - exact)
        assert err <= en, (hex(b), hex(n), float(exact))
        if err == en:
            assert (mag & 1) == 0, "tie must go to the even significand"


def test_combine_brute_force_exact_rounding():
    cfg = Config("comb", 3, 4, 24, 9, 3, routing="zipf", zipf_s=1.2, mask_prob=0.2, seed=21)
    c = make_case(cfg)
    E, R, K = 9, 3, 3
    L = oracle.layout(c.topk_idx, E, R)
    y = workloads.expert_outputs(L.num_rows, 24, seed=22)
    w = workloads.random_weights(np.random.default_rng(23), cfg.num_tokens, K)
    out = oracle.combine(y, c.topk_idx, w, E, R, L.slot)
    yv = oracle.bf16_to_double(y)
    for t in range(cfg.num_tokens):
        for h in range(24):
            terms = []
            for k in range(K):
                e = c.topk_idx[t, k]
                if e < 0:
                    continue
                p = L.slot[t, e // (E // R)]
                terms.append((float(w[t, k]), float(yv[p, h])))
            if not terms:
                assert out[t, h] == 0
            else:
                _exact_bf16_check(out[t, h], terms)


def test_combine_one_hot_weights_return_the_row():
    cfg = CONFIGS["tiny"]
    c = make_case(cfg)
    L = oracle.layout(c.topk_idx, cfg.num_experts, cfg.num_ranks)
    y = workloads.expert_outputs(L.num_rows, cfg.hidden, seed=31)
    w = np.zeros_like(c.topk_weights)
    w[:, 0] = 1.0
    out = oracle.combine(y, c.topk_idx, w, cfg.num_experts, cfg.num_ranks, L.slot)
    El = cfg.num_experts // cfg.num_ranks
    rows = L.slot[np.arange(cfg.num_tokens), c.topk_idx[:, 0] // El]
    assert np.array_equal(out, y[rows])


@pytest.mark.parametrize("name", ["tiny", "skewed"])
def test_round_trip_identity_experts(name):
    """combine(dispatch(x)) == x with identity experts and weights summing to 1
    (the pages' intranode validation: each rank recovers its tokens with
    "combine diff=0")."""
    cfg = CONFIGS[name]
    if name == "skewed":
        cfg = cfg.scaled(64)
    c = make_case(cfg)
    E, R = cfg.num_experts, cfg.num_ranks
    w = c.topk_weights.astype(np.float64)
    w = np.where(c.topk_idx >= 0, w, 0.0)
    s = w.sum(axis=1, keepdims=True)
    keep = s[:, 0] > 0
    w = np.where(s > 0, w / np.where(s > 0, s, 1), 0).astype(np.float32)
    L = oracle.layout(c.topk_idx, E, R)
    d = oracle.dispatch(c.x_bits, c.topk_idx, w, E, R, L.slot, L.num_rows)
    out = oracle.combine(d.recv_x, c.topk_idx, w, E, R, L.slot)
    # equal as values: a -0.0 in x comes back as +0.0 (0 + w * -0 = +0)
    assert np.array_equal(oracle.bf16_to_double(out[keep]), oracle.bf16_to_double(c.x_bits[keep]))
    assert (out[~keep] == 0).all()


def test_round_trip_negative_zero_returns_positive_zero():
    idx = np.array([[0, 1]], np.int64)
    w = np.array([[0.25, 0.75]], np.float32)
    x = np.array([[0x8000, 0x3F80]], np.uint16)  # -0.0, 1.0
    L = oracle.layout(idx, 2, 1)
    d = oracle.dispatch(x, idx, w, 2, 1, L.slot, L.num_rows)
    out = oracle.combine(d.recv_x, idx, w, 2, 1, L.slot)
    assert out.tolist() == [[0x0000, 0x3F80]]


def test_golden_tiny_layout():
    """The tiny workload's layout summary, written by tests/golden/make_golden.py."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_layout.txt")
    want = {}
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, v = line.split(":", 1)
            want[k.strip()] = [int(t) for t in v.split()]
    cfg = CONFIGS["tiny"]
    c = make_case(cfg, with_hidden=False)
    L = oracle.layout(c.topk_idx, cfg.num_experts, cfg.num_ranks)
    assert L.recv_base.tolist() == want["recv_base"]
    assert L.num_tokens_per_rank.ravel().tolist() == want["num_tokens_per_rank"]
    assert L.num_tokens_per_expert.ravel().tolist() == want["num_tokens_per_expert"]
    assert L.slot[:8].ravel().tolist() == want["slot_first_8_tokens"]


def test_combine_ranksum_brute_force_exact_rounding():
    """Unweighted combine (each destination rank's row once): exact rounding of
    the exact sum, on a case with duplicate ranks per token and masked slots."""
    cfg = Config("rsum", 3, 5, 16, 6, 4, routing="zipf", zipf_s=1.2, mask_prob=0.25, seed=41)
    c = make_case(cfg)
    L = oracle.layout(c.topk_idx, 6, 3)
    y = workloads.expert_outputs(L.num_rows, 16, seed=42)
    out = oracle.combine_ranksum(y, L.slot)
    yv = oracle.bf16_to_double(y)
    for t in range(cfg.num_tokens):
        rows = [int(p) for p in L.slot[t] if p >= 0]
        for h in range(16):
            if not rows:
                assert out[t, h] == 0
            else:
                _exact_bf16_check(out[t, h], [(1.0, float(yv[p, h])) for p in rows])


def test_combine_ranksum_equals_weighted_with_one_weight_per_rank():
    """Rank-sum equals the weighted combine when each rank's first slot has
    weight 1 and its other slots weight 0 (a closed-form special case)."""
    cfg = CONFIGS["tiny"]
    c = make_case(cfg, with_hidden=False)
    E, R = cfg.num_experts, cfg.num_ranks
    L = oracle.layout(c.topk_idx, E, R)
    y = workloads.expert_outputs(L.num_rows, cfg.hidden, seed=43)
    w = np.zeros_like(c.topk_weights)
    for t in range(cfg.num_tokens):
        seen = set()
        for k in range(cfg.num_topk):
            r = c.topk_idx[t, k] // (E // R)
            if c.topk_idx[t, k] >= 0 and r not in seen:
                w[t, k] = 1.0
                seen.add(r)
    assert np.array_equal(oracle.combine_ranksum(y, L.slot),
                          oracle.combine(y, c.topk_idx, w, E, R, L.slot))


# --------------------------------------------------------------------------
# low-latency (expert-major) layout, dispatch and combine
# --------------------------------------------------------------------------
def brute_ll_layout(topk_idx, E, R, cap):
    """Walk experts, then source ranks, then tokens, then k, handing out rows."""
    T, K = topk_idx.shape
    Tr = T // R
    slot = np.full((T, K), -1, np.int32)
    count = np.zeros(E, np.int32)
    off = np.zeros((E, R), np.int32)
    bad = 0
    for e in range(E):
        pos = 0
        for s in range(R):
            off[e, s] = pos
            for t in range(s * Tr, (s + 1) * Tr):
                for k in range(K):
                    if topk_idx[t, k] == e:
                        if pos < cap:
                            slot[t, k] = e * cap + pos
                        else:
                            bad |= 2
                        pos += 1
        count[e] = pos
    if ((topk_idx < -1) | (topk_idx >= E)).any():
        bad |= 1
    return slot, count, off, bad


LL_CASES = [Config("ll0", 4, 32, 16, 16, 4, seed=61), Config("ll1", 3, 7, 8, 9, 2, routing="zipf",
            zipf_s=1.2, mask_prob=0.2, seed=62), Config("ll2", 8, 5, 8, 64, 8, seed=63),
            Config("ll3", 1, 40, 8, 5, 3, routing="zipf", zipf_s=1.2, seed=64)]


@pytest.mark.parametrize("cfg", LL_CASES, ids=lambda c: c.name)
def test_ll_layout_matches_brute_force_and_ht_counts(cfg):
    c = make_case(cfg, with_hidden=False)
    E, R, T = cfg.num_experts, cfg.num_ranks, cfg.num_tokens
    got = oracle.ll_layout(c.topk_idx, E, R, T)
    slot, count, off, bad = brute_ll_layout(c.topk_idx, E, R, T)
    np.testing.assert_array_equal(got.ll_slot, slot)
    np.testing.assert_array_equal(got.ll_count, count)
    np.testing.assert_array_equal(got.ll_src_offset, off)
    assert got.err_bits == bad == 0
    # per-expert counts are the column sums of the high-throughput layout's
    # per-source expert counts, and each expert's rows are a bijection onto
    # [e*cap, e*cap + count)
    ht = oracle.layout(c.topk_idx, E, R)
    np.testing.assert_array_equal(got.ll_count, ht.num_tokens_per_expert.sum(axis=0))
    for e in range(E):
        rows = np.sort(got.ll_slot[c.topk_idx == e])
        assert np.array_equal(rows, e * T + np.arange(got.ll_count[e]))


def test_ll_layout_duplicates_and_capacity():
    idx = np.array([[2, 2, 0], [1, 2, -1], [2, 0, 2], [-1, -1, -1]], np.int64)
    got = oracle.ll_layout(idx, 3, 1, 3)
    slot, count, off, bad = brute_ll_layout(idx, 3, 1, 3)
    np.testing.assert_array_equal(got.ll_slot, slot)
    np.testing.assert_array_equal(got.ll_count, count)
    assert got.ll_count.tolist() == [2, 1, 5] and got.err_bits == bad == 2
    # expert 2 rows in (token, k) order: (0,0) (0,1) (1,1) then capacity
    assert got.ll_slot[0].tolist() == [6, 7, 0] and got.ll_slot[1].tolist() == [3, 8, -1]
    assert got.ll_slot[2].tolist() == [-1, 1, -1]


@pytest.mark.parametrize("use_fp8", [False, True])
def test_ll_dispatch_brute_force(use_fp8):
    cfg = Config("lld", 2, 6, 256, 8, 3, seed=65)
    c = make_case(cfg)
    E, R, T = 8, 2, cfg.num_tokens
    L = oracle.ll_layout(c.topk_idx, E, R, T)
    recv, scales, src = oracle.ll_dispatch(c.x_bits, L.ll_slot, E * T, use_fp8=use_fp8)
    for t in range(T):
        for k in range(3):
            p = L.ll_slot[t, k]
            if p < 0:
                continue
            assert src[p] == t
            if use_fp8:
                for b in range(2):
                    qt, st = torch_quantize_block(c.x_bits[t, b * 128:(b + 1) * 128])
                    assert np.array_equal(recv[p, b * 128:(b + 1) * 128], qt)
                    assert scales[p, b] == np.float32(st)
            else:
                assert np.array_equal(recv[p], c.x_bits[t])
    assert (src >= 0).sum() == (L.ll_slot >= 0).sum()


def test_ll_combine_equals_ht_combine_on_copied_rows():
    """With every expert row a copy of its rank's row, the expert-major combine
    has the same terms, in the same k order, as the rank-major one: equal bits."""
    cfg = Config("llc", 4, 16, 24, 16, 4, routing="zipf", zipf_s=1.2, mask_prob=0.1, seed=66)
    c = make_case(cfg, with_hidden=False)
    E, R, T, K = 16, 4, cfg.num_tokens, 4
    ht = oracle.layout(c.topk_idx, E, R)
    ll = oracle.ll_layout(c.topk_idx, E, R, T)
    y_ht = workloads.expert_outputs(ht.num_rows, 24, seed=67)
    y_ll = np.zeros((E * T, 24), np.uint16)
    for t in range(T):
        for k in range(K):
            e = c.topk_idx[t, k]
            if e >= 0:
                y_ll[ll.ll_slot[t, k]] = y_ht[ht.slot[t, e // (E // R)]]
    w = workloads.random_weights(np.random.default_rng(68), T, K)
    assert np.array_equal(oracle.ll_combine(y_ll, w, ll.ll_slot),
                          oracle.combine(y_ht, c.topk_idx, w, E, R, ht.slot))


def test_ll_combine_brute_force_exact_rounding():
    cfg = Config("llx", 2, 6, 8, 6, 3, mask_prob=0.2, seed=69)
    c = make_case(cfg, with_hidden=False)
    L = oracle.ll_layout(c.topk_idx, 6, 2, cfg.num_tokens)
    y = workloads.expert_outputs(6 * cfg.num_tokens, 8, seed=70)
    yv = oracle.bf16_to_double(y)
    for w in (c.topk_weights, None):
        out = oracle.ll_combine(y, w, L.ll_slot)
        for t in range(cfg.num_tokens):
            terms = [(1.0 if w is None else float(w[t, k]), None, L.ll_slot[t, k])
                     for k in range(3) if L.ll_slot[t, k] >= 0]
            for h in range(8):
                if not terms:
                    assert out[t, h] == 0
                else:
                    _exact_bf16_check(out[t, h], [(wk, float(yv[p, h])) for wk, _, p in terms])


def test_ll_round_trip_identity_experts():
    cfg = CONFIGS["decode_fp8"].scaled(8)
    c = make_case(cfg)
    E, R, T = cfg.num_experts, cfg.num_ranks, cfg.num_tokens
    L = oracle.ll_layout(c.topk_idx, E, R, T)
    recv, _, _ = oracle.ll_dispatch(c.x_bits, L.ll_slot, E * T)
    w = c.topk_weights.astype(np.float64)
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    out = oracle.ll_combine(recv, w, L.ll_slot)
    assert np.array_equal(oracle.bf16_to_double(out), oracle.bf16_to_double(c.x_bits))


# ---------------------------------------------------------------------------
# sharded form: one rank's layout of its own tokens (oracle.shard_layout)
# ---------------------------------------------------------------------------
def brute_shard_layout(topk_idx, E, R):
    """Each destination's send run built directly: walk the destinations in
    order and, within each, the tokens in order."""
    T, K = topk_idx.shape
    El = E // R
    members = [set() for _ in range(T)]
    per_expert = [0] * E
    bad = 0
    for t in range(T):
        for k in range(K):
            e = int(topk_idx[t, k])
            if e == -1:
                continue
            if not (0 <= e < E):
                bad = 1
                continue
            members[t].add(e // El)
            per_expert[e] += 1
    slot = np.full((T, R), -1, np.int32)
    base = [0]
    row = 0
    for r in range(R):
        for t in range(T):
            if r in members[t]:
                slot[t, r] = row
                row += 1
        base.append(row)
    return dict(slot=slot, base=np.array(base, np.int32),
                counts=np.diff(np.array(base, np.int32)),
                per_expert=np.array(per_expert, np.int32), bad=bad)


@pytest.mark.parametrize("T,R,E,K,seed", [(0, 4, 16, 4, 1), (1, 1, 3, 2, 2), (7, 3, 6, 2, 3),
                                          (33, 5, 10, 3, 4), (64, 8, 64, 8, 5),
                                          (13, 64, 128, 8, 6), (200, 4, 16, 4, 7)])
def test_shard_layout_matches_brute_force(T, R, E, K, seed):
    rng = np.random.default_rng(seed)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int64)
    idx[rng.random((T, K)) < 0.15] = -1
    if T > 3:
        idx[2, 0] = E + 5  # a bad id: treated as masked and flagged
        idx[3, K - 1] = idx[3, 0]  # a duplicate expert: membership is an OR, counts count slots
    got = oracle.shard_layout(idx, E, R)
    want = brute_shard_layout(idx, E, R)
    np.testing.assert_array_equal(got.send_slot, want["slot"])
    np.testing.assert_array_equal(got.send_base, want["base"])
    np.testing.assert_array_equal(got.send_counts, want["counts"])
    np.testing.assert_array_equal(got.expert_counts, want["per_expert"])
    assert got.err_bits == want["bad"]
    # send_slot is a bijection onto [0, rows)
    live = got.send_slot[got.send_slot >= 0]
    np.testing.assert_array_equal(np.sort(live), np.arange(got.send_base[-1]))


def test_shard_layout_rows_are_the_single_call_rows_of_one_source():
    """With the whole batch as one rank's tokens (T % R == 0), the send slots
    are the single-call layout's slots and the counts its column sums: the
    slot order within a destination is token order either way."""
    cfg = CONFIGS["skewed"].scaled(64)
    c = make_case(cfg, with_hidden=False)
    E, R = cfg.num_experts, cfg.num_ranks
    sh = oracle.shard_layout(c.topk_idx, E, R)
    full = oracle.layout(c.topk_idx, E, R)
    np.testing.assert_array_equal(sh.send_slot, full.slot)
    np.testing.assert_array_equal(sh.send_base, full.recv_base)
    np.testing.assert_array_equal(sh.send_counts, full.num_tokens_per_rank.sum(axis=0))
    np.testing.assert_array_equal(sh.expert_counts, full.num_tokens_per_expert.sum(axis=0))
