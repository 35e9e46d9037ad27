"""Adversarial routing against the oracle: duplicate experts within a token,
out-of-range expert ids, every slot on one expert or on one rank, and whole
tokens masked, on ragged shapes from 1 to 64 ranks.  Each case runs every
rank-major and expert-major entry point through the random sweep's checks
(bit-exact layouts and dispatches, the combine tolerance), including the
error bits, which must be exactly the oracle's (bad ids set
EP_ERRBIT_BAD_EXPERT and are treated as masked)."""
from __future__ import annotations

import numpy as np
import pytest

from test_gpu_random import check_expert_major, check_rank_major
from workloads import Config, make_case

pytestmark = pytest.mark.gpu

# name, R, T_r, H, experts per rank, K
SHAPES = [
    ("r1", 1, 37, 128, 4, 3),
    ("r4", 4, 100, 264, 2, 8),
    ("r8", 8, 65, 128, 3, 12),
    ("r16", 16, 130, 72, 1, 4),
    ("r32", 32, 9, 1024, 2, 8),
    ("r64", 64, 3, 128, 1, 2),
]


def _distinct(rng, T, E, K):
    """K distinct experts per token (K <= E), else with replacement."""
    if K <= E:
        return np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int64)
    return rng.integers(0, E, (T, K)).astype(np.int64)


def _routing(kind: str, rng, T, E, K, El, R):
    if kind == "duplicates":  # few experts, drawn with replacement
        return rng.integers(0, min(E, 3), (T, K)).astype(np.int64)
    if kind == "bad_ids":
        idx = _distinct(rng, T, E, K)
        bad = np.array([-7, -2, E, E + 5, 1 << 40], dtype=np.int64)
        pick = rng.random((T, K)) < 0.1
        idx[pick] = rng.choice(bad, int(pick.sum()))
        return idx
    if kind == "hot_expert":  # every slot names expert 0
        return np.zeros((T, K), np.int64)
    if kind == "one_rank":  # only the last rank's experts
        return rng.integers((R - 1) * El, E, (T, K)).astype(np.int64)
    if kind == "masked_tokens":  # half the tokens send nothing
        idx = _distinct(rng, T, E, K)
        idx[rng.random(T) < 0.5] = -1
        return idx
    if kind == "mixed":  # all of the above at once
        idx = rng.integers(0, E, (T, K)).astype(np.int64)
        idx[rng.random((T, K)) < 0.05] = E + 1
        idx[rng.random((T, K)) < 0.2] = -1
        idx[rng.random(T) < 0.2] = -1
        idx[rng.random(T) < 0.1, :] = 0
        return idx
    raise ValueError(kind)


KINDS = ["duplicates", "bad_ids", "hot_expert", "one_rank", "masked_tokens", "mixed"]
CASES = [(k, s) for k in KINDS for s in SHAPES]


def _case(kind, shape, i):
    name, R, Tr, H, El, K = shape
    cfg = Config(f"adv_{kind}_{name}", R, Tr, H, R * El, K, seed=9100 + i)
    c = make_case(cfg)
    rng = np.random.default_rng(9500 + i)
    c.topk_idx[:] = _routing(kind, rng, cfg.num_tokens, cfg.num_experts, K, El, R)
    return cfg, c


@pytest.mark.parametrize("i", range(len(CASES)), ids=[f"{k}-{s[0]}" for k, s in CASES])
def test_rank_major_adversarial_routing(ep, i):
    kind, shape = CASES[i]
    cfg, c = _case(kind, shape, i)
    check_rank_major(ep, cfg, c)


@pytest.mark.parametrize("i", range(len(CASES)), ids=[f"{k}-{s[0]}" for k, s in CASES])
def test_expert_major_adversarial_routing(ep, i):
    kind, shape = CASES[i]
    cfg, c = _case(kind, shape, i)
    check_expert_major(ep, cfg, c)
