"""Seeded synthetic inputs for the MoE expert-parallel token shuffle.

This module only draws inputs. It holds no layout, dispatch, quantisation or
combine arithmetic. The CPU oracle tests, the CUDA parity tests and the
benchmark all take their inputs from here, so both sides see the same bytes.

Workload shapes follow the MoE workloads that the MSCCL++ EP port benchmarks
against ("[Not ready] MSCCLPP EP implementation", mscclpp pull request 852):
the functional test uses num_ranks*4 experts with top-4 routing, and the
benchmarks use DeepSeek-V3-like shapes (hidden 7168, 256 experts, top-8) for
the high-throughput kernels and 128 tokens per rank for the low-latency FP8
kernels (the commits that add the MSCCLPP_EP_BENCH_EXPERTS/_TOPK knobs and the
MSCCLPP_EP_LL_* overrides).

Recipe (fixed, so that every machine draws the same inputs):
  * one numpy Generator(PCG64(seed)) per case, drawn in this order:
    routing, masking, weights, hidden states;
  * uniform routing: the first K columns of argsort(U[0,1)^{T x E}) per row,
    i.e. K distinct experts in a uniformly random order;
  * Zipf(s) routing: Gumbel-top-k over log p_i with p_i proportional to
    1/(i+1)^s for expert i (popularity rank i, deliberately not permuted, so
    rank 0 owns the hot experts);
  * masking: each top-k slot independently becomes -1 with probability
    mask_prob;
  * weights: softmax over all K slots of N(0,1) draws, computed in float64 and
    stored as float32 (masked slots keep their weight);
  * hidden states: N(0,1) float32 drawn row-chunk by row-chunk, rounded to
    bfloat16 by torch (round to nearest even) and kept as raw uint16 bits.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

_ROW_CHUNK = 4096  # rows of hidden states drawn per generator call


@dataclass(frozen=True)
class Config:
    name: str
    num_ranks: int
    tokens_per_rank: int
    hidden: int
    num_experts: int
    num_topk: int
    routing: str = "uniform"  # "uniform" | "zipf"
    zipf_s: float = 0.0
    mask_prob: float = 0.0
    fp8: bool = False
    seed: int = 0

    @property
    def num_tokens(self) -> int:
        return self.num_ranks * self.tokens_per_rank

    @property
    def experts_per_rank(self) -> int:
        return self.num_experts // self.num_ranks

    def scaled(self, tokens_per_rank: int) -> "Config":
        """Same routing recipe and seed, different number of tokens per rank."""
        return replace(self, tokens_per_rank=tokens_per_rank,
                       name=f"{self.name}@{tokens_per_rank}tpr")


# The five workloads. Seeds 0..4 in this order.
CONFIGS: dict[str, Config] = {
    "tiny": Config("tiny", 4, 128, 256, 16, 4, seed=0),
    "dsv3_prefill": Config("dsv3_prefill", 8, 4096, 7168, 256, 8, seed=1),
    "decode_fp8": Config("decode_fp8", 32, 128, 7168, 256, 8, fp8=True, seed=2),
    "skewed": Config("skewed", 16, 8192, 4096, 64, 6, routing="zipf",
                     zipf_s=1.2, mask_prob=0.05, seed=3),
    "mixtral": Config("mixtral", 8, 16384, 4096, 8, 2, seed=4),
}


@dataclass
class Case:
    cfg: Config
    topk_idx: np.ndarray      # [T, K] int64, -1 = masked slot
    topk_weights: np.ndarray  # [T, K] float32
    x_bits: np.ndarray | None  # [T, H] uint16 (bfloat16 bit patterns)


def _routing(cfg: Config, rng: np.random.Generator) -> np.ndarray:
    T, E, K = cfg.num_tokens, cfg.num_experts, cfg.num_topk
    out = np.empty((T, K), dtype=np.int64)
    if cfg.routing == "uniform":
        for r0 in range(0, T, 16384):
            r1 = min(T, r0 + 16384)
            u = rng.random((r1 - r0, E))
            out[r0:r1] = np.argsort(u, axis=1, kind="stable")[:, :K]
    elif cfg.routing == "zipf":
        logp = -cfg.zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))
        logp -= np.log(np.exp(logp).sum())
        for r0 in range(0, T, 16384):
            r1 = min(T, r0 + 16384)
            g = rng.gumbel(size=(r1 - r0, E))
            out[r0:r1] = np.argsort(-(logp[None, :] + g), axis=1,
                                    kind="stable")[:, :K]
    else:
        raise ValueError(f"unknown routing {cfg.routing!r}")
    return out


def _bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def normal_bf16_bits(rng: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    """N(0,1) float32 rounded to bfloat16, returned as uint16 bit patterns."""
    out = np.empty((rows, cols), dtype=np.uint16)
    for r0 in range(0, rows, _ROW_CHUNK):
        r1 = min(rows, r0 + _ROW_CHUNK)
        out[r0:r1] = _bf16_bits_from_f32(
            rng.standard_normal((r1 - r0, cols), dtype=np.float32))
    return out


def make_case(cfg: Config, with_hidden: bool = True) -> Case:
    """Draw routing, weights and (optionally) hidden states for one config."""
    if cfg.num_experts % cfg.num_ranks:
        raise ValueError("num_experts must be a multiple of num_ranks")
    if cfg.num_topk > cfg.num_experts:
        raise ValueError("num_topk must not exceed num_experts")
    rng = np.random.Generator(np.random.PCG64(cfg.seed))
    T, K = cfg.num_tokens, cfg.num_topk
    topk_idx = _routing(cfg, rng)
    if cfg.mask_prob > 0:
        masked = rng.random((T, K)) < cfg.mask_prob
        topk_idx[masked] = -1
    z = rng.standard_normal((T, K))
    z = np.exp(z - z.max(axis=1, keepdims=True)) if T else z
    w = (z / z.sum(axis=1, keepdims=True)).astype(np.float32) if T else z.astype(np.float32)
    x = normal_bf16_bits(rng, T, cfg.hidden) if with_hidden else None
    return Case(cfg, topk_idx, np.ascontiguousarray(w), x)


def expert_outputs(rows: int, hidden: int, seed: int) -> np.ndarray:
    """Stand-in expert outputs Y [rows, hidden]: N(0,1) rounded to bfloat16 bits."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return normal_bf16_bits(rng, rows, hidden)


def random_weights(rng: np.random.Generator, T: int, K: int) -> np.ndarray:
    """Uniform(0,1) float32 weights, for combine cases that need no softmax."""
    return rng.random((T, K)).astype(np.float32)


def signed_unit_bf16_bits(rows: int, hidden: int, seed: int) -> np.ndarray:
    """Stand-in expert outputs for full-size batches, drawn fast: bfloat16 bit
    patterns with a random sign, exponent 126 or 127 and a random 7-bit
    mantissa, i.e. values uniform over the bf16 grid of +-[0.5, 2).  One
    integer draw per element (no float rounding pass), so a few GB of rows
    take seconds."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = np.empty((rows, hidden), dtype=np.uint16)
    for r0 in range(0, rows, 16384):
        r1 = min(rows, r0 + 16384)
        u = rng.integers(0, 1 << 16, size=(r1 - r0, hidden), dtype=np.uint16)
        # keep the sign (bit 15), the exponent's lowest bit (bit 7) and the
        # mantissa (bits 0..6); set exponent bits 8..14 to 0111111 (0x7E/0x7F)
        np.bitwise_and(u, 0x80FF, out=u)
        np.bitwise_or(u, 0x3F00, out=u)
        out[r0:r1] = u
    return out
