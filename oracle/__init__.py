"""CPU oracle for the MoE expert-parallel token shuffle (test infrastructure).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package. The CUDA library does not call it, and neither side
imports the other. This wrapper marshals numpy arrays into the plain-C oracle
in ep_oracle.c. That file holds all of the arithmetic and cites the passages
it follows.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        P = C.c_void_p
        i64, i32 = C.c_int64, C.c_int
        L.oracle_layout.argtypes = [P, i64, i32, i32, i32, P, P, P, P, P, P]
        L.oracle_num_recv_tokens_per_expert.argtypes = [P, i32, i32, P]
        L.oracle_shard_layout.argtypes = [P, i64, i32, i32, i32, P, P, P, P, P, P]
        L.oracle_dispatch.argtypes = [P, i64, i64, P, P, i32, i32, i32, P, i64, i64, i32,
                                      P, P, P, P, P]
        L.oracle_combine.argtypes = [P, i64, P, P, i64, i32, i32, i32, P, i64, i64, P]
        L.oracle_combine_ranksum.argtypes = [P, i64, i64, i32, P, i64, i64, P]
        L.oracle_ll_layout.argtypes = [P, i64, i32, i32, i32, i64, P, P, P, P]
        L.oracle_ll_dispatch.argtypes = [P, i64, i64, i32, P, i64, i64, i32, P, P, P]
        L.oracle_ll_combine.argtypes = [P, i64, P, i64, i32, P, i64, i64, P]
        L.oracle_quantize_block_e4m3.argtypes = [P, i32, P, P]
        L.oracle_quantize_block_e4m3.restype = None
        for name in ("oracle_e4m3_from_float_n", "oracle_double_to_bf16_n",
                     "oracle_bf16_to_double_n", "oracle_e4m3_to_double_n"):
            getattr(L, name).argtypes = [P, i64, P]
            getattr(L, name).restype = None
        for name in ("oracle_layout", "oracle_num_recv_tokens_per_expert", "oracle_shard_layout",
                     "oracle_dispatch", "oracle_combine", "oracle_combine_ranksum",
                     "oracle_ll_layout", "oracle_ll_dispatch", "oracle_ll_combine"):
            getattr(L, name).restype = C.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"{what}: oracle returned {rc}")


@dataclass
class Layout:
    is_token_in_rank: np.ndarray       # [T, R] uint8
    num_tokens_per_rank: np.ndarray    # [R, R] int32 (row = source rank)
    num_tokens_per_expert: np.ndarray  # [R, E] int32 (row = source rank)
    slot: np.ndarray                   # [T, R] int32, -1 = not sent
    recv_base: np.ndarray              # [R + 1] int32, recv_base[R] = P
    err_bits: int

    @property
    def num_rows(self) -> int:
        return int(self.recv_base[-1])


def layout(topk_idx: np.ndarray, num_experts: int, num_ranks: int) -> Layout:
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    T, K = topk_idx.shape
    R, E = num_ranks, num_experts
    itr = np.empty((T, R), np.uint8)
    ntpr = np.empty((R, R), np.int32)
    ntpe = np.empty((R, E), np.int32)
    slot = np.empty((T, R), np.int32)
    base = np.empty(R + 1, np.int32)
    err = np.zeros(1, np.int32)
    _check(lib().oracle_layout(_p(topk_idx), T, K, E, R, _p(itr), _p(ntpr), _p(ntpe),
                               _p(slot), _p(base), _p(err)), "layout")
    return Layout(itr, ntpr, ntpe, slot, base, int(err[0]))


@dataclass
class ShardLayout:
    is_token_in_rank: np.ndarray  # [T, R] uint8
    send_counts: np.ndarray       # [R] int32
    expert_counts: np.ndarray     # [E] int32
    send_slot: np.ndarray         # [T, R] int32, -1 = not sent
    send_base: np.ndarray         # [R + 1] int32
    err_bits: int


def shard_layout(topk_idx: np.ndarray, num_experts: int, num_ranks: int) -> ShardLayout:
    """One rank's layout of its own tokens over num_ranks destinations."""
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    T, K = topk_idx.shape
    R, E = num_ranks, num_experts
    itr = np.empty((T, R), np.uint8)
    cnt = np.empty(R, np.int32)
    ecnt = np.empty(E, np.int32)
    slot = np.empty((T, R), np.int32)
    base = np.empty(R + 1, np.int32)
    err = np.zeros(1, np.int32)
    _check(lib().oracle_shard_layout(_p(topk_idx), T, K, E, R, _p(itr), _p(cnt), _p(ecnt),
                                     _p(slot), _p(base), _p(err)), "shard_layout")
    return ShardLayout(itr, cnt, ecnt, slot, base, int(err[0]))


def num_recv_tokens_per_expert(num_tokens_per_expert: np.ndarray, num_experts: int,
                               num_ranks: int) -> np.ndarray:
    ntpe = np.ascontiguousarray(num_tokens_per_expert, dtype=np.int32)
    out = np.empty((num_ranks, num_experts // num_ranks), np.int32)
    _check(lib().oracle_num_recv_tokens_per_expert(_p(ntpe), num_experts, num_ranks, _p(out)),
           "num_recv_tokens_per_expert")
    return out


@dataclass
class Dispatched:
    recv_x: np.ndarray             # [P, H] uint16 (bf16 bits) or uint8 (E4M3 codes)
    recv_scales: np.ndarray | None  # [P, H/128] float32 (FP8 only)
    recv_src_idx: np.ndarray       # [P] int32
    recv_topk_idx: np.ndarray      # [P, K] int64
    recv_topk_weights: np.ndarray  # [P, K] float32


def dispatch(x_bits: np.ndarray, topk_idx: np.ndarray, topk_weights: np.ndarray,
             num_experts: int, num_ranks: int, slot: np.ndarray, num_rows: int,
             use_fp8: bool = False, t_range: tuple[int, int] | None = None,
             fill: int | None = 0) -> Dispatched:
    """Dispatch tokens in t_range (default: all); rows of other tokens keep
    `fill` (left uninitialised when fill is None)."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    topk_weights = np.ascontiguousarray(topk_weights, dtype=np.float32)
    slot = np.ascontiguousarray(slot, dtype=np.int32)
    T, H = x_bits.shape
    K = topk_idx.shape[1]
    t0, t1 = t_range if t_range is not None else (0, T)
    if use_fp8:
        recv_x = (np.empty((num_rows, H), np.uint8) if fill is None
                  else np.full((num_rows, H), fill & 0xFF, np.uint8))
        scales = np.zeros((num_rows, H // 128), np.float32)
    else:
        recv_x = (np.empty((num_rows, H), np.uint16) if fill is None
                  else np.full((num_rows, H), fill & 0xFFFF, np.uint16))
        scales = None
    src = np.full(num_rows, -2, np.int32)
    tidx = np.full((num_rows, K), -2, np.int64)
    tw = np.full((num_rows, K), np.nan, np.float32)
    _check(lib().oracle_dispatch(_p(x_bits), T, H, _p(topk_idx), _p(topk_weights), K,
                                 num_experts, num_ranks, _p(slot), t0, t1, int(use_fp8),
                                 _p(recv_x), _p(scales), _p(src), _p(tidx), _p(tw)),
           "dispatch")
    return Dispatched(recv_x, scales, src, tidx, tw)


def combine(y_bits: np.ndarray, topk_idx: np.ndarray, topk_weights: np.ndarray,
            num_experts: int, num_ranks: int, slot: np.ndarray,
            t_range: tuple[int, int] | None = None) -> np.ndarray:
    """Weighted combine; returns out [T, H] uint16 (rows outside t_range are 0)."""
    y_bits = np.ascontiguousarray(y_bits, dtype=np.uint16)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    topk_weights = np.ascontiguousarray(topk_weights, dtype=np.float32)
    slot = np.ascontiguousarray(slot, dtype=np.int32)
    H = y_bits.shape[1]
    T, K = topk_idx.shape
    t0, t1 = t_range if t_range is not None else (0, T)
    out = np.zeros((T, H), np.uint16)
    _check(lib().oracle_combine(_p(y_bits), H, _p(topk_idx), _p(topk_weights), T, K,
                                num_experts, num_ranks, _p(slot), t0, t1, _p(out)),
           "combine")
    return out


def combine_ranksum(y_bits: np.ndarray, slot: np.ndarray,
                    t_range: tuple[int, int] | None = None) -> np.ndarray:
    """Unweighted combine: each destination rank's row once; out [T, H] uint16."""
    y_bits = np.ascontiguousarray(y_bits, dtype=np.uint16)
    slot = np.ascontiguousarray(slot, dtype=np.int32)
    H = y_bits.shape[1]
    T, R = slot.shape
    t0, t1 = t_range if t_range is not None else (0, T)
    out = np.zeros((T, H), np.uint16)
    _check(lib().oracle_combine_ranksum(_p(y_bits), H, T, R, _p(slot), t0, t1, _p(out)),
           "combine_ranksum")
    return out


@dataclass
class LLLayout:
    ll_slot: np.ndarray        # [T, K] int32: row in the expert-major buffer, -1 = none
    ll_count: np.ndarray       # [E] int32: rows each expert receives
    ll_src_offset: np.ndarray  # [E, R] int32: first row of each source within its expert
    err_bits: int


def ll_layout(topk_idx: np.ndarray, num_experts: int, num_ranks: int,
              expert_capacity: int) -> LLLayout:
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    T, K = topk_idx.shape
    E, R = num_experts, num_ranks
    slot = np.empty((T, K), np.int32)
    cnt = np.empty(E, np.int32)
    off = np.empty((E, R), np.int32)
    err = np.zeros(1, np.int32)
    _check(lib().oracle_ll_layout(_p(topk_idx), T, K, E, R, expert_capacity, _p(slot), _p(cnt),
                                  _p(off), _p(err)), "ll_layout")
    return LLLayout(slot, cnt, off, int(err[0]))


def ll_dispatch(x_bits: np.ndarray, ll_slot: np.ndarray, num_rows: int, use_fp8: bool = False,
                t_range: tuple[int, int] | None = None):
    """(recv_x, recv_scales or None, recv_src_idx) over num_rows rows; untouched rows are 0 / -2."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    ll_slot = np.ascontiguousarray(ll_slot, dtype=np.int32)
    T, H = x_bits.shape
    K = ll_slot.shape[1]
    t0, t1 = t_range if t_range is not None else (0, T)
    recv = np.zeros((num_rows, H), np.uint8 if use_fp8 else np.uint16)
    scales = np.zeros((num_rows, H // 128), np.float32) if use_fp8 else None
    src = np.full(num_rows, -2, np.int32)
    _check(lib().oracle_ll_dispatch(_p(x_bits), T, H, K, _p(ll_slot), t0, t1, int(use_fp8),
                                    _p(recv), _p(scales), _p(src)), "ll_dispatch")
    return recv, scales, src


def ll_combine(y_bits: np.ndarray, topk_weights: np.ndarray | None, ll_slot: np.ndarray,
               t_range: tuple[int, int] | None = None) -> np.ndarray:
    y_bits = np.ascontiguousarray(y_bits, dtype=np.uint16)
    ll_slot = np.ascontiguousarray(ll_slot, dtype=np.int32)
    w = None if topk_weights is None else np.ascontiguousarray(topk_weights, dtype=np.float32)
    H = y_bits.shape[1]
    T, K = ll_slot.shape
    t0, t1 = t_range if t_range is not None else (0, T)
    out = np.zeros((T, H), np.uint16)
    _check(lib().oracle_ll_combine(_p(y_bits), H, _p(w), T, K, _p(ll_slot), t0, t1, _p(out)),
           "ll_combine")
    return out


def quantize_block_e4m3(x_bits: np.ndarray) -> tuple[np.ndarray, float]:
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    q = np.empty(x_bits.size, np.uint8)
    s = np.empty(1, np.float32)
    lib().oracle_quantize_block_e4m3(_p(x_bits), x_bits.size, _p(q), _p(s))
    return q, float(s[0])


def e4m3_from_float(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().oracle_e4m3_from_float_n(_p(x), x.size, _p(out))
    return out


def e4m3_to_double(c: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().oracle_e4m3_to_double_n(_p(c), c.size, _p(out))
    return out


def bf16_from_double(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_double_to_bf16_n(_p(x), x.size, _p(out))
    return out


def bf16_to_double(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    out = np.empty(b.shape, np.float64)
    lib().oracle_bf16_to_double_n(_p(b), b.size, _p(out))
    return out
