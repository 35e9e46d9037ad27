"""Single-GPU MoE expert-parallel token shuffle for GB300: Python binding.

A thin ctypes layer over the C ABI in include/ep.h (libep.so, hand-written
CUDA for sm_103a).  It only marshals arguments: it allocates output tensors
with torch and passes raw device pointers and the current CUDA stream.  Every
step of layout, dispatch and combine runs in the library's kernels.  There is
no CPU or PyTorch fallback.  If the library is missing or cannot be loaded,
every call raises.

The three steps follow the high-throughput expert-parallel kernels of
"[Not ready] MSCCLPP EP implementation" (mscclpp pull request 852), section
"Scope" (get_dispatch_layout, intranode_dispatch, intranode_combine), with the
kUseFP8 payload cast of its low-latency dispatch.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libep.so")

EP_OK = 0
EP_ERRBIT_BAD_EXPERT = 1
EP_ERRBIT_CAPACITY = 2
EP_ERRBIT_TIMEOUT = 4
EP_ERRBIT_SCHED = 8
EP_MAX_RANKS = 64
EP_MAX_TOPK = 32
EP_MAX_EXPERTS = 4096

# ep_layout_path_t
LAYOUT_PATHS = {"auto": 0, "multi": 1, "single": 2}

# every entry point declared in include/ep.h
EXPORTED = ("ep_status_string", "ep_workspace_bytes", "ep_get_dispatch_layout",
            "ep_layout_single_launch_fits", "ep_layout_auto_single_launch",
            "ep_get_dispatch_layout_path",
            "ep_get_dispatch_layout_noalloc", "ep_layout_total_rows", "ep_dispatch",
            "ep_combine", "ep_ll_workspace_bytes", "ep_ll_get_dispatch_layout",
            "ep_ll_dispatch", "ep_ll_combine", "ep_debug_set_combine_stall",
            "ep_ll_layout_single_launch_fits", "ep_ll_layout_auto_single_launch",
            "ep_ll_get_dispatch_layout_path", "ep_combine_sched", "ep_ll_combine_sched",
            "ep_layout_dispatch_fused_fits", "ep_layout_dispatch_fused",
            "ep_layout_dispatch_fused_workspace_bytes", "ep_debug_set_fused_stall",
            "ep_shard_workspace_bytes", "ep_shard_layout", "ep_shard_offsets",
            "ep_shard_recv_tokens_per_expert", "ep_debug_e4m3_range")

# 64-bit words of a combine's scheduling counters (EP_COMBINE_SCHED_WORDS)
COMBINE_SCHED_WORDS = 2
# 64-bit words of the fused layout + dispatch's counters (EP_FUSED_SYNC_WORDS)
FUSED_SYNC_WORDS = 640

_lib = None


class EPError(RuntimeError):
    pass


def load(path: str | None = None) -> C.CDLL:
    """Load libep.so (built by combine_get_dispatch_04_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise EPError(f"CUDA library not built: {path} is missing "
                      "(run combine_get_dispatch_04_gb300.build.build())")
    L = C.CDLL(path)
    P, i32, i64, sz = C.c_void_p, C.c_int, C.c_int64, C.c_size_t
    L.ep_status_string.argtypes = [i32]
    L.ep_status_string.restype = C.c_char_p
    L.ep_workspace_bytes.argtypes = [i64, i32, i32]
    L.ep_workspace_bytes.restype = sz
    L.ep_get_dispatch_layout.argtypes = [P, i64, i32, i32, i32, P, P, P, P, P, P, P, sz, P]
    L.ep_layout_single_launch_fits.argtypes = [i64, i32, i32]
    L.ep_layout_single_launch_fits.restype = i32
    L.ep_layout_auto_single_launch.argtypes = [i64, i32, i32]
    L.ep_layout_auto_single_launch.restype = i32
    L.ep_get_dispatch_layout_path.argtypes = [P, i64, i32, i32, i32, P, P, P, P, P, P, P, sz,
                                              i32, P]
    L.ep_layout_total_rows.argtypes = [P, i32, P, P]
    L.ep_dispatch.argtypes = [P, i32, P, P, i64, i32, i32, i32, P, P, i64, i32, P, P, P, P, P,
                              P, P, P]
    L.ep_combine.argtypes = [P, i32, P, P, i64, i32, i32, i32, P, P, P, P]
    L.ep_debug_set_combine_stall.argtypes = [i32]
    L.ep_debug_set_combine_stall.restype = None
    L.ep_ll_workspace_bytes.argtypes = [i64, i32, i32]
    L.ep_ll_workspace_bytes.restype = sz
    L.ep_ll_get_dispatch_layout.argtypes = [P, i64, i32, i32, i32, i64, P, P, P, P, P, sz, P]
    L.ep_ll_get_dispatch_layout_path.argtypes = [P, i64, i32, i32, i32, i64, P, P, P, P, P, sz,
                                                 i32, P]
    for name in ("ep_ll_layout_single_launch_fits", "ep_ll_layout_auto_single_launch"):
        getattr(L, name).argtypes = [i64, i32, i32, i32]
        getattr(L, name).restype = i32
    L.ep_ll_dispatch.argtypes = [P, i32, i64, i32, P, i64, i32, P, P, P, P, P]
    L.ep_ll_combine.argtypes = [P, i32, P, i64, i32, P, P, P, P]
    L.ep_combine_sched.argtypes = [P, i32, P, P, i64, i32, i32, i32, P, P, P, P, P]
    L.ep_ll_combine_sched.argtypes = [P, i32, P, i64, i32, P, P, P, P, P]
    L.ep_layout_dispatch_fused_fits.argtypes = [i64, i32, i32]
    L.ep_layout_dispatch_fused_fits.restype = i32
    L.ep_layout_dispatch_fused_workspace_bytes.argtypes = [i64, i32, i32]
    L.ep_layout_dispatch_fused_workspace_bytes.restype = sz
    L.ep_layout_dispatch_fused.argtypes = [P, i32, P, P, i64, i32, i32, i32, P, P, P, P, P, i64,
                                           i32, P, P, P, P, P, P, P, sz, P, P, P]
    L.ep_debug_set_fused_stall.argtypes = [i32]
    L.ep_debug_set_fused_stall.restype = None
    L.ep_debug_e4m3_range.argtypes = [C.c_uint32, i64, P, P]
    L.ep_shard_workspace_bytes.argtypes = [i64, i32, i32]
    L.ep_shard_workspace_bytes.restype = sz
    L.ep_shard_layout.argtypes = [P, i64, i32, i32, i32, P, P, P, P, P, P, P, sz, P]
    L.ep_shard_offsets.argtypes = [P, i32, i32, P, P]
    L.ep_shard_recv_tokens_per_expert.argtypes = [P, i32, i32, i32, P]
    for name in ("ep_get_dispatch_layout", "ep_get_dispatch_layout_path",
                 "ep_layout_total_rows", "ep_dispatch", "ep_combine",
                 "ep_ll_get_dispatch_layout", "ep_ll_get_dispatch_layout_path",
                 "ep_ll_dispatch", "ep_ll_combine", "ep_combine_sched", "ep_ll_combine_sched",
                 "ep_layout_dispatch_fused", "ep_shard_layout", "ep_shard_offsets",
                 "ep_shard_recv_tokens_per_expert", "ep_debug_e4m3_range"):
        getattr(L, name).restype = i32
    _lib = L
    return L


def lib() -> C.CDLL:
    return load()


# Debug mode (environment EP_DEBUG=1, or set_debug(True)): every call waits
# for its stream and raises at once if the device error word it was given is
# non-zero or the kernels failed, naming the call.  Off by default: calls are
# asynchronous.
_debug = os.environ.get("EP_DEBUG", "0") not in ("", "0")

_ERRBITS = ((EP_ERRBIT_BAD_EXPERT, "an expert id outside [-1, E)"),
            (EP_ERRBIT_CAPACITY, "a row at or beyond the receive capacity"),
            (EP_ERRBIT_TIMEOUT, "a bounded pipeline wait ran out"),
            (EP_ERRBIT_SCHED, "a combine's scheduling counters were in use by another launch"))


def set_debug(on: bool) -> None:
    """Synchronise and check the error word after every call (see above)."""
    global _debug
    _debug = bool(on)


def describe_error_word(value: int) -> str:
    names = [text for bit, text in _ERRBITS if value & bit]
    return ", ".join(names) if names else "no error"


def _debug_check(what: str, err: torch.Tensor | None, device: torch.device):
    if not _debug:
        return
    torch.cuda.current_stream(device).synchronize()  # raises on a kernel fault
    if err is not None and int(err.item()) != 0:
        v = int(err.item())
        raise EPError(f"{what}: device error word {v} ({describe_error_word(v)})")


def _check(status: int, what: str):
    if status != EP_OK:
        msg = lib().ep_status_string(status).decode()
        raise EPError(f"{what} failed: {msg}")


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


def _stream(device: torch.device):
    return C.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None):
    if not t.is_cuda:
        raise EPError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise EPError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise EPError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise EPError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


@dataclass
class Layout:
    """Outputs of get_dispatch_layout (all on the device)."""
    num_tokens_per_rank: torch.Tensor    # [R, R] int32, row = source rank
    num_tokens_per_expert: torch.Tensor  # [R, E] int32, row = source rank
    is_token_in_rank: torch.Tensor       # [T, R] bool
    slot: torch.Tensor                   # [T, R] int32, -1 = not sent
    recv_base: torch.Tensor              # [R + 1] int32, recv_base[R] = P
    num_experts: int
    num_ranks: int
    workspace: torch.Tensor | None = None
    # [2] int64 counters of the dynamically scheduled combine, zero between
    # launches; None: the static schedule.  They serve the combines of the
    # first stream that uses them; combines on any other stream get counters
    # of their own (sched_for), so that combines through one Layout on two
    # streams, or a graph replayed beside eager calls, never share them.
    sched: torch.Tensor | None = None
    # [FUSED_SYNC_WORDS] int64 counters and flags of the one-launch layout +
    # dispatch, zero between launches; per stream like sched
    fused_sync: torch.Tensor | None = None

    @property
    def num_tokens(self) -> int:
        return self.slot.shape[0]


def workspace_bytes(num_tokens: int, num_ranks: int, num_experts: int) -> int:
    return int(lib().ep_workspace_bytes(num_tokens, num_ranks, num_experts))


def single_launch_fits(num_tokens: int, num_ranks: int, num_experts: int) -> bool:
    """True if the one-launch (thread-block cluster) layout applies."""
    return bool(lib().ep_layout_single_launch_fits(num_tokens, num_ranks, num_experts))


def auto_single_launch(num_tokens: int, num_ranks: int, num_experts: int) -> bool:
    """True if path="auto" takes the one-launch layout for this batch."""
    return bool(lib().ep_layout_auto_single_launch(num_tokens, num_ranks, num_experts))


def alloc_combine_sched(device: torch.device) -> torch.Tensor:
    """Zeroed counters for the dynamically scheduled combine (each launch
    leaves them zero again)."""
    return torch.zeros(COMBINE_SCHED_WORDS, dtype=torch.int64, device=device)


def alloc_layout(num_tokens: int, num_experts: int, num_ranks: int,
                 device: torch.device) -> Layout:
    """Output tensors and the multi-launch workspace (allocated for every size,
    so that the same Layout serves either path)."""
    T, R, E = num_tokens, num_ranks, num_experts
    i32 = dict(dtype=torch.int32, device=device)
    # one workspace for the multi-launch layout and the one-launch layout + dispatch
    wsb = max(workspace_bytes(T, R, E),
              int(lib().ep_layout_dispatch_fused_workspace_bytes(T, R, E)), 16)
    ws = torch.empty(wsb, dtype=torch.uint8, device=device)
    return Layout(torch.empty((R, R), **i32), torch.empty((R, E), **i32),
                  torch.empty((T, R), dtype=torch.bool, device=device),
                  torch.empty((T, R), **i32), torch.empty(R + 1, **i32), E, R, ws,
                  alloc_combine_sched(device),
                  torch.zeros(FUSED_SYNC_WORDS, dtype=torch.int64, device=device))


def get_dispatch_layout(topk_idx: torch.Tensor, num_experts: int, num_ranks: int, *,
                        err: torch.Tensor | None = None, out: Layout | None = None,
                        path: str = "auto") -> Layout:
    """Per-rank / per-expert counts, is_token_in_rank and the slot of every
    (token, destination rank) pair.  Enqueued on the current stream.
    path: "auto", "multi" (multi-launch) or "single" (one cluster launch,
    small batches only); all give the same outputs."""
    _need(topk_idx, "topk_idx", torch.int64)
    if topk_idx.dim() != 2:
        raise EPError("topk_idx must be [num_tokens, num_topk]")
    if path not in LAYOUT_PATHS:
        raise EPError(f"path must be one of {sorted(LAYOUT_PATHS)}")
    T, K = topk_idx.shape
    L = out if out is not None else alloc_layout(T, num_experts, num_ranks, topk_idx.device)
    if err is not None:
        _need(err, "err", torch.int32)
    args = (_ptr(topk_idx), T, K, num_experts, num_ranks, _ptr(L.num_tokens_per_rank),
            _ptr(L.num_tokens_per_expert), _ptr(L.is_token_in_rank), _ptr(L.slot),
            _ptr(L.recv_base), _ptr(err), _ptr(L.workspace),
            L.workspace.numel() if L.workspace is not None else 0)
    stream = _stream(topk_idx.device)
    if path == "auto":
        _check(lib().ep_get_dispatch_layout(*args, stream), "ep_get_dispatch_layout")
    else:
        _check(lib().ep_get_dispatch_layout_path(*args, LAYOUT_PATHS[path], stream),
               "ep_get_dispatch_layout_path")
    _debug_check("get_dispatch_layout", err, topk_idx.device)
    return L


def total_rows(layout: Layout) -> int:
    """P = rows of the receive buffer (copies one int32 and synchronises)."""
    v = C.c_int32(0)
    _check(lib().ep_layout_total_rows(_ptr(layout.recv_base), layout.num_ranks, C.byref(v),
                                      _stream(layout.recv_base.device)), "ep_layout_total_rows")
    return int(v.value)


@dataclass
class Dispatched:
    recv_x: torch.Tensor                # [cap, H] bf16, or [cap, H] uint8 E4M3 codes
    recv_scales: torch.Tensor | None    # [cap, H/128] float32 (FP8 only)
    recv_src_idx: torch.Tensor          # [cap] int32
    recv_topk_idx: torch.Tensor         # [cap, K] int64
    recv_topk_weights: torch.Tensor     # [cap, K] float32
    num_recv_tokens_per_expert: torch.Tensor  # [R, E/R] int32
    use_fp8: bool


def worst_case_rows(num_tokens: int, num_topk: int, num_ranks: int) -> int:
    return num_tokens * min(num_topk, num_ranks)


def alloc_dispatched(capacity: int, hidden: int, num_topk: int, num_experts: int,
                     num_ranks: int, use_fp8: bool, device: torch.device) -> Dispatched:
    if use_fp8:
        recv_x = torch.empty((capacity, hidden), dtype=torch.uint8, device=device)
        scales = torch.empty((capacity, hidden // 128), dtype=torch.float32, device=device)
    else:
        recv_x = torch.empty((capacity, hidden), dtype=torch.bfloat16, device=device)
        scales = None
    return Dispatched(recv_x, scales,
                      torch.empty(capacity, dtype=torch.int32, device=device),
                      torch.empty((capacity, num_topk), dtype=torch.int64, device=device),
                      torch.empty((capacity, num_topk), dtype=torch.float32, device=device),
                      torch.empty((num_ranks, num_experts // num_ranks), dtype=torch.int32,
                                  device=device), use_fp8)


def dispatch(x: torch.Tensor, topk_idx: torch.Tensor, topk_weights: torch.Tensor,
             layout: Layout, *, use_fp8: bool = False, capacity: int | None = None,
             err: torch.Tensor | None = None, out: Dispatched | None = None) -> Dispatched:
    """Scatter every token row to its destination ranks' rows (bf16 copy or
    FP8 E4M3 with per-128-channel scales).  Enqueued on the current stream."""
    _need(x, "x", torch.bfloat16)
    T, H = x.shape
    K = topk_idx.shape[1]
    _need(topk_idx, "topk_idx", torch.int64, (T, K))
    _need(topk_weights, "topk_weights", torch.float32, (T, K))
    R, E = layout.num_ranks, layout.num_experts
    _need(layout.slot, "slot", torch.int32, (T, R))
    if out is None:
        cap = capacity if capacity is not None else worst_case_rows(T, K, R)
        out = alloc_dispatched(cap, H, K, E, R, use_fp8, x.device)
    elif out.use_fp8 != use_fp8:
        raise EPError("preallocated dispatch buffers have the wrong payload type")
    cap = out.recv_x.shape[0]
    if err is not None:
        _need(err, "err", torch.int32)
    # a shard's layout has no [R, E] per-source counts: no per-expert receive counts here
    ntpe = getattr(layout, "num_tokens_per_expert", None)
    nrpe = out.num_recv_tokens_per_expert if ntpe is not None else None
    _check(lib().ep_dispatch(
        _ptr(x), H, _ptr(topk_idx), _ptr(topk_weights), T, K, E, R, _ptr(layout.slot),
        _ptr(ntpe), cap, int(use_fp8), _ptr(out.recv_x),
        _ptr(out.recv_scales), _ptr(out.recv_src_idx), _ptr(out.recv_topk_idx),
        _ptr(out.recv_topk_weights), _ptr(nrpe), _ptr(err),
        _stream(x.device)), "ep_dispatch")
    _debug_check("dispatch", err, x.device)
    return out


def _per_stream(s: torch.Tensor, name: str, words: int, device: torch.device) -> torch.Tensor:
    """Counter state `s` serves the first stream that uses it (recorded on
    the tensor, so copies of a Layout agree); any other stream gets a state
    of its own, kept on `s` and zeroed when first needed."""
    _need(s, name, torch.int64, (words,))
    if s.device != device:
        raise EPError(f"the layout's {name} must be on the call's device")
    key = torch.cuda.current_stream(device).cuda_stream
    home = getattr(s, "_ep_home_stream", None)
    if home is None:
        s._ep_home_stream = home = key
    if key == home:
        return s
    others = s.__dict__.setdefault("_ep_other_streams", {})
    if key not in others:
        others[key] = torch.zeros(words, dtype=torch.int64, device=device)
    return others[key]


def sched_for(layout, device: torch.device) -> torch.Tensor | None:
    """The scheduling counters that a combine through `layout` on the current
    stream uses (see _per_stream).  None: the layout asks for the static
    schedule."""
    s = layout.sched
    return None if s is None else _per_stream(s, "sched", COMBINE_SCHED_WORDS, device)


def fused_fits(num_tokens: int, num_ranks: int, num_experts: int) -> bool:
    """True if layout_dispatch (one launch) applies to the batch."""
    return bool(lib().ep_layout_dispatch_fused_fits(num_tokens, num_ranks, num_experts))


def layout_dispatch(x: torch.Tensor, topk_idx: torch.Tensor, topk_weights: torch.Tensor,
                    num_experts: int, num_ranks: int, *, use_fp8: bool = False,
                    capacity: int | None = None, err: torch.Tensor | None = None,
                    layout: Layout | None = None,
                    out: Dispatched | None = None) -> tuple[Layout, Dispatched]:
    """get_dispatch_layout and dispatch in one kernel launch (small batches:
    fused_fits).  Same outputs as the two calls.  Enqueued on the current
    stream."""
    _need(x, "x", torch.bfloat16)
    T, H = x.shape
    _need(topk_idx, "topk_idx", torch.int64)
    K = topk_idx.shape[1]
    _need(topk_idx, "topk_idx", torch.int64, (T, K))
    _need(topk_weights, "topk_weights", torch.float32, (T, K))
    R, E = num_ranks, num_experts
    L = layout if layout is not None else alloc_layout(T, E, R, x.device)
    _need(L.slot, "slot", torch.int32, (T, R))
    if L.fused_sync is None:
        raise EPError("the layout has no fused_sync state")
    sync = _per_stream(L.fused_sync, "fused_sync", FUSED_SYNC_WORDS, x.device)
    if out is None:
        cap = capacity if capacity is not None else worst_case_rows(T, K, R)
        out = alloc_dispatched(cap, H, K, E, R, use_fp8, x.device)
    elif out.use_fp8 != use_fp8:
        raise EPError("preallocated dispatch buffers have the wrong payload type")
    if err is not None:
        _need(err, "err", torch.int32)
    _check(lib().ep_layout_dispatch_fused(
        _ptr(x), H, _ptr(topk_idx), _ptr(topk_weights), T, K, E, R,
        _ptr(L.num_tokens_per_rank), _ptr(L.num_tokens_per_expert), _ptr(L.is_token_in_rank),
        _ptr(L.slot), _ptr(L.recv_base), out.recv_x.shape[0], int(use_fp8), _ptr(out.recv_x),
        _ptr(out.recv_scales), _ptr(out.recv_src_idx), _ptr(out.recv_topk_idx),
        _ptr(out.recv_topk_weights), _ptr(out.num_recv_tokens_per_expert), _ptr(L.workspace),
        L.workspace.numel(), _ptr(sync), _ptr(err), _stream(x.device)),
        "ep_layout_dispatch_fused")
    _debug_check("layout_dispatch", err, x.device)
    return L, out


def combine(y: torch.Tensor, topk_idx: torch.Tensor, topk_weights: torch.Tensor | None,
            layout: Layout, *, err: torch.Tensor | None = None,
            out: torch.Tensor | None = None) -> torch.Tensor:
    """out[t] = bf16(sum_k w[t][k] * y[slot[t][rank(e_k)]]) accumulated in
    float32; with topk_weights=None, the unweighted sum of the token's
    destination-rank rows (each rank once).  Enqueued on the current stream."""
    _need(y, "y", torch.bfloat16)
    H = y.shape[1]
    T, K = topk_idx.shape
    _need(topk_idx, "topk_idx", torch.int64, (T, K))
    if topk_weights is not None:
        _need(topk_weights, "topk_weights", torch.float32, (T, K))
    R, E = layout.num_ranks, layout.num_experts
    _need(layout.slot, "slot", torch.int32, (T, R))
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=y.device)
    _need(out, "out", torch.bfloat16, (T, H))
    if err is not None:
        _need(err, "err", torch.int32)
    sched = sched_for(layout, y.device)
    _check(lib().ep_combine_sched(_ptr(y), H, _ptr(topk_idx), _ptr(topk_weights), T, K, E, R,
                                  _ptr(layout.slot), _ptr(out), _ptr(sched), _ptr(err),
                                  _stream(y.device)), "ep_combine_sched")
    _debug_check("combine", err, y.device)
    return out


# --------------------------------------------------------------------------
# sharded form: one rank's own tokens (the exchange is in .sharded)
# --------------------------------------------------------------------------
@dataclass
class ShardLayout:
    """Outputs of shard_layout (all on the device)."""
    send_counts: torch.Tensor       # [R] int32: tokens sent to each destination rank
    expert_counts: torch.Tensor     # [E] int32: slots naming each expert
    is_token_in_rank: torch.Tensor  # [T, R] bool
    send_slot: torch.Tensor         # [T, R] int32: row in the send buffer, -1 = not sent
    send_base: torch.Tensor         # [R + 1] int32: destination r's run starts here
    num_experts: int
    num_ranks: int
    workspace: torch.Tensor | None = None
    sched: torch.Tensor | None = None  # the local combine's counters (as Layout.sched)

    @property
    def slot(self) -> torch.Tensor:  # dispatch and combine read the send slots as slots
        return self.send_slot


def alloc_shard_layout(num_tokens: int, num_experts: int, num_ranks: int,
                       device: torch.device) -> ShardLayout:
    T, R, E = num_tokens, num_ranks, num_experts
    i32 = dict(dtype=torch.int32, device=device)
    ws = torch.empty(max(int(lib().ep_shard_workspace_bytes(T, R, E)), 16), dtype=torch.uint8,
                     device=device)
    return ShardLayout(torch.empty(R, **i32), torch.empty(E, **i32),
                       torch.empty((T, R), dtype=torch.bool, device=device),
                       torch.empty((T, R), **i32), torch.empty(R + 1, **i32), E, R, ws,
                       alloc_combine_sched(device))


def shard_layout(topk_idx: torch.Tensor, num_experts: int, num_ranks: int, *,
                 err: torch.Tensor | None = None, out: ShardLayout | None = None) -> ShardLayout:
    """One rank's layout of its own tokens over num_ranks destinations (any
    number of tokens): its send buffer is packed destination-major in token
    order.  Enqueued on the current stream."""
    _need(topk_idx, "topk_idx", torch.int64)
    if topk_idx.dim() != 2:
        raise EPError("topk_idx must be [num_tokens, num_topk]")
    T, K = topk_idx.shape
    L = out if out is not None else alloc_shard_layout(T, num_experts, num_ranks,
                                                       topk_idx.device)
    if err is not None:
        _need(err, "err", torch.int32)
    _check(lib().ep_shard_layout(_ptr(topk_idx), T, K, num_experts, num_ranks,
                                 _ptr(L.send_counts), _ptr(L.expert_counts),
                                 _ptr(L.is_token_in_rank), _ptr(L.send_slot), _ptr(L.send_base),
                                 _ptr(err), _ptr(L.workspace), L.workspace.numel(),
                                 _stream(topk_idx.device)), "ep_shard_layout")
    _debug_check("shard_layout", err, topk_idx.device)
    return L


def shard_offsets(counts: np.ndarray, rank: int) -> tuple[np.ndarray, np.ndarray]:
    """Host: from the gathered counts [R, R] (counts[s][r] = tokens of rank s
    sent to rank r), this rank's send offsets (its runs in its send buffer)
    and receive offsets (where each source's run lands), both [R + 1] int64."""
    c = np.ascontiguousarray(counts, dtype=np.int32)
    R = c.shape[0]
    if c.shape != (R, R):
        raise EPError("counts must be [R, R]")
    send = np.empty(R + 1, np.int64)
    recv = np.empty(R + 1, np.int64)
    _check(lib().ep_shard_offsets(c.ctypes.data, R, rank, send.ctypes.data, recv.ctypes.data),
           "ep_shard_offsets")
    return send, recv


def shard_recv_tokens_per_expert(expert_counts: np.ndarray, rank: int) -> np.ndarray:
    """Host: from every rank's expert counts [R, E], the rows this rank
    receives per local expert, [E / R] int32."""
    c = np.ascontiguousarray(expert_counts, dtype=np.int32)
    R, E = c.shape
    out = np.empty(E // R if R and E % R == 0 else 0, np.int32)
    _check(lib().ep_shard_recv_tokens_per_expert(c.ctypes.data, E, R, rank, out.ctypes.data),
           "ep_shard_recv_tokens_per_expert")
    return out


# --------------------------------------------------------------------------
# low-latency (expert-major) layout
# --------------------------------------------------------------------------
@dataclass
class LLLayout:
    """Outputs of ll_get_dispatch_layout (all on the device)."""
    ll_slot: torch.Tensor        # [T, K] int32: row of each slot, -1 = none
    ll_count: torch.Tensor       # [E] int32: rows each expert receives
    ll_src_offset: torch.Tensor  # [E, R] int32: first row of each source within its expert
    num_experts: int
    num_ranks: int
    expert_capacity: int
    workspace: torch.Tensor | None = None
    sched: torch.Tensor | None = None  # as Layout.sched

    @property
    def num_rows(self) -> int:
        """Rows of the expert-major buffer: E * expert_capacity."""
        return self.num_experts * self.expert_capacity


def alloc_ll_layout(num_tokens: int, num_topk: int, num_experts: int, num_ranks: int,
                    expert_capacity: int, device: torch.device) -> LLLayout:
    ws = torch.empty(max(int(lib().ep_ll_workspace_bytes(num_tokens, num_ranks, num_experts)), 16),
                     dtype=torch.uint8, device=device)
    return LLLayout(torch.empty((num_tokens, num_topk), dtype=torch.int32, device=device),
                    torch.empty(num_experts, dtype=torch.int32, device=device),
                    torch.empty((num_experts, num_ranks), dtype=torch.int32, device=device),
                    num_experts, num_ranks, int(expert_capacity), ws,
                    alloc_combine_sched(device))


def ll_single_launch_fits(num_tokens: int, num_topk: int, num_ranks: int,
                          num_experts: int) -> bool:
    """True if the one-launch (thread-block cluster) expert-major layout applies."""
    return bool(lib().ep_ll_layout_single_launch_fits(num_tokens, num_topk, num_ranks,
                                                      num_experts))


def ll_auto_single_launch(num_tokens: int, num_topk: int, num_ranks: int,
                          num_experts: int) -> bool:
    """True if path="auto" takes the one-launch expert-major layout."""
    return bool(lib().ep_ll_layout_auto_single_launch(num_tokens, num_topk, num_ranks,
                                                      num_experts))


def ll_get_dispatch_layout(topk_idx: torch.Tensor, num_experts: int, num_ranks: int,
                           expert_capacity: int | None = None, *,
                           err: torch.Tensor | None = None,
                           out: LLLayout | None = None, path: str = "auto") -> LLLayout:
    """Rows of the expert-major layout (default capacity: T rows per expert).
    path: "auto", "multi" or "single" (one cluster launch, small batches)."""
    _need(topk_idx, "topk_idx", torch.int64)
    if path not in LAYOUT_PATHS:
        raise EPError(f"path must be one of {sorted(LAYOUT_PATHS)}")
    T, K = topk_idx.shape
    if out is not None:
        L = out
        cap = L.expert_capacity
    else:
        cap = T if expert_capacity is None else int(expert_capacity)
        L = alloc_ll_layout(T, K, num_experts, num_ranks, cap, topk_idx.device)
    dev = topk_idx.device
    ws = L.workspace
    if err is not None:
        _need(err, "err", torch.int32)
    args = (_ptr(topk_idx), T, K, num_experts, num_ranks, cap, _ptr(L.ll_slot),
            _ptr(L.ll_count), _ptr(L.ll_src_offset), _ptr(err), _ptr(ws), ws.numel())
    if path == "auto":
        _check(lib().ep_ll_get_dispatch_layout(*args, _stream(dev)), "ep_ll_get_dispatch_layout")
    else:
        _check(lib().ep_ll_get_dispatch_layout_path(*args, LAYOUT_PATHS[path], _stream(dev)),
               "ep_ll_get_dispatch_layout_path")
    _debug_check("ll_get_dispatch_layout", err, dev)
    return L


@dataclass
class LLDispatched:
    recv_x: torch.Tensor              # [E*cap, H] bf16 or uint8 (E4M3)
    recv_scales: torch.Tensor | None  # [E*cap, H/128] float32 (FP8 only)
    recv_src_idx: torch.Tensor        # [E*cap] int32
    use_fp8: bool


def ll_dispatch(x: torch.Tensor, layout: LLLayout, *, use_fp8: bool = False,
                err: torch.Tensor | None = None, out: LLDispatched | None = None) -> LLDispatched:
    _need(x, "x", torch.bfloat16)
    T, H = x.shape
    K = layout.ll_slot.shape[1]
    _need(layout.ll_slot, "ll_slot", torch.int32, (T, K))
    rows = layout.num_rows
    if out is None:
        dev = x.device
        out = LLDispatched(
            torch.empty((rows, H), dtype=torch.uint8 if use_fp8 else torch.bfloat16, device=dev),
            torch.empty((rows, H // 128), dtype=torch.float32, device=dev) if use_fp8 else None,
            torch.empty(rows, dtype=torch.int32, device=dev), use_fp8)
    if err is not None:
        _need(err, "err", torch.int32)
    _check(lib().ep_ll_dispatch(_ptr(x), H, T, K, _ptr(layout.ll_slot), out.recv_x.shape[0],
                                int(use_fp8), _ptr(out.recv_x), _ptr(out.recv_scales),
                                _ptr(out.recv_src_idx), _ptr(err), _stream(x.device)),
           "ep_ll_dispatch")
    _debug_check("ll_dispatch", err, x.device)
    return out


def ll_combine(y: torch.Tensor, topk_weights: torch.Tensor | None, layout: LLLayout, *,
               err: torch.Tensor | None = None, out: torch.Tensor | None = None) -> torch.Tensor:
    _need(y, "y", torch.bfloat16)
    H = y.shape[1]
    T, K = layout.ll_slot.shape
    if y.shape[0] < layout.num_rows:
        raise EPError(f"y must have the layout's {layout.num_rows} rows (E * capacity), "
                      f"got {y.shape[0]}")
    if topk_weights is not None:
        _need(topk_weights, "topk_weights", torch.float32, (T, K))
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=y.device)
    _need(out, "out", torch.bfloat16, (T, H))
    if err is not None:
        _need(err, "err", torch.int32)
    sched = sched_for(layout, y.device)
    _check(lib().ep_ll_combine_sched(_ptr(y), H, _ptr(topk_weights), T, K, _ptr(layout.ll_slot),
                                     _ptr(out), _ptr(sched), _ptr(err), _stream(y.device)),
           "ep_ll_combine_sched")
    _debug_check("ll_combine", err, y.device)
    return out


def debug_e4m3_range(first: int, out: torch.Tensor) -> None:
    """Test hook: out[i] = the FP8 dispatch's E4M3 code for the float32 with
    bit pattern first + i (out: uint8, a multiple of 4 elements).  Enqueued on
    the current stream."""
    _need(out, "out", torch.uint8)
    _check(lib().ep_debug_e4m3_range(int(first), out.numel(), _ptr(out), _stream(out.device)),
           "ep_debug_e4m3_range")
