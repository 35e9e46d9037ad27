"""The sharded form on CPU ranks (gloo, world sizes 2 and 4): every rank holds
its own tokens; the package's host logic (counts exchange, offsets, one
all-to-all-v per buffer and its reverse for combine) runs unchanged, over
gloo, with each rank's local steps (layout of its own tokens, dispatch into
its send buffer, combine) done by the CPU oracle instead of the GPU.  Each
rank's received rows must equal, bit for bit, its destination's rows of the
single-call oracle layout and dispatch (bf16 rows, or FP8 codes and scales,
with the per-row metadata and per-expert counts), and the combined tokens
the single-call oracle combine of the same expert outputs, bit for bit.  The
same run on the GPU's kernels is tests/test_gpu_sharded.py."""
from __future__ import annotations

import json
import os
import socket
import traceback
from types import SimpleNamespace

import numpy as np
import pytest
import torch


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleSteps:
    """A rank's local steps by the CPU oracle, on CPU tensors."""

    def layout(self, topk_idx, num_experts, num_ranks, err=None):
        import oracle
        L = oracle.shard_layout(topk_idx.numpy(), num_experts, num_ranks)
        return SimpleNamespace(
            send_counts=torch.from_numpy(L.send_counts), expert_counts=torch.from_numpy(L.expert_counts),
            send_slot=L.send_slot, send_base=L.send_base, num_experts=num_experts,
            num_ranks=num_ranks)

    def pack(self, x_bits, topk_idx, topk_weights, layout, rows, use_fp8, err=None):
        import oracle
        d = oracle.dispatch(x_bits.numpy(), topk_idx.numpy(), topk_weights.numpy(),
                            layout.num_experts, layout.num_ranks, layout.send_slot, rows,
                            use_fp8=use_fp8)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a))  # noqa: E731
        recv_x = t(d.recv_x.view(np.int16)) if not use_fp8 else t(d.recv_x)
        return SimpleNamespace(recv_x=recv_x, recv_scales=None if d.recv_scales is None else t(d.recv_scales),
                               recv_src_idx=t(d.recv_src_idx), recv_topk_idx=t(d.recv_topk_idx),
                               recv_topk_weights=t(d.recv_topk_weights))

    def combine(self, y_back, topk_idx, topk_weights, layout, err=None):
        import oracle
        y = y_back.numpy().view(np.uint16)
        if topk_weights is None:  # the rank sum
            out = oracle.combine_ranksum(y, layout.send_slot)
        else:
            out = oracle.combine(y, topk_idx.numpy(), topk_weights.numpy(), layout.num_experts,
                                 layout.num_ranks, layout.send_slot)
        return torch.from_numpy(out.view(np.int16))


def _rank_main(rank, world, port, outdir, fp8):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    from datetime import timedelta
    # a rank that fails makes the others' collectives raise, not wait forever
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=timedelta(seconds=60))
    result = {"ok": False}
    try:
        import oracle
        import workloads
        from combine_get_dispatch_04_gb300 import sharded
        from workloads import Config, make_case
        R, Tr = world, 37                      # ragged: T_r % R != 0
        E, K, H = 4 * R, 4, 256
        cfg = Config(f"shard_r{R}", R, Tr, H, E, K, routing="zipf", zipf_s=1.2, mask_prob=0.1,
                     fp8=fp8, seed=4000 + R)
        c = make_case(cfg)                     # every rank draws the same global batch
        a, b = rank * Tr, (rank + 1) * Tr      # ... and keeps its own tokens
        idx = torch.from_numpy(np.ascontiguousarray(c.topk_idx[a:b]))
        w = torch.from_numpy(np.ascontiguousarray(c.topk_weights[a:b]))
        x = torch.from_numpy(np.ascontiguousarray(c.x_bits[a:b]).view(np.int16))
        ep = sharded.ShardedEP(sharded.DistExchange(), OracleSteps())
        recv, handle = ep.dispatch(x, idx, w, E, use_fp8=fp8)

        # the single-call oracle over the whole batch, destination `rank`
        G = oracle.layout(c.topk_idx, E, R)
        P = G.num_rows
        gd = oracle.dispatch(c.x_bits, c.topk_idx, c.topk_weights, E, R, G.slot, P, use_fp8=fp8)
        lo, hi = int(G.recv_base[rank]), int(G.recv_base[rank + 1])
        assert recv.recv_offsets[-1] == hi - lo
        if fp8:
            np.testing.assert_array_equal(recv.recv_x.numpy(), gd.recv_x[lo:hi])
            np.testing.assert_array_equal(recv.recv_scales.numpy().view(np.uint32),
                                          gd.recv_scales[lo:hi].view(np.uint32))
        else:
            np.testing.assert_array_equal(recv.recv_x.numpy().view(np.uint16), gd.recv_x[lo:hi])
        # source-local token index -> global token index, by source segment
        src = recv.recv_src_idx.numpy().astype(np.int64).copy()
        for s in range(R):
            src[recv.recv_offsets[s]:recv.recv_offsets[s + 1]] += s * Tr
        np.testing.assert_array_equal(src, gd.recv_src_idx[lo:hi])
        np.testing.assert_array_equal(recv.recv_topk_idx.numpy(), gd.recv_topk_idx[lo:hi])
        np.testing.assert_array_equal(recv.recv_topk_weights.numpy().view(np.uint32),
                                      gd.recv_topk_weights[lo:hi].view(np.uint32))
        np.testing.assert_array_equal(
            recv.num_recv_tokens_per_expert,
            oracle.num_recv_tokens_per_expert(G.num_tokens_per_expert, E, R)[rank])

        # combine: expert outputs of the global rows, each rank holding its own
        Y = workloads.expert_outputs(P, H, seed=cfg.seed + 9)
        y = torch.from_numpy(np.ascontiguousarray(Y[lo:hi]).view(np.int16))
        out = ep.combine(y, handle)
        want = oracle.combine(Y, c.topk_idx, c.topk_weights, E, R, G.slot)[a:b]
        np.testing.assert_array_equal(out.numpy().view(np.uint16), want)
        want_u = oracle.combine_ranksum(Y, G.slot)[a:b]
        out_u = ep.combine(y, handle, weighted=False)
        np.testing.assert_array_equal(out_u.numpy().view(np.uint16), want_u)
        result = {"ok": True, "rows": hi - lo}
    except Exception:  # reported to the parent, which fails the test
        result = {"ok": False, "error": traceback.format_exc()}
    finally:
        with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
            json.dump(result, f)
        try:
            dist.barrier()
        finally:
            dist.destroy_process_group()


@pytest.mark.parametrize("world,fp8", [(2, False), (4, False), (2, True), (4, True)])
def test_sharded_exchange_reproduces_the_single_call_oracle(tmp_path, world, fp8):
    import torch.multiprocessing as mp
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path), fp8), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(world)]
    for i, r in enumerate(res):
        assert r["ok"], f"rank {i}:\n{r.get('error')}"
    assert sum(r["rows"] for r in res) > 0


def test_shard_offsets_host_function():
    import combine_get_dispatch_04_gb300 as ep
    counts = np.array([[3, 0, 2], [1, 4, 0], [0, 5, 6]], np.int32)
    send, recv = ep.shard_offsets(counts, 1)
    assert send.tolist() == [0, 1, 5, 5]        # rank 1's row, as a prefix
    assert recv.tolist() == [0, 0, 4, 9]        # column 1 over sources 0, 1, 2
    with pytest.raises(ep.EPError):
        ep.shard_offsets(counts, 3)             # rank outside [0, R)
    with pytest.raises(ep.EPError):
        ep.shard_offsets(np.array([[1, -1], [0, 0]], np.int32), 0)
    per = ep.shard_recv_tokens_per_expert(np.arange(12, dtype=np.int32).reshape(2, 6), 1)
    assert per.tolist() == [3 + 9, 4 + 10, 5 + 11]  # experts 3..5 of rank 1, summed over sources


def _rank_main_unequal(rank, world, port, outdir):
    """Ranks with different numbers of tokens (rank 1 has none): each
    destination's received rows against a brute-force assembly of the runs
    (for every source rank in order, its tokens sent to the destination in
    token order), and the combined tokens against the oracle's combine of the
    rank's own tokens over the rows it gets back."""
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    from datetime import timedelta
    # a rank that fails makes the others' collectives raise, not wait forever
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=timedelta(seconds=60))
    result = {"ok": False}
    try:
        import oracle
        from combine_get_dispatch_04_gb300 import sharded
        R, E, K, H = world, 6 * world, 3, 64
        counts = [23, 0, 41][:world]
        rng = np.random.default_rng(77)  # the same draws on every rank
        idx_all = [np.argsort(rng.random((n, E)), axis=1)[:, :K].astype(np.int64) for n in counts]
        for a in idx_all:
            a[rng.random(a.shape) < 0.2] = -1
        w_all = [rng.random((n, K)).astype(np.float32) for n in counts]
        x_all = [rng.integers(0, 1 << 16, (n, H), dtype=np.uint16) & 0xBFFF for n in counts]
        me = rank
        ep = sharded.ShardedEP(sharded.DistExchange(), OracleSteps())
        recv, handle = ep.dispatch(torch.from_numpy(x_all[me].view(np.int16)),
                                   torch.from_numpy(idx_all[me]), torch.from_numpy(w_all[me]), E)
        El = E // R
        want_rows, want_src = [], []
        for s in range(R):
            for t in range(counts[s]):
                ranks = {int(e) // El for e in idx_all[s][t] if e >= 0}
                if me in ranks:
                    want_rows.append(x_all[s][t])
                    want_src.append(t)
        got = recv.recv_x.numpy().view(np.uint16)
        assert got.shape[0] == len(want_rows)
        if want_rows:
            np.testing.assert_array_equal(got, np.stack(want_rows))
            np.testing.assert_array_equal(recv.recv_src_idx.numpy(), np.array(want_src))
        np.testing.assert_array_equal(np.diff(recv.recv_offsets),
                                      [sum(1 for t in range(counts[s])
                                           if me in {int(e) // El for e in idx_all[s][t] if e >= 0})
                                       for s in range(R)])
        # experts: every received row doubled (exact in bf16)
        y = torch.from_numpy((got.astype(np.uint32) + (1 << 7)).astype(np.uint16).view(np.int16)) \
            if got.size else torch.empty((0, H), dtype=torch.int16)
        out = ep.combine(y, handle)
        sl = oracle.shard_layout(idx_all[me], E, R)
        back = np.zeros((int(sl.send_base[-1]), H), np.uint16)
        for t in range(counts[me]):
            for r in range(R):
                if sl.send_slot[t, r] >= 0:
                    back[sl.send_slot[t, r]] = (x_all[me][t].astype(np.uint32) + (1 << 7)).astype(np.uint16)
        want = oracle.combine(back, idx_all[me], w_all[me], E, R, sl.send_slot)
        np.testing.assert_array_equal(out.numpy().view(np.uint16), want)
        result = {"ok": True}
    except Exception:
        result = {"ok": False, "error": traceback.format_exc()}
    finally:
        with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
            json.dump(result, f)
        try:
            dist.barrier()
        finally:
            dist.destroy_process_group()


def test_sharded_exchange_with_unequal_and_empty_ranks(tmp_path):
    import torch.multiprocessing as mp
    world = 3
    mp.spawn(_rank_main_unequal, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for i in range(world):
        r = json.load(open(tmp_path / f"rank{i}.json"))
        assert r["ok"], f"rank {i}:\n{r.get('error')}"
