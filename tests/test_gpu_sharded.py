"""GPU parity of the sharded form's kernels: ep_shard_layout against the
oracle's one-rank layout (bit-exact, any T, bad ids, empty), and whole
sharded dispatch / combine runs of R ranks emulated in one process on one
GPU: one host thread per rank, each on its own stream, calling the package's
ShardedEP unchanged with the CUDA library's steps; the collectives are
replaced by an in-process exchange (device copies between the threads'
buffers, after a synchronise).  Every rank's received rows must equal its
destination's rows of the single-call oracle bit for bit (bf16 or FP8 codes
and scales, metadata, per-expert counts), and its combined tokens the
single-call oracle combine within the combine tolerance."""
from __future__ import annotations

import os

import threading

import numpy as np
import pytest
import torch

import oracle
import workloads
from ep_testlib import assert_combine_close, bits_of, combine_bound
from test_gpu_adversarial import CASES as _ADV, _case as _adv_case
from workloads import Config, make_case

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,R,E,K,seed", [(1, 1, 3, 2, 1), (301, 4, 16, 4, 2), (129, 8, 64, 8, 3),
                                          (1000, 64, 128, 8, 4), (4096, 32, 256, 8, 5)])
def test_shard_layout_matches_oracle(ep, T, R, E, K, seed):
    rng = np.random.default_rng(seed)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int64)
    idx[rng.random((T, K)) < 0.1] = -1
    if T > 3:
        idx[2, 0] = E + 7  # a bad id
    want = oracle.shard_layout(idx, E, R)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = ep.shard_layout(torch.from_numpy(idx).cuda(), E, R, err=err)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(L.send_slot.cpu().numpy(), want.send_slot)
    np.testing.assert_array_equal(L.send_base.cpu().numpy(), want.send_base)
    np.testing.assert_array_equal(L.send_counts.cpu().numpy(), want.send_counts)
    np.testing.assert_array_equal(L.expert_counts.cpu().numpy(), want.expert_counts)
    np.testing.assert_array_equal(L.is_token_in_rank.view(torch.uint8).cpu().numpy(),
                                  want.is_token_in_rank)
    assert int(err.item()) == want.err_bits


def test_shard_layout_empty(ep):
    L = ep.shard_layout(torch.empty((0, 4), dtype=torch.int64, device="cuda"), 16, 4)
    torch.cuda.synchronize()
    assert not L.send_counts.any() and not L.expert_counts.any() and not L.send_base.any()


class ThreadExchange:
    """The collectives for R ranks that are host threads of one process."""

    def __init__(self, shared, rank, world):
        self.sh, self.rank, self.world = shared, rank, world

    def _sync(self):
        torch.cuda.current_stream().synchronize()
        self.sh["barrier"].wait()

    def all_gather_rows(self, row):
        self.sh["rows"][self.rank] = row
        self._sync()
        out = torch.stack([r.clone() for r in self.sh["rows"]])
        self._sync()
        return out

    def all_to_all_rows(self, out, inp, out_splits, in_splits):
        self.sh["a2a"][self.rank] = (inp, np.concatenate([[0], np.cumsum(in_splits)]))
        self._sync()
        pos = 0
        for s in range(self.world):
            src, off = self.sh["a2a"][s]
            n = int(off[self.rank + 1] - off[self.rank])
            assert n == int(out_splits[s])
            if n:
                out[pos:pos + n].copy_(src[int(off[self.rank]):int(off[self.rank]) + n])
            pos += n
        self._sync()


def masked_case(cfg, masked_ranks=(), with_hidden=True, routing=None):
    """The workload's case (with the given top-k ids instead of its own, if
    any), with every slot of the tokens of masked_ranks set to -1."""
    c = make_case(cfg, with_hidden=with_hidden)
    if routing is not None:
        c.topk_idx[:] = routing
    Tr = cfg.tokens_per_rank
    for r in masked_ranks:
        c.topk_idx[r * Tr:(r + 1) * Tr] = -1
    return c


def run_ranks(ep, cfg, fp8, y_global, masked_ranks=(), routing=None):
    from combine_get_dispatch_04_gb300 import sharded
    c = masked_case(cfg, masked_ranks, routing=routing)
    R, Tr, E = cfg.num_ranks, cfg.tokens_per_rank, cfg.num_experts
    shared = {"barrier": threading.Barrier(R), "rows": [None] * R, "a2a": [None] * R}
    results, errors = [None] * R, []

    def rank_main(rank):
        try:
            torch.cuda.set_device(0)
            with torch.cuda.stream(torch.cuda.Stream()):
                a, b = rank * Tr, (rank + 1) * Tr
                idx = torch.from_numpy(np.ascontiguousarray(c.topk_idx[a:b])).cuda()
                w = torch.from_numpy(np.ascontiguousarray(c.topk_weights[a:b])).cuda()
                x = torch.from_numpy(np.ascontiguousarray(c.x_bits[a:b]).view(np.int16)).cuda() \
                    .view(torch.bfloat16)
                err = torch.zeros(1, dtype=torch.int32, device="cuda")
                sep = sharded.ShardedEP(ThreadExchange(shared, rank, R))
                recv, handle = sep.dispatch(x, idx, w, E, use_fp8=fp8, err=err)
                lo = int(recv_base_global[rank])
                n = int(recv.recv_offsets[-1])
                y = torch.from_numpy(np.ascontiguousarray(y_global[lo:lo + n]).view(np.int16)).cuda() \
                    .view(torch.bfloat16)
                out = sep.combine(y, handle, err=err)
                torch.cuda.current_stream().synchronize()
                results[rank] = (recv, out, int(err.item()))
        except Exception as e:  # noqa: BLE001 -- reported below
            errors.append((rank, repr(e)))
            shared["barrier"].abort()

    G = oracle.layout(c.topk_idx, E, R)
    recv_base_global = G.recv_base
    threads = [threading.Thread(target=rank_main, args=(r,)) for r in range(R)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    return c, G, results


@pytest.mark.parametrize("cfg", [
    Config("shard_gpu_bf16", 4, 301, 1024, 16, 4, routing="zipf", zipf_s=1.2, mask_prob=0.05,
           seed=4100),
    Config("shard_gpu_fp8", 4, 129, 1024, 32, 6, fp8=True, seed=4101),
    Config("shard_gpu_decode", 8, 128, 7168, 64, 8, fp8=True, seed=4102),
], ids=lambda c: c.name)
def test_sharded_ranks_on_one_gpu_match_the_single_call_oracle(ep, cfg):
    check_sharded_against_single_call(ep, cfg)


@pytest.mark.parametrize("fp8", [False, True])
def test_sharded_rank_with_every_slot_masked(ep, fp8):
    """A rank whose tokens all go nowhere sends no rows: its dispatch writes
    into an empty send buffer and its combine reads no row (all its tokens
    come back as zeros); the other ranks still exchange with it."""
    cfg = Config("shard_gpu_masked_rank", 4, 96, 256, 16, 4, fp8=fp8, seed=4103)
    check_sharded_against_single_call(ep, cfg, masked_ranks=(1,))


def check_sharded_against_single_call(ep, cfg, masked_ranks=(), routing=None):
    R, Tr, E, H = cfg.num_ranks, cfg.tokens_per_rank, cfg.num_experts, cfg.hidden
    c0 = masked_case(cfg, masked_ranks, with_hidden=False, routing=routing)
    P = oracle.layout(c0.topk_idx, E, R).num_rows
    Y = workloads.expert_outputs(max(P, 1), H, seed=cfg.seed + 9)
    c, G, results = run_ranks(ep, cfg, cfg.fp8, Y, masked_ranks, routing)
    gd = oracle.dispatch(c.x_bits, c.topk_idx, c.topk_weights, E, R, G.slot, P, use_fp8=cfg.fp8)
    nrpe = oracle.num_recv_tokens_per_expert(G.num_tokens_per_expert, E, R)
    want_out = oracle.combine(Y, c.topk_idx, c.topk_weights, E, R, G.slot)
    bound = combine_bound(oracle.bf16_to_double(Y), c.topk_idx, c.topk_weights, G.slot, E // R,
                          np.arange(cfg.num_tokens))
    for rank, (recv, out, err) in enumerate(results):
        # bad ids in the rank's own tokens, as its shard layout reports them
        assert err == oracle.shard_layout(c.topk_idx[rank * Tr:(rank + 1) * Tr], E, R).err_bits
        lo, hi = int(G.recv_base[rank]), int(G.recv_base[rank + 1])
        if cfg.fp8:
            np.testing.assert_array_equal(recv.recv_x.cpu().numpy(), gd.recv_x[lo:hi])
            np.testing.assert_array_equal(recv.recv_scales.cpu().numpy().view(np.uint32),
                                          gd.recv_scales[lo:hi].view(np.uint32))
        else:
            np.testing.assert_array_equal(bits_of(recv.recv_x), gd.recv_x[lo:hi])
        src = recv.recv_src_idx.cpu().numpy().astype(np.int64)
        for s in range(R):
            src[recv.recv_offsets[s]:recv.recv_offsets[s + 1]] += s * Tr
        np.testing.assert_array_equal(src, gd.recv_src_idx[lo:hi])
        np.testing.assert_array_equal(recv.recv_topk_idx.cpu().numpy(), gd.recv_topk_idx[lo:hi])
        np.testing.assert_array_equal(recv.recv_topk_weights.cpu().numpy().view(np.uint32),
                                      gd.recv_topk_weights[lo:hi].view(np.uint32))
        np.testing.assert_array_equal(recv.num_recv_tokens_per_expert, nrpe[rank])
        a, b = rank * Tr, (rank + 1) * Tr
        assert_combine_close(bits_of(out), want_out[a:b], bound[a:b])


@pytest.mark.parametrize("i", range(int(os.environ.get("EP_SHARDED_CASES", "64"))))
def test_sharded_random_shapes(ep, i):
    """The random sweep's generator, kept to at most 16 ranks (one host thread
    each): bf16 rows, and FP8 where H % 128 == 0."""
    from test_gpu_random import random_config
    j = i
    cfg = random_config(j)
    while cfg.num_ranks > 16:  # the next shapes of the same sweep
        j += 100
        cfg = random_config(j)
    for fp8 in ([False, True] if cfg.hidden % 128 == 0 else [False]):
        c = cfg.__class__(**{**cfg.__dict__, "fp8": fp8})
        test_sharded_ranks_on_one_gpu_match_the_single_call_oracle(ep, c)


@pytest.mark.parametrize("i", [i for i, (_, shape) in enumerate(_ADV) if shape[1] <= 16],
                         ids=lambda i: "{}-{}".format(_ADV[i][0], _ADV[i][1][0]))
def test_sharded_adversarial_routing(ep, i):
    """The adversarial routings (duplicate experts, bad ids, one hot expert or
    rank, masked tokens) through the sharded exchange, up to 16 ranks: ranks
    that send or receive nothing included."""
    kind, shape = _ADV[i]
    cfg, c = _adv_case(kind, shape, i)
    for fp8 in ([False, True] if cfg.hidden % 128 == 0 else [False]):
        check_sharded_against_single_call(ep, cfg.__class__(**{**cfg.__dict__, "fp8": fp8}),
                                          routing=c.topk_idx)
