"""Splitting one packed batch across ranks (linear_attention_chunkwise_gb300.shard), on CPU.

The split's own properties (every sequence on exactly one rank, contiguous, cu_seqlens rebased, tokens
balanced), then a world-size-2 gloo run: each rank computes the prefill of its shard with the fp64
oracle from its own slices of the packed inputs, the ranks gather their outputs, and the concatenation
must equal the single-rank result bit for bit (sequences never exchange data, so nothing on the data
path needs a collective; the gather here is only the test's check).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from linear_attention_chunkwise_gb300 import shard, synth

LENGTHS = [300, 0, 64, 1, 129, 200, 700, 5, 0, 90]
H = 2


def _cu(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


@pytest.mark.parametrize("world", [1, 2, 3, 4, 7, 16])
def test_split_covers_every_sequence_once_and_balances_tokens(world):
    cu = _cu(LENGTHS)
    shards = shard.split_sequences(cu, world)
    assert len(shards) == world
    assert shards[0].seq_begin == 0 and shards[-1].seq_end == len(LENGTHS)
    for a, b in zip(shards, shards[1:]):
        assert a.seq_end == b.seq_begin and a.tok_end == b.tok_begin
    total = int(cu[-1])
    for s in shards:
        assert s.cu_seqlens[0] == 0 and s.cu_seqlens.dtype == np.int32
        np.testing.assert_array_equal(s.cu_seqlens, cu[s.seq_begin:s.seq_end + 1] - cu[s.seq_begin])
        assert s.num_tokens == int(cu[s.seq_end] - cu[s.seq_begin])
        # by midpoints: rank r's first token lies within half the longest sequence of r T / W
        assert abs(s.tok_begin - s.rank * total / world) <= max(LENGTHS) / 2


def test_split_edge_cases():
    assert [s.num_seqs for s in shard.split_sequences([0], 3)] == [0, 0, 0]
    assert [s.num_seqs for s in shard.split_sequences([0, 0, 0], 2)] == [2, 0]
    one = shard.split_sequences([0, 1000], 4)
    assert sum(s.num_seqs for s in one) == 1
    with pytest.raises(ValueError):
        shard.split_sequences([1, 5], 2)
    with pytest.raises(ValueError):
        shard.split_sequences([0, 5, 3], 2)
    assert shard.split_heads(32, 3) == [(0, 11), (11, 22), (22, 32)]
    assert shard.split_heads(2, 4) == [(0, 1), (1, 2), (2, 2), (2, 2)]


def _inputs():
    p = synth.prefill_inputs(LENGTHS, H, s0_std=0.02, seed=77, device="cpu")
    f = lambda t: None if t is None else t.float().numpy()
    return f(p.q), f(p.k), f(p.v), f(p.log_alpha), f(p.beta), f(p.S0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        q, k, v, la, beta, S0 = _inputs()
        sh = shard.split_sequences(_cu(LENGTHS), world)[rank]
        o, sf = oracle.kda_prefill(sh.tokens(q), sh.tokens(k), sh.tokens(v), sh.tokens(la), sh.tokens(beta),
                                   sh.cu_seqlens, sh.seqs(S0), nthreads=1)
        parts = [None] * world
        dist.all_gather_object(parts, (rank, o, sf))
        if rank == 0:
            out["parts"] = parts
    finally:
        dist.destroy_process_group()


def test_two_ranks_reproduce_the_single_rank_prefill():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        parts = out["parts"]
    q, k, v, la, beta, S0 = _inputs()
    o_ref, sf_ref = oracle.kda_prefill(q, k, v, la, beta, _cu(LENGTHS), S0, nthreads=1)
    parts = sorted(parts, key=lambda x: x[0])
    assert all(p[1].shape[0] > 0 for p in parts)  # both ranks got work
    np.testing.assert_array_equal(np.concatenate([p[1] for p in parts]), o_ref)
    np.testing.assert_array_equal(np.concatenate([p[2] for p in parts]), sf_ref)
