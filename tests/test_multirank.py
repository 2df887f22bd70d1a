"""Multi-rank host logic on CPU: world size 2 over the gloo backend.

Two things run across ranks. The benchmark's reductions: the slowest rank's
time, rank 0's step count, and the whole-job rate. And decode context
parallelism (vLLM mla_attention API docs, MLAAttention.forward): q heads are
all-gathered, each rank attends over its shard of every request's tokens, and
the ranks' (out, lse) pairs are all-gathered and combined; each rank keeps
its own heads. On CPU the oracle stands in for each rank's decode; the shard
lengths come from the library's host function, and the exchange produces the
rank-major layout mla_dcp_combine takes. Child processes are started with
``spawn``.
"""

import math
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)


def _timing_worker(rank, world, port):
    import bench
    _init(rank, world, port)
    try:
        # The slowest rank's time, whichever rank it is.
        assert bench.max_over_ranks(1.5 + rank, world, "cpu") == 1.5 + world - 1
        assert bench.max_over_ranks(9.0 - rank, world, "cpu") == 9.0
        assert bench.agree_on_steps(100 + 7 * rank, world, "cpu") == 100
        # Each rank decodes its own copy of the batch: units add up over ranks.
        assert bench.whole_job_rate(1000, world, 10, 2.0) == 1000 * world * 10 / 2e-3
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _paged(rng, rows_per_req, page_size):
    pages = [-(-len(r) // page_size) for r in rows_per_req]
    nb = sum(pages) + 2
    cache = np.full((nb, page_size, 576), np.nan)
    table = np.full((len(pages), max(pages + [1])), -1, dtype=np.int64)
    perm = rng.permutation(nb)
    k = 0
    for b, rows in enumerate(rows_per_req):
        for j in range(pages[b]):
            table[b, j] = perm[k]
            chunk = rows[j * page_size:(j + 1) * page_size]
            cache[perm[k], :len(chunk)] = chunk
            k += 1
    return cache, table


def _dcp_worker(rank, world, port, interleave):
    from mla_latent_cache_paged_gb300 import binding
    from oracle import dcp_combine, dcp_owner, mla_decode_reference
    _init(rank, world, port)
    try:
        rng = np.random.default_rng(4242)      # same global problem on every rank
        lens = [1, 3, 64, 130, 257]
        heads, page = 4, 16
        scale = 1 / math.sqrt(192)
        dense = [rng.standard_normal((L, 576)) for L in lens]
        q_all = rng.standard_normal((len(lens), heads, 576))
        hs = slice(rank * heads // world, (rank + 1) * heads // world)

        # The rank's shard: the tokens the placement gives it, in local order,
        # in a paged pool of its own.
        local_lens = binding.dcp_local_seq_lens(lens, world, rank, interleave)
        shard = []
        for b, L in enumerate(lens):
            mine = sorted((dcp_owner(t, world, interleave)[1], t) for t in range(L)
                          if dcp_owner(t, world, interleave)[0] == rank)
            assert [j for j, _ in mine] == list(range(len(mine)))
            assert len(mine) == local_lens[b]
            shard.append(dense[b][[t for _, t in mine]])
        cache_r, table_r = _paged(np.random.default_rng(rank), shard, page)

        # Query all-gather over heads: each rank starts with its own heads.
        q_parts = [torch.zeros((len(lens), heads // world, 576), dtype=torch.float64)
                   for _ in range(world)]
        dist.all_gather(q_parts, torch.from_numpy(q_all[:, hs]).contiguous())
        q = torch.cat(q_parts, dim=1).numpy()
        np.testing.assert_array_equal(q, q_all)

        out_r, lse_r = mla_decode_reference(q, cache_r, table_r, local_lens, scale)

        # Exchange of the ranks' results: rank-major, as mla_dcp_combine takes them.
        outs = [torch.zeros(out_r.shape, dtype=torch.float64) for _ in range(world)]
        lses = [torch.zeros(lse_r.shape, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(outs, torch.from_numpy(out_r))
        dist.all_gather(lses, torch.from_numpy(lse_r))
        out_parts = torch.stack(outs).numpy()
        lse_parts = torch.stack(lses).numpy()
        assert out_parts.shape == (world, len(lens), heads, 512)
        assert np.isneginf(lse_parts[:, 0]).sum() == (world - 1) * heads   # 1 token, 1 owner
        out, lse = dcp_combine(out_parts, lse_parts)

        cache, table = _paged(np.random.default_rng(99), dense, page)
        ref_out, ref_lse = mla_decode_reference(q_all, cache, table, lens, scale)
        np.testing.assert_allclose(out[:, hs], ref_out[:, hs], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[:, hs], ref_lse[:, hs], rtol=1e-12, atol=1e-12)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_bench_reductions_over_two_ranks():
    mp.spawn(_timing_worker, args=(WORLD, _free_port()), nprocs=WORLD, join=True)


@pytest.mark.parametrize("interleave", [1, 16])
def test_dcp_decode_over_two_ranks_equals_unsplit(interleave):
    mp.spawn(_dcp_worker, args=(WORLD, _free_port(), interleave), nprocs=WORLD, join=True)
