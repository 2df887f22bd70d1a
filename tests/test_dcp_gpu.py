"""Decode context parallelism modelled on one GPU, and the merge at other widths.

Each rank's shard (the tokens the placement of vLLM's mla_attention page,
MLACommonMetadataBuilder, gives it) is laid out in a page pool of its own;
mla_decode runs once per shard with the shard lengths from
mla_dcp_local_seq_lens, and mla_dcp_combine merges the stacked results.
Checked against the oracle: the unsplit definition over the whole sequences,
and the oracle's own per-rank results.
"""

import numpy as np
import pytest

from mla_latent_cache_paged_gb300 import binding
from mla_latent_cache_paged_gb300.workloads import (BF16_NAN, Workload, bf16_bits_to_f64,
                                                    bf16_tensor_bits, f32_to_bf16_bits,
                                                    make_workload)
from oracle import dcp_combine, dcp_decode_partials, dcp_owner, merge_partials
from parity_util import (assert_lse_close, assert_out_close, bf16_ulp, oracle_rows,
                         run_decode, value_abs_max)

pytestmark = pytest.mark.gpu


def _shard(w, world, rank, interleave, seed):
    """The rank's shard of workload `w` as a workload of its own (same q)."""
    ps = w.page_size
    local_lens = binding.dcp_local_seq_lens(w.seq_lens, world, rank, interleave)
    rows = []
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        mine = sorted((dcp_owner(t, world, interleave)[1], t) for t in range(L)
                      if dcp_owner(t, world, interleave)[0] == rank)
        assert len(mine) == local_lens[b]
        t = np.array([t for _, t in mine], dtype=np.int64)
        rows.append(w.cache_bits[w.block_table[b, t // ps], t % ps] if len(t) else
                    np.zeros((0, 576), np.uint16))
    pages = [-(-len(r) // ps) for r in rows]
    nb = max(1, sum(pages))
    rng = np.random.default_rng(seed)
    perm = rng.permutation(nb).astype(np.int32)
    table = np.full((w.batch, max([1] + pages)), -1, dtype=np.int32)
    cache = np.full((nb, ps, 576), BF16_NAN, dtype=np.uint16)   # tail rows: NaN
    k = 0
    for b, r in enumerate(rows):
        for j in range(pages[b]):
            table[b, j] = perm[k]
            chunk = r[j * ps:(j + 1) * ps]
            cache[perm[k], :len(chunk)] = chunk
            k += 1
    return Workload(name=f"{w.name}_r{rank}of{world}", batch=w.batch, num_heads=w.num_heads,
                    seq_lens=local_lens, block_table=table, num_blocks=nb, q_bits=w.q_bits,
                    cache_bits=cache, softmax_scale=w.softmax_scale, num_kv_splits=0,
                    page_size=ps)


@pytest.mark.parametrize("world,interleave", [(2, 1), (2, 64), (4, 16), (3, 1)])
def test_dcp_on_one_gpu_equals_the_unsplit_oracle(world, interleave):
    import torch
    w = make_workload("dcp", 4, 128, [1, 100, 1000, 4097], seed=71)
    outs, lses = [], []
    for r in range(world):
        wr = _shard(w, world, r, interleave, seed=100 + r)
        _, _, _, t = run_decode(wr)
        outs.append(t["out"])
        lses.append(t["lse"])
    out_parts = torch.stack(outs)
    lse_parts = torch.stack(lses)
    out, lse = binding.mla_dcp_combine(out_parts, lse_parts)
    torch.cuda.synchronize()
    got = bf16_bits_to_f64(bf16_tensor_bits(out))

    reqs = range(w.batch)
    ref_out, ref_lse = oracle_rows(w, reqs)
    vmax = value_abs_max(w, reqs)
    assert_out_close(got, ref_out, f"dcp R={world} I={interleave}", vmax)
    assert_lse_close(lse.double().cpu().numpy(), ref_lse, "dcp lse")

    # The oracle's own per-rank results: each rank's GPU decode matches them,
    # and so does their combine.
    q, cache = w.q_f64(), w.cache_f64()
    o_r, l_r = dcp_decode_partials(q, cache, w.block_table, w.seq_lens, w.softmax_scale,
                                   world, interleave)
    for r in range(world):
        got_r = bf16_bits_to_f64(bf16_tensor_bits(outs[r]))
        assert_out_close(got_r, o_r[r], f"rank {r}", vmax)
        assert_lse_close(lses[r].double().cpu().numpy(), l_r[r], f"rank {r} lse")
    c_out, c_lse = dcp_combine(o_r, l_r)
    np.testing.assert_allclose(c_out, ref_out, rtol=1e-10, atol=1e-10)
    # The one-token request lives on rank 0 alone.
    assert np.isneginf(lses[1][0].cpu().numpy()).all()


def _bf16(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


@pytest.mark.parametrize("world,batch,heads,v_dim", [
    (1, 2, 8, 512), (2, 3, 16, 512), (8, 2, 5, 136), (3, 17, 128, 512), (5, 20, 128, 8),
    (4, 2, 3, 1032), (2, 17, 128, 512), (1, 17, 128, 512)])
def test_dcp_combine_against_the_oracle(world, batch, heads, v_dim):
    """Combine of bf16 rank results, both grid shapes (rows below and above 2048)."""
    import torch
    rng = np.random.default_rng(world * 1000 + v_dim)
    o_bits = _bf16(rng.standard_normal((world, batch, heads, v_dim)))
    ls = (rng.standard_normal((world, batch, heads)) * 3).astype(np.float32)
    ls[:, 0, 0] = -np.inf                          # every rank empty: neutral result
    if world > 1:
        ls[1:, 1, :] = -np.inf                     # only rank 0 holds request 1
        o_bits[1:, 1] = BF16_NAN                   # empty ranks' contents are never read
    o_bits[:, 0, 0] = BF16_NAN
    out_parts = torch.from_numpy(o_bits.view(np.int16)).view(torch.bfloat16).cuda()
    out, lse = binding.mla_dcp_combine(out_parts, torch.from_numpy(ls).cuda())
    torch.cuda.synchronize()
    o_ref = np.where(np.isneginf(ls)[..., None], 0.0, bf16_bits_to_f64(o_bits))
    ref_out, ref_lse = dcp_combine(o_ref, ls.astype(np.float64))
    got = bf16_bits_to_f64(bf16_tensor_bits(out))
    # Exact weighted sum, then one rounding to bf16: within one bf16 ulp.
    err = np.abs(got - ref_out)
    assert (err <= bf16_ulp(ref_out) + 1e-5).all(), err.max()
    assert_lse_close(lse.double().cpu().numpy(), ref_lse, "combine lse")
    assert np.all(got[0, 0] == 0) and np.isneginf(lse[0, 0].item())
    if world > 1:
        np.testing.assert_array_equal(bf16_tensor_bits(out)[1], o_bits[0, 1])


@pytest.mark.parametrize("batch,heads,S,v_dim", [(2, 6, 5, 8), (3, 4, 7, 136),
                                                 (17, 128, 3, 136), (2, 2, 4, 2048),
                                                 (17, 128, 2, 512), (16, 128, 4, 512),
                                                 (17, 128, 5, 512)])
def test_merge_splits_at_other_widths(batch, heads, S, v_dim):
    import torch
    rng = np.random.default_rng(S * 7 + v_dim)
    o = rng.standard_normal((batch, heads, S, v_dim)).astype(np.float32)
    ls = (rng.standard_normal((batch, heads, S)) * 2).astype(np.float32)
    ls[0, 0, 1:] = -np.inf
    o[0, 0, 1:] = np.nan
    out, lse = binding.mla_merge_splits(torch.from_numpy(o).cuda(), torch.from_numpy(ls).cuda())
    torch.cuda.synchronize()
    o_ref = np.where(np.isneginf(ls)[..., None], 0.0, o.astype(np.float64))
    ref_out, ref_lse = merge_partials(o_ref, ls.astype(np.float64))
    got = bf16_bits_to_f64(bf16_tensor_bits(out))
    err = np.abs(got - ref_out)
    assert (err <= bf16_ulp(ref_out) + 1e-5).all(), err.max()
    assert_lse_close(lse.double().cpu().numpy(), ref_lse, "merge lse")
