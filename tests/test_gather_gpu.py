"""GPU: the page-table indexing, checked bit for bit against NumPy indexing:
the plain gather hook, and the tensor-core decode kernel's own TMA loaders."""

import numpy as np
import pytest

from mla_latent_cache_paged_gb300 import binding
from mla_latent_cache_paged_gb300.workloads import bf16_tensor_bits, make_workload, to_torch

pytestmark = pytest.mark.gpu

SENTINEL = 0x1234


@pytest.mark.parametrize("lens", [[1, 63, 64, 65, 1000], [256], [0, 5, 4096]])
def test_gather_pages_bit_exact(lens):
    import torch
    w = make_workload("gather", len(lens), 1, lens, seed=41, extra_blocks=6)
    _, cache, table, seq = to_torch(w)
    T = max(max(lens), 1) + 3
    dst = torch.full((w.batch, T, 576), SENTINEL, dtype=torch.int16, device="cuda")
    dst = dst.view(torch.bfloat16)
    ws = torch.zeros(binding.STATUS_BYTES, dtype=torch.uint8, device="cuda")
    binding.debug_gather_pages(cache, table, seq, dst, ws)
    torch.cuda.synchronize()
    assert binding.read_error(ws) == 0
    got = bf16_tensor_bits(dst)
    for b, L in enumerate(lens):
        t = np.arange(L)
        want = w.cache_bits[w.block_table[b, t // 64], t % 64]
        assert np.array_equal(got[b, :L], want), b
        assert np.all(got[b, L:] == SENTINEL), b


def test_gather_reports_bad_block_ids():
    import torch
    w = make_workload("gather_bad", 2, 1, [100, 10], seed=42)
    _, cache, table, seq = to_torch(w)
    table[0, 1] = w.num_blocks
    dst = torch.zeros((2, 128, 576), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(binding.STATUS_BYTES, dtype=torch.uint8, device="cuda")
    binding.debug_gather_pages(cache, table, seq, dst, ws)
    assert binding.read_error(ws) == binding.MLA_ERR_BAD_BLOCK_ID


@pytest.mark.parametrize("lens,splits,schedule,num_sms", [
    ([1, 63, 64, 65, 1000, 4096], 1, "split", 152),
    ([1, 63, 64, 65, 1000, 4096], 3, "split", 8),
    ([700, 0, 129, 2000, 5, 64], 0, "balanced", 10),
    ([4096, 3000], 0, "balanced", 152),
])
def test_decode_loader_receives_every_row_bit_exact(lens, splits, schedule, num_sms):
    """The tensor-core decode kernel's own page loaders (its segment walk,
    block-table reads, tensor map, 64 x 64 boxes at row block * 64 and the
    swizzled rings), run alone: each CTA of a pair copies out every page it
    received; both must hold exactly the cache rows NumPy indexing gives, and
    nothing past a request's length."""
    import torch
    w = make_workload("loader", len(lens), 128, lens, seed=45 + len(lens) + num_sms,
                      extra_blocks=5, num_kv_splits=splits)
    _, cache, table, seq = to_torch(w)
    plan = binding.make_plan(w.batch, 128, w.max_blocks_per_seq, seq_lens_host=w.seq_lens,
                             max_seq_len=w.max_seq_len, num_kv_splits=splits,
                             schedule=schedule, num_sms=num_sms)
    assert plan.kernel == binding.MLA_KERNEL_TC
    assert (plan.sched_pairs > 0) == (schedule == "balanced")
    T = max(max(lens), 1) + 5
    dst = torch.full((2, w.batch, T, 576), SENTINEL, dtype=torch.int16, device="cuda")
    dst = dst.view(torch.bfloat16)
    ws = binding.new_status_workspace()
    binding.debug_loader_pages(plan, cache, table, seq, dst, ws)
    torch.cuda.synchronize()
    assert binding.read_error(ws) == 0
    got = bf16_tensor_bits(dst)
    for b, L in enumerate(lens):
        t = np.arange(L)
        want = w.cache_bits[w.block_table[b, t // 64], t % 64]
        for r in range(2):
            assert np.array_equal(got[r, b, :L], want), (r, b)
            assert np.all(got[r, b, L:] == SENTINEL), (r, b)


def test_decode_loader_zero_fills_and_reports_a_bad_block():
    import torch
    w = make_workload("loader_bad", 2, 128, [200, 64], seed=46, num_kv_splits=1)
    _, cache, table, seq = to_torch(w)
    table[0, 1] = w.num_blocks + 3
    plan = binding.make_plan(2, 128, w.max_blocks_per_seq, num_kv_splits=1)
    dst = torch.full((2, 2, 256, 576), SENTINEL, dtype=torch.int16, device="cuda")
    dst = dst.view(torch.bfloat16)
    ws = binding.new_status_workspace()
    binding.debug_loader_pages(plan, cache, table, seq, dst, ws)
    assert binding.read_error(ws) == binding.MLA_ERR_BAD_BLOCK_ID
    got = bf16_tensor_bits(dst)
    for r in range(2):
        assert np.all(got[r, 0, 64:128] == 0)          # the bad page reads as zeros
        t = np.arange(64)
        assert np.array_equal(got[r, 0, :64], w.cache_bits[w.block_table[0, 0], t])
        assert np.array_equal(got[r, 0, 128:192], w.cache_bits[w.block_table[0, 2], t])
        assert np.array_equal(got[r, 0, 192:200], w.cache_bits[w.block_table[0, 3], t[:8]])
        assert np.all(got[r, 0, 200:] == SENTINEL)
