"""GPU: the page-table indexing, checked bit for bit against NumPy indexing."""

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
