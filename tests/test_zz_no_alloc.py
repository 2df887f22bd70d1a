"""GPU: mla_decode_noalloc, the decode for callers that cannot allocate.

Such callers (allocation-free serving loops, runtimes that own all device
memory, bindings that pass only the operation's tensors) give no workspace;
the library's fixed scratch array stands in for it. These checks call the
entry point through the C ABI twice in a row and compare it with mla_decode
(which uses a caller workspace) on the same inputs. This file is collected
last so that a failure here cannot hide the other tests' results.
"""

import numpy as np
import pytest

from mla_latent_cache_paged_gb300 import binding, build
from mla_latent_cache_paged_gb300.workloads import bf16_bits_to_f64, bf16_tensor_bits, make_workload, to_torch
from parity_util import assert_lse_close, assert_out_close, value_abs_max

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("heads,lens,splits", [
    (128, [100, 1000, 5000], 4),     # split partials live in the fixed scratch
    (128, [64, 700], 1),
    (16, [300, 9], 3),                # CUDA-core kernel
])
def test_noalloc_matches_mla_decode_twice(heads, lens, splits):
    import torch
    build.build()
    w = make_workload("noalloc", len(lens), heads, lens, seed=77 + splits, extra_blocks=2,
                      num_kv_splits=splits)
    q, cache, table, seq = to_torch(w)
    plan = binding.make_plan(w.batch, heads, w.max_blocks_per_seq, seq_lens_host=w.seq_lens,
                             max_seq_len=w.max_seq_len, num_kv_splits=splits)
    ws = binding.new_workspace(plan)
    ref_out, ref_lse = binding.mla_decode(q, cache, table, seq, w.softmax_scale, plan=plan,
                                          workspace=ws)
    torch.cuda.synchronize()
    assert binding.read_error(ws) == 0
    ref = bf16_bits_to_f64(bf16_tensor_bits(ref_out))
    vmax = value_abs_max(w, range(w.batch))
    status = torch.full((2,), 12345, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out, lse = binding.mla_decode_noalloc(q, cache, table, seq, w.softmax_scale, plan=plan,
                                              device_status=status)
        torch.cuda.synchronize()
        assert int(status[0].item()) == 0
        got = bf16_bits_to_f64(bf16_tensor_bits(out))
        assert_out_close(got, ref, "noalloc vs mla_decode", vmax)
        assert_lse_close(lse.double().cpu().numpy(), ref_lse.double().cpu().numpy(), "noalloc lse")


def test_noalloc_rejects_plans_beyond_its_scratch():
    build.build()
    plan = binding.make_plan(4, 128, 2048, num_kv_splits=64)   # 4*128*64*2052 B of partials
    assert plan.workspace_bytes > (32 << 20)
    import torch
    q = torch.zeros((4, 128, 576), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((8, 64, 576), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((4, 2048), dtype=torch.int32, device="cuda")
    seq = torch.zeros((4,), dtype=torch.int32, device="cuda")
    with pytest.raises(binding.MlaError) as info:
        binding.mla_decode_noalloc(q, cache, table, seq, 0.07, plan=plan)
    assert info.value.status == binding.MLA_ERR_SCRATCH_LIMIT
