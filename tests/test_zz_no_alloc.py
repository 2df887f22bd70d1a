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
    # The stated bounds: 32,632 bf16 split rows fit (B=32, N=128: S=7 fits, S=8
    # does not); with fp32 rows 16,348 (S=3 fits, S=4 does not).
    fp32 = binding.MLA_PLAN_FP32_PARTIALS
    assert binding.make_plan(32, 128, 64, num_kv_splits=7).workspace_bytes <= (32 << 20)
    assert binding.make_plan(32, 128, 64, num_kv_splits=8).workspace_bytes > (32 << 20)
    assert binding.make_plan(32, 128, 64, num_kv_splits=3,
                             extra_flags=fp32).workspace_bytes <= (32 << 20)
    assert binding.make_plan(32, 128, 64, num_kv_splits=4,
                             extra_flags=fp32).workspace_bytes > (32 << 20)
    import torch
    q = torch.zeros((4, 128, 576), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((8, 64, 576), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((4, 2048), dtype=torch.int32, device="cuda")
    seq = torch.zeros((4,), dtype=torch.int32, device="cuda")
    with pytest.raises(binding.MlaError) as info:
        binding.mla_decode_noalloc(q, cache, table, seq, 0.07, plan=plan)
    assert info.value.status == binding.MLA_ERR_SCRATCH_LIMIT


def _balanced_case(seed):
    lens = [1000, 3000, 64, 2000, 1, 700, 129, 4096]
    w = make_workload("noalloc_bal", len(lens), 128, lens, seed=seed, extra_blocks=2,
                      num_kv_splits=0)
    return w


def test_noalloc_page_balanced_writes_only_its_two_status_words():
    """A page-balanced plan: the merge's per-request counters stay in the
    library's scratch. device_status is the first two words of a larger
    buffer filled with a sentinel; every other word must keep it."""
    import torch
    build.build()
    w = _balanced_case(501)
    q, cache, table, seq = to_torch(w)
    plan = binding.make_plan(w.batch, 128, w.max_blocks_per_seq, seq_lens_host=w.seq_lens,
                             max_seq_len=w.max_seq_len, schedule="balanced", num_sms=64)
    assert plan.sched_pairs == 32 and plan.workspace_bytes <= (32 << 20)
    ws = binding.new_workspace(plan)
    ref_out, ref_lse = binding.mla_decode(q, cache, table, seq, w.softmax_scale, plan=plan,
                                          workspace=ws)
    torch.cuda.synchronize()
    assert binding.read_error(ws) == 0
    ref = bf16_bits_to_f64(bf16_tensor_bits(ref_out))
    vmax = value_abs_max(w, range(w.batch))
    guard = torch.full((4096,), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out, lse = binding.mla_decode_noalloc(q, cache, table, seq, w.softmax_scale, plan=plan,
                                              device_status=guard[:2])
        torch.cuda.synchronize()
        words = guard.cpu().numpy()
        assert words[0] == 0 and words[1] == 0, words[:2]
        assert np.all(words[2:] == 0x5A5A5A5A), np.nonzero(words[2:] != 0x5A5A5A5A)
        got = bf16_bits_to_f64(bf16_tensor_bits(out))
        assert_out_close(got, ref, "noalloc balanced vs mla_decode", vmax)
        assert_lse_close(lse.double().cpu().numpy(), ref_lse.double().cpu().numpy(),
                         "noalloc balanced lse")


def test_noalloc_after_a_timed_out_call_starts_from_clean_counters():
    """A call that times out leaves the balanced merge's counters part-way in
    the library's scratch (no caller can reset that array). The test flag
    MLA_PLAN_DEBUG_WITHHOLD_LOAD makes one call time out without a fault;
    the next ordinary call must still match mla_decode."""
    import torch
    build.build()
    w = _balanced_case(502)
    q, cache, table, seq = to_torch(w)
    kw = dict(seq_lens_host=w.seq_lens, max_seq_len=w.max_seq_len, schedule="balanced",
              num_sms=64)
    plan = binding.make_plan(w.batch, 128, w.max_blocks_per_seq, **kw)
    bad = binding.make_plan(w.batch, 128, w.max_blocks_per_seq,
                            extra_flags=binding.MLA_PLAN_DEBUG_WITHHOLD_LOAD, **kw)
    ws = binding.new_workspace(plan)
    ref_out, ref_lse = binding.mla_decode(q, cache, table, seq, w.softmax_scale, plan=plan,
                                          workspace=ws)
    torch.cuda.synchronize()
    assert binding.read_error(ws) == 0
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    binding.mla_decode_noalloc(q, cache, table, seq, w.softmax_scale, plan=bad,
                               device_status=status)
    torch.cuda.synchronize()
    assert int(status[0].item()) == binding.MLA_ERR_TIMEOUT
    for _ in range(2):
        out, lse = binding.mla_decode_noalloc(q, cache, table, seq, w.softmax_scale, plan=plan,
                                              device_status=status)
        torch.cuda.synchronize()
        assert int(status[0].item()) == 0
        assert_out_close(bf16_bits_to_f64(bf16_tensor_bits(out)),
                         bf16_bits_to_f64(bf16_tensor_bits(ref_out)), "noalloc after timeout",
                         value_abs_max(w, range(w.batch)))
        assert_lse_close(lse.double().cpu().numpy(), ref_lse.double().cpu().numpy(),
                         "noalloc after timeout lse")
