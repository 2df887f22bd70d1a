"""GPU: failure detection without a fault, through the C ABI.

Every wait inside the tensor-core decode kernel is bounded. The test flag
MLA_PLAN_DEBUG_WITHHOLD_LOAD makes CTA 0 skip its first K-ring load (a flag
that nothing sets) and shortens the call's wait limit to 2 ms: the score
warp's wait for that page runs out, the kernel records MLA_ERR_TIMEOUT with
the wait's site (8, the K-ring wait), every role drains what it issued, TMEM
is freed and the kernel returns. The context stays usable: after
mla_workspace_init the same workspace decodes to the oracle again.
"""

import numpy as np
import pytest

from mla_latent_cache_paged_gb300 import binding
from mla_latent_cache_paged_gb300.workloads import (bf16_bits_to_f64, bf16_tensor_bits,
                                                    make_workload, to_torch)
from parity_util import assert_lse_close, assert_out_close, oracle_rows, value_abs_max

pytestmark = pytest.mark.gpu

K_RING_WAIT_SITE = 8


@pytest.mark.parametrize("schedule,splits", [("split", 1), ("split", 3), ("balanced", 0)])
def test_decode_wait_runs_out_and_the_workspace_recovers(schedule, splits):
    import torch
    lens = [700, 1000, 65, 2048, 1]
    w = make_workload("withhold", len(lens), 128, lens, seed=811 + splits, extra_blocks=2,
                      num_kv_splits=splits)
    q, cache, table, seq = to_torch(w)
    kw = dict(seq_lens_host=w.seq_lens, max_seq_len=w.max_seq_len, num_kv_splits=splits,
              schedule=schedule, num_sms=16)
    bad = binding.make_plan(w.batch, 128, w.max_blocks_per_seq,
                            extra_flags=binding.MLA_PLAN_DEBUG_WITHHOLD_LOAD, **kw)
    plan = binding.make_plan(w.batch, 128, w.max_blocks_per_seq, **kw)
    assert plan.kernel == binding.MLA_KERNEL_TC
    assert (plan.sched_pairs > 0) == (schedule == "balanced")
    ws = binding.new_workspace(plan)
    binding.mla_decode(q, cache, table, seq, w.softmax_scale, plan=bad, workspace=ws)
    torch.cuda.synchronize()                      # the context is still usable
    words = ws[:8].view(torch.int32).cpu().numpy()
    assert words[0] == binding.MLA_ERR_TIMEOUT and words[1] == K_RING_WAIT_SITE, words
    assert binding.read_error(ws) == binding.MLA_ERR_TIMEOUT
    # Recovery in the same workspace: re-initialise its status header (the
    # balanced merge may have left counters part-way), then decode normally.
    binding.load_library().mla_workspace_init(binding._ptr(ws), ws.numel(),
                                              binding._stream_ptr(None))
    for _ in range(2):
        out, lse = binding.mla_decode(q, cache, table, seq, w.softmax_scale, plan=plan,
                                      workspace=ws)
        torch.cuda.synchronize()
        assert binding.read_error(ws) == 0
        header = ws[:binding.STATUS_BYTES].view(torch.int32).cpu().numpy()
        assert not header.any(), np.nonzero(header)
        ref_out, ref_lse = oracle_rows(w, range(w.batch))
        assert_out_close(bf16_bits_to_f64(bf16_tensor_bits(out)), ref_out, "after the timeout",
                         value_abs_max(w, range(w.batch)))
        assert_lse_close(lse.double().cpu().numpy(), ref_lse, "after the timeout")
