"""GPU parity of the page-balanced schedule (sched_pairs > 0) against the oracle.

The schedule cuts the batch's pages, request after request, into C contiguous
ranges (range c = pages [c*P//C, (c+1)*P//C)), one per CTA pair; requests that
cross a range boundary leave partial rows that a merge kernel combines. The
final output is checked against the oracle; the partial rows are checked
against the oracle on exactly the token ranges the cut gives them.
"""

import numpy as np
import pytest

from mla_latent_cache_paged_gb300.workloads import (bf16_bits_to_f64, bf16_tensor_bits,
                                                    make_workload, to_torch)
from parity_util import (assert_lse_close, assert_out_close, assert_out_rel_rms, oracle_rows,
                         run_decode, value_abs_max)

pytestmark = pytest.mark.gpu

PS = 64


SEG_COST = 5   # units of fixed cost per request with pages (the header's cut rule)


def balanced_pieces(lens, pairs):
    """Host restatement of the cut: {request: [(slot, t_lo, t_hi), ...]} for the
    requests whose pages cross a range boundary, and the set of requests whose
    pages lie inside one range."""
    pages = [-(-int(L) // PS) for L in lens]
    units = [pg + SEG_COST if pg > 0 else 0 for pg in pages]
    pfx = np.concatenate([[0], np.cumsum(units)]).astype(np.int64)
    total = int(pfx[-1])
    begin = [c * total // pairs for c in range(pairs + 1)]
    pieces, whole = {}, set()
    for b, L in enumerate(lens):
        if pages[b] == 0:
            continue
        pb, pe = int(pfx[b]) + SEG_COST, int(pfx[b + 1])   # units holding the pages
        cs = [c for c in range(pairs) if begin[c] < pe and begin[c + 1] > pb]
        if len(cs) == 1:
            whole.add(b)
            continue
        pieces[b] = []
        for c in cs:
            lo, hi = max(begin[c], pb), min(begin[c + 1], pe)
            slot = 2 * c if begin[c] >= int(pfx[b]) else 2 * c + 1
            pieces[b].append((slot, (lo - pb) * PS, min(int(L), (hi - pb) * PS)))
    return pieces, whole


@pytest.mark.parametrize("lens,num_sms", [
    ([1, 63, 64, 65, 300, 1000], 6),
    ([1000, 1, 2000, 0, 129], 4),
    ([0, 0, 700], 8),
    ([4096], 16),
    ([64] * 9, 6),
    ([5, 3000, 17, 64, 1, 999, 2048, 77], 152),
])
def test_balanced_parity(lens, num_sms):
    w = make_workload("balanced", len(lens), 128, lens, seed=300 + len(lens) + num_sms,
                      extra_blocks=3, num_kv_splits=0)
    got, lse, plan, _ = run_decode(w, schedule="balanced", num_sms=num_sms)
    assert plan.sched_pairs == min(num_sms // 2, sum(-(-L // PS) for L in lens))
    assert plan.grid_ctas == 2 * plan.sched_pairs
    ref_out, ref_lse = oracle_rows(w, range(w.batch))
    assert_out_close(got, ref_out, "balanced", value_abs_max(w, range(w.batch)))
    assert_out_rel_rms(got, ref_out, "balanced")
    assert_lse_close(lse, ref_lse, "balanced lse")


def test_balanced_partials_cover_their_ranges():
    import torch
    lens = [1000, 1, 2000, 0, 129, 640]
    w = make_workload("bal_parts", len(lens), 128, lens, seed=77, extra_blocks=2, num_kv_splits=0)
    _, _, plan, t = run_decode(w, schedule="balanced", num_sms=10)
    C, N = plan.sched_pairs, w.num_heads
    pieces, whole = balanced_pieces(lens, C)
    assert pieces, "the cut should split at least one request"
    ws = t["ws"]
    rows = 2 * C * N
    o_part = ws[plan.partial_offset:plan.partial_offset + rows * 512 * 4]
    o_part = o_part.view(torch.float32).view(2 * C, N, 512).double().cpu().numpy()
    l_part = ws[plan.lse_partial_offset:plan.lse_partial_offset + rows * 4]
    l_part = l_part.view(torch.float32).view(2 * C, N).double().cpu().numpy()
    for b, plist in pieces.items():
        for slot, lo, hi in plist:
            # The oracle over tokens [lo, hi) of request b: the same request
            # with its block table advanced by lo/64 pages (lo is page-aligned).
            sub = make_workload("bal_sub", 1, N, [hi - lo], seed=1, extra_blocks=0, num_kv_splits=1)
            sub.q_bits = w.q_bits[b:b + 1]
            sub.cache_bits = w.cache_bits
            sub.num_blocks = w.num_blocks
            table = np.full((1, w.block_table.shape[1]), -1, dtype=w.block_table.dtype)
            n = -(-(hi - lo) // PS)
            table[0, :n] = w.block_table[b, lo // PS:lo // PS + n]
            sub.block_table = table
            sub.softmax_scale = w.softmax_scale
            ref_o, ref_l = oracle_rows(sub, [0])
            assert_lse_close(l_part[slot], ref_l[0], f"lse piece b={b} slot={slot}")
            # fp32 partial normalised by the bf16 weights the P.V MMA used:
            # the bound is the one the bf16 output is held to.
            err = np.abs(o_part[slot] - ref_o[0]).max()
            assert err < 2e-2, (b, slot, err)



def test_balanced_merge_counters_return_to_zero():
    """The merge of the balanced schedule waits on per-request counters in the
    workspace's status header; every call must leave them at zero, so that the
    same workspace serves the next call (bit-identical results)."""
    import torch
    from mla_latent_cache_paged_gb300 import binding
    lens = [1000, 1, 2000, 0, 129, 640, 3000, 77]
    w = make_workload("bal_ctr", len(lens), 128, lens, seed=91, extra_blocks=2, num_kv_splits=0)
    _, _, plan, t = run_decode(w, schedule="balanced", num_sms=10)
    ws = t["ws"]
    words = ws[:binding.STATUS_BYTES].view(torch.int32).cpu().numpy()
    assert not words[2:].any(), np.nonzero(words[2:])
    first_out, first_lse = t["out"].clone(), t["lse"].clone()
    for _ in range(3):
        out, lse = binding.mla_decode(t["q"], t["cache"], t["table"], t["lens"], w.softmax_scale,
                                      plan=plan, workspace=ws)
        torch.cuda.synchronize()
        assert binding.read_error(ws) == 0
        assert torch.equal(out, first_out) and torch.equal(lse, first_lse)
    words = ws[:binding.STATUS_BYTES].view(torch.int32).cpu().numpy()
    assert not words[2:].any(), np.nonzero(words[2:])


def test_merge_wait_runs_out_and_reports_a_timeout():
    """Failure detection without a fault: the balanced merge waits (bounded,
    4 s) for a request's pieces through a counter in the status header. A
    counter started far below zero never reaches its target, so the wait runs
    out: the call reports MLA_ERR_TIMEOUT (detail 20: the merge's wait), the
    context stays usable, and after mla_workspace_init the same plan decodes
    correctly again."""
    import torch
    from mla_latent_cache_paged_gb300 import binding
    ready_word = 64          # status header: int32 word 64 + b counts request b's pieces
    lens = [4096, 4096]
    w = make_workload("bal_timeout", len(lens), 128, lens, seed=93, num_kv_splits=0)
    q, cache, table, lens_d = to_torch(w)
    plan = binding.make_plan(w.batch, w.num_heads, w.max_blocks_per_seq,
                             seq_lens_host=w.seq_lens, schedule="balanced")
    assert plan.sched_pairs > 1
    ws = binding.new_workspace(plan)
    ws[:binding.STATUS_BYTES].view(torch.int32)[ready_word + 0] = -(1 << 30)
    binding.mla_decode(q, cache, table, lens_d, w.softmax_scale, plan=plan, workspace=ws)
    torch.cuda.synchronize()
    words = ws[:8].view(torch.int32).cpu().numpy()
    assert words[0] == binding.MLA_ERR_TIMEOUT and words[1] == 20, words
    assert binding.read_error(ws) == binding.MLA_ERR_TIMEOUT
    assert binding.load_library().mla_workspace_init(binding._ptr(ws), ws.numel(),
                                                     binding._stream_ptr(None)) == 0
    out, lse = binding.mla_decode(q, cache, table, lens_d, w.softmax_scale, plan=plan,
                                  workspace=ws)
    torch.cuda.synchronize()
    assert binding.read_error(ws) == 0
    header = ws[:binding.STATUS_BYTES].view(torch.int32).cpu().numpy()
    assert not header.any(), np.nonzero(header)
    ref_out, ref_lse = oracle_rows(w, range(w.batch))
    assert_out_close(bf16_bits_to_f64(bf16_tensor_bits(out)), ref_out, "after the timeout",
                     value_abs_max(w, range(w.batch)))
    assert_lse_close(lse.double().cpu().numpy(), ref_lse, "after the timeout")
