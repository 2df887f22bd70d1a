"""The boundary calls are graph-capturable (no host synchronisation inside).

A whole decode step -- front end (q absorption, q_pe concat, cache insert),
decode (+ its merge), up-projection -- is captured into one CUDA graph and
replayed; every replay matches the same calls run eagerly, bit for bit, also
after the graph's input buffers are refilled with new values. The
page-balanced schedule's merge keeps per-request counters in the workspace,
which must be back at zero after every replay for the next one to work.
"""

import numpy as np
import pytest

from mla_latent_cache_paged_gb300 import binding
from mla_latent_cache_paged_gb300.workloads import make_workload, to_torch

pytestmark = pytest.mark.gpu


def _step(inp, cache, table, lens, scale, plan, ws, status, outs):
    binding.mla_q_absorb_concat_cache(inp["q"], inp["w_uk_t"], inp["kv_c"], inp["k_pe"],
                                      inp["slots"], cache, workspace=status, out=outs["mqa_q"])
    binding.mla_decode(outs["mqa_q"], cache, table, lens, scale, plan=plan, out=outs["lat"],
                       lse=outs["lse"], workspace=ws)
    binding.mla_v_up_proj(outs["lat"], inp["w_uv"], workspace=status, out=outs["o"])


@pytest.mark.parametrize("schedule,splits", [("split", 4), ("balanced", 0)])
def test_decode_step_replays_in_a_cuda_graph(schedule, splits):
    import torch
    B, N = 6, 128
    lens_host = [64, 200, 1, 1000, 130, 77]
    w = make_workload("graph", B, N, lens_host, seed=1700)
    _, cache, table, lens = to_torch(w)
    gen = torch.Generator(device="cuda").manual_seed(1701)

    def inputs():
        t = lambda *s, sc=1.0: (torch.randn(s, generator=gen, device="cuda") * sc).to(torch.bfloat16)
        # The new token is each request's last cached token (position L - 1):
        # the insert writes its row before the decode reads it.
        slot = [int(w.block_table[b, (L - 1) // 64]) * 64 + (L - 1) % 64 for b, L in enumerate(lens_host)]
        return dict(q=t(B, N, 192), w_uk_t=t(N, 128, 512, sc=128 ** -0.5),
                    kv_c=t(B, 512), k_pe=t(B, 64), w_uv=t(N, 512, 128, sc=512 ** -0.5),
                    slots=torch.tensor(slot, dtype=torch.int64, device="cuda"))

    plan = binding.make_plan(B, N, w.max_blocks_per_seq, seq_lens_host=w.seq_lens,
                             num_kv_splits=splits, schedule=schedule)
    assert (plan.sched_pairs > 0) == (schedule == "balanced")
    ws = binding.new_workspace(plan)
    status = binding.new_status_workspace()
    new_outs = lambda: dict(mqa_q=torch.empty((B, N, 576), dtype=torch.bfloat16, device="cuda"),
                            lat=torch.empty((B, N, 512), dtype=torch.bfloat16, device="cuda"),
                            lse=torch.empty((B, N), dtype=torch.float32, device="cuda"),
                            o=torch.empty((B, N, 128), dtype=torch.bfloat16, device="cuda"))
    static_in, static_out = inputs(), new_outs()
    cache_g = cache.clone()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _step(static_in, cache_g, table, lens, w.softmax_scale, plan, ws, status, static_out)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _step(static_in, cache_g, table, lens, w.softmax_scale, plan, ws, status, static_out)

    for rnd in range(3):
        if rnd:
            fresh = inputs()
            for k in static_in:
                static_in[k].copy_(fresh[k])
        cache_e = cache.clone()
        eager = new_outs()
        ws_e = binding.new_workspace(plan)
        _step(static_in, cache_e, table, lens, w.softmax_scale, plan, ws_e, status, eager)
        cache_g.copy_(cache)
        graph.replay()
        torch.cuda.synchronize()
        assert binding.read_error(ws) == 0 and binding.read_error(status) == 0
        for k in eager:
            np.testing.assert_array_equal(static_out[k].view(torch.int16 if k != "lse" else torch.int32)
                                          .cpu().numpy(),
                                          eager[k].view(torch.int16 if k != "lse" else torch.int32)
                                          .cpu().numpy(), err_msg=f"{k} replay {rnd}")
        assert torch.equal(cache_g.view(torch.int16), cache_e.view(torch.int16))


@pytest.mark.parametrize("kind", ["fp8", "v_up_proj"])
def test_fp8_decode_and_fused_up_projection_replay_in_a_cuda_graph(kind):
    """mla_decode_fp8 (page-balanced plan, its merge's counters) and
    mla_decode_v_up_proj (split plan: the decode, then the merge fused into
    the up-projection) captured into a graph and replayed: every replay
    matches the same call run eagerly bit for bit, with new q each time."""
    import torch
    B, N = 6, 128
    lens_host = [64, 200, 1, 1000, 130, 77]
    fp8 = kind == "fp8"
    w = make_workload("graph2", B, N, lens_host, seed=1710, extra_blocks=2,
                      cache_dtype="fp8" if fp8 else "bf16")
    q, cache, table, lens = to_torch(w)
    plan = binding.make_plan(B, N, w.max_blocks_per_seq, seq_lens_host=w.seq_lens,
                             num_kv_splits=0 if fp8 else 4,
                             schedule="balanced" if fp8 else "split", num_sms=16)
    assert (plan.sched_pairs > 0) == fp8
    gen = torch.Generator(device="cuda").manual_seed(1711)
    w_uv = (torch.randn((N, 512, 128), generator=gen, device="cuda") * 512 ** -0.5).to(
        torch.bfloat16)
    ws = binding.new_workspace(plan)

    def new_outs():
        return dict(o=torch.empty((B, N, 128 if not fp8 else 512), dtype=torch.bfloat16,
                                  device="cuda"),
                    lse=torch.empty((B, N), dtype=torch.float32, device="cuda"))

    def call(qq, o, workspace):
        if fp8:
            binding.mla_decode_fp8(qq, cache, table, lens, w.softmax_scale, w.k_scale, plan=plan,
                                   out=o["o"], lse=o["lse"], workspace=workspace)
        else:
            binding.mla_decode_v_up_proj(qq, cache, table, lens, w.softmax_scale, w_uv,
                                         plan=plan, workspace=workspace, out=o["o"],
                                         lse=o["lse"])

    q_static = q.clone()
    out_static = new_outs()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(q_static, out_static, ws)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(q_static, out_static, ws)
    for rnd in range(3):
        if rnd:
            q_static.copy_((torch.randn(q.shape, generator=gen, device="cuda")).to(torch.bfloat16))
        eager = new_outs()
        ws_e = binding.new_workspace(plan)
        call(q_static, eager, ws_e)
        graph.replay()
        torch.cuda.synchronize()
        assert binding.read_error(ws) == 0 and binding.read_error(ws_e) == 0
        assert torch.equal(out_static["o"], eager["o"]), (kind, rnd)
        assert torch.equal(out_static["lse"], eager["lse"]), (kind, rnd)
        header = ws[:binding.STATUS_BYTES].view(torch.int32).cpu().numpy()
        assert not header.any(), np.nonzero(header)
