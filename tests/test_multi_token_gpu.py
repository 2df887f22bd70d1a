"""Uniform multi-token decode through the C ABI against the oracle.

vLLM mla_attention API docs, QueryLenSupport.UNIFORM: every request has T
query tokens at positions L - T .. L - 1; causal blocks see the tokens up to
their own position, non-causal blocks see all L. Ragged lengths include
requests shorter than T (rows that see nothing: zero output, -inf LSE).
"""

import numpy as np
import pytest

from mla_latent_cache_paged_gb300 import binding
from mla_latent_cache_paged_gb300.workloads import (bf16_bits_to_f64, bf16_tensor_bits,
                                                    f32_to_bf16_bits, make_workload, to_torch)
from oracle import mla_decode_multi_token_reference
from parity_util import assert_lse_close, assert_out_close, assert_out_rel_rms, value_abs_max

pytestmark = pytest.mark.gpu


def _run(w, T, causal, q_bits, **plan_kw):
    import torch
    _, cache, table, lens = to_torch(w)
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).cuda()
    plan = binding.make_plan_multi_token(w.batch, T, w.num_heads, w.max_blocks_per_seq,
                                         seq_lens_host=w.seq_lens, causal=causal, **plan_kw)
    ws = binding.new_workspace(plan)
    out, lse = binding.mla_decode_multi_token(q, cache, table, lens, w.softmax_scale,
                                              causal=causal, plan=plan, workspace=ws)
    torch.cuda.synchronize()
    assert binding.read_error(ws) == 0
    return bf16_bits_to_f64(bf16_tensor_bits(out)), lse.double().cpu().numpy(), plan


@pytest.mark.parametrize("T,causal,N,plan_kw", [
    # T * N > 128: B * T rows of N heads.
    (2, True, 128, {}),
    (4, True, 128, {"num_kv_splits": 4}),
    (3, True, 128, {"num_kv_splits": 1}),
    (2, True, 64, {"schedule": "balanced", "expand": True}),
    # T * N <= 128: the tokens' heads as the rows of one decode.
    (3, False, 16, {}),
    (2, True, 64, {"schedule": "balanced"}),
    (4, True, 16, {}),
    (8, True, 16, {"num_kv_splits": 4}),
    (3, True, 40, {"num_kv_splits": 1}),
    (2, True, 32, {"force_simt": True}),
    (4, True, 16, {"force_simt": True, "num_kv_splits": 3}),
])
def test_multi_token_against_the_oracle(T, causal, N, plan_kw):
    lens = [1, 2, 63, 64, 65, 300, 1000, 0]
    w = make_workload("mt", len(lens), N, lens, seed=1400 + 10 * T + N)
    rng = np.random.default_rng(1500 + T)
    q_bits = f32_to_bf16_bits(rng.standard_normal((len(lens), T, N, 576)).astype(np.float32))
    got, lse, plan = _run(w, T, causal, q_bits, **plan_kw)
    packed = T * N <= 128 and not plan_kw.get("expand", False)
    assert (plan.num_heads, plan.batch) == ((T * N, w.batch) if packed else (N, w.batch * T))
    ref, ref_lse = mla_decode_multi_token_reference(bf16_bits_to_f64(q_bits), w.cache_f64(),
                                                    w.block_table, w.seq_lens, w.softmax_scale,
                                                    causal=causal)
    vmax = value_abs_max(w, range(w.batch))[:, None]           # [B, 1, 1, 512]
    assert_out_close(got, ref, f"T={T} causal={causal}", vmax)
    assert_lse_close(lse, ref_lse, "multi-token lse")
    if causal:
        # The one-token request: only its last query token sees anything.
        assert np.isneginf(lse[0, :T - 1]).all() and np.isfinite(lse[0, T - 1]).all()
        assert (got[0, :T - 1] == 0).all()
    # The empty request: every query token sees nothing.
    assert np.isneginf(lse[-1]).all() and (got[-1] == 0).all()


def _random_mt_case(i):
    rng = np.random.default_rng(7000 + i)
    T = int(rng.integers(1, 9))
    causal = bool(rng.random() < 0.7)
    N = int(rng.choice([1, 5, 16, 32, 64, 100, 128]))
    B = int(rng.integers(1, 7))
    edge = [0, 1, max(T - 1, 0), T, 63, 64, 65]
    lens = [int(rng.choice(edge)) if rng.random() < 0.4 else int(rng.integers(1, 1200))
            for _ in range(B)]
    kind = str(rng.choice(["auto", "split", "balanced", "expand", "simt"]))
    kw = {"num_sms": int(rng.choice([8, 30, 152]))}
    if kind == "split":
        kw["num_kv_splits"] = int(rng.choice([1, 2, 3, 5]))
    elif kind == "balanced":
        kw["schedule"] = "balanced"
    elif kind == "expand":
        kw["expand"] = True
        kw["schedule"] = str(rng.choice(["auto", "balanced"]))
    elif kind == "simt":
        kw["force_simt"] = True
        kw["num_kv_splits"] = int(rng.choice([1, 2]))
    return T, causal, N, lens, kw


@pytest.mark.parametrize("i", range(40))
def test_multi_token_random_case_against_the_oracle(i):
    """Seeded random multi-token problems: T 1-8, causal or not, head counts
    from 1 to 128 (both the packed and the row-expanded form), ragged lengths
    with requests shorter than T, every schedule, both kernels, several SM
    counts."""
    T, causal, N, lens, kw = _random_mt_case(i)
    # (one spare block: a batch whose requests are all empty still passes a
    # cache of at least one block, as the interface asks)
    w = make_workload("mt_rand", len(lens), N, lens, seed=7100 + i, extra_blocks=1)
    rng = np.random.default_rng(7200 + i)
    q_bits = f32_to_bf16_bits(rng.standard_normal((len(lens), T, N, 576)).astype(np.float32))
    got, lse, plan = _run(w, T, causal, q_bits, **kw)
    ref, ref_lse = mla_decode_multi_token_reference(bf16_bits_to_f64(q_bits), w.cache_f64(),
                                                    w.block_table, w.seq_lens, w.softmax_scale,
                                                    causal=causal)
    vmax = value_abs_max(w, range(w.batch))[:, None]
    what = f"case {i}: T={T} causal={causal} N={N} lens={lens} {kw}"
    assert_out_close(got, ref, what, vmax, plan.sched_pairs == 0 and plan.num_kv_splits > 1)
    assert_out_rel_rms(got, ref, what)
    assert_lse_close(lse, ref_lse, what)
