"""GPU parity over a seeded random sweep of small problems, through the C ABI.

Each case draws its own batch, head count, lengths (with empty, one-token and
page-edge lengths mixed in), split count, schedule, SM count (so the number
of CTA pairs and the page-balanced cut vary), softmax scale (zero and
negative included), kernel and cache type (bf16, or fp8 E4M3 on the
tensor-core kernel), and is checked against the oracle: bf16 out within
max(2e-2, one bf16 ulp, 2^-8 max_t |V[t, d]|) (the weight-rounding allowance
of the bf16 tests; with the split schedule's bf16 partial rows, rounded
twice, max(2e-2, one ulp + 2^-8 max_t |V[t, d]|)), the whole output's RMS
error within 1e-2 of its RMS, and LSE within 1e-3.
"""

import numpy as np
import pytest

from mla_latent_cache_paged_gb300 import binding
from mla_latent_cache_paged_gb300.workloads import (bf16_bits_to_f64, bf16_tensor_bits,
                                                    make_workload, to_torch)
from parity_util import (assert_lse_close, assert_out_close, assert_out_rel_rms, oracle_rows,
                         oracle_rows_fp8, value_abs_max, value_abs_max_fp8)

pytestmark = pytest.mark.gpu

EDGE_LENS = [0, 1, 63, 64, 65, 127, 128, 129]


def _case(i):
    rng = np.random.default_rng(9000 + i)
    B = int(rng.integers(1, 10))
    N = int(rng.choice([1, 3, 16, 31, 64, 100, 128]))
    lens = []
    for _ in range(B):
        if rng.random() < 0.35:
            lens.append(int(rng.choice(EDGE_LENS)))
        else:
            lens.append(int(rng.integers(1, 1500)))
    fp8 = rng.random() < 0.35
    simt = (not fp8) and rng.random() < 0.2
    splits = int(rng.choice([0, 0, 0, 1, 2, 3, 5, 8]))
    schedule = "auto"
    if splits == 0 and not simt:
        schedule = str(rng.choice(["auto", "split", "balanced", "balanced"]))
    num_sms = int(rng.choice([4, 16, 30, 152]))
    scale = float(rng.choice([1 / np.sqrt(192), 0.3, 0.0, -0.07]))
    return dict(B=B, N=N, lens=lens, fp8=fp8, simt=simt, splits=splits, schedule=schedule,
                num_sms=num_sms, scale=scale, seed=9100 + i)


@pytest.mark.parametrize("i", range(200))
def test_random_case_against_the_oracle(i):
    import torch
    c = _case(i)
    w = make_workload("sweep", c["B"], c["N"], c["lens"], seed=c["seed"], extra_blocks=3,
                      num_kv_splits=c["splits"], cache_dtype="fp8" if c["fp8"] else "bf16")
    w.softmax_scale = c["scale"]
    q, cache, table, lens = to_torch(w)
    plan = binding.make_plan(w.batch, w.num_heads, w.max_blocks_per_seq,
                             seq_lens_host=w.seq_lens, max_seq_len=w.max_seq_len,
                             num_kv_splits=c["splits"], num_sms=c["num_sms"],
                             force_simt=c["simt"], schedule=c["schedule"])
    if c["schedule"] == "balanced" and sum(c["lens"]) > 0:
        assert plan.sched_pairs > 0
    ws = binding.new_workspace(plan)
    if c["fp8"]:
        out, lse = binding.mla_decode_fp8(q, cache, table, lens, w.softmax_scale, w.k_scale,
                                          plan=plan, workspace=ws)
    else:
        out, lse = binding.mla_decode(q, cache, table, lens, w.softmax_scale, plan=plan,
                                      workspace=ws)
    torch.cuda.synchronize()
    status = binding.read_error(ws)
    assert status == 0, (c, binding.status_string(status))
    header = ws[:binding.STATUS_BYTES].view(torch.int32).cpu().numpy()
    assert not header.any(), (c, np.nonzero(header))
    reqs = range(w.batch)
    if c["fp8"]:
        ref_out, ref_lse = oracle_rows_fp8(w, reqs)
        vmax = value_abs_max_fp8(w, reqs)
    else:
        ref_out, ref_lse = oracle_rows(w, reqs)
        vmax = value_abs_max(w, reqs)
    what = f"case {i}: {c} plan S={plan.num_kv_splits} pairs={plan.sched_pairs}"
    got = bf16_bits_to_f64(bf16_tensor_bits(out))
    bf16_partials = plan.sched_pairs == 0 and plan.num_kv_splits > 1
    assert_out_close(got, ref_out, what, vmax, bf16_partials)
    assert_out_rel_rms(got, ref_out, what)
    assert_lse_close(lse.double().cpu().numpy(), ref_lse, what)
