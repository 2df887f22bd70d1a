"""GPU parity of mla_decode_fp8 (E4M3 latent cache, per-tensor scale) against
the oracle's fp8 definition, through the C ABI.

The tensor cores take f16 operands here (q, the widened cache entries, the
softmax weights); the bounds are the decode's: bf16 out within 2e-2 and LSE
within 1e-3 on the N(0, 1) configurations, the x8-outlier configuration
keeping the weight-rounding allowance of the bf16 tests.
"""

import numpy as np
import pytest

from mla_latent_cache_paged_gb300 import binding
from mla_latent_cache_paged_gb300.workloads import (bf16_tensor_bits, get_workload,
                                                    make_workload, to_torch)
from parity_util import (OUT_ATOL, assert_lse_close, assert_out_close, assert_out_rel_rms,
                         max_abs_err, oracle_rows_fp8, run_decode_fp8, value_abs_max_fp8)

pytestmark = pytest.mark.gpu


def _fp8(name, batch, heads, lens, seed, splits, extra=3, **kw):
    return make_workload(name, batch, heads, lens, seed=seed, extra_blocks=extra,
                         num_kv_splits=splits, cache_dtype="fp8", **kw)


def _check(w, got, lse, strict=True):
    reqs = range(w.batch)
    ref_out, ref_lse = oracle_rows_fp8(w, reqs)
    if strict:
        err = np.abs(got - ref_out)
        assert err.max() <= OUT_ATOL, (w.name, float(err.max()))
    else:
        assert_out_close(got, ref_out, w.name, value_abs_max_fp8(w, reqs))
    assert_lse_close(lse, ref_lse, w.name)
    assert_out_rel_rms(got, ref_out, w.name)
    return max_abs_err(got, ref_out), max_abs_err(lse, ref_lse)


@pytest.mark.parametrize("heads,lens,splits,schedule", [
    (16, [256], 1, "auto"),
    (128, [1, 63, 64, 65, 300, 1000], 1, "auto"),
    (128, [1, 63, 64, 65, 300, 1000], 3, "auto"),
    (128, [1, 63, 64, 65, 300, 1000], 32, "auto"),
    (5, [130, 7], 2, "auto"),
    (64, [517, 2048], 0, "auto"),
    (128, [0, 100], 1, "auto"),
    (128, [0, 100, 0], 4, "auto"),
    (128, [5, 3000, 17, 64, 1, 999, 2048, 77], 0, "balanced"),
])
def test_fp8_small_parity(heads, lens, splits, schedule):
    w = _fp8(f"fp8_small_n{heads}", len(lens), heads, lens, 2000 + heads + len(lens), splits)
    got, lse, plan, _ = run_decode_fp8(w, schedule=schedule,
                                       num_sms=16 if schedule == "balanced" else None)
    assert (plan.sched_pairs > 0) == (schedule == "balanced")
    _check(w, got, lse)


def test_fp8_single_token_returns_its_dequantized_row_bit_exact():
    """L = 1: the output is the token's value row times k_scale; with a
    power-of-two k_scale that product is exact and so is its bf16 rounding."""
    import torch
    from mla_latent_cache_paged_gb300.workloads import f32_to_bf16_bits
    from oracle import dequantize_e4m3_cache
    w = _fp8("fp8_one_token", 3, 128, [1, 1, 1], 7, 1, extra=2)
    w.k_scale = 2.0 ** -5
    got, lse, _, t = run_decode_fp8(w)
    out_bits = bf16_tensor_bits(t["out"])
    for b in range(3):
        row = dequantize_e4m3_cache(w.cache_bits[w.block_table[b, 0], 0, :512], w.k_scale)
        want = f32_to_bf16_bits(row.astype(np.float32))
        assert np.array_equal(out_bits[b], np.broadcast_to(want, (128, 512))), b


def test_fp8_every_finite_code_widens_exactly():
    """L = 1 with the token's 512 value codes running through every finite
    E4M3 code, forwards in one request and backwards in the other (the two
    NaN codes, 0x7f and 0xff, replaced by 0): each output element is its
    code's value times the power-of-two k_scale, exactly. (Values, not bits:
    the code for -0 comes out as +0, since the P.V sum adds the masked
    tokens' +0 products to it.)"""
    from mla_latent_cache_paged_gb300.workloads import bf16_bits_to_f64
    from oracle import dequantize_e4m3_cache
    w = _fp8("fp8_codes", 2, 16, [1, 1], 8, 1, extra=2)
    codes = np.arange(256, dtype=np.uint8)
    codes[[0x7F, 0xFF]] = 0
    rows = [np.concatenate([codes, codes[::-1]]), np.concatenate([codes[::-1], codes])]
    for b in range(2):
        w.cache_bits[w.block_table[b, 0], 0, :512] = rows[b]
    w.k_scale = 2.0 ** -5
    _, _, _, t = run_decode_fp8(w)
    got = bf16_bits_to_f64(bf16_tensor_bits(t["out"]))
    for b in range(2):
        want = dequantize_e4m3_cache(rows[b], w.k_scale)
        bad = np.nonzero(got[b] != want[None, :])
        assert bad[0].size == 0, (b, bad[1][:8], got[b][bad][:8], want[bad[1][:8]])


def test_fp8_page_permutation_gives_bit_identical_output():
    lens = [70, 640, 129]
    w1 = _fp8("fp8_perm", 3, 128, lens, 11, 1, extra=5)
    rng = np.random.default_rng(99)
    nb = w1.num_blocks + 4
    perm = rng.permutation(nb)
    cache2 = np.full((nb, 64, 576), 0x7F, dtype=np.uint8)
    table2 = np.full_like(w1.block_table, -1)
    pos = 0
    for b, L in enumerate(lens):
        for j in range(-(-L // 64)):
            cache2[perm[pos]] = w1.cache_bits[w1.block_table[b, j]]
            table2[b, j] = perm[pos]
            pos += 1
    w2 = _fp8("fp8_perm", 3, 128, lens, 11, 1, extra=5)
    w2.cache_bits, w2.block_table, w2.num_blocks = cache2, table2, nb
    _, _, _, t1 = run_decode_fp8(w1)
    _, _, _, t2 = run_decode_fp8(w2)
    assert np.array_equal(bf16_tensor_bits(t1["out"]), bf16_tensor_bits(t2["out"]))
    assert np.array_equal(t1["lse"].cpu().numpy(), t2["lse"].cpu().numpy())


@pytest.mark.parametrize("scale", [0.0, -0.05, 0.3])
def test_fp8_zero_negative_and_large_scales(scale):
    w = _fp8("fp8_scales", 3, 128, [700, 65, 1], 57, 1, extra=2)
    w.softmax_scale = scale
    got, lse, _, _ = run_decode_fp8(w)
    ref_out, ref_lse = oracle_rows_fp8(w, range(w.batch))
    assert_out_close(got, ref_out, f"fp8 scale {scale}", value_abs_max_fp8(w, range(w.batch)))
    assert_lse_close(lse, ref_lse, f"fp8 scale {scale} lse")


def test_fp8_query_beyond_f16_range_is_reported():
    import torch
    w = _fp8("fp8_range", 2, 128, [200, 64], 31, 1)
    q, cache, table, lens = to_torch(w)
    q[1, 5, 300] = 1.0e5
    plan = binding.make_plan(2, 128, w.max_blocks_per_seq, num_kv_splits=1)
    ws = binding.new_workspace(plan)
    binding.mla_decode_fp8(q, cache, table, lens, w.softmax_scale, w.k_scale, plan=plan,
                           workspace=ws)
    assert binding.read_error(ws) == binding.MLA_ERR_RANGE
    words = ws[:8].view(torch.int32).cpu().numpy()
    assert binding.read_error(ws) == 0


def test_fp8_bad_block_id_is_reported_not_faulted():
    import torch
    w = _fp8("fp8_bad_block", 2, 128, [200, 64], 32, 1, extra=0)
    q, cache, table, lens = to_torch(w)
    table[0, 1] = w.num_blocks + 1000
    table[1, 0] = -5
    plan = binding.make_plan(2, 128, w.max_blocks_per_seq, num_kv_splits=1)
    ws = binding.new_workspace(plan)
    out, lse = binding.mla_decode_fp8(q, cache, table, lens, w.softmax_scale, w.k_scale,
                                      plan=plan, workspace=ws)
    assert binding.read_error(ws) == binding.MLA_ERR_BAD_BLOCK_ID
    assert torch.isfinite(out.float()).all()


def test_fp8_rejects_a_cuda_core_plan_and_a_bad_scale():
    import torch
    w = _fp8("fp8_args", 1, 16, [64], 33, 1, extra=0)
    q, cache, table, lens = to_torch(w)
    simt = binding.make_plan(1, 16, w.max_blocks_per_seq, num_kv_splits=1, force_simt=True)
    with pytest.raises(binding.MlaError) as e:
        binding.mla_decode_fp8(q, cache, table, lens, w.softmax_scale, w.k_scale, plan=simt)
    assert e.value.status == binding.MLA_ERR_UNSUPPORTED
    plan = binding.make_plan(1, 16, w.max_blocks_per_seq, num_kv_splits=1)
    for bad in (0.0, -1.0, float("inf")):
        with pytest.raises(binding.MlaError) as e:
            binding.mla_decode_fp8(q, cache, table, lens, w.softmax_scale, bad, plan=plan)
        assert e.value.status == binding.MLA_ERR_INVALID_ARG


FULL_SIZE_FP8 = [
    ("b1_n16_l256_pool8_fp8", True),
    ("b32_n128_l1k-4k_fp8", True),
    ("b128_n128_l8192_fp8", True),
    ("b4_n128_l32k_s64_fp8", True),
    ("b4_n128_l64k_s64_fp8", True),
    ("b4_n128_l96k_s64_fp8", True),
    ("b4_n128_l128k_s64_fp8", True),
    ("b256_n128_logu16-32k_outliers_fp8", False),
]


@pytest.mark.parametrize("name,strict", FULL_SIZE_FP8)
def test_fp8_full_size_configs(name, strict):
    """Every config with an fp8 cache, in the benchmark's launch configuration,
    every request against the oracle."""
    w = get_workload(name)
    got, lse, plan, _ = run_decode_fp8(w)
    e_out, e_lse = _check(w, got, lse, strict)
    print(f"{name}: S={plan.num_kv_splits} pairs={plan.sched_pairs} k_scale={w.k_scale:.4g} "
          f"max|out err|={e_out:.3g} max|lse err|={e_lse:.3g}")
