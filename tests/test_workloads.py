"""Seeded input generator: bf16 rounding, page-table layout, poison rows."""

import numpy as np

from mla_latent_cache_paged_gb300.workloads import (BF16_NAN, WORKLOADS, bf16_bits_to_f32,
                                                    f32_to_bf16_bits, get_workload,
                                                    make_workload)


def test_bf16_round_to_nearest_even():
    one = np.float32(1.0)
    eps = np.float32(2.0 ** -8)        # half a bf16 ulp at 1.0
    vals = np.array([one, one + eps, one + 3 * eps, one + np.float32(2.0 ** -7),
                     -2.5, 0.0, np.inf, np.nan], dtype=np.float32)
    bits = f32_to_bf16_bits(vals)
    assert bits[0] == 0x3F80
    assert bits[1] == 0x3F80           # tie -> even
    assert bits[2] == 0x3F82           # tie -> even (upwards)
    assert bits[3] == 0x3F81
    assert bits[4] == 0xC020
    assert bits[5] == 0x0000
    assert bits[6] == 0x7F80
    assert bits[7] == BF16_NAN
    back = bf16_bits_to_f32(bits[:7])
    np.testing.assert_array_equal(back, np.array([1, 1, 1 + 2 ** -6, 1 + 2 ** -7, -2.5, 0, np.inf],
                                                 dtype=np.float32))


def test_block_table_is_a_permutation_with_sentinels():
    w = make_workload("t", 3, 4, [1, 64, 130], seed=1, extra_blocks=2)
    pages = [1, 1, 3]
    used = np.concatenate([w.block_table[b, :p] for b, p in enumerate(pages)])
    assert len(set(used.tolist())) == len(used) == 5
    assert used.min() >= 0 and used.max() < w.num_blocks == 7
    for b, p in enumerate(pages):
        rest = w.block_table[b, p:]
        assert np.all((rest < 0) | (rest >= w.num_blocks))
    # tail rows of partial last pages are NaN poison; full pages are not
    last = w.block_table[0, 0]
    assert np.all(w.cache_bits[last, 1:] == BF16_NAN)
    assert not np.any(w.cache_bits[last, 0] == BF16_NAN)
    assert not np.any(w.cache_bits[w.block_table[1, 0]] == BF16_NAN)


def test_outlier_rows_are_scaled_by_eight():
    a = make_workload("t", 2, 2, [300, 500], seed=3, outlier_frac=0.0, poison=False)
    b = make_workload("t", 2, 2, [300, 500], seed=3, outlier_frac=0.01, poison=False)
    fa = bf16_bits_to_f32(a.cache_bits).reshape(-1, 576)
    fb = bf16_bits_to_f32(b.cache_bits).reshape(-1, 576)
    changed = np.where(np.any(fa != fb, axis=1))[0]
    assert len(changed) == 8           # floor(0.01 * 800)
    np.testing.assert_array_equal(fb[changed], fa[changed] * 8)


def test_named_workloads_have_stated_shapes():
    shapes = {name: get_workload(name, with_data=False) for name in WORKLOADS}
    c1 = shapes["b1_n16_l256_pool8"]
    assert c1.batch == 1 and c1.num_heads == 16 and c1.num_blocks == 8 and c1.total_tokens == 256
    c2 = shapes["b32_n128_l1k-4k"]
    assert c2.batch == 32 and c2.seq_lens.min() >= 1024 and c2.seq_lens.max() <= 4096
    c3 = shapes["b128_n128_l8192"]
    assert c3.total_tokens == 128 * 8192 and c3.num_blocks == 16384
    c5 = shapes["b256_n128_logu16-32k_outliers"]
    assert c5.batch == 256 and c5.seq_lens.min() >= 16 and c5.seq_lens.max() <= 32768


def test_e4m3_quantizer_matches_torch_and_saturates():
    import torch
    from mla_latent_cache_paged_gb300.workloads import f32_to_e4m3_bits
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(1 << 16).astype(np.float32) * 60,
                        rng.standard_normal(1 << 12).astype(np.float32) * 0.01,
                        np.array([0.0, -0.0, 2 ** -10, 3 * 2 ** -10, 447.0], np.float32)])
    got = f32_to_e4m3_bits(x)
    inr = np.abs(x) <= 448
    ref = torch.from_numpy(x[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got[inr], ref)
    big = f32_to_e4m3_bits(np.array([464.0, 1e9, -1e9, np.nan], np.float32))
    assert big.tolist() == [0x7E, 0x7E, 0xFE, 0x7F]


def test_fp8_workloads_share_the_bf16_layout():
    from mla_latent_cache_paged_gb300.workloads import get_workload
    a = get_workload("b1_n16_l256_pool8")
    b = get_workload("b1_n16_l256_pool8_fp8")
    assert b.cache_dtype == "fp8" and b.cache_bits.dtype == np.uint8
    assert np.array_equal(a.block_table, b.block_table) and np.array_equal(a.q_bits, b.q_bits)
    assert 0 < b.k_scale < 1
    # tail rows past L hold the NaN code
    assert a.seq_lens[0] % 64 == 0 or np.all(b.cache_bits[b.block_table[0, -1], 64:] == 0x7F)
