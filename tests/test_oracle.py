"""Pins for the CPU oracle: it is checked against things other than itself.

Hand-worked golden cases, pure-Python brute force, closed forms, torch's
float64 SDPA, exact identities (MHA == absorbed MQA, split+merge == unsplit,
page-table permutation invariance). CPU only.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import (absorb_query, dcp_combine, dcp_decode_partials,
                    dcp_local_seq_lens, dcp_owner, gather_request_latent,
                    merge_partials, mha_compute_friendly, mla_decode_multi_token_reference,
                    mla_decode_reference,
                    mla_decode_split_partials, q_absorb_concat_cache, split_token_ranges,
                    up_project, v_up_proj)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _exact(text):
    """Evaluate the fixtures' exact forms: 'ln 6', '4 ln 2', '0', '-inf'."""
    text = text.strip()
    if text == "-inf":
        return -math.inf
    if "ln" not in text:
        return float(text)
    coef, _, arg = text.partition("ln")
    coef = float(coef) if coef.strip() else 1.0
    return coef * math.log(float(arg))


def _paged_from_dense(rng, dense_rows_per_req, page_size, extra_blocks=3, fill=77.0):
    """Scatter dense per-request rows into a randomly permuted page pool."""
    pages = [-(-len(r) // page_size) for r in dense_rows_per_req]
    nb = sum(pages) + extra_blocks
    width = dense_rows_per_req[0].shape[1]
    cache = np.full((nb, page_size, width), fill, dtype=np.float64)
    perm = rng.permutation(nb)
    table = np.full((len(pages), max(pages + [1])), -1, dtype=np.int64)
    pos = 0
    for b, rows in enumerate(dense_rows_per_req):
        for j in range(pages[b]):
            blk = perm[pos]
            pos += 1
            table[b, j] = blk
            chunk = rows[j * page_size:(j + 1) * page_size]
            cache[blk, :len(chunk)] = chunk
    return cache, table


# ---------------------------------------------------------------- golden cases

def test_golden_hand_worked_decode():
    with open(os.path.join(GOLDEN, "decode_hand_worked.json")) as f:
        g = json.load(f)
    cache = np.array(g["cache"], dtype=np.float64)
    table = np.array(g["block_table"], dtype=np.int64)
    seq = np.array(g["seq_lens"])
    q = np.array(g["q"], dtype=np.float64)
    for b in range(len(seq)):
        got = gather_request_latent(cache, table[b], seq[b], g["page_size"])
        np.testing.assert_array_equal(got, np.array(g["gathered"][b], dtype=np.float64))
    out, lse = mla_decode_reference(q, cache, table, seq, math.log(2.0),
                                    kv_lora_rank=g["kv_lora_rank"])
    np.testing.assert_allclose(out, np.array(g["expected_out"]), rtol=0, atol=1e-14)
    exact = np.array([[_exact(x) for x in row] for row in g["expected_lse_exact"]])
    np.testing.assert_allclose(lse, exact, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.array(g["expected_lse"]), rtol=0, atol=1e-14)


def test_golden_hand_worked_merge():
    with open(os.path.join(GOLDEN, "merge_hand_worked.json")) as f:
        g = json.load(f)
    o_part = np.array(g["o_part"], dtype=np.float64)
    lse_part = np.array([[_exact(x) for x in row] for row in g["lse_part_exact"]])
    out, lse = merge_partials(o_part, lse_part)
    np.testing.assert_allclose(out, np.array(g["expected_out"]), rtol=0, atol=1e-14)
    exact = np.array([_exact(x) for x in g["expected_lse_exact"]])
    assert np.isneginf(lse[2]) and np.isneginf(exact[2])
    np.testing.assert_allclose(lse[:2], exact[:2], rtol=0, atol=1e-14)


# ------------------------------------------------------------- brute force

def _brute_force(q, rows, scale, lkv):
    """Pure-Python loops: no numpy, no vectorisation, straight from the sum."""
    n_heads = len(q)
    outs, lses = [], []
    for h in range(n_heads):
        s = [scale * sum(q[h][d] * rows[t][d] for d in range(len(q[h])))
             for t in range(len(rows))]
        big = max(s)
        z = sum(math.exp(x - big) for x in s)
        lses.append(big + math.log(z))
        outs.append([sum(math.exp(s[t] - big) / z * rows[t][d] for t in range(len(rows)))
                     for d in range(lkv)])
    return outs, lses


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    lkv, rope, ps, n = 6, 3, 4, 3
    lens = [1, 5, 9]
    dense = [rng.standard_normal((L, lkv + rope)) for L in lens]
    cache, table = _paged_from_dense(rng, dense, ps)
    q = rng.standard_normal((len(lens), n, lkv + rope))
    scale = 0.37
    out, lse = mla_decode_reference(q, cache, table, lens, scale, kv_lora_rank=lkv)
    for b in range(len(lens)):
        bo, bl = _brute_force(q[b].tolist(), dense[b].tolist(), scale, lkv)
        np.testing.assert_allclose(out[b], np.array(bo), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[b], np.array(bl), rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------- closed forms

def test_zero_query_gives_mean_and_log_length():
    rng = np.random.default_rng(5)
    lens = [1, 7, 64, 130]
    dense = [rng.standard_normal((L, 576)) for L in lens]
    cache, table = _paged_from_dense(rng, dense, 64)
    q = np.zeros((len(lens), 4, 576))
    out, lse = mla_decode_reference(q, cache, table, lens, 0.072)
    for b, L in enumerate(lens):
        np.testing.assert_allclose(lse[b], math.log(L), rtol=0, atol=1e-13)
        np.testing.assert_allclose(out[b], np.broadcast_to(dense[b][:, :512].mean(0), (4, 512)),
                                   rtol=1e-12, atol=1e-12)


def test_single_token_returns_its_latent_row():
    rng = np.random.default_rng(6)
    dense = [rng.standard_normal((1, 576))]
    cache, table = _paged_from_dense(rng, dense, 64)
    q = rng.standard_normal((1, 8, 576))
    scale = 1 / math.sqrt(192)
    out, lse = mla_decode_reference(q, cache, table, [1], scale)
    np.testing.assert_array_equal(out[0], np.broadcast_to(dense[0][0, :512], (8, 512)))
    np.testing.assert_allclose(lse[0], scale * (q[0] @ dense[0][0]), rtol=1e-14, atol=1e-14)


def test_identical_rows_give_uniform_weights():
    rng = np.random.default_rng(7)
    row = rng.standard_normal(576)
    L = 100
    dense = [np.tile(row, (L, 1))]
    cache, table = _paged_from_dense(rng, dense, 64)
    q = rng.standard_normal((1, 3, 576))
    scale = 0.05
    out, lse = mla_decode_reference(q, cache, table, [L], scale)
    np.testing.assert_allclose(out[0], np.broadcast_to(row[:512], (3, 512)), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse[0], scale * (q[0] @ row) + math.log(L), rtol=1e-13, atol=1e-13)


def test_empty_request_is_neutral():
    rng = np.random.default_rng(8)
    cache = rng.standard_normal((2, 64, 576))
    table = np.array([[0, 1]])
    out, lse = mla_decode_reference(rng.standard_normal((1, 2, 576)), cache, table, [0], 0.1)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


# ------------------------------------------------- library special case

def test_matches_torch_sdpa_float64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(9)
    lens = [3, 64, 65, 200]
    n = 16
    dense = [rng.standard_normal((L, 576)) for L in lens]
    cache, table = _paged_from_dense(rng, dense, 64)
    q = rng.standard_normal((len(lens), n, 576))
    scale = 1 / math.sqrt(192)
    out, lse = mla_decode_reference(q, cache, table, lens, scale)
    for b, L in enumerate(lens):
        qt = torch.from_numpy(q[b]).view(1, n, 1, 576)
        kt = torch.from_numpy(dense[b]).view(1, 1, L, 576).expand(1, n, L, 576)
        vt = torch.from_numpy(dense[b][:, :512]).view(1, 1, L, 512).expand(1, n, L, 512)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        np.testing.assert_allclose(out[b], ref.view(n, 512).numpy(), rtol=1e-11, atol=1e-12)
        ref_lse = torch.logsumexp(scale * (qt.view(n, 576) @ kt[0, 0].T), dim=-1)
        np.testing.assert_allclose(lse[b], ref_lse.numpy(), rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------- identities

def test_absorbed_mqa_equals_compute_friendly_mha():
    """forward_mqa followed by the W_UV up-projection equals forward_mha."""
    rng = np.random.default_rng(10)
    n, p, r, v, lkv, L = 4, 16, 8, 16, 32, 37
    w_uk = rng.standard_normal((lkv, n, p)) / math.sqrt(lkv)
    w_uv = rng.standard_normal((lkv, n, v)) / math.sqrt(lkv)
    q_nope = rng.standard_normal((n, p))
    q_pe = rng.standard_normal((n, r))
    kv_c = rng.standard_normal((L, lkv))
    k_pe = rng.standard_normal((L, r))
    scale = (p + r) ** -0.5
    ref_out, ref_lse = mha_compute_friendly(q_nope, q_pe, kv_c, k_pe, w_uk, w_uv, scale)

    ql_nope = absorb_query(q_nope[None], w_uk)[0]                   # [N, Lkv]
    q_abs = np.concatenate([ql_nope, q_pe], axis=1)[None]           # [1, N, Lkv+R]
    cache, table = _paged_from_dense(rng, [np.concatenate([kv_c, k_pe], axis=1)], 8)
    lat, lse = mla_decode_reference(q_abs, cache, table, [L], scale, kv_lora_rank=lkv)
    out = up_project(lat, w_uv)[0]
    np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse[0], ref_lse, rtol=1e-12, atol=1e-13)


def test_absorb_query_against_explicit_sum():
    rng = np.random.default_rng(11)
    q_nope = rng.standard_normal((2, 3, 5))
    w_uk = rng.standard_normal((7, 3, 5))
    got = absorb_query(q_nope, w_uk)
    for s in range(2):
        for nh in range(3):
            for l in range(7):
                want = sum(q_nope[s, nh, h] * w_uk[l, nh, h] for h in range(5))
                assert abs(got[s, nh, l] - want) < 1e-12


@pytest.mark.parametrize("num_splits", [1, 2, 3, 7, 64])
def test_split_then_merge_equals_unsplit(num_splits):
    rng = np.random.default_rng(100 + num_splits)
    lens = [1, 63, 64, 65, 300, 1000]
    dense = [rng.standard_normal((L, 576)) for L in lens]
    cache, table = _paged_from_dense(rng, dense, 64)
    q = rng.standard_normal((len(lens), 4, 576))
    scale = 1 / math.sqrt(192)
    ref_out, ref_lse = mla_decode_reference(q, cache, table, lens, scale)
    o_part, lse_part = mla_decode_split_partials(q, cache, table, lens, scale, num_splits)
    if num_splits >= 7:
        assert np.isneginf(lse_part).any(), "expected some empty splits"
    out, lse = merge_partials(o_part, lse_part)
    np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_merge_neutral_element_changes_nothing():
    rng = np.random.default_rng(12)
    o = rng.standard_normal((5, 3, 8))
    ls = rng.standard_normal((5, 3))
    base_out, base_lse = merge_partials(o, ls)
    o2 = np.concatenate([o, np.zeros((5, 1, 8))], axis=1)
    ls2 = np.concatenate([ls, np.full((5, 1), -np.inf)], axis=1)
    out, lse = merge_partials(o2, ls2)
    np.testing.assert_allclose(out, base_out, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(lse, base_lse, rtol=1e-14, atol=1e-14)


def test_split_ranges_cover_and_align():
    for L in [0, 1, 63, 64, 65, 1000, 8192, 131072]:
        for S in [1, 2, 3, 7, 32, 64]:
            rngs = split_token_ranges(L, S, 64)
            assert len(rngs) == S
            assert rngs[0][0] == 0 and rngs[-1][1] == L
            for (lo, hi), (lo2, _) in zip(rngs, rngs[1:]):
                assert hi == lo2 and lo <= hi
            for lo, hi in rngs:
                assert lo % 64 == 0 or lo == L


def test_page_permutation_is_bitwise_invariant():
    rng = np.random.default_rng(13)
    lens = [5, 128, 190]
    dense = [rng.standard_normal((L, 576)) for L in lens]
    q = rng.standard_normal((3, 8, 576))
    c1, t1 = _paged_from_dense(np.random.default_rng(1), dense, 64)
    c2, t2 = _paged_from_dense(np.random.default_rng(2), dense, 64, extra_blocks=9)
    assert not np.array_equal(t1[:, :1], t2[:, :1])
    o1, l1 = mla_decode_reference(q, c1, t1, lens, 0.07)
    o2, l2 = mla_decode_reference(q, c2, t2, lens, 0.07)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_rope_columns_enter_scores_but_not_values():
    """K is the whole 576-wide entry; V is only its first 512 columns."""
    rng = np.random.default_rng(14)
    dense = [rng.standard_normal((40, 576))]
    cache, table = _paged_from_dense(rng, dense, 64)
    q = rng.standard_normal((1, 2, 576))
    o1, l1 = mla_decode_reference(q, cache, table, [40], 0.1)
    cache2 = cache.copy()
    cache2[..., 512:] *= 2.0          # changes scores only
    o2, l2 = mla_decode_reference(q, cache2, table, [40], 0.1)
    assert not np.allclose(l1, l2)
    q3 = q.copy()
    q3[..., 512:] = 0.0
    cache3 = cache.copy()
    cache3[..., 512:] = 123.0         # with q_pe = 0 the rope columns cannot matter
    o3, l3 = mla_decode_reference(q3, cache, table, [40], 0.1)
    o4, l4 = mla_decode_reference(q3, cache3, table, [40], 0.1)
    np.testing.assert_array_equal(o3, o4)
    np.testing.assert_array_equal(l3, l4)
    assert o1.shape[-1] == 512


# ------------------------------------------------ decode context parallelism

def test_dcp_placement_hand_worked():
    """Runs of `interleave` tokens dealt round-robin (worked by hand)."""
    # world 2, interleave 2, 10 tokens: runs 0..4 -> ranks 0,1,0,1,0.
    got = [dcp_owner(t, 2, 2) for t in range(10)]
    assert got == [(0, 0), (0, 1), (1, 0), (1, 1), (0, 2), (0, 3),
                   (1, 2), (1, 3), (0, 4), (0, 5)]
    # world 3, interleave 1 (one token per run), 7 tokens.
    got = [dcp_owner(t, 3, 1) for t in range(7)]
    assert got == [(0, 0), (1, 0), (2, 0), (0, 1), (1, 1), (2, 1), (0, 2)]
    # world 1 keeps every token where it was.
    assert all(dcp_owner(t, 1, 4) == (0, t) for t in range(9))
    np.testing.assert_array_equal(dcp_local_seq_lens([10, 7, 0], 2, 2),
                                  [[6, 4, 0], [4, 3, 0]])


def test_dcp_local_lengths_bound_and_conservation():
    """Every token is on exactly one rank, local indices are dense, and no
    shard is longer than the bound the pages print for it: ceil(L / (R * I)) * I
    (vLLM mla_attention API docs, MLACommonMetadataBuilder.build); rank 0
    reaches it whenever the last virtual block gives it a whole run."""
    for world in [1, 2, 3, 4, 8]:
        for interleave in [1, 2, 16, 64]:
            lens = [0, 1, 5, 63, 64, 65, 129, 1000, 1031]
            counts = dcp_local_seq_lens(lens, world, interleave)
            np.testing.assert_array_equal(counts.sum(axis=0), lens)
            for b, L in enumerate(lens):
                bound = -(-L // (world * interleave)) * interleave
                assert counts[:, b].max() <= bound
                if L % (world * interleave) == 0 or L % (world * interleave) >= interleave:
                    assert counts[0, b] == bound
                seen = [set() for _ in range(world)]
                for t in range(L):
                    r, j = dcp_owner(t, world, interleave)
                    seen[r].add(j)
                for r in range(world):
                    assert seen[r] == set(range(counts[r, b]))


@pytest.mark.parametrize("world,interleave", [(1, 1), (2, 1), (2, 64), (3, 2), (4, 16)])
def test_dcp_combine_equals_unsplit(world, interleave):
    rng = np.random.default_rng(200 + 7 * world + interleave)
    lens = [1, 3, 64, 65, 300]
    dense = [rng.standard_normal((L, 576)) for L in lens]
    cache, table = _paged_from_dense(rng, dense, 64)
    q = rng.standard_normal((len(lens), 4, 576))
    scale = 1 / math.sqrt(192)
    ref_out, ref_lse = mla_decode_reference(q, cache, table, lens, scale)
    o_r, l_r = dcp_decode_partials(q, cache, table, lens, scale, world, interleave)
    assert o_r.shape == (world, len(lens), 4, 512) and l_r.shape == (world, len(lens), 4)
    if world > 1:
        assert np.isneginf(l_r[:, 0]).any(), "a 1-token request leaves ranks empty"
    out, lse = dcp_combine(o_r, l_r)
    if world == 1:
        np.testing.assert_array_equal(out, ref_out)
        np.testing.assert_array_equal(lse, ref_lse)
    np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_dcp_rank_result_is_attention_over_its_own_tokens():
    """Rank r's result equals the definition applied to the dense rows it holds."""
    rng = np.random.default_rng(210)
    L = 37
    rows = rng.standard_normal((L, 576))
    cache, table = _paged_from_dense(rng, [rows], 8)
    q = rng.standard_normal((1, 3, 576))
    o_r, l_r = dcp_decode_partials(q, cache, table, [L], 0.1, 3, 2)
    for r in range(3):
        mine = [t for t in range(L) if (t // 2) % 3 == r]
        c1, t1 = _paged_from_dense(rng, [rows[mine]], 8)
        o, l = mla_decode_reference(q, c1, t1, [len(mine)], 0.1)
        np.testing.assert_allclose(o_r[r], o, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(l_r[r], l, rtol=1e-13, atol=1e-13)


# -------------------------------------------- front end and up-projection

def test_q_absorb_against_explicit_sums_over_the_printed_layout():
    """ql_nope[b, n, l] = sum_p q_nope[b, n, p] * W_UK_T[n, p, l], with W_UK_T
    (N, P, Lkv) as the page lays it out; q_pe lands after the Lkv columns."""
    rng = np.random.default_rng(300)
    B, N, P, R, L = 3, 2, 4, 2, 5
    q = rng.standard_normal((B, N, P + R))
    w_uk_t = rng.standard_normal((N, P, L))
    mqa_q, _ = q_absorb_concat_cache(q, w_uk_t, np.zeros((B, L)), np.zeros((B, R)),
                                     [-1] * B, np.zeros((1, 4, L + R)), qk_nope_head_dim=P)
    assert mqa_q.shape == (B, N, L + R)
    for b in range(B):
        for n in range(N):
            for l in range(L):
                want = sum(q[b, n, p] * w_uk_t[n, p, l] for p in range(P))
                assert abs(mqa_q[b, n, l] - want) < 1e-12
            np.testing.assert_array_equal(mqa_q[b, n, L:], q[b, n, P:])


def test_v_up_proj_against_explicit_sums_over_the_printed_layout():
    """out[b, n, v] = sum_l x[b, n, l] * W_UV[n, l, v], W_UV laid out (N, Lkv, V)."""
    rng = np.random.default_rng(301)
    B, N, L, V = 2, 3, 5, 4
    x = rng.standard_normal((B, N, L))
    w_uv = rng.standard_normal((N, L, V))
    out = v_up_proj(x, w_uv)
    for b in range(B):
        for n in range(N):
            for v in range(V):
                want = sum(x[b, n, l] * w_uv[n, l, v] for l in range(L))
                assert abs(out[b, n, v] - want) < 1e-12


def test_cache_insert_hand_worked():
    """Slots 3, padding (-1) and 8 + 5 with 8-row pages: rows (0, 3) and
    (1, 5) take [kv_c | k_pe]; every other row keeps its bits."""
    rng = np.random.default_rng(302)
    cache = rng.standard_normal((3, 8, 6))
    kv_c = np.arange(12.0).reshape(3, 4)
    k_pe = -np.arange(6.0).reshape(3, 2) - 1
    q = rng.standard_normal((3, 1, 4 + 2))
    _, new = q_absorb_concat_cache(q, rng.standard_normal((1, 4, 4)), kv_c, k_pe,
                                   [3, -1, 13], cache, qk_nope_head_dim=4)
    np.testing.assert_array_equal(new[0, 3], [0, 1, 2, 3, -1, -2])
    np.testing.assert_array_equal(new[1, 5], [8, 9, 10, 11, -5, -6])
    keep = np.ones(cache.shape[:2], dtype=bool)
    keep[0, 3] = keep[1, 5] = False
    np.testing.assert_array_equal(new[keep], cache[keep])
    assert not np.array_equal(new, cache)


def test_decode_step_with_front_end_equals_compute_friendly_mha():
    """Front end (absorb, concat, insert of the new token) -> decode over the
    cache, now holding the new token -> up-projection equals MHA over the
    cached tokens plus the new one, with the weights in the layouts the page
    prepares: W_UK_T = W_UK.permute(1, 2, 0), W_UV transposed to (N, Lkv, V)."""
    rng = np.random.default_rng(303)
    n, p, r, v, lkv, L, ps = 4, 16, 8, 16, 32, 21, 8
    w_uk = rng.standard_normal((lkv, n, p)) / math.sqrt(lkv)
    w_uv = rng.standard_normal((lkv, n, v)) / math.sqrt(lkv)
    kv_c = rng.standard_normal((L + 1, lkv))          # the last row is the new token's
    k_pe = rng.standard_normal((L + 1, r))
    q = rng.standard_normal((1, n, p + r))
    scale = (p + r) ** -0.5
    ref_out, ref_lse = mha_compute_friendly(q[0, :, :p], q[0, :, p:], kv_c, k_pe, w_uk, w_uv,
                                            scale)

    cache, table = _paged_from_dense(rng, [np.concatenate([kv_c[:L], k_pe[:L]], axis=1)], ps,
                                     extra_blocks=2)
    # The new token goes to row L % ps of the request's last page (L = 21:
    # page 2 of 3, which already holds rows 16..20).
    slot = int(table[0, L // ps]) * ps + L % ps
    mqa_q, cache2 = q_absorb_concat_cache(q, np.transpose(w_uk, (1, 2, 0)), kv_c[L:], k_pe[L:],
                                          [slot], cache, qk_nope_head_dim=p)
    lat, lse = mla_decode_reference(mqa_q, cache2, table, [L + 1], scale, kv_lora_rank=lkv)
    out = v_up_proj(lat, np.transpose(w_uv, (1, 0, 2)))[0]
    np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse[0], ref_lse, rtol=1e-12, atol=1e-13)


# ------------------------------------------------ multi-token (uniform) decode

def test_multi_token_hand_worked():
    """Two query tokens over a two-token cache, scale ln 2 (worked by hand).
    Causal: token 0 sits at position 0 and sees only row 0 (out = V[0],
    lse = 2 ln 2 since q0.k0 = 2); token 1 sees both rows with q1.k = (0, 1):
    weights 1/3, 2/3 and lse = ln 3. Non-causal: token 0 sees both rows too,
    q0.k = (2, 2): weights 1/2, 1/2 and lse = 2 ln 2 + ln 2 = 3 ln 2."""
    # Entries [v0, v1 | rope]: Lkv = 2, R = 1.
    cache = np.array([[[1.0, 0.0, 2.0], [0.0, 1.0, 2.0]]])     # k0 = (1,0,2), k1 = (0,1,2)
    table = np.array([[0]])
    q = np.array([[[[0.0, 0.0, 1.0]], [[-2.0, -1.0, 1.0]]]])   # q0.k = (2, 2); q1.k = (0, 1)
    out, lse = mla_decode_multi_token_reference(q, cache, table, [2], math.log(2),
                                                causal=True, kv_lora_rank=2)
    np.testing.assert_allclose(out[0, 0, 0], [1.0, 0.0], atol=1e-15)
    assert abs(lse[0, 0, 0] - 2 * math.log(2)) < 1e-14
    np.testing.assert_allclose(out[0, 1, 0], [1 / 3, 2 / 3], atol=1e-15)
    assert abs(lse[0, 1, 0] - math.log(3)) < 1e-14
    out, lse = mla_decode_multi_token_reference(q, cache, table, [2], math.log(2),
                                                causal=False, kv_lora_rank=2)
    np.testing.assert_allclose(out[0, 0, 0], [0.5, 0.5], atol=1e-15)
    assert abs(lse[0, 0, 0] - 3 * math.log(2)) < 1e-14


@pytest.mark.parametrize("causal", [True, False])
def test_multi_token_equals_single_token_over_the_visible_tokens(causal):
    rng = np.random.default_rng(400 + causal)
    T, lens = 3, [1, 2, 3, 64, 65, 130]
    dense = [rng.standard_normal((L, 576)) for L in lens]
    cache, table = _paged_from_dense(rng, dense, 64)
    q = rng.standard_normal((len(lens), T, 4, 576))
    out, lse = mla_decode_multi_token_reference(q, cache, table, lens, 0.07, causal=causal)
    for i in range(T):
        vis = [max(0, L - T + 1 + i) if causal else L for L in lens]
        o1, l1 = mla_decode_reference(q[:, i], cache, table, vis, 0.07)
        np.testing.assert_allclose(out[:, i], o1, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(lse[:, i], l1, rtol=1e-13, atol=1e-13)
    if causal:
        assert np.isneginf(lse[0, :2]).all() and np.isfinite(lse[0, 2]).all()
    o_single, l_single = mla_decode_reference(q[:, 0], cache, table, lens, 0.07)
    o_t1, l_t1 = mla_decode_multi_token_reference(q[:, :1], cache, table, lens, 0.07,
                                                  causal=causal)
    np.testing.assert_allclose(o_t1[:, 0], o_single, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(l_t1[:, 0], l_single, rtol=1e-13, atol=1e-13)


def test_multi_token_matches_torch_sdpa_with_the_causal_block_mask():
    import torch
    rng = np.random.default_rng(402)
    T, L, N = 4, 37, 3
    rows = rng.standard_normal((L, 576))
    cache, table = _paged_from_dense(rng, [rows], 16)
    q = rng.standard_normal((1, T, N, 576))
    out, lse = mla_decode_multi_token_reference(q, cache, table, [L], 0.05, causal=True)
    mask = torch.arange(L)[None, :] <= (L - T + torch.arange(T))[:, None]      # [T, L]
    qt = torch.from_numpy(q[0]).permute(1, 0, 2)                                 # [N, T, D]
    k = torch.from_numpy(rows)[None].expand(N, L, 576)
    v = torch.from_numpy(rows[:, :512])[None].expand(N, L, 512)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, k, v, attn_mask=mask, scale=0.05)
    np.testing.assert_allclose(out[0].transpose(1, 0, 2), ref.numpy(), rtol=1e-12, atol=1e-12)
    scores = (qt @ k.transpose(1, 2)) * 0.05
    ref_lse = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1)   # [N, T]
    np.testing.assert_allclose(lse[0].T, ref_lse.numpy(), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- fp8 (E4M3) cache

def _code(text):
    return int(text, 16)


def test_e4m3_golden_codes():
    from oracle import e4m3_to_float
    with open(os.path.join(GOLDEN, "e4m3_decode.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        got = float(e4m3_to_float(np.array([_code(case["code"])], dtype=np.uint8))[0])
        want = case["value"]
        if want == "nan":
            assert math.isnan(got), case
        else:
            assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), case


def test_e4m3_every_code_matches_torch_float8_e4m3fn():
    """Library special case: torch's float8_e4m3fn decodes the same 256 codes."""
    import torch
    from oracle import e4m3_to_float
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = e4m3_to_float(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_order_and_symmetry():
    from oracle import e4m3_to_float
    pos = e4m3_to_float(np.arange(0x7F, dtype=np.uint8))          # 0x00 .. 0x7E
    assert np.all(np.diff(pos) > 0) and pos[-1] == 448.0
    neg = e4m3_to_float(np.arange(0x80, 0xFF, dtype=np.uint8))
    np.testing.assert_array_equal(neg, -pos)
    # 126 distinct positive finite values, plus zero
    assert len(set(pos.tolist())) == 127


def test_golden_hand_worked_fp8_decode():
    from oracle import mla_decode_reference_fp8
    with open(os.path.join(GOLDEN, "decode_fp8_hand_worked.json")) as f:
        g = json.load(f)
    codes = np.array([[[_code(c) for c in row] for row in blk] for blk in g["cache_codes"]],
                     dtype=np.uint8)
    table = np.array(g["block_table"], dtype=np.int64)
    seq = np.array(g["seq_lens"])
    q = np.array(g["q"], dtype=np.float64)
    from oracle import dequantize_e4m3_cache
    deq = dequantize_e4m3_cache(codes, g["k_scale"])
    got_rows = gather_request_latent(deq, table[0], seq[0], g["page_size"])
    np.testing.assert_array_equal(got_rows, np.array(g["dequantized_rows"], dtype=np.float64))
    out, lse = mla_decode_reference_fp8(q, codes, table, seq, math.log(2.0), g["k_scale"],
                                        kv_lora_rank=g["kv_lora_rank"])
    np.testing.assert_allclose(out, np.array(g["expected_out"]), rtol=0, atol=1e-14)
    exact = np.array([[_exact(x) for x in row] for row in g["expected_lse_exact"]])
    np.testing.assert_allclose(lse, exact, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.array(g["expected_lse"]), rtol=0, atol=1e-14)


@pytest.mark.parametrize("log2_scale", [-3, 0, 2])
def test_fp8_decode_equals_bf16_decode_on_exact_values(log2_scale):
    """With a power-of-two k_scale every dequantized entry is a bf16 number
    (3 mantissa bits in 7, exponents in range), so the fp8 definition must
    equal the bf16 one on the bf16 encoding of the same values, bit for bit
    in float64."""
    from oracle import dequantize_e4m3_cache, mla_decode_reference_fp8
    from mla_latent_cache_paged_gb300.workloads import bf16_bits_to_f64, f32_to_bf16_bits
    rng = np.random.default_rng(40 + log2_scale)
    nb, ps, width = 7, 4, 24
    codes = rng.integers(0, 256, size=(nb, ps, width), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38              # no NaN codes in the live rows
    k_scale = 2.0 ** log2_scale
    deq = dequantize_e4m3_cache(codes, k_scale)
    bf16 = bf16_bits_to_f64(f32_to_bf16_bits(deq.astype(np.float32)))
    assert np.array_equal(bf16, deq)                   # the values are bf16 numbers
    table = np.array([[3, 0, 6], [5, 1, -1]])
    seq = [10, 7]
    q = rng.standard_normal((2, 3, width))
    a_out, a_lse = mla_decode_reference_fp8(q, codes, table, seq, 0.05, k_scale, kv_lora_rank=16)
    b_out, b_lse = mla_decode_reference(q, bf16, table, seq, 0.05, kv_lora_rank=16)
    assert np.array_equal(a_out, b_out) and np.array_equal(a_lse, b_lse)
