"""The steps on either side of the decode, through the C ABI, against the oracle.

Front end (mla_q_absorb_concat_cache: q absorption by W_UK_T, q_pe concat,
the new tokens' cache insert) and the up-projection (mla_v_up_proj by W_UV),
per-head batched matmuls on the tensor cores. Inputs are seeded bf16; the
oracle widens the same bits to float64. A result accumulated in fp32 and
rounded once to bf16 is within one bf16 ulp of the exact value (plus a
small absolute term for the fp32 sum of 128 or 512 products).
"""

import numpy as np
import pytest

from mla_latent_cache_paged_gb300 import binding
from mla_latent_cache_paged_gb300.workloads import (bf16_bits_to_f64, bf16_tensor_bits,
                                                    f32_to_bf16_bits, make_workload, to_torch)
from oracle import mla_decode_reference, q_absorb_concat_cache, v_up_proj
from parity_util import bf16_ulp

pytestmark = pytest.mark.gpu

FP32_SUM_ATOL = 1e-4


def _bf16(rng, shape, scale=1.0):
    return f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def _dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _assert_within_one_ulp(got_bits, ref, what):
    got = bf16_bits_to_f64(got_bits)
    err = np.abs(got - ref)
    tol = bf16_ulp(ref) + FP32_SUM_ATOL
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} outside one ulp; worst "
                           f"{float(err.max())} at {np.unravel_index(err.argmax(), err.shape)}")


@pytest.mark.parametrize("B,N", [(1, 1), (5, 16), (128, 128), (200, 8), (300, 3), (129, 37),
                                 (384, 2), (511, 7), (64, 128)])
def test_front_end_against_the_oracle(B, N):
    import torch
    rng = np.random.default_rng(1000 + 7 * B + N)
    q = _bf16(rng, (B, N, 192))
    w = _bf16(rng, (N, 128, 512), 1 / np.sqrt(128))
    kv_c = _bf16(rng, (B, 512))
    k_pe = _bf16(rng, (B, 64))
    nb = (B + 1) // 2 + 3
    cache = _bf16(rng, (nb, 64, 576))
    # Distinct slots in random order, every fourth request a padding slot.
    slots = rng.permutation(nb * 64)[:B].astype(np.int64)
    slots[::4] = -1
    cache_d = _dev(cache)
    ws = binding.new_status_workspace()
    out = binding.mla_q_absorb_concat_cache(_dev(q), _dev(w), _dev(kv_c), _dev(k_pe),
                                            torch.from_numpy(slots).cuda(), cache_d,
                                            workspace=ws)
    torch.cuda.synchronize()
    assert binding.read_error(ws) == 0
    ref_q, ref_cache = q_absorb_concat_cache(bf16_bits_to_f64(q), bf16_bits_to_f64(w),
                                             bf16_bits_to_f64(kv_c), bf16_bits_to_f64(k_pe),
                                             slots, bf16_bits_to_f64(cache))
    got = bf16_tensor_bits(out)
    _assert_within_one_ulp(got[..., :512], ref_q[..., :512], "ql_nope")
    np.testing.assert_array_equal(got[..., 512:], q[..., 128:])          # q_pe: copied bits
    got_cache = bf16_tensor_bits(cache_d)
    np.testing.assert_array_equal(bf16_bits_to_f64(got_cache), ref_cache)   # insert: bit-exact


def test_front_end_without_insert_and_with_a_bad_slot():
    import torch
    rng = np.random.default_rng(1100)
    B, N, nb = 6, 4, 2
    q = _bf16(rng, (B, N, 192))
    w = _bf16(rng, (N, 128, 512), 1 / np.sqrt(128))
    ws = binding.new_status_workspace()
    out = binding.mla_q_absorb_concat_cache(_dev(q), _dev(w), workspace=ws)
    torch.cuda.synchronize()
    assert binding.read_error(ws) == 0
    ref_q, _ = q_absorb_concat_cache(bf16_bits_to_f64(q), bf16_bits_to_f64(w), np.zeros((B, 512)),
                                     np.zeros((B, 64)), [-1] * B, np.zeros((1, 64, 576)))
    _assert_within_one_ulp(bf16_tensor_bits(out)[..., :512], ref_q[..., :512], "no insert")

    cache = _bf16(rng, (nb, 64, 576))
    kv_c, k_pe = _bf16(rng, (B, 512)), _bf16(rng, (B, 64))
    slots = np.array([0, 5, nb * 64, 70, -1, nb * 64 + 1000], dtype=np.int64)
    cache_d = _dev(cache)
    binding.mla_q_absorb_concat_cache(_dev(q), _dev(w), _dev(kv_c), _dev(k_pe),
                                      torch.from_numpy(slots).cuda(), cache_d, workspace=ws)
    torch.cuda.synchronize()
    assert binding.read_error(ws) == binding.MLA_ERR_BAD_BLOCK_ID
    good = np.where((slots >= 0) & (slots < nb * 64), slots, -1)
    _, ref_cache = q_absorb_concat_cache(bf16_bits_to_f64(q), bf16_bits_to_f64(w),
                                         bf16_bits_to_f64(kv_c), bf16_bits_to_f64(k_pe), good,
                                         bf16_bits_to_f64(cache))
    np.testing.assert_array_equal(bf16_bits_to_f64(bf16_tensor_bits(cache_d)), ref_cache)


@pytest.mark.parametrize("B,N", [(1, 1), (3, 8), (128, 128), (257, 5), (127, 100), (384, 3),
                                 (640, 1), (255, 64)])
def test_v_up_proj_against_the_oracle(B, N):
    import torch
    rng = np.random.default_rng(1200 + 7 * B + N)
    x = _bf16(rng, (B, N, 512))
    w = _bf16(rng, (N, 512, 128), 1 / np.sqrt(512))
    ws = binding.new_status_workspace()
    out = binding.mla_v_up_proj(_dev(x), _dev(w), workspace=ws)
    torch.cuda.synchronize()
    assert binding.read_error(ws) == 0
    ref = v_up_proj(bf16_bits_to_f64(x), bf16_bits_to_f64(w))
    _assert_within_one_ulp(bf16_tensor_bits(out), ref, "v_up_proj")


def test_decode_step_front_end_decode_up_projection():
    """The three calls in sequence on one stream: the new token is inserted,
    then attended to, then up-projected. The oracle runs the same step in
    float64, rounding the two intermediates the device keeps in bf16 (mqa_q
    and the latent output) to bf16 as the device does."""
    import torch
    B, N = 4, 128
    lens = np.array([63, 64, 200, 1000], dtype=np.int32)
    w_l = make_workload("step", B, N, lens + 1, seed=1300)      # room for the new token
    rng = np.random.default_rng(1301)
    q_in = _bf16(rng, (B, N, 192))
    w_uk_t = _bf16(rng, (N, 128, 512), 1 / np.sqrt(128))
    w_uv = _bf16(rng, (N, 512, 128), 1 / np.sqrt(512))
    kv_c, k_pe = _bf16(rng, (B, 512)), _bf16(rng, (B, 64))
    t = lens.astype(np.int64)
    slots = w_l.block_table[np.arange(B), t // 64].astype(np.int64) * 64 + t % 64

    _, cache, table, seq = to_torch(w_l)
    ws = binding.new_status_workspace()
    mqa_q = binding.mla_q_absorb_concat_cache(_dev(q_in), _dev(w_uk_t), _dev(kv_c), _dev(k_pe),
                                              torch.from_numpy(slots).cuda(), cache,
                                              workspace=ws)
    lat, lse = binding.mla_decode(mqa_q, cache, table, seq, w_l.softmax_scale)
    out = binding.mla_v_up_proj(lat, _dev(w_uv), workspace=ws)
    torch.cuda.synchronize()
    assert binding.read_error(ws) == 0

    ref_q, ref_cache = q_absorb_concat_cache(bf16_bits_to_f64(q_in), bf16_bits_to_f64(w_uk_t),
                                             bf16_bits_to_f64(kv_c), bf16_bits_to_f64(k_pe),
                                             slots, w_l.cache_f64())
    ref_q = bf16_bits_to_f64(f32_to_bf16_bits(ref_q.astype(np.float32)))
    ref_lat, ref_lse = mla_decode_reference(ref_q, ref_cache, w_l.block_table, w_l.seq_lens,
                                            w_l.softmax_scale)
    ref_lat = bf16_bits_to_f64(f32_to_bf16_bits(ref_lat.astype(np.float32)))
    ref = v_up_proj(ref_lat, bf16_bits_to_f64(w_uv))
    got = bf16_bits_to_f64(bf16_tensor_bits(out))
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 1e-2, rel
    np.testing.assert_allclose(lse.double().cpu().numpy(), ref_lse, atol=5e-3)


# ------------------------------------------------ merge fused with the up-projection

@pytest.mark.parametrize("B,N,S", [(1, 1, 1), (3, 5, 3), (130, 128, 2), (32, 128, 32),
                                   (4, 16, 64), (7, 3, 512)])
def test_merge_splits_v_up_proj_against_the_oracle(B, N, S):
    """The merged rows (returned through latent_out) are within one bf16 ulp
    of the oracle's merge, and the output is within one ulp of the oracle's
    up-projection of those very rows; neutral partials (-inf LSE, NaN rows)
    carry no weight, and a row whose partials are all neutral gives 0."""
    import torch
    from oracle import merge_partials
    rng = np.random.default_rng(1400 + B + N + S)
    o = rng.standard_normal((B, N, S, 512)).astype(np.float32)
    ls = (rng.standard_normal((B, N, S)) * 3).astype(np.float32)
    ls[0, 0, :] = -np.inf
    if S > 1:
        ls[-1, -1, ::2] = -np.inf
        o[-1, -1, ::2] = np.nan
    o[0, 0] = np.nan
    w = _bf16(rng, (N, 512, 128), 1 / np.sqrt(512))
    ws = binding.new_status_workspace()
    lat = torch.empty((B, N, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, N), dtype=torch.float32, device="cuda")
    out = binding.mla_merge_splits_v_up_proj(torch.from_numpy(o).cuda(),
                                             torch.from_numpy(ls).cuda(), _dev(w),
                                             workspace=ws, lse=lse, latent_out=lat)
    torch.cuda.synchronize()
    assert binding.read_error(ws) == 0
    o_ref = np.where(np.isneginf(ls)[..., None], 0.0, o.astype(np.float64))
    ref_lat, ref_lse = merge_partials(o_ref, ls.astype(np.float64))
    _assert_within_one_ulp(bf16_tensor_bits(lat), ref_lat, "merged rows")
    got_lse = lse.double().cpu().numpy()
    assert np.isneginf(got_lse[0, 0]) and np.isneginf(ref_lse[0, 0])
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(got_lse[fin], ref_lse[fin], rtol=0, atol=1e-5)
    ref = v_up_proj(bf16_bits_to_f64(bf16_tensor_bits(lat)), bf16_bits_to_f64(w))
    _assert_within_one_ulp(bf16_tensor_bits(out), ref, "fused up-projection")
    assert np.all(bf16_tensor_bits(out)[0, 0] == 0)


@pytest.mark.parametrize("splits", [1, 4])
def test_decode_v_up_proj_matches_the_separate_calls_and_the_oracle(splits):
    """mla_decode_v_up_proj: a split plan merges straight into the
    up-projection (no latent rows written), S = 1 goes through latent_out.
    Against mla_decode + mla_v_up_proj on the same inputs, and against the
    oracle's decode and up-projection with the latent rounded to bf16."""
    import torch
    from parity_util import oracle_rows
    B, N = 5, 128
    lens = [1, 100, 700, 2048, 65]
    w_l = make_workload("decode_up", B, N, lens, seed=1500 + splits, extra_blocks=2,
                        num_kv_splits=splits)
    rng = np.random.default_rng(1501)
    w_uv = _dev(_bf16(rng, (N, 512, 128), 1 / np.sqrt(512)))
    q, cache, table, seq = to_torch(w_l)
    plan = binding.make_plan(B, N, w_l.max_blocks_per_seq, seq_lens_host=w_l.seq_lens,
                             max_seq_len=w_l.max_seq_len, num_kv_splits=splits, schedule="split")
    assert plan.num_kv_splits == splits
    ws = binding.new_workspace(plan)
    lat = torch.empty((B, N, 512), dtype=torch.bfloat16, device="cuda")
    if splits == 1:
        with pytest.raises(binding.MlaError):    # the latent rows have nowhere to go
            binding.mla_decode_v_up_proj(q, cache, table, seq, w_l.softmax_scale, w_uv,
                                         plan=plan, workspace=ws)
    out = binding.mla_decode_v_up_proj(q, cache, table, seq, w_l.softmax_scale, w_uv, plan=plan,
                                       workspace=ws, latent_out=lat if splits == 1 else None)
    torch.cuda.synchronize()
    assert binding.read_error(ws) == 0
    sep_lat, _ = binding.mla_decode(q, cache, table, seq, w_l.softmax_scale, plan=plan,
                                    workspace=ws)
    sep = binding.mla_v_up_proj(sep_lat, w_uv, workspace=ws)
    torch.cuda.synchronize()
    got = bf16_bits_to_f64(bf16_tensor_bits(out))
    ref_sep = bf16_bits_to_f64(bf16_tensor_bits(sep))
    if splits == 1:
        assert torch.equal(out, sep)                 # the same two kernels
    else:
        # the fused merge sums the splits in the same order as one of the
        # merge kernel's layouts, not necessarily this one: a merged row may
        # round one ulp apart
        assert np.abs(got - ref_sep).max() <= 2e-2
    ref_lat, _ = oracle_rows(w_l, range(B))
    ref_lat = bf16_bits_to_f64(f32_to_bf16_bits(ref_lat.astype(np.float32)))
    ref = v_up_proj(ref_lat, bf16_bits_to_f64(bf16_tensor_bits(w_uv)))
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 1e-2, rel
