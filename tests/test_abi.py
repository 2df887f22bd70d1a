"""The C ABI without a GPU: symbols, struct layout, planner, host-side checks."""

import ctypes
import os
import re
import subprocess
import tempfile

import numpy as np
import pytest

from mla_latent_cache_paged_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla_decode.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def _declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(mla_\w+)\s*\(", text, re.M)))


def test_every_declared_function_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 8
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(binding.EXPORTED_SYMBOLS)
    version = int(re.search(r"#define MLA_DECODE_ABI_VERSION (\d+)", open(HEADER).read()).group(1))
    assert lib.mla_abi_version() == version


def test_plan_struct_layout_matches_the_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "mla_decode.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu\\n\", sizeof(mla_decode_plan_t),"
        " offsetof(mla_decode_plan_t, flags), offsetof(mla_decode_plan_t, workspace_bytes),"
        " offsetof(mla_decode_plan_t, lse_partial_offset), offsetof(mla_decode_plan_t, sched_pairs),"
        " offsetof(mla_decode_plan_t, reserved));"
        "return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                    str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    P = binding.MlaDecodePlan
    want = [ctypes.sizeof(P), P.flags.offset, P.workspace_bytes.offset,
            P.lse_partial_offset.offset, P.sched_pairs.offset, P.reserved.offset]
    assert got == want


def _plan(lib, batch=4, heads=128, max_blocks=32, max_seq=2048, lens=None, splits=0,
          sms=152, flags=0, kv=512, rope=64, ps=64):
    plan = binding.MlaDecodePlan()
    ptr = ctypes.c_void_p(0)
    keep = None
    if lens is not None:
        keep = np.ascontiguousarray(np.asarray(lens, np.int32))
        ptr = ctypes.c_void_p(keep.ctypes.data)
    rc = lib.mla_decode_plan(batch, heads, kv, rope, ps, max_blocks, max_seq, ptr, splits, sms,
                             flags, ctypes.byref(plan))
    return rc, plan


def test_plan_fixed_splits_and_workspace_layout(lib):
    rows = 4 * 128 * 64
    rc, p = _plan(lib, batch=4, heads=128, splits=64)
    assert rc == 0 and p.num_kv_splits == 64
    assert p.partial_offset == binding.STATUS_BYTES   # status header, then the partials
    # bf16 partial rows by default, then the fp32 LSEs
    assert p.lse_partial_offset == p.partial_offset + rows * 512 * 2
    assert p.workspace_bytes == p.lse_partial_offset + rows * 4
    assert p.workspace_bytes % 256 == 0
    rc, p32 = _plan(lib, batch=4, heads=128, splits=64, flags=binding.MLA_PLAN_FP32_PARTIALS)
    assert rc == 0 and p32.lse_partial_offset == p32.partial_offset + rows * 512 * 4
    assert p32.workspace_bytes == p32.lse_partial_offset + rows * 4
    rc, p1 = _plan(lib, splits=1)
    assert rc == 0 and p1.num_kv_splits == 1 and p1.workspace_bytes == binding.STATUS_BYTES


def test_planner_choice_is_bounded_and_deterministic(lib):
    for batch, seq in [(1, 256), (32, 4096), (128, 8192), (4, 131072), (256, 32768)]:
        mb = -(-seq // 64)
        rc, p = _plan(lib, batch=batch, max_blocks=mb, max_seq=seq)
        assert rc == 0
        assert 1 <= p.num_kv_splits <= min(64, mb)
        rc2, p2 = _plan(lib, batch=batch, max_blocks=mb, max_seq=seq)
        assert p2.num_kv_splits == p.num_kv_splits
    # a long single request must be split to use the GPU
    rc, p = _plan(lib, batch=1, max_blocks=2048, max_seq=131072)
    assert p.num_kv_splits > 8


def test_planner_uses_host_lengths(lib):
    lens = [16] * 255 + [32768]
    rc, p = _plan(lib, batch=256, max_blocks=512, max_seq=32768, lens=lens)
    assert rc == 0 and p.num_kv_splits >= 1
    rc, _ = _plan(lib, batch=2, max_blocks=4, max_seq=256, lens=[10, 300])
    assert rc == binding.MLA_ERR_INVALID_ARG


def test_plan_force_simt_flag(lib):
    rc, p = _plan(lib, flags=binding.MLA_PLAN_FORCE_SIMT)
    assert rc == 0 and p.kernel == binding.MLA_KERNEL_SIMT
    assert p.grid_ctas == 8 * p.batch * p.num_kv_splits


@pytest.mark.parametrize("kw,code", [
    (dict(kv=256), binding.MLA_ERR_UNSUPPORTED),
    (dict(rope=32), binding.MLA_ERR_UNSUPPORTED),
    (dict(ps=16), binding.MLA_ERR_UNSUPPORTED),
    (dict(heads=129), binding.MLA_ERR_UNSUPPORTED),
    (dict(heads=0), binding.MLA_ERR_INVALID_ARG),
    (dict(batch=-1), binding.MLA_ERR_INVALID_ARG),
    (dict(max_blocks=0), binding.MLA_ERR_INVALID_ARG),
    (dict(max_seq=2049), binding.MLA_ERR_INVALID_ARG),
    (dict(splits=-2), binding.MLA_ERR_INVALID_ARG),
    (dict(splits=1025), binding.MLA_ERR_UNSUPPORTED),
    (dict(sms=0), binding.MLA_ERR_INVALID_ARG),
])
def test_plan_rejects_bad_arguments(lib, kw, code):
    rc, _ = _plan(lib, **kw)
    assert rc == code


def test_decode_rejects_bad_arguments_before_touching_the_device(lib):
    rc, p = _plan(lib, batch=2, heads=16, max_blocks=4, max_seq=256, splits=1)
    assert rc == 0
    fake = ctypes.c_void_p(0x10000)      # never dereferenced: checks fail first
    null = ctypes.c_void_p(0)
    args = lambda **o: [ctypes.byref(o.get("plan", p)), o.get("q", fake), o.get("cache", fake),
                        o.get("nb", 8), o.get("bt", fake), o.get("sl", fake),
                        o.get("scale", 0.07), o.get("out", fake), o.get("lse", null),
                        o.get("ws", fake), o.get("wsb", 4096), null]
    assert lib.mla_decode(*args(q=null)) == binding.MLA_ERR_INVALID_ARG
    assert lib.mla_decode(*args(out=null)) == binding.MLA_ERR_INVALID_ARG
    assert lib.mla_decode(*args(nb=0)) == binding.MLA_ERR_INVALID_ARG
    assert lib.mla_decode(*args(scale=float("nan"))) == binding.MLA_ERR_INVALID_ARG
    assert lib.mla_decode(*args(q=ctypes.c_void_p(0x10008))) == binding.MLA_ERR_INVALID_ARG
    assert lib.mla_decode(*args(ws=null)) == binding.MLA_ERR_WORKSPACE
    assert lib.mla_decode(*args(wsb=16)) == binding.MLA_ERR_WORKSPACE
    assert lib.mla_decode(*args(ws=ctypes.c_void_p(0x10010))) == binding.MLA_ERR_WORKSPACE
    bad = binding.MlaDecodePlan.from_buffer_copy(p)
    bad.kv_lora_rank = 320
    assert lib.mla_decode(*args(plan=bad)) == binding.MLA_ERR_UNSUPPORTED
    bad = binding.MlaDecodePlan.from_buffer_copy(p)
    bad.num_kv_splits = 0
    assert lib.mla_decode(*args(plan=bad)) == binding.MLA_ERR_INVALID_ARG


def test_merge_and_gather_reject_bad_arguments(lib):
    fake = ctypes.c_void_p(0x10000)
    null = ctypes.c_void_p(0)
    assert lib.mla_merge_splits(fake, fake, 1, 1, 0, 512, fake, null, null) == \
        binding.MLA_ERR_INVALID_ARG
    assert lib.mla_merge_splits(fake, fake, 1, 1, 2, 500, fake, null, null) == \
        binding.MLA_ERR_UNSUPPORTED
    assert lib.mla_merge_splits(null, fake, 1, 1, 2, 512, fake, null, null) == \
        binding.MLA_ERR_INVALID_ARG
    assert lib.mla_debug_gather_pages(fake, 4, fake, fake, 1, 0, 64, fake, fake, 256, null) == \
        binding.MLA_ERR_INVALID_ARG
    assert lib.mla_debug_gather_pages(fake, 4, fake, fake, 1, 1, 64, fake, null, 256, null) == \
        binding.MLA_ERR_WORKSPACE


def test_dcp_combine_rejects_bad_arguments(lib):
    fake = ctypes.c_void_p(0x10000)
    null = ctypes.c_void_p(0)
    assert lib.mla_dcp_combine(fake, fake, 0, 1, 1, 512, fake, null, null) == \
        binding.MLA_ERR_INVALID_ARG
    assert lib.mla_dcp_combine(fake, fake, 2, 1, 1, 500, fake, null, null) == \
        binding.MLA_ERR_UNSUPPORTED
    assert lib.mla_dcp_combine(null, fake, 2, 1, 1, 512, fake, null, null) == \
        binding.MLA_ERR_INVALID_ARG
    assert lib.mla_dcp_combine(ctypes.c_void_p(0x10004), fake, 2, 1, 1, 512, fake, null,
                               null) == binding.MLA_ERR_INVALID_ARG
    assert lib.mla_dcp_combine(null, null, 2, 0, 1, 512, null, null, null) == binding.MLA_OK


def test_merge_and_combine_reject_row_counts_past_int32(lib):
    fake = ctypes.c_void_p(0x10000)
    null = ctypes.c_void_p(0)
    big = 1 << 24                                   # 2^24 requests x 2^8 heads = 2^32 rows
    assert lib.mla_merge_splits(fake, fake, big, 256, 2, 512, fake, null, null) == \
        binding.MLA_ERR_UNSUPPORTED
    assert lib.mla_dcp_combine(fake, fake, 2, big, 256, 512, fake, null, null) == \
        binding.MLA_ERR_UNSUPPORTED


def test_dcp_local_seq_lens_match_the_oracle_placement():
    """Host-side shard lengths, bit-exact against counting every token's owner."""
    from oracle import dcp_local_seq_lens as oracle_counts
    rng = np.random.default_rng(31)
    lens = np.concatenate([[0, 1, 2, 63, 64, 65, 127, 128, 129, 4096, 4097],
                           rng.integers(0, 5000, 20)]).astype(np.int32)
    for world in [1, 2, 3, 4, 8]:
        for interleave in [1, 2, 8, 64]:
            want = oracle_counts(lens, world, interleave)
            for rank in range(world):
                got = binding.dcp_local_seq_lens(lens, world, rank, interleave)
                np.testing.assert_array_equal(got, want[rank])


@pytest.mark.parametrize("world,rank,interleave,lens", [
    (0, 0, 1, [4]), (2, 2, 1, [4]), (2, -1, 1, [4]), (2, 0, 0, [4]), (2, 0, 1, [4, -1])])
def test_dcp_local_seq_lens_rejects_bad_arguments(lib, world, rank, interleave, lens):
    arr = np.asarray(lens, dtype=np.int32)
    out = np.full(len(lens), 99, dtype=np.int32)
    rc = lib.mla_dcp_local_seq_lens(ctypes.c_void_p(arr.ctypes.data), len(lens), world, rank,
                                    interleave, ctypes.c_void_p(out.ctypes.data))
    assert rc == binding.MLA_ERR_INVALID_ARG
    assert (out == 99).all()


def test_front_end_and_up_projection_reject_bad_arguments(lib):
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    null = ctypes.c_void_p(0)
    ws = ctypes.c_void_p(0x20000)
    big = binding.STATUS_BYTES
    qa = lib.mla_q_absorb_concat_cache
    assert qa(fake, fake, null, null, null, null, 0, 2, 129, fake, ws, big, null) == \
        binding.MLA_ERR_INVALID_ARG
    assert qa(null, fake, null, null, null, null, 0, 2, 4, fake, ws, big, null) == \
        binding.MLA_ERR_INVALID_ARG
    assert qa(fake, fake, null, null, fake, null, 4, 2, 4, fake, ws, big, null) == \
        binding.MLA_ERR_INVALID_ARG                     # slots without the cache rows
    assert qa(fake, fake, null, null, null, null, 0, 2, 4, fake, ws, 256, null) == \
        binding.MLA_ERR_WORKSPACE
    assert qa(fake, fake, null, null, null, null, 0, 2, 4, fake, odd, big, null) == \
        binding.MLA_ERR_WORKSPACE
    assert qa(odd, fake, null, null, null, null, 0, 2, 4, fake, ws, big, null) == \
        binding.MLA_ERR_INVALID_ARG
    assert qa(null, null, null, null, null, null, 0, 0, 4, null, null, 0, null) == binding.MLA_OK
    up = lib.mla_v_up_proj
    assert up(fake, fake, 2, 0, fake, ws, big, null) == binding.MLA_OK
    assert up(fake, fake, -1, 4, fake, ws, big, null) == binding.MLA_ERR_INVALID_ARG
    assert up(fake, null, 2, 4, fake, ws, big, null) == binding.MLA_ERR_INVALID_ARG
    assert up(fake, fake, 2, 4, fake, null, big, null) == binding.MLA_ERR_WORKSPACE
    assert up(fake, fake, 2, 4, odd, ws, big, null) == binding.MLA_ERR_INVALID_ARG


def test_multi_token_scratch_size_and_argument_checks(lib):
    assert lib.mla_multi_token_scratch_bytes(3, 2, 10) == 256 + 256      # 240 B + 24 B, each rounded
    assert lib.mla_multi_token_scratch_bytes(64, 4, 128) == 64 * 4 * 128 * 4 + 1024
    assert lib.mla_multi_token_scratch_bytes(3, 0, 10) == 0
    assert lib.mla_multi_token_scratch_bytes(-1, 2, 10) == 0
    plan = binding.make_plan(6, 128, 4, num_sms=152)
    fake = ctypes.c_void_p(0x10000)
    null = ctypes.c_void_p(0)
    call = lib.mla_decode_multi_token
    # A plan of 6 rows of 128 heads: the B * T-row form (T * N = 128 * T > 128).
    args = lambda q_len, scratch, nbytes, n=128: (ctypes.byref(plan), q_len, n, 1, fake, fake, 8,
                                                  fake, fake, 0.1, fake, null, fake, 1 << 20,
                                                  scratch, nbytes, null)
    assert call(*args(4, fake, 1 << 20)) == binding.MLA_ERR_INVALID_ARG     # 6 rows, T = 4
    assert call(*args(0, fake, 1 << 20)) == binding.MLA_ERR_INVALID_ARG
    assert call(*args(3, null, 1 << 20)) == binding.MLA_ERR_WORKSPACE
    assert call(*args(3, fake, 64)) == binding.MLA_ERR_WORKSPACE
    assert call(*args(3, ctypes.c_void_p(0x10010), 1 << 20)) == binding.MLA_ERR_WORKSPACE
    assert call(*args(3, fake, 1 << 20, n=0)) == binding.MLA_ERR_INVALID_ARG
    assert call(*args(3, fake, 1 << 20, n=64)) == binding.MLA_ERR_INVALID_ARG   # neither shape


def test_multi_token_row_lengths_match_the_oracle_visibility():
    """Host row lengths (used for the plan) against counting, per row, the
    tokens the oracle's definition lets query token i see."""
    lens = [0, 1, 2, 3, 5, 64, 100]
    for T in [1, 2, 3, 4]:
        for causal in [True, False]:
            got = binding.multi_token_row_lens(lens, T, causal)
            want = []
            for L in lens:
                for i in range(T):
                    want.append(sum(1 for t in range(L) if (not causal) or t <= L - T + i))
            np.testing.assert_array_equal(got, want)


def test_status_strings(lib):
    for code in range(-7, 1):
        assert lib.mla_status_string(code)
    assert b"block" in lib.mla_status_string(binding.MLA_ERR_BAD_BLOCK_ID)


def test_binding_fails_loudly_without_the_library(tmp_path):
    with pytest.raises(RuntimeError):
        binding.load_library(str(tmp_path / "missing.so"))


def test_plan_balanced_schedule(lib):
    # Headline shape: 128 requests of 128 pages on 152 SMs -> 76 CTA pairs.
    rc, plan = _plan(lib, batch=128, max_blocks=128, max_seq=8192, lens=[8192] * 128)
    assert rc == 0
    assert (plan.sched_pairs, plan.grid_ctas, plan.num_kv_splits) == (76, 152, 1)
    rows = 2 * 76 * 128
    assert plan.partial_offset == binding.STATUS_BYTES
    assert plan.lse_partial_offset == binding.STATUS_BYTES + rows * 512 * 4
    assert plan.workspace_bytes == plan.lse_partial_offset + rows * 4
    # The split-only flag, the CUDA-core kernel and an explicit S keep the split schedule.
    for kw in (dict(flags=binding.MLA_PLAN_SPLIT_ONLY), dict(flags=binding.MLA_PLAN_FORCE_SIMT),
               dict(splits=2)):
        rc, p2 = _plan(lib, batch=128, max_blocks=128, max_seq=8192, lens=[8192] * 128, **kw)
        assert rc == 0 and p2.sched_pairs == 0, kw
    # More requests than the offsets table holds: split schedule.
    rc, p3 = _plan(lib, batch=600, max_blocks=4, max_seq=256, lens=[256] * 600,
                   flags=binding.MLA_PLAN_FORCE_BALANCED)
    assert rc == 0 and p3.sched_pairs == 0
    # Forced: at most one pair per page.
    rc, p4 = _plan(lib, batch=2, max_blocks=4, max_seq=256, lens=[100, 30],
                   flags=binding.MLA_PLAN_FORCE_BALANCED)
    assert rc == 0 and p4.sched_pairs == 3 and p4.grid_ctas == 6


def test_decode_rejects_a_plan_that_does_not_follow_from_its_sizes(lib):
    rc, plan = _plan(lib, batch=128, max_blocks=128, max_seq=8192, lens=[8192] * 128)
    assert rc == 0
    dummy = ctypes.c_void_p(1 << 20)
    for field, value in (("grid_ctas", plan.grid_ctas + 2), ("sched_pairs", 300),
                         ("workspace_bytes", plan.workspace_bytes - 256),
                         ("num_kv_splits", 2)):
        bad = binding.MlaDecodePlan.from_buffer_copy(plan)
        setattr(bad, field, value)
        rc = lib.mla_decode(ctypes.byref(bad), dummy, dummy, 16, dummy, dummy,
                            ctypes.c_float(0.1), dummy, None, dummy,
                            ctypes.c_size_t(1 << 40), None)
        assert rc == binding.MLA_ERR_INVALID_ARG, field
