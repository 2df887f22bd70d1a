"""Seeded synthetic inputs for absorbed MLA decode over a paged latent cache.

This module only draws numbers and lays them out; it holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle may use it.

Recipe (every config is bf16, Lkv=512, R=64, page_size=64, scale=1/sqrt(192)):
  * q and every cache row ~ N(0, 1) drawn as float32 from ``numpy`` PCG64
    (``default_rng(seed)``), rounded to bf16 round-to-nearest-even. The same
    bf16 bit patterns go to the device and (widened) to the oracle.
  * The page pool holds ``sum_b ceil(L_b / 64)`` blocks plus ``extra_blocks``;
    pages are assigned to requests, in request order, from one random
    permutation of the pool, so logical and physical order never agree.
  * Unused block-table entries hold out-of-range sentinels and the rows past
    ``L_b`` in a request's last page hold NaN, so any read of them shows up.
  * ``outlier_frac`` scales that fraction of the cached token rows (all 576
    columns) by 8, which is exact in bf16.
  * fp8 caches (``cache_dtype="fp8"``): the same float32 draws (and the same
    x8 rows) are stored as E4M3 codes of ``x / k_scale`` (round to nearest
    even, saturated at +-448) with one per-tensor ``k_scale = amax / 448``
    over the pool (float32); tail rows hold the NaN code 0x7F. q stays bf16.
Config names describe their shapes; ``WORKLOADS`` lists them.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

KV_LORA_RANK = 512
ROPE_DIM = 64
HEAD_DIM = KV_LORA_RANK + ROPE_DIM
PAGE_SIZE = 64
DEFAULT_SCALE = 1.0 / math.sqrt(192.0)
BF16_NAN = np.uint16(0x7FC0)
E4M3_NAN = np.uint8(0x7F)
E4M3_MAX = 448.0


def f32_to_bf16_bits(x):
    """Round float32 values to bf16 (round to nearest, ties to even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    nan = (u & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    if nan.any():
        r[nan] = BF16_NAN
    return r


def f32_to_e4m3_bits(x):
    """Round float32 values to E4M3 codes (sign, 4 exponent bits with bias 7,
    3 mantissa bits; subnormals m * 2^-9): round to nearest, ties to even,
    magnitudes beyond 448 saturated to 448, NaN to 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    nan = np.isnan(x)
    sign = np.signbit(x)
    a = np.minimum(np.abs(np.where(nan, 0.0, x)), E4M3_MAX)
    frac, exp = np.frexp(a)                       # a = frac * 2^exp, frac in [0.5, 1)
    e = exp - 1                                   # a = (2 * frac) * 2^e
    normal = (e >= -6) & (a > 0)
    # normal: mantissa steps of 2^(e-3); subnormal: steps of 2^-9
    step = np.exp2(np.where(normal, e - 3, -9).astype(np.float64))
    k = np.rint(a / step).astype(np.int64)        # half to even
    # normal: k in [8, 16]; 16 carries into the next exponent
    ee = np.where(normal, e + 7, 0)
    carry = normal & (k == 16)
    ee = np.where(carry, ee + 1, ee)
    k = np.where(carry, 8, k)
    # subnormal: k in [0, 8]; 8 is the smallest normal (e field 1, m 0)
    sub_to_normal = (~normal) & (k == 8)
    ee = np.where(sub_to_normal, 1, ee)
    m = np.where(normal | sub_to_normal, k - 8, k)
    m = np.where(sub_to_normal, 0, m)
    code = ((ee.astype(np.int64) << 3) | m).astype(np.int64)
    code = np.where(sign, code | 0x80, code)
    code = np.where(nan, 0x7F, code)
    return code.astype(np.uint8)


def bf16_bits_to_f32(bits):
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


@dataclasses.dataclass
class Workload:
    name: str
    batch: int
    num_heads: int
    seq_lens: np.ndarray          # int32 [B]
    block_table: np.ndarray       # int32 [B, max_blocks_per_seq]
    num_blocks: int
    q_bits: np.ndarray            # uint16 [B, N, 576] (bf16 patterns)
    cache_bits: np.ndarray        # uint16 [num_blocks, 64, 576]
    softmax_scale: float = DEFAULT_SCALE
    num_kv_splits: int = 0        # 0: the planner chooses
    cache_dtype: str = "bf16"     # "bf16" (uint16 codes) or "fp8" (uint8 E4M3 codes)
    k_scale: float = 1.0          # per-tensor scale of an fp8 cache
    page_size: int = PAGE_SIZE
    kv_lora_rank: int = KV_LORA_RANK
    rope_dim: int = ROPE_DIM

    @property
    def total_tokens(self):
        return int(np.asarray(self.seq_lens, dtype=np.int64).sum())

    @property
    def max_blocks_per_seq(self):
        return int(self.block_table.shape[1])

    @property
    def max_seq_len(self):
        return int(np.max(self.seq_lens)) if self.batch else 0

    def q_f64(self):
        return bf16_bits_to_f64(self.q_bits)

    def cache_f64(self):
        return bf16_bits_to_f64(self.cache_bits)


def _normal_f32(rng, shape, chunk_elems=1 << 26):
    """N(0,1) float32 draws, generated in the same chunks as _normal_bf16."""
    total = int(np.prod(shape))
    out = np.empty(total, dtype=np.float32)
    pos = 0
    while pos < total:
        n = min(chunk_elems, total - pos)
        out[pos:pos + n] = rng.standard_normal(n, dtype=np.float32)
        pos += n
    return out.reshape(shape)


def _normal_bf16(rng, shape, chunk_elems=1 << 26):
    """N(0,1) float32 draws rounded to bf16, generated in chunks."""
    total = int(np.prod(shape))
    out = np.empty(total, dtype=np.uint16)
    pos = 0
    while pos < total:
        n = min(chunk_elems, total - pos)
        out[pos:pos + n] = f32_to_bf16_bits(rng.standard_normal(n, dtype=np.float32))
        pos += n
    return out.reshape(shape)


def make_workload(name, batch, num_heads, seq_lens, *, seed, page_size=PAGE_SIZE,
                  extra_blocks=0, outlier_frac=0.0, num_kv_splits=0,
                  softmax_scale=DEFAULT_SCALE, max_blocks_per_seq=None,
                  poison=True, with_data=True, cache_dtype="bf16"):
    """Build one seeded workload (see the module docstring for the recipe)."""
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32).reshape(batch)
    pages = [-(-int(L) // page_size) for L in seq_lens]
    used = int(sum(pages))
    num_blocks = used + int(extra_blocks)
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max([1] + pages)
    perm = rng.permutation(num_blocks).astype(np.int32)
    block_table = np.empty((batch, max_blocks_per_seq), dtype=np.int32)
    # Sentinels in unused entries: alternate -1 and an id past the pool.
    sentinel = np.where(np.arange(max_blocks_per_seq) % 2 == 0, -1,
                        num_blocks + 7).astype(np.int32)
    block_table[:] = sentinel
    pos = 0
    for b, p in enumerate(pages):
        block_table[b, :p] = perm[pos:pos + p]
        pos += p
    q_bits = cache_bits = None
    k_scale = 1.0
    if cache_dtype not in ("bf16", "fp8"):
        raise ValueError(f"cache_dtype must be bf16 or fp8, not {cache_dtype!r}")
    if with_data:
        q_bits = _normal_bf16(rng, (batch, num_heads, HEAD_DIM))
        fp8 = cache_dtype == "fp8"
        if fp8:
            cache_f32 = _normal_f32(rng, (num_blocks, page_size, HEAD_DIM))
        else:
            cache_bits = _normal_bf16(rng, (num_blocks, page_size, HEAD_DIM))
        if outlier_frac > 0.0:
            # token rows that hold real tokens, as (block, row) pairs
            rows = []
            for b in range(batch):
                L = int(seq_lens[b])
                t = np.arange(L, dtype=np.int64)
                rows.append(block_table[b, t // page_size].astype(np.int64) * page_size
                            + t % page_size)
            valid = np.concatenate(rows) if rows else np.zeros(0, np.int64)
            k = int(math.floor(outlier_frac * valid.size))
            pick = rng.choice(valid, size=k, replace=False) if k else valid[:0]
            if fp8:
                flat32 = cache_f32.reshape(-1, HEAD_DIM)
                flat32[pick] = flat32[pick] * np.float32(8.0)
            else:
                flat = cache_bits.reshape(-1, HEAD_DIM)
                vals = bf16_bits_to_f32(flat[pick]) * np.float32(8.0)
                flat[pick] = f32_to_bf16_bits(vals)
        if fp8:
            amax = float(np.abs(cache_f32).max()) if cache_f32.size else 1.0
            k_scale = float(np.float32(amax / E4M3_MAX)) if amax > 0 else 1.0
            cache_bits = np.empty(cache_f32.shape, dtype=np.uint8)
            flat_in = cache_f32.reshape(-1)
            flat_out = cache_bits.reshape(-1)
            for pos in range(0, flat_in.size, 1 << 24):
                flat_out[pos:pos + (1 << 24)] = f32_to_e4m3_bits(
                    flat_in[pos:pos + (1 << 24)] / np.float32(k_scale))
            del cache_f32
        if poison:
            for b in range(batch):
                L = int(seq_lens[b])
                if L % page_size:
                    last = block_table[b, L // page_size]
                    cache_bits[last, L % page_size:, :] = E4M3_NAN if fp8 else BF16_NAN
    return Workload(name=name, batch=batch, num_heads=num_heads, seq_lens=seq_lens,
                    block_table=block_table, num_blocks=num_blocks, q_bits=q_bits,
                    cache_bits=cache_bits, softmax_scale=softmax_scale,
                    num_kv_splits=num_kv_splits, page_size=page_size,
                    cache_dtype=cache_dtype, k_scale=k_scale)


def _c1(with_data=True):
    # B=1, N=16, L=256: 4 pages at random ids of an 8-block pool, S=1.
    return make_workload("b1_n16_l256_pool8", 1, 16, [256], seed=20260001,
                         extra_blocks=4, num_kv_splits=1, with_data=with_data)


def _c2(with_data=True):
    rng = np.random.default_rng(20260002 + 100)
    lens = rng.integers(1024, 4096, size=32, endpoint=True)
    return make_workload("b32_n128_l1k-4k", 32, 128, lens, seed=20260002,
                         num_kv_splits=32, with_data=with_data)


def _c3(with_data=True):
    return make_workload("b128_n128_l8192", 128, 128, [8192] * 128, seed=20260003,
                         num_kv_splits=0, with_data=with_data)


def _c3_small(with_data=True):
    # The headline shape at 16 requests (151 MB of cache, still larger than
    # L2): the small case for full-section profiles of the same kernel.
    return make_workload("b16_n128_l8192", 16, 128, [8192] * 16, seed=20260006,
                         num_kv_splits=0, with_data=with_data)


def _c3_mid(with_data=True):
    # The headline shape at 32 requests: 604 MB of bf16 cache (302 MB as fp8),
    # larger than L2 either way; the small case for full-section profiles.
    return make_workload("b32_n128_l8192", 32, 128, [8192] * 32, seed=20260007,
                         num_kv_splits=0, with_data=with_data)


def _c4(length):
    def build(with_data=True):
        return make_workload(f"b4_n128_l{length // 1024}k_s64", 4, 128, [length] * 4,
                             seed=20260004 * 10 + length // 32768,
                             num_kv_splits=64, with_data=with_data)
    return build


def _c5(with_data=True):
    rng = np.random.default_rng(20260005 + 100)
    u = rng.uniform(math.log(16), math.log(32768), size=256)
    lens = np.clip(np.rint(np.exp(u)), 16, 32768).astype(np.int32)
    return make_workload("b256_n128_logu16-32k_outliers", 256, 128, lens,
                         seed=20260005, outlier_frac=0.01, num_kv_splits=0,
                         with_data=with_data)


def _fp8(build):
    """The same workload with an fp8 (E4M3, per-tensor scale) cache."""
    def make(with_data=True):
        w0 = build(with_data=False)
        return make_workload(w0.name + "_fp8", w0.batch, w0.num_heads, w0.seq_lens,
                             seed=_SEEDS[w0.name], extra_blocks=w0.num_blocks - sum(
                                 -(-int(L) // w0.page_size) for L in w0.seq_lens),
                             outlier_frac=_OUTLIERS.get(w0.name, 0.0),
                             num_kv_splits=w0.num_kv_splits, with_data=with_data,
                             cache_dtype="fp8")
    return make


WORKLOADS = {
    "b1_n16_l256_pool8": _c1,
    "b32_n128_l1k-4k": _c2,
    "b128_n128_l8192": _c3,
    "b16_n128_l8192": _c3_small,
    "b32_n128_l8192": _c3_mid,
    "b4_n128_l32k_s64": _c4(32768),
    "b4_n128_l64k_s64": _c4(65536),
    "b4_n128_l96k_s64": _c4(98304),
    "b4_n128_l128k_s64": _c4(131072),
    "b256_n128_logu16-32k_outliers": _c5,
}

_SEEDS = {"b1_n16_l256_pool8": 20260001, "b32_n128_l1k-4k": 20260002,
          "b128_n128_l8192": 20260003, "b16_n128_l8192": 20260006, "b32_n128_l8192": 20260007,
          "b4_n128_l32k_s64": 20260004 * 10 + 1, "b4_n128_l64k_s64": 20260004 * 10 + 2,
          "b4_n128_l96k_s64": 20260004 * 10 + 3, "b4_n128_l128k_s64": 20260004 * 10 + 4,
          "b256_n128_logu16-32k_outliers": 20260005}
_OUTLIERS = {"b256_n128_logu16-32k_outliers": 0.01}
for _name in list(WORKLOADS):
    WORKLOADS[_name + "_fp8"] = _fp8(WORKLOADS[_name])

HEADLINE = "b128_n128_l8192"


def get_workload(name, with_data=True):
    return WORKLOADS[name](with_data=with_data)


def to_torch(w, device="cuda"):
    """Device tensors of a workload: q (bf16), latent_cache (bf16, or uint8 E4M3
    codes for an fp8 cache), block_table, seq_lens (int32)."""
    import torch
    q = torch.from_numpy(w.q_bits.view(np.int16)).view(torch.bfloat16).to(device)
    if w.cache_dtype == "fp8":
        cache = torch.from_numpy(np.ascontiguousarray(w.cache_bits)).to(device)
    else:
        cache = torch.from_numpy(w.cache_bits.view(np.int16)).view(torch.bfloat16).to(device)
    table = torch.from_numpy(np.ascontiguousarray(w.block_table)).to(device)
    lens = torch.from_numpy(np.ascontiguousarray(w.seq_lens)).to(device)
    return q, cache, table, lens


def bf16_tensor_bits(t):
    """uint16 bit patterns (numpy) of a bf16 torch tensor."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
