"""Plain float64 CPU oracle for absorbed ("forward_mqa") MLA decode.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module. It is slow on purpose and shares no code, constant or helper with the
CUDA library: it is written straight from the definitions on the pages.

Every input array holds the values the device sees (bf16 numbers already
widened to float64 by the caller); every result is float64.

Notation (vLLM ``mla_attention`` API docs, module docstring, "More Extent
Definitions"): ``Lkv`` latent width (512 in DSV3), ``R`` RoPE width (64),
``N`` heads, ``P``/``V`` nope / value head dims (128).

Pins (see ``tests/test_oracle.py``):
  * ``mla_decode_reference`` -- hand-derived golden cases, pure-Python brute
    force, closed forms, torch ``scaled_dot_product_attention`` in float64,
    page-table permutation invariance, and the MHA == absorbed-MQA identity.
  * ``mla_decode_split_partials`` + ``merge_partials`` -- split-and-merge equals
    the unsplit definition for many split counts, including empty splits; the
    neutral element (zero output, ``-inf`` LSE) is checked directly.
  * ``gather_request_latent`` -- golden page-table fixture and permutation.
  * ``mha_compute_friendly`` / ``absorb_query`` / ``up_project`` -- the
    identity between the two computing approaches, plus torch SDPA.
  * ``dcp_owner`` / ``dcp_local_seq_lens`` -- a hand-worked placement, the
    per-rank bound the pages print for a shard's length, conservation of
    tokens; ``dcp_decode_partials`` + ``dcp_combine`` -- equal to the unsplit
    definition for every world size and interleave tried, and world 1 is the
    unsplit result itself.
  * ``q_absorb_concat_cache`` / ``v_up_proj`` -- explicit sums over the
    weights' printed layouts on tiny inputs, a hand-worked cache insert, and
    the whole decode step (front end, decode, up-projection) equal to the
    compute-friendly MHA over the cache plus the new token.
  * ``mla_decode_multi_token_reference`` -- T = 1 is the single-token
    definition; each query token equals the single-token definition over the
    tokens it sees; torch SDPA in float64 with the causal block mask; a
    hand-worked two-token case.
  * ``e4m3_to_float`` -- a golden table of codes worked by hand from the
    format, every one of the 256 codes against torch's ``float8_e4m3fn``,
    order and sign symmetry; ``mla_decode_reference_fp8`` -- a hand-worked
    fp8 case, and equality (bit for bit in float64) with the bf16 definition
    when the scale is a power of two, so that every dequantized value is
    also a bf16 number.
No function here is "parity unpinned".
"""

from __future__ import annotations

import math

import numpy as np


def gather_request_latent(cache, block_table_row, seq_len, page_size=None):
    """Rows ``[0, seq_len)`` of one request's latent cache, in logical order.

    Token ``t`` lives in row ``t % page_size`` of physical block
    ``block_table_row[t // page_size]``.

    Cache layout ``[num_blocks, page_size, Lkv + R]`` with one KV head: vLLM
    ``mla/common.py`` (vllm-cpu 0.8.5.post2), ``MLACommonBackend.get_kv_cache_shape``;
    ModelOpt ``mla_attention_decode`` parameters ``latent_cache`` and
    ``block_table`` ([batch, max_blocks_per_seq] page table). The pages name
    the page table but never print the index formula; the page-aligned reading
    here is the one the chunked-context gather uses (vLLM ``mla_attention``
    API docs, ``build_mla_chunked_context_metadata``: a split request advances
    in block-aligned steps). Entries past ``ceil(seq_len / page_size)`` and
    rows past ``seq_len`` are never touched.
    """
    cache = np.asarray(cache)
    if page_size is None:
        page_size = cache.shape[1]
    seq_len = int(seq_len)
    rows = []
    for t in range(seq_len):
        block = int(block_table_row[t // page_size])
        rows.append(cache[block, t % page_size, :])
    if not rows:
        return np.zeros((0, cache.shape[2]), dtype=np.float64)
    return np.stack(rows).astype(np.float64)


def _attend_one(q_heads, k_rows, softmax_scale, kv_lora_rank):
    """softmax(scale * q K^T) V with K = full entry, V = first Lkv columns.

    vLLM ``mla_attention`` API docs, module docstring, "Data-Movement Friendly
    Approach (i.e. forward_mqa)": MQA with QK head dim Lkv + R and V head dim
    Lkv, ``sdpa(cat[ql_nope, q_pe], cat[kv_c, k_pe], kv_c)``. The scale is the
    caller's (ModelOpt ``mla_attention_decode``, ``softmax_scale``). Returns
    ``out [N, Lkv]`` and the natural-log LSE ``[N]`` of the scaled scores
    (ModelOpt ``mla_attention_decode``, ``return_lse``). An empty key set gives
    the merge's neutral element: zero output, ``-inf`` LSE (vLLM
    ``mla_attention`` API docs, ``neutralize_empty_context_partials``).
    """
    n_heads = q_heads.shape[0]
    if k_rows.shape[0] == 0:
        return (np.zeros((n_heads, kv_lora_rank), dtype=np.float64),
                np.full((n_heads,), -np.inf, dtype=np.float64))
    scores = softmax_scale * (q_heads @ k_rows.T)            # [N, L]
    m = scores.max(axis=1, keepdims=True)                    # [N, 1]
    e = np.exp(scores - m)
    denom = e.sum(axis=1, keepdims=True)
    lse = (m + np.log(denom))[:, 0]
    v_rows = k_rows[:, :kv_lora_rank]                         # V = kv_c
    out = (e / denom) @ v_rows
    return out, lse


def mla_decode_reference(q, cache, block_table, seq_lens, softmax_scale,
                         kv_lora_rank=512):
    """Absorbed MLA decode, by definition: ``out [B, N, Lkv]``, ``lse [B, N]``.

    For request ``b`` with ``L = seq_lens[b]`` every query head attends to all
    ``L`` cached tokens (no causal mask: the new token is inserted before the
    attention runs -- vLLM ``mla_attention`` API docs, ``MLAAttention.forward``,
    ``do_kv_cache_update``). Interface: ModelOpt
    ``modelopt.torch.kernels.quantization.attention.mla``,
    ``mla_attention_decode`` (q ``[batch, num_heads, kv_lora_rank +
    qk_rope_head_dim]``, returns ``out [batch, num_heads, kv_lora_rank]`` and
    ``lse [batch, num_heads]``).
    """
    q = np.asarray(q, dtype=np.float64)
    batch, n_heads, _ = q.shape
    out = np.zeros((batch, n_heads, kv_lora_rank), dtype=np.float64)
    lse = np.zeros((batch, n_heads), dtype=np.float64)
    for b in range(batch):
        k_rows = gather_request_latent(cache, block_table[b], seq_lens[b])
        out[b], lse[b] = _attend_one(q[b], k_rows, softmax_scale, kv_lora_rank)
    return out, lse


def split_token_ranges(seq_len, num_splits, page_size):
    """Token ranges of the ``num_splits`` splits of one request.

    ModelOpt ``mla_attention_decode``, ``num_kv_splits``: a fixed split count
    along the token axis. The pages do not print the partition; the reading
    used here keeps splits page-aligned: split ``s`` covers
    ``[s*C, min((s+1)*C, L))`` with ``C = page_size * ceil(ceil(L/page_size) / S)``.
    Splits past the end are empty.
    """
    seq_len = int(seq_len)
    pages = -(-seq_len // page_size)
    chunk = page_size * (-(-pages // num_splits)) if pages else 0
    ranges = []
    for s in range(num_splits):
        lo = min(s * chunk, seq_len)
        hi = min((s + 1) * chunk, seq_len)
        ranges.append((lo, hi))
    return ranges


def mla_decode_split_partials(q, cache, block_table, seq_lens, softmax_scale,
                              num_splits, kv_lora_rank=512):
    """Split-KV partials: ``o_part [B, N, S, Lkv]`` (normalised) and
    ``lse_part [B, N, S]``.

    Each split attends over its own token range exactly as
    ``mla_decode_reference`` does over the whole sequence; empty splits give
    the neutral element (zero output, ``-inf`` LSE).
    """
    q = np.asarray(q, dtype=np.float64)
    cache = np.asarray(cache)
    page_size = cache.shape[1]
    batch, n_heads, _ = q.shape
    o_part = np.zeros((batch, n_heads, num_splits, kv_lora_rank), dtype=np.float64)
    lse_part = np.full((batch, n_heads, num_splits), -np.inf, dtype=np.float64)
    for b in range(batch):
        k_all = gather_request_latent(cache, block_table[b], seq_lens[b], page_size)
        for s, (lo, hi) in enumerate(split_token_ranges(seq_lens[b], num_splits, page_size)):
            o_part[b, :, s, :], lse_part[b, :, s] = _attend_one(
                q[b], k_all[lo:hi], softmax_scale, kv_lora_rank)
    return o_part, lse_part


def merge_partials(o_part, lse_part):
    """LSE-weighted merge of split partials along axis -2 / -1.

    ``o_part [..., S, V]``, ``lse_part [..., S]`` -> ``out [..., V]``,
    ``lse [...]``. vLLM names this ``merge_attn_states`` (``mla_attention`` API
    docs, module docstring "Chunked Prefill" and ``accumulate_mla_context_chunk``)
    but prints no formula; the one used is the exact identity for partials
    normalised by their own softmax sums:
    ``lse = M + ln sum_s exp(lse_s - M)``, ``M = max_s lse_s``,
    ``out = sum_s exp(lse_s - lse) * o_s``. A zero output with ``-inf`` LSE
    carries no weight (``neutralize_empty_context_partials``); when every
    partial is neutral, the result is neutral too.
    """
    o_part = np.asarray(o_part, dtype=np.float64)
    lse_part = np.asarray(lse_part, dtype=np.float64)
    lead = lse_part.shape[:-1]
    out = np.zeros(lead + (o_part.shape[-1],), dtype=np.float64)
    lse = np.full(lead, -np.inf, dtype=np.float64)
    for idx in np.ndindex(*lead):
        ls = lse_part[idx]
        big = ls.max()
        if big == -np.inf:
            continue
        total = big + math.log(np.exp(ls - big).sum())
        lse[idx] = total
        weights = np.exp(ls - total)
        out[idx] = weights @ o_part[idx]
    return out, lse


def absorb_query(q_nope, w_uk):
    """``ql_nope = einsum("snh,lnh->snl", q_nope, W_UK)``.

    vLLM ``mla_attention`` API docs, module docstring, "Data-Movement Friendly
    Approach": ``q_nope [Sq, N, P]``, ``W_UK [Lkv, N, P]`` -> ``[Sq, N, Lkv]``.
    """
    return np.einsum("snh,lnh->snl", np.asarray(q_nope, np.float64),
                     np.asarray(w_uk, np.float64))


def up_project(latent_out, w_uv):
    """``o = einsum("snl,lnv->snv", sdpa_o, W_UV)`` (same section as above)."""
    return np.einsum("snl,lnv->snv", np.asarray(latent_out, np.float64),
                     np.asarray(w_uv, np.float64))


def mha_compute_friendly(q_nope, q_pe, kv_c, k_pe, w_uk, w_uv, softmax_scale):
    """The compute-friendly path ("forward_mha") for one query token.

    vLLM ``mla_attention`` API docs, module docstring, "Compute Friendly
    Approach": ``k_nope = kv_c @ W_UK``, ``v = kv_c @ W_UV``, then MHA with QK
    head dim P + R over ``cat[k_nope, k_pe expanded over heads]``.
    Shapes: ``q_nope [N, P]``, ``q_pe [N, R]``, ``kv_c [L, Lkv]``,
    ``k_pe [L, R]``, ``W_UK [Lkv, N, P]``, ``W_UV [Lkv, N, V]``.
    Returns ``out [N, V]`` and ``lse [N]``.
    """
    q_nope = np.asarray(q_nope, np.float64)
    q_pe = np.asarray(q_pe, np.float64)
    kv_c = np.asarray(kv_c, np.float64)
    k_pe = np.asarray(k_pe, np.float64)
    w_uk = np.asarray(w_uk, np.float64)
    w_uv = np.asarray(w_uv, np.float64)
    n_heads = q_nope.shape[0]
    k_nope = np.einsum("tl,lnp->tnp", kv_c, w_uk)            # [L, N, P]
    v = np.einsum("tl,lnv->tnv", kv_c, w_uv)                 # [L, N, V]
    out = np.zeros((n_heads, w_uv.shape[2]), dtype=np.float64)
    lse = np.zeros((n_heads,), dtype=np.float64)
    for h in range(n_heads):
        q_h = np.concatenate([q_nope[h], q_pe[h]])
        k_h = np.concatenate([k_nope[:, h, :], k_pe], axis=1)  # k_pe shared by heads
        scores = softmax_scale * (k_h @ q_h)
        m = scores.max()
        e = np.exp(scores - m)
        lse[h] = m + math.log(e.sum())
        out[h] = (e / e.sum()) @ v[:, h, :]
    return out, lse


# Decode context parallelism (DCP): every rank holds a shard of every
# request's tokens, attends over its shard, and the ranks' (out, lse) pairs are
# combined with the same LSE merge as split-KV (vLLM ``mla_attention`` API
# docs, ``MLAAttention.forward``: ``forward_mqa`` per rank, then
# ``dcp_manager.combine`` with the per-rank ``lse``).

def dcp_owner(t, world, interleave):
    """Rank that holds token ``t`` and the token's index in that rank's shard.

    vLLM ``mla_attention`` API docs, ``MLACommonMetadataBuilder.__init__`` and
    ``build``: tokens are dealt to the ``world`` ranks in runs of
    ``cp_kv_cache_interleave_size`` (the local block), so one virtual block of
    ``interleave * world`` tokens holds one local block per rank. The pages do
    not print the placement; the reading used is the plain round-robin one:
    run ``t // interleave`` goes to rank ``run % world`` and lands after the
    ``run // world`` runs that rank already holds.
    """
    run = t // interleave
    return run % world, (run // world) * interleave + t % interleave


def dcp_local_seq_lens(seq_lens, world, interleave):
    """Tokens of each request on each rank, ``[world, B]``, by counting owners.

    Brute force over every token: ``counts[r, b]`` is the number of
    ``t < seq_lens[b]`` with ``dcp_owner(t)[0] == r``.
    """
    counts = np.zeros((world, len(seq_lens)), dtype=np.int64)
    for b, seq_len in enumerate(seq_lens):
        for t in range(int(seq_len)):
            counts[dcp_owner(t, world, interleave)[0], b] += 1
    return counts


def dcp_decode_partials(q, cache, block_table, seq_lens, softmax_scale, world,
                        interleave, kv_lora_rank=512):
    """Per-rank results of DCP decode: ``out [world, B, N, Lkv]`` (each
    normalised over the rank's own tokens) and ``lse [world, B, N]``.

    Rank ``r`` attends over the tokens ``dcp_owner`` gives it, in the order of
    their local indices; a rank without tokens of a request gives the merge's
    neutral element (zero output, ``-inf`` LSE).
    """
    q = np.asarray(q, dtype=np.float64)
    page_size = np.asarray(cache).shape[1]
    batch, n_heads, _ = q.shape
    out = np.zeros((world, batch, n_heads, kv_lora_rank), dtype=np.float64)
    lse = np.full((world, batch, n_heads), -np.inf, dtype=np.float64)
    for b in range(batch):
        k_all = gather_request_latent(cache, block_table[b], seq_lens[b], page_size)
        shards = [[] for _ in range(world)]
        for t in range(int(seq_lens[b])):
            r, j = dcp_owner(t, world, interleave)
            assert j == len(shards[r])
            shards[r].append(t)
        for r in range(world):
            out[r, b], lse[r, b] = _attend_one(q[b], k_all[shards[r]], softmax_scale,
                                               kv_lora_rank)
    return out, lse


def dcp_combine(out_parts, lse_parts):
    """Combine the ranks' results: ``out [world, B, N, V]``, ``lse [world, B, N]``
    -> ``out [B, N, V]``, ``lse [B, N]``; the ``merge_partials`` identity taken
    over the rank axis."""
    return merge_partials(np.moveaxis(np.asarray(out_parts), 0, -2),
                          np.moveaxis(np.asarray(lse_parts), 0, -1))


# The steps on either side of the decode (vLLM ``mla_attention`` API docs,
# ``MLAAttention.forward_impl`` and ``_v_up_proj``; raon-1-mini MLA page,
# ``_decode_concat_cache`` and the weight preparation after loading).

def q_absorb_concat_cache(q, w_uk_t, kv_c, k_pe, slot_mapping, cache,
                          qk_nope_head_dim=128):
    """Decode front end: ``mqa_q [B, N, Lkv + R]`` and the cache after the
    new tokens' insert.

    ``q [B, N, P + R]`` is split into ``q_nope`` (P) and ``q_pe`` (R);
    ``ql_nope = bmm(q_nope (N, B, P), W_UK_T (N, P, Lkv))``, transposed back to
    ``(B, N, Lkv)``, with ``W_UK_T = W_UK.permute(1, 2, 0)`` of the
    ``(Lkv, N, P)`` weight; ``mqa_q = cat[ql_nope, q_pe]``. Each request's new
    token ``[kv_c | k_pe]`` is written to row ``slot % page_size`` of block
    ``slot // page_size`` (the page-to-token reading of the decode); the pages
    print no rule for padded tokens, and the reading used is vLLM's padding
    slot id: a negative slot writes nothing. Returns new arrays; the inputs are
    not modified.
    """
    q = np.asarray(q, dtype=np.float64)
    w_uk = np.transpose(np.asarray(w_uk_t, dtype=np.float64), (2, 0, 1))   # (Lkv, N, P)
    ql_nope = absorb_query(q[..., :qk_nope_head_dim], w_uk)
    mqa_q = np.concatenate([ql_nope, q[..., qk_nope_head_dim:]], axis=-1)
    new_cache = np.array(cache, dtype=np.float64, copy=True)
    page_size = new_cache.shape[1]
    kv_c = np.asarray(kv_c, dtype=np.float64)
    k_pe = np.asarray(k_pe, dtype=np.float64)
    lkv = kv_c.shape[-1]
    for b, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        new_cache[slot // page_size, slot % page_size, :lkv] = kv_c[b]
        new_cache[slot // page_size, slot % page_size, lkv:] = k_pe[b]
    return mqa_q, new_cache


def v_up_proj(x, w_uv):
    """``out [B, N, V] = bmm(x (N, B, Lkv), W_UV (N, Lkv, V))`` transposed back,
    with ``W_UV`` the ``(Lkv, N, V)`` weight transposed to ``(N, Lkv, V)``."""
    return up_project(x, np.transpose(np.asarray(w_uv, dtype=np.float64), (1, 0, 2)))


def mla_decode_multi_token_reference(q, cache, block_table, seq_lens, softmax_scale,
                                     causal=True, kv_lora_rank=512):
    """Uniform multi-token decode: ``q [B, T, N, Lkv + R]`` -> ``out [B, T, N,
    Lkv]``, ``lse [B, T, N]``.

    vLLM ``mla_attention`` API docs, ``QueryLenSupport.UNIFORM`` (every request
    has the same query length T > 1) and ``MLACommonMetadataBuilder.build``
    (``causal``; a non-causal query block is also allowed). The T new tokens
    are already in the cache (they are inserted before the attention), so
    request b holds ``L = seq_lens[b]`` tokens and its query token i sits at
    position ``L - T + i``. Reading: with ``causal`` it attends to the tokens
    ``t <= L - T + i``, else to all ``t < L``; a query token that sees no
    token gives the neutral element (zero output, ``-inf`` LSE). Written as
    one masked score matrix ``[T, L]`` per request and head.
    """
    q = np.asarray(q, dtype=np.float64)
    batch, qlen, n_heads, _ = q.shape
    out = np.zeros((batch, qlen, n_heads, kv_lora_rank), dtype=np.float64)
    lse = np.full((batch, qlen, n_heads), -np.inf, dtype=np.float64)
    for b in range(batch):
        L = int(seq_lens[b])
        k_rows = gather_request_latent(cache, block_table[b], L)
        if L == 0:
            continue
        pos = np.arange(L)
        for h in range(n_heads):
            scores = softmax_scale * (q[b, :, h, :] @ k_rows.T)          # [T, L]
            if causal:
                visible = pos[None, :] <= (L - qlen + np.arange(qlen))[:, None]
                scores = np.where(visible, scores, -np.inf)
            for i in range(qlen):
                row = scores[i]
                if not np.isfinite(row).any():
                    continue
                m = row.max()
                e = np.exp(row - m)
                s = e.sum()
                lse[b, i, h] = m + math.log(s)
                out[b, i, h] = (e / s) @ k_rows[:, :kv_lora_rank]
    return out, lse


def e4m3_to_float(bits):
    """8-bit floating point E4M3 codes -> float64 values.

    The pages store a plain per-tensor fp8 latent cache as bytes and have the
    attention read it "as E4M3" (raon-1-mini MLA page,
    ``_attn_read_kv_cache``; vLLM ``mla_attention`` API docs,
    ``MLAAttention.forward_impl``: ``kv_cache.view(current_platform.fp8_dtype())``).
    The format is not printed there; this is the OCP 8-bit floating point
    E4M3 encoding, the finite variant NVIDIA hardware and torch's
    ``float8_e4m3fn`` use: bit 7 the sign, bits 6..3 the exponent e (bias 7),
    bits 2..0 the mantissa m. e = 0 encodes the subnormals m * 2^-9; otherwise
    the value is (1 + m / 8) * 2^(e - 7). There are no infinities; the codes
    with all seven low bits set (0x7F, 0xFF) are NaN, so the largest finite
    magnitude is 1.75 * 2^8 = 448.
    """
    b = np.asarray(bits).astype(np.int64) & 0xFF
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    val = sign * mag
    return np.where((b & 0x7F) == 0x7F, np.nan, val)


def dequantize_e4m3_cache(cache_bits, k_scale):
    """A per-tensor-scaled fp8 cache as float64: ``e4m3(code) * k_scale``.

    vLLM ``mla_attention`` API docs, ``MLAAttention.forward``: the cache
    update and the attention take the layer's single ``_k_scale`` with the
    cache dtype (per-tensor scale); the stored code times that scale is the
    latent entry.
    """
    return e4m3_to_float(cache_bits) * float(k_scale)


def mla_decode_reference_fp8(q, cache_bits, block_table, seq_lens, softmax_scale, k_scale,
                             kv_lora_rank=512):
    """Absorbed MLA decode over an fp8 (E4M3, per-tensor ``k_scale``) latent
    cache: the definition of ``mla_decode_reference`` applied to the
    dequantized cache. K is the whole dequantized entry and V its first
    ``Lkv`` columns; the query stays in its own precision (a backend that
    takes a quantized query is optional on the vLLM page:
    ``supports_quant_query_input``)."""
    return mla_decode_reference(q, dequantize_e4m3_cache(cache_bits, k_scale), block_table,
                                seq_lens, softmax_scale, kv_lora_rank)
