"""Thin ctypes binding of libmla_decode (include/mla_decode.h).

Only argument marshalling lives here: torch tensors become device pointers,
the current torch stream becomes the ``stream`` argument, and non-zero
status codes become ``MlaError``. Every arithmetic step runs in the CUDA
library; if the library is missing the calls raise instead of falling back.
"""

from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

MLA_OK = 0
MLA_ERR_INVALID_ARG = -1
MLA_ERR_UNSUPPORTED = -2
MLA_ERR_WORKSPACE = -3
MLA_ERR_CUDA = -4
MLA_ERR_BAD_BLOCK_ID = -5
MLA_ERR_BAD_SEQ_LEN = -6
MLA_ERR_TIMEOUT = -7
MLA_ERR_SCRATCH_LIMIT = -8
MLA_ERR_RANGE = -9

MLA_KERNEL_SIMT = 1
MLA_KERNEL_TC = 2
MLA_PLAN_FORCE_SIMT = 0x1
MLA_PLAN_SPLIT_ONLY = 0x2
MLA_PLAN_FORCE_BALANCED = 0x4
MLA_PLAN_FP32_PARTIALS = 0x8
MLA_PLAN_DEBUG_WITHHOLD_LOAD = 0x100

KV_LORA_RANK = 512
ROPE_DIM = 64
HEAD_DIM = KV_LORA_RANK + ROPE_DIM
PAGE_SIZE = 64
STATUS_BYTES = 8192

EXPORTED_SYMBOLS = (
    "mla_decode_plan", "mla_workspace_init", "mla_decode", "mla_merge_splits",
    "mla_read_error", "mla_status_string", "mla_abi_version", "mla_debug_gather_pages",
    "mla_decode_noalloc", "mla_dcp_local_seq_lens", "mla_dcp_combine",
    "mla_q_absorb_concat_cache", "mla_v_up_proj", "mla_multi_token_scratch_bytes",
    "mla_decode_multi_token", "mla_debug_loader_pages", "mla_multi_token_row_lens",
    "mla_decode_fp8", "mla_merge_splits_v_up_proj", "mla_decode_v_up_proj",
)


class MlaError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class MlaDecodePlan(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("kv_lora_rank", ctypes.c_int32),
        ("rope_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("max_seq_len", ctypes.c_int32),
        ("num_kv_splits", ctypes.c_int32),
        ("kernel", ctypes.c_int32),
        ("num_sms", ctypes.c_int32),
        ("grid_ctas", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("workspace_bytes", ctypes.c_uint64),
        ("partial_offset", ctypes.c_uint64),
        ("lse_partial_offset", ctypes.c_uint64),
        ("sched_pairs", ctypes.c_int32),
        ("reserved", ctypes.c_uint32 * 7),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_ if name != "reserved"}


_LIB = None


def load_library(path=None):
    """Load libmla_decode.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (mla_latent_cache_paged_gb300.build)")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz, f32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                             ctypes.c_float)
    lib.mla_decode_plan.argtypes = [i32, i32, i32, i32, i32, i32, i32, vp, i32, i32,
                                    ctypes.c_uint32, ctypes.POINTER(MlaDecodePlan)]
    lib.mla_workspace_init.argtypes = [vp, sz, vp]
    lib.mla_decode.argtypes = [ctypes.POINTER(MlaDecodePlan), vp, vp, i64, vp, vp, f32, vp, vp,
                               vp, sz, vp]
    lib.mla_decode_fp8.argtypes = [ctypes.POINTER(MlaDecodePlan), vp, vp, i64, vp, vp, f32, f32,
                                   vp, vp, vp, sz, vp]
    lib.mla_merge_splits.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp]
    lib.mla_merge_splits_v_up_proj.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, sz,
                                               vp]
    lib.mla_decode_v_up_proj.argtypes = [ctypes.POINTER(MlaDecodePlan), vp, vp, i64, vp, vp, f32,
                                         vp, vp, vp, vp, vp, sz, vp]
    lib.mla_read_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int), vp]
    lib.mla_status_string.argtypes = [i32]
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_abi_version.argtypes = []
    lib.mla_debug_gather_pages.argtypes = [vp, i64, vp, vp, i32, i32, i32, vp, vp, sz, vp]
    lib.mla_decode_noalloc.argtypes = [ctypes.POINTER(MlaDecodePlan), vp, vp, i64, vp, vp, f32, vp,
                                       vp, vp, vp]
    lib.mla_dcp_local_seq_lens.argtypes = [vp, i32, i32, i32, i32, vp]
    lib.mla_dcp_combine.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp]
    lib.mla_q_absorb_concat_cache.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, i32, vp, vp, sz,
                                              vp]
    lib.mla_v_up_proj.argtypes = [vp, vp, i32, i32, vp, vp, sz, vp]
    lib.mla_debug_loader_pages.argtypes = [ctypes.POINTER(MlaDecodePlan), vp, i64, vp, vp, i32,
                                           vp, vp, sz, vp]
    lib.mla_multi_token_scratch_bytes.argtypes = [i32, i32, i32]
    lib.mla_multi_token_row_lens.argtypes = [vp, i32, i32, i32, vp]
    lib.mla_decode_multi_token.argtypes = [ctypes.POINTER(MlaDecodePlan), i32, i32, i32, vp, vp,
                                           i64, vp, vp, f32, vp, vp, vp, sz, vp, sz, vp]
    for name in EXPORTED_SYMBOLS:
        if name not in ("mla_status_string", "mla_multi_token_scratch_bytes"):
            getattr(lib, name).restype = ctypes.c_int
    lib.mla_multi_token_scratch_bytes.restype = ctypes.c_size_t
    if path == LIB_PATH:
        _LIB = lib
    return lib


def status_string(status):
    try:
        return load_library().mla_status_string(int(status)).decode()
    except RuntimeError:
        return "library not loaded"


def _check(status, what):
    if status != MLA_OK:
        raise MlaError(status, what)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_plan(batch, num_heads, max_blocks_per_seq, max_seq_len=None, *, seq_lens_host=None,
              num_kv_splits=0, num_sms=None, force_simt=False, schedule="auto", extra_flags=0):
    """Call mla_decode_plan (host only; no device work).

    ``schedule``: "auto" (the planner's estimate), "split" (never the
    page-balanced schedule) or "balanced" (the page-balanced schedule wherever
    it applies; needs num_kv_splits = 0). ``extra_flags``: further MLA_PLAN_*
    bits (tests use MLA_PLAN_DEBUG_WITHHOLD_LOAD).
    """
    if schedule not in ("auto", "split", "balanced"):
        raise ValueError(f"schedule must be auto, split or balanced, not {schedule!r}")
    lib = load_library()
    if max_seq_len is None:
        max_seq_len = max_blocks_per_seq * PAGE_SIZE
    if num_sms is None:
        import torch
        num_sms = (torch.cuda.get_device_properties(0).multi_processor_count
                   if torch.cuda.is_available() else 152)
    lens_ptr = ctypes.c_void_p(0)
    keep = None
    if seq_lens_host is not None:
        import numpy as np
        keep = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
        lens_ptr = ctypes.c_void_p(keep.ctypes.data)
    plan = MlaDecodePlan()
    rc = lib.mla_decode_plan(int(batch), int(num_heads), KV_LORA_RANK, ROPE_DIM, PAGE_SIZE,
                             int(max_blocks_per_seq), int(max_seq_len), lens_ptr,
                             int(num_kv_splits), int(num_sms),
                             (MLA_PLAN_FORCE_SIMT if force_simt else 0) |
                             (MLA_PLAN_SPLIT_ONLY if schedule == "split" else 0) |
                             (MLA_PLAN_FORCE_BALANCED if schedule == "balanced" else 0) |
                             int(extra_flags),
                             ctypes.byref(plan))
    del keep
    _check(rc, "mla_decode_plan")
    return plan


def new_workspace(plan, device=None, stream=None):
    """Allocate (through torch) and initialise a workspace for `plan`."""
    import torch
    nbytes = max(int(plan.workspace_bytes), STATUS_BYTES)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
    _check(load_library().mla_workspace_init(_ptr(ws), nbytes, _stream_ptr(stream)),
           "mla_workspace_init")
    return ws


def _check_tensor(t, name, dtype, shape=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def mla_decode(q, latent_cache, block_table, seq_lens, softmax_scale, *, plan=None,
               num_kv_splits=0, out=None, lse=None, return_lse=True, workspace=None,
               stream=None, force_simt=False):
    """Absorbed MLA decode. Returns ``(out bf16 [B,N,512], lse fp32 [B,N] | None)``.

    Mirrors the argument list of ModelOpt's ``mla_attention_decode``; the work
    is one ``mla_decode`` call of the C library on the current stream.
    """
    import torch
    B, N, D = q.shape
    if D != HEAD_DIM:
        raise ValueError(f"q last dim must be {HEAD_DIM}")
    _check_tensor(q, "q", torch.bfloat16)
    _check_tensor(latent_cache, "latent_cache", torch.bfloat16)
    if latent_cache.dim() != 3 or latent_cache.shape[1:] != (PAGE_SIZE, HEAD_DIM):
        raise ValueError("latent_cache must be [num_blocks, 64, 576]")
    _check_tensor(block_table, "block_table", torch.int32)
    _check_tensor(seq_lens, "seq_lens", torch.int32, (B,))
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_blocks_per_seq]")
    if plan is None:
        plan = make_plan(B, N, block_table.shape[1], num_kv_splits=num_kv_splits,
                         force_simt=force_simt)
    if out is None:
        out = torch.empty((B, N, KV_LORA_RANK), dtype=torch.bfloat16, device=q.device)
    _check_tensor(out, "out", torch.bfloat16, (B, N, KV_LORA_RANK))
    if lse is None and return_lse:
        lse = torch.empty((B, N), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_tensor(lse, "lse", torch.float32, (B, N))
    if workspace is None:
        workspace = new_workspace(plan, q.device, stream)
    rc = load_library().mla_decode(
        ctypes.byref(plan), _ptr(q), _ptr(latent_cache), int(latent_cache.shape[0]),
        _ptr(block_table), _ptr(seq_lens), float(softmax_scale), _ptr(out), _ptr(lse),
        _ptr(workspace), int(workspace.numel()), _stream_ptr(stream))
    _check(rc, "mla_decode")
    return out, lse


def mla_decode_fp8(q, latent_cache_fp8, block_table, seq_lens, softmax_scale, k_scale, *,
                   plan=None, num_kv_splits=0, out=None, lse=None, return_lse=True,
                   workspace=None, stream=None):
    """Absorbed MLA decode over an fp8 cache (uint8 E4M3 codes ``[num_blocks,
    64, 576]`` with a per-tensor ``k_scale``). Returns ``(out bf16 [B,N,512],
    lse fp32 [B,N] | None)``; one ``mla_decode_fp8`` call."""
    import torch
    B, N, D = q.shape
    if D != HEAD_DIM:
        raise ValueError(f"q last dim must be {HEAD_DIM}")
    _check_tensor(q, "q", torch.bfloat16)
    _check_tensor(latent_cache_fp8, "latent_cache_fp8", torch.uint8)
    if latent_cache_fp8.dim() != 3 or latent_cache_fp8.shape[1:] != (PAGE_SIZE, HEAD_DIM):
        raise ValueError("latent_cache_fp8 must be [num_blocks, 64, 576]")
    _check_tensor(block_table, "block_table", torch.int32)
    _check_tensor(seq_lens, "seq_lens", torch.int32, (B,))
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_blocks_per_seq]")
    if plan is None:
        plan = make_plan(B, N, block_table.shape[1], num_kv_splits=num_kv_splits)
    if out is None:
        out = torch.empty((B, N, KV_LORA_RANK), dtype=torch.bfloat16, device=q.device)
    _check_tensor(out, "out", torch.bfloat16, (B, N, KV_LORA_RANK))
    if lse is None and return_lse:
        lse = torch.empty((B, N), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_tensor(lse, "lse", torch.float32, (B, N))
    if workspace is None:
        workspace = new_workspace(plan, q.device, stream)
    rc = load_library().mla_decode_fp8(
        ctypes.byref(plan), _ptr(q), _ptr(latent_cache_fp8), int(latent_cache_fp8.shape[0]),
        _ptr(block_table), _ptr(seq_lens), float(softmax_scale), float(k_scale), _ptr(out),
        _ptr(lse), _ptr(workspace), int(workspace.numel()), _stream_ptr(stream))
    _check(rc, "mla_decode_fp8")
    return out, lse


def multi_token_row_lens(seq_lens_host, q_len, causal=True):
    """Tokens each (request, query token) row sees, row r = b * T + i, from
    ``mla_multi_token_row_lens`` (host C; numpy int32 ``[B * T]``)."""
    import numpy as np
    lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32).reshape(-1))
    rows = np.empty(lens.size * int(q_len), dtype=np.int32)
    rc = load_library().mla_multi_token_row_lens(
        ctypes.c_void_p(lens.ctypes.data), int(lens.size), int(q_len), 1 if causal else 0,
        ctypes.c_void_p(rows.ctypes.data))
    _check(rc, "mla_multi_token_row_lens")
    return rows


def make_plan_multi_token(batch, q_len, num_heads, max_blocks_per_seq, *, seq_lens_host=None,
                          causal=True, expand=None, **kw):
    """A plan for a uniform multi-token decode: the T query tokens' heads as
    the rows of one decode when T * N <= 128 (each page read once), else
    B * T rows of N heads. ``expand=True`` forces the second form."""
    if expand is None:
        expand = int(q_len) * int(num_heads) > 128
    if not expand:
        if seq_lens_host is not None:
            kw["seq_lens_host"] = seq_lens_host
        return make_plan(batch, int(q_len) * int(num_heads), max_blocks_per_seq, **kw)
    if seq_lens_host is not None:
        rows = multi_token_row_lens(seq_lens_host, q_len, causal)
        kw.setdefault("max_seq_len", int(rows.max()) if rows.size else 0)
        kw["seq_lens_host"] = rows
    return make_plan(int(batch) * int(q_len), num_heads, max_blocks_per_seq, **kw)


def mla_decode_multi_token(q, latent_cache, block_table, seq_lens, softmax_scale, *,
                           causal=True, plan=None, num_kv_splits=0, out=None, lse=None,
                           return_lse=True, workspace=None, scratch=None, stream=None):
    """Uniform multi-token decode: ``q [B, T, N, 576]`` -> ``(out [B, T, N, 512],
    lse [B, T, N] | None)``; one ``mla_decode_multi_token`` call."""
    import torch
    B, T, N, D = q.shape
    if D != HEAD_DIM:
        raise ValueError(f"q last dim must be {HEAD_DIM}")
    _check_tensor(q, "q", torch.bfloat16)
    _check_tensor(latent_cache, "latent_cache", torch.bfloat16)
    _check_tensor(block_table, "block_table", torch.int32)
    _check_tensor(seq_lens, "seq_lens", torch.int32, (B,))
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_blocks_per_seq]")
    if plan is None:
        plan = make_plan_multi_token(B, T, N, block_table.shape[1], causal=causal,
                                     num_kv_splits=num_kv_splits)
    if out is None:
        out = torch.empty((B, T, N, KV_LORA_RANK), dtype=torch.bfloat16, device=q.device)
    _check_tensor(out, "out", torch.bfloat16, (B, T, N, KV_LORA_RANK))
    if lse is None and return_lse:
        lse = torch.empty((B, T, N), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_tensor(lse, "lse", torch.float32, (B, T, N))
    if workspace is None:
        workspace = new_workspace(plan, q.device, stream)
    lib = load_library()
    if scratch is None and plan.num_heads != T * N:
        nbytes = int(lib.mla_multi_token_scratch_bytes(B, T, block_table.shape[1]))
        scratch = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    rc = lib.mla_decode_multi_token(
        ctypes.byref(plan), int(T), int(N), 1 if causal else 0, _ptr(q), _ptr(latent_cache),
        int(latent_cache.shape[0]), _ptr(block_table), _ptr(seq_lens), float(softmax_scale),
        _ptr(out), _ptr(lse), _ptr(workspace), int(workspace.numel()), _ptr(scratch),
        int(scratch.numel()) if scratch is not None else 0, _stream_ptr(stream))
    _check(rc, "mla_decode_multi_token")
    return out, lse


def mla_merge_splits(o_part, lse_part, *, out=None, lse=None, return_lse=True, stream=None):
    """LSE merge of fp32 partials ``[B,N,S,V]`` / ``[B,N,S]`` -> bf16 ``[B,N,V]``, fp32 ``[B,N]``."""
    import torch
    B, N, S, V = o_part.shape
    _check_tensor(o_part, "o_part", torch.float32)
    _check_tensor(lse_part, "lse_part", torch.float32, (B, N, S))
    if out is None:
        out = torch.empty((B, N, V), dtype=torch.bfloat16, device=o_part.device)
    _check_tensor(out, "out", torch.bfloat16, (B, N, V))
    if lse is None and return_lse:
        lse = torch.empty((B, N), dtype=torch.float32, device=o_part.device)
    rc = load_library().mla_merge_splits(_ptr(o_part), _ptr(lse_part), B, N, S, V, _ptr(out),
                                         _ptr(lse), _stream_ptr(stream))
    _check(rc, "mla_merge_splits")
    return out, lse


def mla_merge_splits_v_up_proj(o_part, lse_part, w_uv, *, workspace, out=None, lse=None,
                               latent_out=None, stream=None):
    """Split merge and up-projection in one launch: fp32 ``[B,N,S,512]`` /
    ``[B,N,S]`` partials and ``W_UV [N,512,128]`` -> bf16 ``out [B,N,128]``
    (``lse`` and the merged ``latent_out`` rows only if given)."""
    import torch
    B, N, S, V = o_part.shape
    _check_tensor(o_part, "o_part", torch.float32)
    _check_tensor(lse_part, "lse_part", torch.float32, (B, N, S))
    _check_tensor(w_uv, "w_uv", torch.bfloat16, (N, 512, 128))
    if V != KV_LORA_RANK:
        raise ValueError("partials must be 512 wide")
    if out is None:
        out = torch.empty((B, N, 128), dtype=torch.bfloat16, device=o_part.device)
    _check_tensor(out, "out", torch.bfloat16, (B, N, 128))
    rc = load_library().mla_merge_splits_v_up_proj(
        _ptr(o_part), _ptr(lse_part), B, N, S, _ptr(w_uv), _ptr(out), _ptr(lse),
        _ptr(latent_out), _ptr(workspace), int(workspace.numel()), _stream_ptr(stream))
    _check(rc, "mla_merge_splits_v_up_proj")
    return out


def mla_decode_v_up_proj(q, latent_cache, block_table, seq_lens, softmax_scale, w_uv, *, plan,
                         workspace, out=None, lse=None, latent_out=None, stream=None):
    """Decode then up-projection (fused with the split merge for split plans):
    returns bf16 ``out [B, N, 128]``."""
    import torch
    B, N, _ = q.shape
    _check_tensor(w_uv, "w_uv", torch.bfloat16, (N, 512, 128))
    if out is None:
        out = torch.empty((B, N, 128), dtype=torch.bfloat16, device=q.device)
    _check_tensor(out, "out", torch.bfloat16, (B, N, 128))
    rc = load_library().mla_decode_v_up_proj(
        ctypes.byref(plan), _ptr(q), _ptr(latent_cache), int(latent_cache.shape[0]),
        _ptr(block_table), _ptr(seq_lens), float(softmax_scale), _ptr(w_uv), _ptr(out), _ptr(lse),
        _ptr(latent_out), _ptr(workspace), int(workspace.numel()), _stream_ptr(stream))
    _check(rc, "mla_decode_v_up_proj")
    return out


def dcp_local_seq_lens(seq_lens_host, world, rank, interleave):
    """Tokens of each request on ``rank`` of ``world`` (runs of ``interleave``
    tokens dealt round-robin): int32 numpy ``[B]``, computed on the host."""
    import numpy as np
    lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
    local = np.empty_like(lens)
    rc = load_library().mla_dcp_local_seq_lens(
        ctypes.c_void_p(lens.ctypes.data), int(lens.size), int(world), int(rank),
        int(interleave), ctypes.c_void_p(local.ctypes.data))
    _check(rc, "mla_dcp_local_seq_lens")
    return local


def mla_dcp_combine(out_parts, lse_parts, *, out=None, lse=None, return_lse=True, stream=None):
    """Combine the ranks' results, bf16 ``[R,B,N,V]`` / fp32 ``[R,B,N]`` ->
    bf16 ``[B,N,V]``, fp32 ``[B,N]``."""
    import torch
    R, B, N, V = out_parts.shape
    _check_tensor(out_parts, "out_parts", torch.bfloat16)
    _check_tensor(lse_parts, "lse_parts", torch.float32, (R, B, N))
    if out is None:
        out = torch.empty((B, N, V), dtype=torch.bfloat16, device=out_parts.device)
    _check_tensor(out, "out", torch.bfloat16, (B, N, V))
    if lse is None and return_lse:
        lse = torch.empty((B, N), dtype=torch.float32, device=out_parts.device)
    rc = load_library().mla_dcp_combine(_ptr(out_parts), _ptr(lse_parts), R, B, N, V, _ptr(out),
                                        _ptr(lse), _stream_ptr(stream))
    _check(rc, "mla_dcp_combine")
    return out, lse


def new_status_workspace(device=None, stream=None):
    """A bare status header (for the calls that need no other workspace)."""
    import torch
    ws = torch.empty(STATUS_BYTES, dtype=torch.uint8, device=device or "cuda")
    _check(load_library().mla_workspace_init(_ptr(ws), STATUS_BYTES, _stream_ptr(stream)),
           "mla_workspace_init")
    return ws


def mla_q_absorb_concat_cache(q, w_uk_t, kv_c=None, k_pe=None, slot_mapping=None,
                              latent_cache=None, *, workspace, out=None, stream=None):
    """Decode front end: ``mqa_q [B, N, 576]`` from ``q [B, N, 192]`` and
    ``W_UK_T [N, 128, 512]``; with ``slot_mapping`` (int64 ``[B]``) the new
    tokens' ``[kv_c | k_pe]`` go into ``latent_cache`` in the same launch."""
    import torch
    B, N, _ = q.shape
    _check_tensor(q, "q", torch.bfloat16, (B, N, 192))
    _check_tensor(w_uk_t, "w_uk_t", torch.bfloat16, (N, 128, 512))
    num_blocks = 0
    if slot_mapping is not None:
        _check_tensor(slot_mapping, "slot_mapping", torch.int64, (B,))
        _check_tensor(kv_c, "kv_c", torch.bfloat16, (B, 512))
        _check_tensor(k_pe, "k_pe", torch.bfloat16, (B, 64))
        _check_tensor(latent_cache, "latent_cache", torch.bfloat16)
        num_blocks = latent_cache.shape[0]
    if out is None:
        out = torch.empty((B, N, 576), dtype=torch.bfloat16, device=q.device)
    _check_tensor(out, "out", torch.bfloat16, (B, N, 576))
    rc = load_library().mla_q_absorb_concat_cache(
        _ptr(q), _ptr(w_uk_t), _ptr(kv_c), _ptr(k_pe), _ptr(slot_mapping), _ptr(latent_cache),
        num_blocks, B, N, _ptr(out), _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check(rc, "mla_q_absorb_concat_cache")
    return out


def mla_v_up_proj(x, w_uv, *, workspace, out=None, stream=None):
    """Up-projection: ``out [B, N, 128]`` from ``x [B, N, 512]`` and ``W_UV [N, 512, 128]``."""
    import torch
    B, N, _ = x.shape
    _check_tensor(x, "x", torch.bfloat16, (B, N, 512))
    _check_tensor(w_uv, "w_uv", torch.bfloat16, (N, 512, 128))
    if out is None:
        out = torch.empty((B, N, 128), dtype=torch.bfloat16, device=x.device)
    _check_tensor(out, "out", torch.bfloat16, (B, N, 128))
    rc = load_library().mla_v_up_proj(_ptr(x), _ptr(w_uv), B, N, _ptr(out), _ptr(workspace),
                                      workspace.numel(), _stream_ptr(stream))
    _check(rc, "mla_v_up_proj")
    return out


def read_error(workspace, stream=None):
    """Synchronise and return (and clear) the device status word of `workspace`."""
    st = ctypes.c_int(0)
    _check(load_library().mla_read_error(_ptr(workspace), ctypes.byref(st), _stream_ptr(stream)),
           "mla_read_error")
    return st.value


def debug_gather_pages(latent_cache, block_table, seq_lens, dst, workspace, stream=None):
    """Test hook: dense gather of every request's rows into ``dst [B, T, 576]``."""
    import torch
    _check_tensor(latent_cache, "latent_cache", torch.bfloat16)
    _check_tensor(dst, "dst", torch.bfloat16)
    B = block_table.shape[0]
    rc = load_library().mla_debug_gather_pages(
        _ptr(latent_cache), int(latent_cache.shape[0]), _ptr(block_table), _ptr(seq_lens), B,
        int(block_table.shape[1]), int(dst.shape[1]), _ptr(dst), _ptr(workspace),
        int(workspace.numel()), _stream_ptr(stream))
    _check(rc, "mla_debug_gather_pages")
    return dst


def debug_loader_pages(plan, latent_cache, block_table, seq_lens, dst, workspace, stream=None):
    """Test hook: the tensor-core kernel's page loaders alone under ``plan``;
    ``dst`` bf16 ``[2, B, T, 576]`` receives, per CTA rank, the rows it loaded."""
    import torch
    _check_tensor(latent_cache, "latent_cache", torch.bfloat16)
    _check_tensor(dst, "dst", torch.bfloat16)
    if dst.dim() != 4 or dst.shape[0] != 2 or dst.shape[1] != plan.batch or dst.shape[3] != 576:
        raise ValueError("dst must be [2, B, T, 576]")
    rc = load_library().mla_debug_loader_pages(
        ctypes.byref(plan), _ptr(latent_cache), int(latent_cache.shape[0]), _ptr(block_table),
        _ptr(seq_lens), int(dst.shape[2]), _ptr(dst), _ptr(workspace), int(workspace.numel()),
        _stream_ptr(stream))
    _check(rc, "mla_debug_loader_pages")
    return dst


def mla_decode_noalloc(q, latent_cache, block_table, seq_lens, softmax_scale, *, plan,
                       out=None, lse=None, device_status=None, stream=None):
    """The decode without a workspace, for callers that cannot allocate device
    memory (see ``mla_decode_noalloc`` in include/mla_decode.h): scratch comes
    from a fixed array inside the library. ``out``/``lse``/``device_status``
    may be given preallocated; nothing here allocates when all three are."""
    import torch
    B, N, _ = q.shape
    if out is None:
        out = torch.empty((B, N, KV_LORA_RANK), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, N), dtype=torch.float32, device=q.device)
    rc = load_library().mla_decode_noalloc(
        ctypes.byref(plan), _ptr(q), _ptr(latent_cache), int(latent_cache.shape[0]),
        _ptr(block_table), _ptr(seq_lens), float(softmax_scale), _ptr(out), _ptr(lse),
        _ptr(device_status), _stream_ptr(stream))
    _check(rc, "mla_decode_noalloc")
    return out, lse
