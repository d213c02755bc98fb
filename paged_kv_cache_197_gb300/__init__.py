"""Paged KV-cache decode on GB300: Python binding of the C ABI in include/pa.h.

Every function here only marshals arguments (torch tensors -> pointers and sizes)
and calls the function of the same name in libpa.so; all of the work runs in the
library's CUDA kernels.  There is no CPU fallback: if the library is missing or
its call fails, an exception is raised.

Layouts (see include/pa.h):
  query, out        [S][Hq][D] bf16
  k_cache, v_cache  [N][Hkv][bs][D] bf16 or int8
  k_scale, v_scale  [N][Hkv][bs] fp32 (int8 caches)
  block_tables      [S][M] int32, context_lens [S] int32, slot_mapping [T] int64
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

PKG = Path(__file__).resolve().parent
LIBRARY = PKG / "libpa.so"

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_OUT_OF_RANGE, PA_ERR_CUDA = range(5)
PA_KV_BF16, PA_KV_INT8, PA_KV_FP8 = 0, 1, 2
PA_FLAG_SLOT_OUT_OF_RANGE = 1
PA_FLAG_BLOCK_OUT_OF_RANGE = 2
PA_FLAG_CONTEXT_OUT_OF_RANGE = 4
PA_FLAG_PREFIX_MISMATCH = 8
PA_FLAG_QUERY_OUT_OF_RANGE = 16
PA_FLAG_TIMEOUT = 32
PA_FLAG_FP16_RANGE = 64
PA_FLAG_WORKSPACE_SHORT = 128

EXPORTED = ["pa_version", "pa_status_string", "pa_last_error_string", "pa_reshape_and_cache",
            "pa_quantize_kv", "pa_quantize_kv_fp8", "pa_copy_blocks", "pa_decode_workspace_size", "pa_decode",
            "pa_decode_noalloc", "pa_decode_shared_prefix_workspace_size", "pa_decode_shared_prefix",
            "pa_multi_token_workspace_size", "pa_multi_token_workspace_size_for_tokens",
            "pa_multi_token_attention"]
PA_NOALLOC_SCRATCH_BYTES = 16 << 20


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"[status {status}] {message}")
        self.status = status


_LIB: ctypes.CDLL | None = None


def load_library(path: Path | str | None = None) -> ctypes.CDLL:
    """Load libpa.so (built by __graft_entry__.build()); raise if it is absent."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = Path(path) if path is not None else LIBRARY
    if not p.exists():
        raise RuntimeError(f"{p} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(str(p))
    vp, i32, i64, sz, f32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                             ctypes.c_float)
    lib.pa_version.restype = i32
    lib.pa_status_string.argtypes = [i32]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_last_error_string.restype = ctypes.c_char_p
    lib.pa_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]
    lib.pa_reshape_and_cache.restype = i32
    lib.pa_quantize_kv.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]
    lib.pa_quantize_kv.restype = i32
    lib.pa_quantize_kv_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]
    lib.pa_quantize_kv_fp8.restype = i32
    lib.pa_copy_blocks.argtypes = [vp, vp, vp, vp, vp, i32, i32, sz, i32, vp]
    lib.pa_copy_blocks.restype = i32
    lib.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.pa_decode_workspace_size.restype = sz
    lib.pa_decode.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32, i32,
                              i32, f32, i32, vp, sz, vp, vp]
    lib.pa_decode.restype = i32
    lib.pa_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32,
                                      i32, i32, f32, i32, vp, vp]
    lib.pa_decode_noalloc.restype = i32
    lib.pa_decode_shared_prefix_workspace_size.argtypes = [i32] * 9
    lib.pa_decode_shared_prefix_workspace_size.restype = sz
    lib.pa_decode_shared_prefix.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32,
                                            i32, i32, i32, f32, i32, vp, vp, i32, i32, i32, vp, sz,
                                            vp, vp]
    lib.pa_decode_shared_prefix.restype = i32
    lib.pa_multi_token_workspace_size.argtypes = [i32] * 9
    lib.pa_multi_token_workspace_size.restype = sz
    lib.pa_multi_token_workspace_size_for_tokens.argtypes = [i32] * 9 + [i64]
    lib.pa_multi_token_workspace_size_for_tokens.restype = sz
    lib.pa_multi_token_attention.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, vp, vp, i32,
                                             i32, i32, i32, i32, i32, i32, f32, i32, i32, vp, sz,
                                             vp, vp]
    lib.pa_multi_token_attention.restype = i32
    if path is None:
        _LIB = lib
    return lib


def _check(status: int) -> None:
    if status != PA_OK:
        lib = load_library()
        raise PagedAttentionError(status, lib.pa_last_error_string().decode())


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _cuda(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int | None = None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dimensions, got {t.dim()}")


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _flag(err_flag):
    if err_flag is not None:
        _cuda(err_flag, "err_flag", torch.int32)
    return _ptr(err_flag)


def pa_version() -> int:
    return int(load_library().pa_version())


def pa_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, err_flag=None,
                         stream=None) -> None:
    """Append the bf16 rows key/value [T][Hkv][D] into slots of a bf16 paged cache."""
    for t, n in ((key, "key"), (value, "value")):
        _cuda(t, n, torch.bfloat16, 3)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _cuda(t, n, torch.bfloat16, 4)
    _cuda(slot_mapping, "slot_mapping", torch.int64, 1)
    T, Hkv, D = key.shape
    N, Hkv2, bs, D2 = k_cache.shape
    if value.shape != key.shape or v_cache.shape != k_cache.shape or (Hkv2, D2) != (Hkv, D) \
            or slot_mapping.shape[0] != T:
        raise ValueError("pa_reshape_and_cache: shape mismatch")
    lib = load_library()
    _check(lib.pa_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(slot_mapping), T, Hkv, D, bs, N, _flag(err_flag),
                                    _stream(stream, key.device)))


def pa_quantize_kv(key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, err_flag=None,
                   stream=None) -> None:
    """Quantise bf16 rows [T][Hkv][D] to int8 with a per-(token, kv head) scale and append."""
    for t, n in ((key, "key"), (value, "value")):
        _cuda(t, n, torch.bfloat16, 3)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _cuda(t, n, torch.int8, 4)
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _cuda(t, n, torch.float32, 3)
    _cuda(slot_mapping, "slot_mapping", torch.int64, 1)
    T, Hkv, D = key.shape
    N, Hkv2, bs, D2 = k_cache.shape
    if value.shape != key.shape or v_cache.shape != k_cache.shape or (Hkv2, D2) != (Hkv, D) \
            or tuple(k_scale.shape) != (N, Hkv, bs) or v_scale.shape != k_scale.shape \
            or slot_mapping.shape[0] != T:
        raise ValueError("pa_quantize_kv: shape mismatch")
    lib = load_library()
    _check(lib.pa_quantize_kv(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                              _ptr(v_scale), _ptr(slot_mapping), T, Hkv, D, bs, N, _flag(err_flag),
                              _stream(stream, key.device)))


FP8_DTYPES = (torch.uint8,) + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ())


def kv_dtype_of(cache: torch.Tensor) -> int:
    """PA_KV_* code of a cache tensor: bf16, int8, or fp8 e4m3 bytes (uint8 or float8_e4m3fn)."""
    if cache.dtype == torch.bfloat16:
        return PA_KV_BF16
    if cache.dtype == torch.int8:
        return PA_KV_INT8
    if cache.dtype in FP8_DTYPES:
        return PA_KV_FP8
    raise TypeError(f"unsupported cache dtype {cache.dtype}")


def pa_quantize_kv_fp8(key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, err_flag=None,
                       stream=None) -> None:
    """Quantise bf16 rows [T][Hkv][D] to fp8 e4m3 with a per-(token, kv head) scale and append."""
    for t, n in ((key, "key"), (value, "value")):
        _cuda(t, n, torch.bfloat16, 3)
    if k_cache.dtype not in FP8_DTYPES:
        raise TypeError("fp8 caches are uint8 or float8_e4m3fn tensors")
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _cuda(t, n, k_cache.dtype, 4)
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _cuda(t, n, torch.float32, 3)
    _cuda(slot_mapping, "slot_mapping", torch.int64, 1)
    T, Hkv, D = key.shape
    N, Hkv2, bs, D2 = k_cache.shape
    if value.shape != key.shape or v_cache.shape != k_cache.shape or (Hkv2, D2) != (Hkv, D) \
            or tuple(k_scale.shape) != (N, Hkv, bs) or v_scale.shape != k_scale.shape \
            or slot_mapping.shape[0] != T:
        raise ValueError("pa_quantize_kv_fp8: shape mismatch")
    lib = load_library()
    _check(lib.pa_quantize_kv_fp8(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                  _ptr(v_scale), _ptr(slot_mapping), T, Hkv, D, bs, N, _flag(err_flag),
                                  _stream(stream, key.device)))


def pa_copy_blocks(k_cache, v_cache, block_mapping, k_scale=None, v_scale=None,
                   stream=None) -> None:
    """Copy whole physical blocks (src, dst) of both caches (and scales, if given).

    block_mapping is a HOST sequence of (src, dst) pairs (tensor, ndarray or list)."""
    kv_dtype_of(k_cache)
    _cuda(k_cache, "k_cache", k_cache.dtype)
    _cuda(v_cache, "v_cache", k_cache.dtype)
    if v_cache.shape != k_cache.shape:
        raise ValueError("pa_copy_blocks: cache shapes differ")
    pairs = torch.as_tensor(block_mapping, dtype=torch.int64, device="cpu").reshape(-1, 2).contiguous()
    N = k_cache.shape[0]
    block_bytes = k_cache.numel() * k_cache.element_size() // N
    scale_elems = 0
    if k_scale is not None or v_scale is not None:
        if k_scale is None or v_scale is None:
            raise ValueError("give both scale arrays or neither")
        _cuda(k_scale, "k_scale", torch.float32)
        _cuda(v_scale, "v_scale", torch.float32)
        if k_scale.shape[0] != N or v_scale.shape != k_scale.shape:
            raise ValueError("pa_copy_blocks: scale shapes")
        scale_elems = k_scale.numel() // N
    lib = load_library()
    _check(lib.pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                              pairs.data_ptr(), pairs.shape[0], N, block_bytes, scale_elems,
                              _stream(stream, k_cache.device)))


def pa_decode_workspace_size(S: int, Hq: int, Hkv: int, D: int, bs: int, kv_dtype: int,
                             max_context_len: int) -> int:
    return int(load_library().pa_decode_workspace_size(S, Hq, Hkv, D, bs, kv_dtype,
                                                       max_context_len))


def pa_decode(out, query, k_cache, v_cache, block_tables, context_lens, scale: float,
              max_context_len: int, workspace=None, k_scale=None, v_scale=None, err_flag=None,
              stream=None) -> None:
    """Paged decode attention; writes out [S][Hq][D] bf16."""
    _cuda(out, "out", torch.bfloat16, 3)
    _cuda(query, "query", torch.bfloat16, 3)
    kv_dtype = kv_dtype_of(k_cache)
    _cuda(k_cache, "k_cache", k_cache.dtype, 4)
    _cuda(v_cache, "v_cache", k_cache.dtype, 4)
    _cuda(block_tables, "block_tables", torch.int32, 2)
    _cuda(context_lens, "context_lens", torch.int32, 1)
    if kv_dtype != PA_KV_BF16:
        if k_scale is None or v_scale is None:
            raise ValueError("an int8 or fp8 cache needs k_scale and v_scale")
        _cuda(k_scale, "k_scale", torch.float32, 3)
        _cuda(v_scale, "v_scale", torch.float32, 3)
    S, Hq, D = query.shape
    N, Hkv, bs, D2 = k_cache.shape
    M = block_tables.shape[1]
    if out.shape != query.shape or v_cache.shape != k_cache.shape or D2 != D \
            or block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise ValueError("pa_decode: shape mismatch")
    ws_bytes = 0
    if workspace is not None:
        _cuda(workspace, "workspace", workspace.dtype)
        ws_bytes = workspace.numel() * workspace.element_size()
    lib = load_library()
    _check(lib.pa_decode(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                         _ptr(v_scale), kv_dtype, _ptr(block_tables), M, _ptr(context_lens), S, Hq,
                         Hkv, D, bs, N, float(scale), int(max_context_len), _ptr(workspace),
                         ws_bytes, _flag(err_flag), _stream(stream, query.device)))


def pa_decode_noalloc(out, query, k_cache, v_cache, block_tables, context_lens, scale: float,
                      max_context_len: int, k_scale=None, v_scale=None, err_flag=None,
                      stream=None) -> None:
    """pa_decode for callers that cannot allocate: the library's own fixed scratch array
    (PA_NOALLOC_SCRATCH_BYTES per GPU) replaces the workspace.  Calls sharing a device
    must not overlap on the GPU."""
    _cuda(out, "out", torch.bfloat16, 3)
    _cuda(query, "query", torch.bfloat16, 3)
    kv_dtype = kv_dtype_of(k_cache)
    _cuda(k_cache, "k_cache", k_cache.dtype, 4)
    _cuda(v_cache, "v_cache", k_cache.dtype, 4)
    _cuda(block_tables, "block_tables", torch.int32, 2)
    _cuda(context_lens, "context_lens", torch.int32, 1)
    if kv_dtype != PA_KV_BF16:
        if k_scale is None or v_scale is None:
            raise ValueError("an int8 or fp8 cache needs k_scale and v_scale")
        _cuda(k_scale, "k_scale", torch.float32, 3)
        _cuda(v_scale, "v_scale", torch.float32, 3)
    S, Hq, D = query.shape
    N, Hkv, bs, D2 = k_cache.shape
    if out.shape != query.shape or v_cache.shape != k_cache.shape or D2 != D \
            or block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise ValueError("pa_decode_noalloc: shape mismatch")
    lib = load_library()
    _check(lib.pa_decode_noalloc(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(k_scale), _ptr(v_scale), kv_dtype, _ptr(block_tables),
                                 block_tables.shape[1], _ptr(context_lens), S, Hq, Hkv, D, bs, N,
                                 float(scale), int(max_context_len), _flag(err_flag),
                                 _stream(stream, query.device)))


def pa_decode_shared_prefix_workspace_size(S: int, Hq: int, Hkv: int, D: int, bs: int,
                                           kv_dtype: int, max_context_len: int,
                                           max_group_size: int, max_prefix_len: int) -> int:
    return int(load_library().pa_decode_shared_prefix_workspace_size(
        S, Hq, Hkv, D, bs, kv_dtype, max_context_len, max_group_size, max_prefix_len))


def pa_decode_shared_prefix(out, query, k_cache, v_cache, block_tables, context_lens,
                            scale: float, max_context_len: int, group_start, group_prefix_len,
                            max_group_size: int, max_prefix_len: int, workspace=None,
                            k_scale=None, v_scale=None, err_flag=None, stream=None) -> None:
    """Paged decode of a batch whose groups of consecutive sequences share prefix blocks;
    the same result as pa_decode.  group_start [n_groups + 1] and group_prefix_len
    [n_groups] are int32 device tensors; workspace defaults to a fresh allocation."""
    _cuda(out, "out", torch.bfloat16, 3)
    _cuda(query, "query", torch.bfloat16, 3)
    kv_dtype = kv_dtype_of(k_cache)
    _cuda(k_cache, "k_cache", k_cache.dtype, 4)
    _cuda(v_cache, "v_cache", k_cache.dtype, 4)
    _cuda(block_tables, "block_tables", torch.int32, 2)
    _cuda(context_lens, "context_lens", torch.int32, 1)
    _cuda(group_start, "group_start", torch.int32, 1)
    _cuda(group_prefix_len, "group_prefix_len", torch.int32, 1)
    if kv_dtype != PA_KV_BF16:
        if k_scale is None or v_scale is None:
            raise ValueError("an int8 or fp8 cache needs k_scale and v_scale")
        _cuda(k_scale, "k_scale", torch.float32, 3)
        _cuda(v_scale, "v_scale", torch.float32, 3)
    S, Hq, D = query.shape
    N, Hkv, bs, D2 = k_cache.shape
    M = block_tables.shape[1]
    n_groups = group_prefix_len.shape[0]
    if out.shape != query.shape or v_cache.shape != k_cache.shape or D2 != D \
            or block_tables.shape[0] != S or context_lens.shape[0] != S \
            or group_start.shape[0] != n_groups + 1:
        raise ValueError("pa_decode_shared_prefix: shape mismatch")
    if workspace is None:
        n = pa_decode_shared_prefix_workspace_size(S, Hq, Hkv, D, bs, kv_dtype, max_context_len,
                                                   max_group_size, max_prefix_len)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=query.device)
    _cuda(workspace, "workspace", workspace.dtype)
    ws_bytes = workspace.numel() * workspace.element_size()
    lib = load_library()
    _check(lib.pa_decode_shared_prefix(
        _ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        kv_dtype, _ptr(block_tables), M, _ptr(context_lens), S, Hq, Hkv, D, bs, N, float(scale),
        int(max_context_len), _ptr(group_start), _ptr(group_prefix_len), n_groups,
        int(max_group_size), int(max_prefix_len), _ptr(workspace), ws_bytes, _flag(err_flag),
        _stream(stream, query.device)))


def pa_multi_token_workspace_size(S: int, T: int, Hq: int, Hkv: int, D: int, bs: int,
                                  kv_dtype: int, max_context_len: int, max_query_len: int) -> int:
    return int(load_library().pa_multi_token_workspace_size(
        S, T, Hq, Hkv, D, bs, kv_dtype, max_context_len, max_query_len))


def pa_multi_token_workspace_size_for_tokens(S: int, T: int, Hq: int, Hkv: int, D: int, bs: int,
                                             kv_dtype: int, max_context_len: int, max_query_len: int,
                                             total_context_tokens: int) -> int:
    return int(load_library().pa_multi_token_workspace_size_for_tokens(
        S, T, Hq, Hkv, D, bs, kv_dtype, max_context_len, max_query_len, int(total_context_tokens)))


def pa_multi_token_attention(out, query, k_cache, v_cache, block_tables, context_lens,
                             query_start, scale: float, max_context_len: int,
                             max_query_len: int, workspace=None, k_scale=None, v_scale=None,
                             err_flag=None, stream=None, total_context_tokens=None) -> None:
    """Several new tokens per sequence attend the paged cache, each up to its own
    position: query/out [T][Hq][D] bf16, sequence s owning rows
    query_start[s] .. query_start[s+1]-1.  workspace defaults to a fresh allocation."""
    _cuda(out, "out", torch.bfloat16, 3)
    _cuda(query, "query", torch.bfloat16, 3)
    kv_dtype = kv_dtype_of(k_cache)
    _cuda(k_cache, "k_cache", k_cache.dtype, 4)
    _cuda(v_cache, "v_cache", k_cache.dtype, 4)
    _cuda(block_tables, "block_tables", torch.int32, 2)
    _cuda(context_lens, "context_lens", torch.int32, 1)
    _cuda(query_start, "query_start", torch.int32, 1)
    if kv_dtype != PA_KV_BF16:
        if k_scale is None or v_scale is None:
            raise ValueError("an int8 or fp8 cache needs k_scale and v_scale")
        _cuda(k_scale, "k_scale", torch.float32, 3)
        _cuda(v_scale, "v_scale", torch.float32, 3)
    T, Hq, D = query.shape
    N, Hkv, bs, D2 = k_cache.shape
    S = context_lens.shape[0]
    M = block_tables.shape[1]
    if out.shape != query.shape or v_cache.shape != k_cache.shape or D2 != D \
            or block_tables.shape[0] != S or query_start.shape[0] != S + 1:
        raise ValueError("pa_multi_token_attention: shape mismatch")
    if workspace is None:
        if total_context_tokens is None:
            n = pa_multi_token_workspace_size(S, T, Hq, Hkv, D, bs, kv_dtype, max_context_len,
                                              max_query_len)
        else:
            n = pa_multi_token_workspace_size_for_tokens(S, T, Hq, Hkv, D, bs, kv_dtype,
                                                         max_context_len, max_query_len,
                                                         total_context_tokens)
        workspace = torch.empty(n, dtype=torch.uint8, device=query.device) if n else None
    ws_bytes = 0
    if workspace is not None:
        _cuda(workspace, "workspace", workspace.dtype)
        ws_bytes = workspace.numel() * workspace.element_size()
    lib = load_library()
    _check(lib.pa_multi_token_attention(
        _ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        kv_dtype, _ptr(block_tables), M, _ptr(context_lens), _ptr(query_start), S, T, Hq, Hkv, D, bs, N,
        float(scale), int(max_context_len), int(max_query_len), _ptr(workspace), ws_bytes,
        _flag(err_flag), _stream(stream, query.device)))


def decode_workspace(query, k_cache, max_context_len: int) -> torch.Tensor | None:
    """Allocate (with torch) the scratch pa_decode needs for these shapes, or None."""
    S, Hq, D = query.shape
    N, Hkv, bs, _ = k_cache.shape
    kv_dtype = kv_dtype_of(k_cache)
    n = pa_decode_workspace_size(S, Hq, Hkv, D, bs, kv_dtype, max_context_len)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=query.device)


# ------------------------------------------------------------------ block manager
PA_ERR_NO_SPACE = 5
BLOCK_MANAGER_EXPORTED = ["pa_bm_create", "pa_bm_destroy", "pa_bm_add_sequence", "pa_bm_append",
                          "pa_bm_fork", "pa_bm_free", "pa_bm_block_table", "pa_bm_get_stats"]


class BlockManagerStats(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int64) for name in (
        "num_blocks", "free_blocks", "cached_blocks", "used_blocks", "used_slots", "cow_copies",
        "prefix_lookup_blocks", "prefix_hit_blocks", "evictions")]

    def as_dict(self) -> dict:
        return {name: int(getattr(self, name)) for name, _ in self._fields_}


def _bm_lib() -> ctypes.CDLL:
    lib = load_library()
    if not getattr(lib, "_bm_ready", False):
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        lib.pa_bm_create.argtypes = [i32, i32, ctypes.POINTER(vp)]
        lib.pa_bm_create.restype = i32
        lib.pa_bm_destroy.argtypes = [vp]
        lib.pa_bm_destroy.restype = None
        lib.pa_bm_add_sequence.argtypes = [vp, i64, vp, i32, ctypes.POINTER(i32)]
        lib.pa_bm_add_sequence.restype = i32
        lib.pa_bm_append.argtypes = [vp, i64, vp, i32, vp, vp, i32, ctypes.POINTER(i32)]
        lib.pa_bm_append.restype = i32
        lib.pa_bm_fork.argtypes = [vp, i64, i64]
        lib.pa_bm_fork.restype = i32
        lib.pa_bm_free.argtypes = [vp, i64]
        lib.pa_bm_free.restype = i32
        lib.pa_bm_block_table.argtypes = [vp, i64, vp, i32, ctypes.POINTER(i32), ctypes.POINTER(i64)]
        lib.pa_bm_block_table.restype = i32
        lib.pa_bm_get_stats.argtypes = [vp, ctypes.POINTER(BlockManagerStats)]
        lib.pa_bm_get_stats.restype = i32
        lib._bm_ready = True
    return lib


class BlockManager:
    """Host block manager of include/pa_blocks.h (pool, tables, copy-on-write, prefix
    cache, LRU eviction).  Token ids and slots are plain Python ints / lists."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = _bm_lib()
        self._h = ctypes.c_void_p()
        _check(self._lib.pa_bm_create(num_blocks, block_size, ctypes.byref(self._h)))
        self.num_blocks, self.block_size = num_blocks, block_size

    def close(self):
        if self._h:
            self._lib.pa_bm_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass

    @staticmethod
    def _ids(tokens):
        if tokens is None:
            return None, 0
        arr = (ctypes.c_int32 * len(tokens))(*tokens)
        return arr, len(tokens)

    def add_sequence(self, seq_id: int, prompt=None) -> int:
        """Register a sequence; returns the number of prompt tokens found cached."""
        arr, n = self._ids(prompt)
        cached = ctypes.c_int(0)
        _check(self._lib.pa_bm_add_sequence(self._h, seq_id, arr, n, ctypes.byref(cached)))
        return cached.value

    def append(self, seq_id: int, n: int | None = None, tokens=None):
        """Append tokens (ids optional); returns (slots, cow_pairs)."""
        if tokens is not None:
            n = len(tokens)
        arr, _ = self._ids(tokens)
        slots = (ctypes.c_int64 * max(n, 1))()
        cow = (ctypes.c_int64 * 2)()
        n_cow = ctypes.c_int(0)
        _check(self._lib.pa_bm_append(self._h, seq_id, arr, n, slots, cow, 1, ctypes.byref(n_cow)))
        pairs = [(cow[0], cow[1])] if n_cow.value else []
        return list(slots)[:n], pairs

    def fork(self, parent: int, child: int) -> None:
        _check(self._lib.pa_bm_fork(self._h, parent, child))

    def free(self, seq_id: int) -> None:
        _check(self._lib.pa_bm_free(self._h, seq_id))

    def block_table(self, seq_id: int):
        n = ctypes.c_int(0)
        length = ctypes.c_int64(0)
        _check(self._lib.pa_bm_block_table(self._h, seq_id, None, 0, ctypes.byref(n), ctypes.byref(length)))
        table = (ctypes.c_int32 * max(n.value, 1))()
        _check(self._lib.pa_bm_block_table(self._h, seq_id, table, n.value, ctypes.byref(n),
                                           ctypes.byref(length)))
        return list(table)[: n.value], length.value

    def stats(self) -> dict:
        out = BlockManagerStats()
        _check(self._lib.pa_bm_get_stats(self._h, ctypes.byref(out)))
        return out.as_dict()
