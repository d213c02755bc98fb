"""CPU oracle for the paged KV-cache decode path -- TEST INFRASTRUCTURE ONLY.

The oracle is a plain C (fp64) restatement of what the GPU library computes; see
``pa_oracle.c`` for the definitions and the passages of the source pages they
follow.  Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may build, load or call it.  The product library never imports it,
and it imports nothing from the product.

Arrays are numpy, C-contiguous.  bf16 tensors travel as ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SOURCE = HERE / "pa_oracle.c"
LIBRARY = HERE / "liboracle.so"

KV_BF16 = 0
KV_INT8 = 1
KV_FP8 = 2

_BASE_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(source: Path | str = SOURCE, output: Path | str = LIBRARY, openmp: bool = True) -> Path:
    """Compile the oracle with gcc into a shared library and return its path.

    OpenMP is used when the compiler supports it; the result is identical either
    way (each (sequence, kv head) pair is computed by one thread in a fixed order).
    """
    source, output = Path(source), Path(output)
    cc = os.environ.get("CC", "gcc")
    if shutil.which(cc) is None:
        raise RuntimeError(f"oracle build needs a C compiler ({cc!r} not found)")
    tmp = output.with_suffix(f".{os.getpid()}.tmp.so")
    attempts = [_BASE_FLAGS + ["-fopenmp"]] if openmp else []
    attempts.append(list(_BASE_FLAGS))
    last = None
    for flags in attempts:
        cmd = [cc, *flags, str(source), "-o", str(tmp), "-lm"]
        proc = subprocess.run(cmd, capture_output=True, text=True)
        if proc.returncode == 0:
            os.replace(tmp, output)
            return output
        last = proc.stderr
    raise RuntimeError(f"oracle build failed:\n{last}")


def _ptr(a: np.ndarray | None) -> ctypes.c_void_p:
    if a is None:
        return ctypes.c_void_p(0)
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("oracle arrays must be C-contiguous")
    return ctypes.c_void_p(a.ctypes.data)


def _need(a: np.ndarray, dtype, name: str) -> None:
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"{name}: expected {np.dtype(dtype)}, got {a.dtype}")
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError(f"{name}: must be C-contiguous")


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: Path | str = LIBRARY):
        self.path = Path(path)
        lib = ctypes.CDLL(str(self.path))
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_version.restype = i32
        lib.oracle_num_threads.restype = i32
        lib.oracle_set_num_threads.argtypes = [i32]
        lib.oracle_set_num_threads.restype = None
        lib.oracle_slot.argtypes = [vp, i64, i32]
        lib.oracle_slot.restype = i64
        lib.oracle_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i64]
        lib.oracle_reshape_and_cache.restype = i64
        lib.oracle_quantize_kv.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i64]
        lib.oracle_quantize_kv.restype = i64
        lib.oracle_quantize_pool.argtypes = [vp, vp, vp, i64, i32]
        lib.oracle_quantize_pool.restype = None
        lib.oracle_quantize_kv_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i64]
        lib.oracle_quantize_kv_fp8.restype = i64
        lib.oracle_quantize_pool_fp8.argtypes = [vp, vp, vp, i64, i32]
        lib.oracle_quantize_pool_fp8.restype = None
        lib.oracle_fp8_encode.argtypes = [ctypes.c_float]
        lib.oracle_fp8_encode.restype = ctypes.c_uint8
        lib.oracle_fp8_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_fp8_decode.restype = dbl
        lib.oracle_copy_blocks.argtypes = [vp, vp, vp, vp, vp, i32, i64, i32]
        lib.oracle_copy_blocks.restype = i32
        lib.oracle_paged_attention.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, vp,
                                               i32, i32, i32, i32, i32, dbl]
        lib.oracle_paged_attention.restype = i32
        lib.oracle_attention_weights.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, vp,
                                                 i32, i32, i32, i32, i32, dbl, i32, i32]
        lib.oracle_attention_weights.restype = i32
        lib.oracle_paged_prefill.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, vp, vp, i32,
                                             i32, i32, i32, i32, i32, dbl]
        lib.oracle_paged_prefill.restype = i32
        self.lib = lib

    @property
    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        """Threads of later calls (timing only: the results do not depend on it)."""
        self.lib.oracle_set_num_threads(int(n))

    # ---------------------------------------------------------------- indexing
    def slot(self, table: np.ndarray, pos: int, bs: int) -> int:
        table = np.ascontiguousarray(table, dtype=np.int32)
        return int(self.lib.oracle_slot(_ptr(table), int(pos), int(bs)))

    # ------------------------------------------------------------------ append
    def reshape_and_cache(self, key, value, k_cache, v_cache, slot_mapping, bs: int) -> int:
        """In-place append of bf16 rows ``key``/``value`` [T][Hkv][D] (uint16 bits)."""
        for a, n in ((key, "key"), (value, "value"), (k_cache, "k_cache"), (v_cache, "v_cache")):
            _need(a, np.uint16, n)
        _need(slot_mapping, np.int64, "slot_mapping")
        T, Hkv, D = key.shape
        N = k_cache.shape[0]
        return int(self.lib.oracle_reshape_and_cache(
            _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
            T, Hkv, D, int(bs), N))

    def quantize_kv(self, key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, bs: int) -> int:
        """In-place int8 quantise-and-append of bf16 rows [T][Hkv][D]."""
        _need(key, np.uint16, "key")
        _need(value, np.uint16, "value")
        _need(k_cache, np.int8, "k_cache")
        _need(v_cache, np.int8, "v_cache")
        _need(k_scale, np.float32, "k_scale")
        _need(v_scale, np.float32, "v_scale")
        _need(slot_mapping, np.int64, "slot_mapping")
        T, Hkv, D = key.shape
        N = k_cache.shape[0]
        return int(self.lib.oracle_quantize_kv(
            _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
            _ptr(slot_mapping), T, Hkv, D, int(bs), N))

    def quantize_pool(self, src: np.ndarray, fp8: bool = False):
        """Quantise every D-row of a bf16 array (uint16 bits, last axis D).

        Returns (codes of the same shape -- int8, or uint8 e4m3 with fp8 --, scales
        float32 of shape[:-1])."""
        _need(src, np.uint16, "src")
        D = src.shape[-1]
        rows = src.size // D
        codes = np.empty(src.shape, dtype=np.uint8 if fp8 else np.int8)
        scales = np.empty(src.shape[:-1], dtype=np.float32)
        fn = self.lib.oracle_quantize_pool_fp8 if fp8 else self.lib.oracle_quantize_pool
        fn(_ptr(src), _ptr(codes), _ptr(scales), rows, D)
        return codes, scales

    def quantize_kv_fp8(self, key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, bs: int) -> int:
        """In-place fp8 (e4m3) quantise-and-append of bf16 rows [T][Hkv][D]."""
        _need(key, np.uint16, "key")
        _need(value, np.uint16, "value")
        _need(k_cache, np.uint8, "k_cache")
        _need(v_cache, np.uint8, "v_cache")
        _need(k_scale, np.float32, "k_scale")
        _need(v_scale, np.float32, "v_scale")
        _need(slot_mapping, np.int64, "slot_mapping")
        T, Hkv, D = key.shape
        N = k_cache.shape[0]
        return int(self.lib.oracle_quantize_kv_fp8(
            _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
            _ptr(slot_mapping), T, Hkv, D, int(bs), N))

    def fp8_encode(self, x: float) -> int:
        return int(self.lib.oracle_fp8_encode(float(x)))

    def fp8_decode(self, code: int) -> float:
        return float(self.lib.oracle_fp8_decode(int(code)))

    # -------------------------------------------------------------------- COW
    def copy_blocks(self, k_cache, v_cache, block_mapping, k_scale=None, v_scale=None) -> None:
        """In-place copy of whole blocks (src, dst) pairs; caches are [N][...] arrays."""
        _need(block_mapping, np.int64, "block_mapping")
        N = k_cache.shape[0]
        block_bytes = k_cache.nbytes // N
        scale_elems = 0 if k_scale is None else k_scale.size // k_scale.shape[0]
        rc = self.lib.oracle_copy_blocks(
            _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_mapping),
            block_mapping.shape[0], block_bytes, scale_elems)
        if rc != 0:
            raise RuntimeError(f"oracle_copy_blocks failed: {rc}")

    # --------------------------------------------------------------- attention
    def paged_attention(self, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                        k_scale=None, v_scale=None) -> np.ndarray:
        """fp64 output [S][Hq][D] of paged decode attention."""
        _need(q, np.uint16, "q")
        _need(block_tables, np.int32, "block_tables")
        _need(context_lens, np.int32, "context_lens")
        kv_dtype = {np.dtype(np.int8): KV_INT8, np.dtype(np.uint8): KV_FP8}.get(k_cache.dtype, KV_BF16)
        if kv_dtype == KV_BF16:
            _need(k_cache, np.uint16, "k_cache")
            _need(v_cache, np.uint16, "v_cache")
        else:
            _need(v_cache, k_cache.dtype, "v_cache")
            _need(k_scale, np.float32, "k_scale")
            _need(v_scale, np.float32, "v_scale")
        S, Hq, D = q.shape
        _, Hkv, bs, D2 = k_cache.shape
        if D2 != D:
            raise ValueError("head_dim mismatch between q and cache")
        M = block_tables.shape[1] if block_tables.ndim == 2 else 0
        out = np.zeros((S, Hq, D), dtype=np.float64)
        rc = self.lib.oracle_paged_attention(
            _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
            kv_dtype, _ptr(block_tables), M, _ptr(context_lens), S, Hq, Hkv, D, bs, float(scale))
        if rc != 0:
            raise RuntimeError(f"oracle_paged_attention failed: {rc}")
        return out

    def paged_prefill(self, q, k_cache, v_cache, block_tables, context_lens, query_start,
                      scale: float, k_scale=None, v_scale=None) -> np.ndarray:
        """fp64 output [T][Hq][D] of multi-token paged attention: the rows
        query_start[s] .. query_start[s+1]-1 are sequence s's newest tokens, each
        attending the tokens up to its own position."""
        _need(q, np.uint16, "q")
        _need(block_tables, np.int32, "block_tables")
        _need(context_lens, np.int32, "context_lens")
        _need(query_start, np.int32, "query_start")
        kv_dtype = {np.dtype(np.int8): KV_INT8, np.dtype(np.uint8): KV_FP8}.get(k_cache.dtype, KV_BF16)
        if kv_dtype == KV_BF16:
            _need(k_cache, np.uint16, "k_cache")
            _need(v_cache, np.uint16, "v_cache")
        else:
            _need(v_cache, k_cache.dtype, "v_cache")
            _need(k_scale, np.float32, "k_scale")
            _need(v_scale, np.float32, "v_scale")
        T, Hq, D = q.shape
        S = context_lens.shape[0]
        if query_start.shape[0] != S + 1:
            raise ValueError("query_start must hold S + 1 offsets")
        _, Hkv, bs, D2 = k_cache.shape
        if D2 != D:
            raise ValueError("head_dim mismatch between q and cache")
        M = block_tables.shape[1] if block_tables.ndim == 2 else 0
        out = np.zeros((T, Hq, D), dtype=np.float64)
        rc = self.lib.oracle_paged_prefill(
            _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
            kv_dtype, _ptr(block_tables), M, _ptr(context_lens), _ptr(query_start), S, T, Hq,
            Hkv, D, bs, float(scale))
        if rc != 0:
            raise RuntimeError(f"oracle_paged_prefill failed: {rc}")
        return out

    def attention_weights(self, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                          s: int, h: int, k_scale=None, v_scale=None) -> np.ndarray:
        kv_dtype = {np.dtype(np.int8): KV_INT8, np.dtype(np.uint8): KV_FP8}.get(k_cache.dtype, KV_BF16)
        S, Hq, D = q.shape
        _, Hkv, bs, _ = k_cache.shape
        M = block_tables.shape[1]
        w = np.zeros(max(int(context_lens[s]), 1), dtype=np.float64)
        rc = self.lib.oracle_attention_weights(
            _ptr(w), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
            kv_dtype, _ptr(block_tables), M, _ptr(context_lens), S, Hq, Hkv, D, bs,
            float(scale), int(s), int(h))
        if rc != 0:
            raise RuntimeError(f"oracle_attention_weights failed: {rc}")
        return w[: int(context_lens[s])]


_DEFAULT: Oracle | None = None


def load(path: Path | str | None = None) -> Oracle:
    """Load the oracle library, building it first when it is missing or stale."""
    global _DEFAULT
    if path is not None:
        return Oracle(path)
    if _DEFAULT is None:
        if not LIBRARY.exists() or LIBRARY.stat().st_mtime < SOURCE.stat().st_mtime:
            build()
        _DEFAULT = Oracle(LIBRARY)
    return _DEFAULT
