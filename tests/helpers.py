"""Shared test steps: run one decode step through the GPU library, and the same step
through the CPU oracle, on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import workloads

BF16_MAX_ABS, BF16_MEAN_ABS = 2e-2, 2e-3   # bf16 cache: output vs fp64 oracle
INT8_MAX_ABS, INT8_MEAN_ABS = 5e-2, 2e-3   # int8 / fp8 cache: vs the oracle on the same codes


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def int8_pool_rows(pool: torch.Tensor) -> torch.Tensor:
    """[N][Hkv][bs][D] -> [N*bs][Hkv][D] (rows in slot order) for a quantise-append of a
    whole pool."""
    N, Hkv, bs, D = pool.shape
    return pool.permute(0, 2, 1, 3).reshape(N * bs, Hkv, D).contiguous()


def gpu_step(case: workloads.PagedCase, device, max_context_len=None, poison_int8=True,
             groups=None):
    """COW copy, append (or quantise-append), decode on the GPU.

    ``groups`` = (group_start, group_prefix_len, max_group_size, max_prefix_len) decodes
    through pa_decode_shared_prefix instead of pa_decode.
    Returns dict(out, k_cache, v_cache, k_scale, v_scale, flag) on the device."""
    import paged_kv_cache_197_gb300 as pa

    c = case.to(device)
    flag = torch.zeros(1, dtype=torch.int32, device=device)
    k_scale = v_scale = None
    if case.kv_dtype == "bf16":
        k_cache, v_cache = c.k_pool.clone(), c.v_pool.clone()
    else:
        N, Hkv, bs, D = case.k_pool.shape
        fp8 = case.kv_dtype == "fp8"
        quant = pa.pa_quantize_kv_fp8 if fp8 else pa.pa_quantize_kv
        k_cache = torch.empty((N, Hkv, bs, D), dtype=torch.uint8 if fp8 else torch.int8, device=device)
        v_cache = torch.empty_like(k_cache)
        k_scale = torch.empty((N, Hkv, bs), dtype=torch.float32, device=device)
        v_scale = torch.empty_like(k_scale)
        slots = torch.arange(N * bs, dtype=torch.int64, device=device)
        quant(int8_pool_rows(c.k_pool), int8_pool_rows(c.v_pool), k_cache, v_cache,
              k_scale, v_scale, slots, err_flag=flag)
        if poison_int8:
            bad = ~workloads.valid_slot_mask(case.meta["content_tables"], case.context_lens - 1,
                                             case.bs, case.N).to(device)
            k_scale.permute(0, 2, 1)[bad] = float("nan")
            v_scale.permute(0, 2, 1)[bad] = float("nan")
    if case.cow_pairs.shape[0]:
        pa.pa_copy_blocks(k_cache, v_cache, case.cow_pairs, k_scale=k_scale, v_scale=v_scale)
    if case.kv_dtype == "bf16":
        pa.pa_reshape_and_cache(c.new_key, c.new_value, k_cache, v_cache, c.slot_mapping,
                                err_flag=flag)
    else:
        quant = pa.pa_quantize_kv_fp8 if case.kv_dtype == "fp8" else pa.pa_quantize_kv
        quant(c.new_key, c.new_value, k_cache, v_cache, k_scale, v_scale, c.slot_mapping,
              err_flag=flag)
    if max_context_len is None:
        max_context_len = int(case.context_lens.max()) if case.S else 0
    out = torch.full_like(c.q, float("nan"))
    if groups is not None:
        starts, plens, max_group, max_prefix = groups
        gs = torch.as_tensor(starts, dtype=torch.int32).to(device)
        gp = torch.as_tensor(plens, dtype=torch.int32).to(device)
        pa.pa_decode_shared_prefix(out, c.q, k_cache, v_cache, c.block_tables, c.context_lens,
                                   case.scale, max_context_len, gs, gp, max_group, max_prefix,
                                   k_scale=k_scale, v_scale=v_scale, err_flag=flag)
    else:
        ws = pa.decode_workspace(c.q, k_cache, max_context_len)
        pa.pa_decode(out, c.q, k_cache, v_cache, c.block_tables, c.context_lens, case.scale,
                     max_context_len, workspace=ws, k_scale=k_scale, v_scale=v_scale,
                     err_flag=flag)
    torch.cuda.synchronize(device)
    return dict(out=out, k_cache=k_cache, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale,
                flag=int(flag.item()))


def oracle_caches(case: workloads.PagedCase, orc, poison_int8=True):
    """The oracle's own caches after COW copy and append (bf16 bits, or int8 codes+scales)."""
    ks = vs = None
    if case.kv_dtype == "bf16":
        kc, vc = bits(case.k_pool), bits(case.v_pool)
    else:
        fp8 = case.kv_dtype == "fp8"
        kc, ks = orc.quantize_pool(bits(case.k_pool), fp8=fp8)
        vc, vs = orc.quantize_pool(bits(case.v_pool), fp8=fp8)
        if poison_int8:
            bad = ~workloads.valid_slot_mask(case.meta["content_tables"], case.context_lens - 1,
                                             case.bs, case.N).numpy()
            ks.transpose(0, 2, 1)[bad] = np.nan
            vs.transpose(0, 2, 1)[bad] = np.nan
    if case.cow_pairs.shape[0]:
        orc.copy_blocks(kc, vc, case.cow_pairs.cpu().numpy(), k_scale=ks, v_scale=vs)
    slots = case.slot_mapping.cpu().numpy()
    if case.kv_dtype == "bf16":
        bad = orc.reshape_and_cache(bits(case.new_key), bits(case.new_value), kc, vc, slots, case.bs)
    elif case.kv_dtype == "fp8":
        bad = orc.quantize_kv_fp8(bits(case.new_key), bits(case.new_value), kc, vc, ks, vs, slots, case.bs)
    else:
        bad = orc.quantize_kv(bits(case.new_key), bits(case.new_value), kc, vc, ks, vs, slots, case.bs)
    assert bad == 0
    return kc, vc, ks, vs


def oracle_out(case, orc, caches, seqs=None) -> np.ndarray:
    kc, vc, ks, vs = caches
    q = bits(case.q)
    tables = case.block_tables.cpu().numpy()
    lens = case.context_lens.cpu().numpy()
    if seqs is not None:
        q = np.ascontiguousarray(q[seqs])
        tables = np.ascontiguousarray(tables[seqs])
        lens = np.ascontiguousarray(lens[seqs])
    return orc.paged_attention(q, kc, vc, tables, lens, case.scale, k_scale=ks, v_scale=vs)


def compare(got: torch.Tensor, ref: np.ndarray, kv_dtype: str):
    g = got.float().cpu().double().numpy()
    assert np.all(np.isfinite(g)), "non-finite output"
    err = np.abs(g - ref)
    max_abs, mean_abs = (BF16_MAX_ABS, BF16_MEAN_ABS) if kv_dtype == "bf16" else (INT8_MAX_ABS, INT8_MEAN_ABS)
    assert err.max() <= max_abs, f"max abs error {err.max():.3e} > {max_abs}"
    assert err.mean() <= mean_abs, f"mean abs error {err.mean():.3e} > {mean_abs}"
    return float(err.max()), float(err.mean())


def compare_row_scaled(got: torch.Tensor, ref: np.ndarray, kv_dtype: str):
    """The stated tolerances applied to the error in units of each output row's own
    magnitude, max(1, max_d |ref[row][d]|).  Rows that attend values of magnitude A > 1
    carry every error source (bf16 rounding of the output, fp16 staging, fp32
    accumulation) scaled by A, so the unit-magnitude bars hold for err / A; rows of
    magnitude below 1 keep the absolute bars."""
    g = got.float().cpu().double().numpy()
    assert np.all(np.isfinite(g)), "non-finite output"
    norm = np.maximum(1.0, np.abs(ref).max(axis=-1, keepdims=True))
    err = np.abs(g - ref) / norm
    max_abs, mean_abs = (BF16_MAX_ABS, BF16_MEAN_ABS) if kv_dtype == "bf16" else (INT8_MAX_ABS, INT8_MEAN_ABS)
    assert err.max() <= max_abs, f"max row-scaled error {err.max():.3e} > {max_abs}"
    assert err.mean() <= mean_abs, f"mean row-scaled error {err.mean():.3e} > {mean_abs}"
    return float(err.max()), float(err.mean())


def gpu_multi_step(case: workloads.PagedCase, device, max_query_len=None, max_context_len=None,
                   workspace_bytes=None):
    """Append every new token, then multi-token attention, on the GPU.  Output rows of
    no sequence stay NaN.  Returns dict(out, k_cache, v_cache, flag)."""
    import paged_kv_cache_197_gb300 as pa

    c = case.to(device)
    flag = torch.zeros(1, dtype=torch.int32, device=device)
    k_scale = v_scale = None
    if case.kv_dtype == "bf16":
        k_cache, v_cache = c.k_pool.clone(), c.v_pool.clone()
        pa.pa_reshape_and_cache(c.new_key, c.new_value, k_cache, v_cache, c.slot_mapping,
                                err_flag=flag)
    else:  # quantise the pool, poison the scales of empty slots as the oracle does, append
        N, Hkv, bs, D = case.k_pool.shape
        fp8 = case.kv_dtype == "fp8"
        quant = pa.pa_quantize_kv_fp8 if fp8 else pa.pa_quantize_kv
        k_cache = torch.empty((N, Hkv, bs, D), dtype=torch.uint8 if fp8 else torch.int8, device=device)
        v_cache = torch.empty_like(k_cache)
        k_scale = torch.empty((N, Hkv, bs), dtype=torch.float32, device=device)
        v_scale = torch.empty_like(k_scale)
        quant(int8_pool_rows(c.k_pool), int8_pool_rows(c.v_pool), k_cache, v_cache, k_scale, v_scale,
              torch.arange(N * bs, dtype=torch.int64, device=device), err_flag=flag)
        bad = ~workloads.valid_slot_mask(case.meta["content_tables"], case.context_lens - 1,
                                         case.bs, case.N).to(device)
        k_scale.permute(0, 2, 1)[bad] = float("nan")
        v_scale.permute(0, 2, 1)[bad] = float("nan")
        quant(c.new_key, c.new_value, k_cache, v_cache, k_scale, v_scale, c.slot_mapping, err_flag=flag)
    if max_context_len is None:
        max_context_len = int(case.context_lens.max())
    if max_query_len is None:
        max_query_len = max(1, max(case.meta["query_lens"]))
    out = torch.full_like(c.q, float("nan"))
    ws = None
    if workspace_bytes is not None:  # a given size (else the binding sizes it)
        ws = torch.empty(workspace_bytes, dtype=torch.uint8, device=device)
    pa.pa_multi_token_attention(out, c.q, k_cache, v_cache, c.block_tables, c.context_lens,
                                c.query_start, case.scale, max_context_len, max_query_len,
                                workspace=ws, k_scale=k_scale, v_scale=v_scale, err_flag=flag)
    torch.cuda.synchronize(device)
    return dict(out=out, k_cache=k_cache, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale,
                flag=int(flag.item()))


def oracle_multi_out(case, orc, caches) -> np.ndarray:
    kc, vc, ks, vs = caches
    return orc.paged_prefill(bits(case.q), kc, vc, case.block_tables.cpu().numpy(),
                             case.context_lens.cpu().numpy(), case.query_start.cpu().numpy(),
                             case.scale, k_scale=ks, v_scale=vs)


def covered_rows(case) -> np.ndarray:
    qs = case.query_start.cpu().numpy()
    return np.concatenate([np.arange(qs[s], qs[s + 1]) for s in range(len(qs) - 1)] + [np.zeros(0, int)])
