"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (an application that owns every allocation, a fixed memory budget,
capture code that may not allocate) cannot hand pa_decode a workspace, so this
entry point uses a fixed scratch array built into the library.  Its output must
match pa_decode's, within the tolerance the parity tests use, on two calls in a
row (the second call reuses the array the first one left behind).  This file is
collected last on purpose.
"""
import numpy as np
import pytest
import torch

import helpers
import workloads

pytestmark = pytest.mark.gpu


def test_noalloc_matches_pa_decode():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_kv_cache_197_gb300 as pa

    dev = torch.device("cuda:0")
    cases = [
        workloads.build_case("noalloc-bf16", S=8, Hq=16, Hkv=2, D=128, bs=16,
                             context_lens=[1, 40, 511, 513, 1200, 2047, 3000, 64], seed=41,
                             poison=False),
        workloads.build_case("noalloc-gqa", S=5, Hq=32, Hkv=4, D=128, bs=16,
                             context_lens=[2600, 700, 1900, 33, 1025], seed=42, poison=False),
    ]
    for call in range(2):
        case = cases[call].to(dev)
        k, v = case.k_pool, case.v_pool
        max_ctx = int(case.context_lens.max())
        need = pa.pa_decode_workspace_size(case.S, case.Hq, case.Hkv, case.D, case.bs,
                                           pa.PA_KV_BF16, max_ctx)
        assert 0 < need <= pa.PA_NOALLOC_SCRATCH_BYTES  # the scratch is really used
        ref = torch.empty_like(case.q)
        ws = pa.decode_workspace(case.q, k, max_ctx)
        pa.pa_decode(ref, case.q, k, v, case.block_tables, case.context_lens, case.scale, max_ctx,
                     workspace=ws)
        got = torch.full_like(case.q, float("nan"))
        flag = torch.zeros(1, dtype=torch.int32, device=dev)
        pa.pa_decode_noalloc(got, case.q, k, v, case.block_tables, case.context_lens, case.scale,
                             max_ctx, err_flag=flag)
        torch.cuda.synchronize(dev)
        assert flag.item() == 0
        err = (got.double() - ref.double()).abs().cpu().numpy()
        assert np.isfinite(err).all()
        assert err.max() <= helpers.BF16_MAX_ABS and err.mean() <= helpers.BF16_MEAN_ABS


@pytest.mark.parametrize("kv_dtype", ["int8", "fp8"])
def test_noalloc_matches_pa_decode_8bit(kv_dtype):
    """The same comparison with an int8 and an fp8 cache (the scratch size depends on the
    cache type through the partition plan), two calls in a row, under the 8-bit bar."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_kv_cache_197_gb300 as pa

    dev = torch.device("cuda:0")
    fp8 = kv_dtype == "fp8"
    quant = pa.pa_quantize_kv_fp8 if fp8 else pa.pa_quantize_kv
    for call, lens in enumerate(([1, 40, 700, 1300, 2047, 3000], [2600, 33, 1900, 1025])):
        case = workloads.build_case(f"noalloc-{kv_dtype}-{call}", S=len(lens), Hq=32, Hkv=8, D=128,
                                    bs=32, context_lens=lens, seed=43 + call, poison=False,
                                    kv_dtype=kv_dtype).to(dev)
        N, Hkv, bs, D = case.k_pool.shape
        k = torch.empty((N, Hkv, bs, D), dtype=torch.uint8 if fp8 else torch.int8, device=dev)
        v = torch.empty_like(k)
        ks = torch.empty((N, Hkv, bs), dtype=torch.float32, device=dev)
        vs = torch.empty_like(ks)
        quant(helpers.int8_pool_rows(case.k_pool), helpers.int8_pool_rows(case.v_pool), k, v, ks, vs,
              torch.arange(N * bs, dtype=torch.int64, device=dev))
        max_ctx = int(case.context_lens.max())
        need = pa.pa_decode_workspace_size(case.S, case.Hq, case.Hkv, case.D, case.bs,
                                           pa.kv_dtype_of(k), max_ctx)
        assert 0 < need <= pa.PA_NOALLOC_SCRATCH_BYTES
        ref = torch.empty_like(case.q)
        pa.pa_decode(ref, case.q, k, v, case.block_tables, case.context_lens, case.scale, max_ctx,
                     workspace=pa.decode_workspace(case.q, k, max_ctx), k_scale=ks, v_scale=vs)
        got = torch.full_like(case.q, float("nan"))
        flag = torch.zeros(1, dtype=torch.int32, device=dev)
        pa.pa_decode_noalloc(got, case.q, k, v, case.block_tables, case.context_lens, case.scale,
                             max_ctx, k_scale=ks, v_scale=vs, err_flag=flag)
        torch.cuda.synchronize(dev)
        assert flag.item() == 0
        err = (got.double() - ref.double()).abs().cpu().numpy()
        assert np.isfinite(err).all()
        assert err.max() <= helpers.INT8_MAX_ABS and err.mean() <= helpers.INT8_MEAN_ABS


def test_noalloc_rejects_oversized_scratch():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_kv_cache_197_gb300 as pa

    dev = torch.device("cuda:0")
    S, Hq, Hkv, D, bs, max_ctx = 256, 32, 8, 128, 32, 32768
    assert pa.pa_decode_workspace_size(S, Hq, Hkv, D, bs, pa.PA_KV_BF16, max_ctx) > pa.PA_NOALLOC_SCRATCH_BYTES
    q = torch.zeros((S, Hq, D), dtype=torch.bfloat16, device=dev)
    cache = torch.zeros((4, Hkv, bs, D), dtype=torch.bfloat16, device=dev)
    tables = torch.zeros((S, max_ctx // bs), dtype=torch.int32, device=dev)
    lens = torch.zeros(S, dtype=torch.int32, device=dev)
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.pa_decode_noalloc(torch.empty_like(q), q, cache, cache, tables, lens, 0.1, max_ctx)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
