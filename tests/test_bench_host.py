"""Host-side pieces of bench.py and of the oracle's timing knobs, on the CPU: the
multi-token kernel attribution follows the library's dispatch rule, the single-core
oracle timing restores the thread count, and the oracle's result does not depend on
how many threads compute it."""
import numpy as np
import pytest
import torch

import workloads


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def _multi(kv_dtype, D, Hq, Hkv, qlen):
    return workloads.build_multi_case(f"src-{kv_dtype}-{D}-{Hq}-{Hkv}-{qlen}", S=1, Hq=Hq, Hkv=Hkv, D=D,
                                      bs=16, context_lens=[200], query_lens=[qlen], seed=3,
                                      kv_dtype=kv_dtype, poison=False)


@pytest.mark.parametrize("kv_dtype,D,Hq,Hkv,qlen,src", [
    ("bf16", 128, 64, 8, 2, "pa_multi_tc.cu"),   # 16 columns per kv head
    ("bf16", 128, 16, 8, 4, "pa_multi.cu"),      # 8 columns
    ("bf16", 64, 64, 8, 16, "pa_multi.cu"),      # head_dim 64
    ("fp8", 128, 64, 8, 4, "pa_decode.cu"),      # 32 columns (8-bit tcgen05 needs 64): rows mode
    ("fp8", 128, 64, 8, 8, "pa_multi_tc.cu"),    # 64 columns
    ("int8", 128, 32, 8, 16, "pa_multi_tc.cu"),
    ("int8", 64, 8, 2, 8, "pa_decode.cu"),       # head_dim 64, 8 new tokens: rows mode
    ("int8", 64, 8, 2, 9, "pa_multi.cu"),        # 9 new tokens: the mma.sync kernel
])
def test_multi_kernel_source_follows_dispatch(kv_dtype, D, Hq, Hkv, qlen, src):
    import bench

    assert bench.multi_kernel_source(_multi(kv_dtype, D, Hq, Hkv, qlen)) == src


def test_eight_bit_tensor_core_calls_carry_the_pool():
    """The library side of the same rule: an 8-bit call that bench.py attributes to the
    tcgen05 kernel needs the dequantised pool in its workspace, one it attributes to the
    mma.sync kernel does not (same shapes with a bf16 cache as the reference)."""
    import paged_kv_cache_197_gb300 as pa

    import bench

    for qlen in (4, 8):
        case = _multi("fp8", 128, 64, 8, qlen)
        args = (1, qlen, 64, 8, 128, 16)
        grow = (pa.pa_multi_token_workspace_size(*args, pa.PA_KV_FP8, 200, qlen) -
                pa.pa_multi_token_workspace_size(*args, pa.PA_KV_BF16, 200, qlen))
        assert (grow > 0) == (bench.multi_kernel_source(case) == "pa_multi_tc.cu")


def test_single_core_timing_restores_threads(oracle):
    import bench

    case = workloads.tiny(device="cpu", poison=False)
    inputs = bench.oracle_sample_inputs(case)
    before = oracle.num_threads
    one = bench.time_oracle(case, inputs, 0.05, threads=1)
    assert one["cores"] == 1 and one["value"] > 0
    assert oracle.num_threads == before


def test_oracle_result_independent_of_threads(oracle):
    """Each (sequence, kv head) pair is computed by one thread in a fixed order, so the
    thread count changes no bit."""
    case = workloads.build_case("threads", S=6, Hq=8, Hkv=2, D=64, bs=16,
                                context_lens=[1, 17, 90, 300, 5, 1000], seed=9, poison=False)
    q, kc, vc = _bits(case.q), _bits(case.k_pool), _bits(case.v_pool)
    tables, lens = case.block_tables.numpy(), case.context_lens.numpy()
    before = oracle.num_threads
    try:
        oracle.set_num_threads(1)
        one = oracle.paged_attention(q, kc, vc, tables, lens, case.scale)
        oracle.set_num_threads(max(2, before))
        many = oracle.paged_attention(q, kc, vc, tables, lens, case.scale)
    finally:
        oracle.set_num_threads(before)
    assert np.array_equal(one, many)
