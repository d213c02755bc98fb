"""GPU parity on caches whose per-token scales span several decades.

The pages' 8-bit caches carry a scale recomputed for every token (ia-vox-magazine,
"Quantization du KV cache"), so one sequence may hold tokens of very different
magnitude.  N(0, 1) workloads keep every scale within a factor of about two; here each
cached row (one token of one kv head) is rescaled to its own magnitude, drawn
log-uniformly over several decades, after a few outlier channels per kv head were
amplified.  The GPU output is compared with the oracle on the same codes and scales,
with the stated bars applied per output row in units of that row's magnitude
(helpers.compare_row_scaled).

  - pa_decode (exact 8-bit path, no fp16 range limit): magnitudes 1e-3 .. 1e3;
  - narrow pa_multi_token_attention calls (exact codes, scales in fp32): 1e-3 .. 1e3;
  - prefill-shaped multi-token calls attend bf16(code x scale): 1e-3 .. 1e3, against
    the oracle on those values;
  - pa_decode_shared_prefix stages a shared prefix as fp16 code x scale, documented for
    scales inside fp16's normal range: magnitudes 0.03 .. 3000 (every scale between
    2^-14 and 65504 / 448);
  - beyond fp16's range the shared-prefix path raises PA_FLAG_FP16_RANGE, while
    pa_decode and the multi-token path still match the oracle.
"""
import numpy as np
import pytest
import torch

import helpers
import paged_kv_cache_197_gb300 as pa_mod
import workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
DECODE_RANGE = (1e-3, 1e3)
STAGED_RANGE = (0.03, 3000.0)


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    pa_mod.load_library()


def _decode(case, orc, groups=None, expect_flag=0):
    got = helpers.gpu_step(case, DEV, groups=groups)
    caches = helpers.oracle_caches(case, orc)
    if case.kv_dtype != "bf16":  # the wide scales themselves, bit for bit
        assert np.array_equal(got["k_scale"].cpu().numpy().view(np.uint32), caches[2].view(np.uint32))
        assert np.array_equal(got["v_scale"].cpu().numpy().view(np.uint32), caches[3].view(np.uint32))
    assert got["flag"] == expect_flag, got["flag"]
    if expect_flag:
        return None
    ref = helpers.oracle_out(case, orc, caches)
    return helpers.compare_row_scaled(got["out"], ref, case.kv_dtype)


def _spread(case) -> float:
    """Decades spanned by the cached rows' magnitudes (checks the inputs are wide)."""
    a = case.k_pool.float().abs().nan_to_num(0.0).amax(dim=-1)
    a = a[a > 0]
    return float(torch.log10(a.max() / a.min()))


@pytest.mark.parametrize("kv_dtype", ["int8", "fp8", "bf16"])
@pytest.mark.parametrize("D,bs,Hq,Hkv", [(128, 16, 32, 4), (128, 32, 8, 8), (64, 16, 16, 2),
                                          (64, 32, 40, 4)])
def test_decode(oracle, kv_dtype, D, bs, Hq, Hkv):
    lens = [1, 17, 300, 1300, 2100, 4500]
    case = workloads.build_case(f"wide-{kv_dtype}-{D}-{bs}-{Hq}", S=len(lens), Hq=Hq, Hkv=Hkv, D=D,
                                bs=bs, context_lens=lens, seed=D + bs + Hq + 500,
                                kv_dtype=kv_dtype)
    workloads.widen_scales(case, *DECODE_RANGE, seed=D + Hq)
    assert _spread(case) > 5.5
    _decode(case, oracle)


@pytest.mark.parametrize("kv_dtype", ["int8", "fp8"])
@pytest.mark.parametrize("D,bs,Hq,Hkv", [(128, 16, 32, 8), (64, 32, 16, 2)])
def test_shared_prefix(oracle, kv_dtype, D, bs, Hq, Hkv):
    prefix = 21 * 32
    own = [1, 16, 17, 100, 333, 700]
    lens = [prefix + o for o in own]
    case = workloads.build_case(f"wide-pfx-{kv_dtype}-{D}", S=len(lens), Hq=Hq, Hkv=Hkv, D=D, bs=bs,
                                context_lens=lens, seed=71 + D, prefix_tokens=prefix, cow=True,
                                kv_dtype=kv_dtype)
    workloads.widen_scales(case, *STAGED_RANGE, seed=72 + D)
    assert _spread(case) > 4.5
    _decode(case, oracle, groups=([0, case.S], [prefix], case.S, prefix))


def _multi(case, orc, expect_flag=0):
    got = helpers.gpu_multi_step(case, DEV)
    assert got["flag"] == expect_flag, got["flag"]
    if expect_flag:
        return None
    caches = helpers.oracle_caches(case, orc)
    ref = helpers.oracle_multi_out(case, orc, caches)
    rows = helpers.covered_rows(case)
    return helpers.compare_row_scaled(got["out"][torch.as_tensor(rows, device=DEV)], ref[rows],
                                      case.kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["int8", "fp8"])
def test_multi_token_narrow(oracle, kv_dtype):
    """Draft verification (few new tokens per sequence: the mma.sync kernel, exact codes,
    scales in fp32), per-token magnitudes over six decades."""
    lens, qlen = [5, 100, 1300, 2100], [4, 3, 4, 2]
    case = workloads.build_multi_case(f"wide-verify-{kv_dtype}", S=len(lens), Hq=32, Hkv=8, D=128,
                                      bs=16, context_lens=lens, query_lens=qlen, seed=81,
                                      kv_dtype=kv_dtype)
    workloads.widen_scales(case, *DECODE_RANGE, seed=82)
    _multi(case, oracle)


def _bf16_dequantised(codes, scales, kv_dtype, orc) -> np.ndarray:
    """bf16 bits of code x scale (fp32 product, rounded once to bf16): the values a
    prefill-shaped 8-bit call attends (include/pa.h)."""
    if kv_dtype == "fp8":
        table = np.array([orc.fp8_decode(c) for c in range(256)], dtype=np.float32)
        vals = table[codes]
    else:
        vals = codes.astype(np.float32)
    x = vals * scales[..., None].astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


@pytest.mark.parametrize("kv_dtype", ["int8", "fp8"])
def test_multi_token_prefill(oracle, kv_dtype):
    """Prefill-shaped calls (the 8-bit blocks dequantised to bf16, then the tcgen05
    kernel), per-token magnitudes over six decades: compared with the oracle on the same
    dequantised values, bf16(code x scale) -- the reading this path takes."""
    lens, qlen = [300, 1000], [300, 130]
    case = workloads.build_multi_case(f"wide-prefill-{kv_dtype}", S=len(lens), Hq=16, Hkv=4, D=128,
                                      bs=16, context_lens=lens, query_lens=qlen, seed=83,
                                      kv_dtype=kv_dtype)
    workloads.widen_scales(case, *DECODE_RANGE, seed=84)
    got = helpers.gpu_multi_step(case, DEV)
    assert got["flag"] == 0
    kc, vc, ks, vs = helpers.oracle_caches(case, oracle)
    assert np.array_equal(got["k_cache"].cpu().numpy(), kc)
    assert np.array_equal(got["k_scale"].cpu().numpy().view(np.uint32), ks.view(np.uint32))
    kq = _bf16_dequantised(kc, np.nan_to_num(ks), kv_dtype, oracle)
    vq = _bf16_dequantised(vc, np.nan_to_num(vs), kv_dtype, oracle)
    ref = oracle.paged_prefill(helpers.bits(case.q), kq, vq, case.block_tables.cpu().numpy(),
                               case.context_lens.cpu().numpy(), case.query_start.cpu().numpy(), case.scale)
    rows = helpers.covered_rows(case)
    helpers.compare_row_scaled(got["out"][torch.as_tensor(rows, device=DEV)], ref[rows], "bf16")


@pytest.mark.parametrize("kv_dtype", ["int8", "fp8"])
def test_fp16_range_flag(oracle, kv_dtype):
    """Rows of magnitude 1e5..2e5: their scales put code x scale beyond fp16's 65504, so
    the shared-prefix path, which stages a shared prefix as fp16 code x scale, raises
    PA_FLAG_FP16_RANGE; pa_decode and narrow multi-token calls, which keep the codes
    exact and apply the scales in fp32, still match the oracle."""
    prefix = 64
    lens = [prefix + 40, prefix + 9]
    case = workloads.build_case(f"f16-range-{kv_dtype}", S=2, Hq=16, Hkv=2, D=128, bs=16,
                                context_lens=lens, seed=91, prefix_tokens=prefix, kv_dtype=kv_dtype)
    workloads.widen_scales(case, 1e5, 2e5, seed=92)
    _decode(case, oracle)
    _decode(case, oracle, groups=([0, 2], [prefix], 2, prefix), expect_flag=pa_mod.PA_FLAG_FP16_RANGE)
    multi = workloads.build_multi_case(f"f16-range-multi-{kv_dtype}", S=2, Hq=16, Hkv=2, D=128, bs=16,
                                       context_lens=[50, 70], query_lens=[2, 3], seed=93,
                                       kv_dtype=kv_dtype)
    workloads.widen_scales(multi, 1e5, 2e5, seed=94)
    _multi(multi, oracle)
