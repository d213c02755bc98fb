"""The C-ABI library builds, loads and exports every function include/pa.h declares;
host-side argument checks answer without touching a GPU."""
import re
from pathlib import Path

import pytest
import torch

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_197_gb300 import _build

    _build.build()
    import paged_kv_cache_197_gb300 as pa

    return pa.load_library()


def declared_functions():
    names = set()
    for header in sorted((ROOT / "include").glob("*.h")):
        text = re.sub(r"/\*.*?\*/", "", header.read_text(), flags=re.S)
        names |= set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    import paged_kv_cache_197_gb300 as pa

    names = declared_functions()
    assert names, "no declarations found"
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert sorted(pa.EXPORTED + pa.BLOCK_MANAGER_EXPORTED) == names


def test_version_and_strings(lib):
    assert lib.pa_version() == 1
    for code in range(5):
        assert lib.pa_status_string(code)


def test_no_extension_fails_loudly(tmp_path):
    import paged_kv_cache_197_gb300 as pa

    with pytest.raises(RuntimeError):
        pa.load_library(tmp_path / "missing.so")


def test_decode_host_checks(lib):
    import paged_kv_cache_197_gb300 as pa

    fake = 1 << 20  # never dereferenced: every call below fails its host checks

    def call(S=2, Hq=8, Hkv=2, D=128, bs=16, N=4, M=4, max_ctx=64, kv=pa.PA_KV_BF16,
             scale=0.1, ws=0, ws_bytes=0, out=fake):
        return lib.pa_decode(out, fake, fake, fake, None, None, kv, fake, M, fake, S, Hq, Hkv, D,
                             bs, N, scale, max_ctx, ws, ws_bytes, None, None)

    assert call(D=96) == pa.PA_ERR_UNSUPPORTED
    assert b"head_dim" in lib.pa_last_error_string()
    assert call(bs=8) == pa.PA_ERR_UNSUPPORTED
    assert call(Hq=6, Hkv=4) == pa.PA_ERR_INVALID_ARG
    assert call(kv=7) == pa.PA_ERR_UNSUPPORTED
    assert call(max_ctx=-1) == pa.PA_ERR_INVALID_ARG
    assert call(max_ctx=65, M=4, bs=16) == pa.PA_ERR_OUT_OF_RANGE
    assert call(kv=pa.PA_KV_INT8) == pa.PA_ERR_INVALID_ARG  # scales missing
    assert call(out=fake + 2) == pa.PA_ERR_INVALID_ARG  # misaligned
    assert call(scale=float("nan")) == pa.PA_ERR_INVALID_ARG
    assert call(max_ctx=4000, M=400) == pa.PA_ERR_INVALID_ARG  # workspace missing
    assert call(S=0) == pa.PA_OK  # nothing to do, nothing queued


def part_tokens(units, max_ctx, slots=304):
    """The partition length pa_decode chooses (a model of its policy)."""
    import math

    if units >= 6 * slots and max_ctx <= 4096:
        return max(max_ctx, 1)
    best, best_p = -1.0, 256
    for cand in (4096, 3072, 2048, 1536, 1024, 768, 512, 384, 256):
        n = max(1, -(-max_ctx // cand))
        waves = units * n / slots
        if waves < 3:
            continue
        ln = min(cand, max(max_ctx, 1))
        score = waves / math.ceil(waves) * ln / (ln + 64)
        if score > best + 1e-9:
            best, best_p = score, cand
    return best_p


def single_part_tokens(units, max_ctx, sms=152, per_sm=3):
    """The partition length of a split bf16 or int8 decode, which runs on the
    single-buffered kernel (four CTAs per SM for bf16, three for int8): n balanced
    partitions of the longest context scored by (last-wave fill) x len / (len + 512)
    with >= 1.5 waves."""
    import math

    ctx = max(max_ctx, 1)
    best, best_p = -1.0, None
    for n in range(1, (ctx + 255) // 256 + 1):
        cand = min(4096, max(256, -(-(-(-ctx // n)) // 64) * 64))
        if -(-ctx // cand) != n:
            continue
        waves = units * n / (per_sm * sms)
        if waves < 1.5 and cand != 256:
            continue
        ln = min(cand, ctx)
        score = waves / math.ceil(waves) * ln / (ln + 512)
        if score > best + 1e-9:
            best, best_p = score, cand
    return best_p


def test_workspace_size(lib):
    """Partition length: no split when the units alone give 6 waves of 2 CTAs per SM (152
    SMs without a GPU) and contexts are <= 4096 tokens; else the best of (last-wave fill)
    x (len / (len + 64)) among lengths giving >= 3 waves.  A split bf16 or int8 decode
    then runs on the single-buffered kernel with its own partitions
    (single_part_tokens); fp8 keeps the first.  The workspace holds (D + 2) fp32 per
    query head and partition."""
    import math

    import paged_kv_cache_197_gb300 as pa

    def parts(units, max_ctx, slots=304, kv=pa.PA_KV_FP8):
        p = max(1, -(-max_ctx // part_tokens(units, max_ctx, slots)))
        if p > 1 and kv != pa.PA_KV_FP8:
            per_sm = 4 if kv == pa.PA_KV_BF16 else 3
            p = max(1, -(-max_ctx // single_part_tokens(units, max_ctx, per_sm=per_sm)))
        return p

    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for S, Hq, Hkv, D, max_ctx in [(64, 40, 40, 128, 2048), (64, 40, 40, 128, 200), (20, 64, 8, 128, 8000), (256, 32, 8, 128, 32768), (2, 8, 2, 64, 1000),
                                   (50, 32, 8, 128, 2512)]:
        for kv in (pa.PA_KV_BF16, pa.PA_KV_INT8, pa.PA_KV_FP8):
            P = parts(S * Hkv * ((Hq // Hkv + 7) // 8), max_ctx, kv=kv)
            rows = S * Hq * P
            expect = 0 if P == 1 else up(up(rows * D * 4) + rows * 2 * 4)
            assert pa.pa_decode_workspace_size(S, Hq, Hkv, D, 16, kv, max_ctx) == expect, (S, kv)
    assert parts(160, 8000) == 11  # fp8: 768-token partitions for the 70B-shaped shape
    assert parts(160, 8000, kv=pa.PA_KV_BF16) == 7  # bf16, four CTAs per SM: 1152-token
    assert parts(160, 8000, kv=pa.PA_KV_INT8) == 5  # int8, three: 1600-token partitions
    assert pa.pa_decode_workspace_size(1, 3, 2, 128, 16, 0, 100) == 0  # invalid -> 0


def test_shared_prefix_workspace_and_checks(lib):
    """Workspace of the prefix-aware decode: S int32 group ids and S start offsets, then
    (D + 2) fp32 per query head and prefix chunk (256 tokens for a bf16 cache with
    head_dim 128, the tcgen05 path; else 128), then (D + 2) fp32 per query
    head and own-token partition; partitions sized for max_context_len - max_prefix_len
    (one partition when that is at most 1024 tokens; rounded up to 64 tokens), counted
    over max_context_len; each region 256-byte aligned.  Host checks refuse what the kernels do not take."""
    import paged_kv_cache_197_gb300 as pa

    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for S, Hq, Hkv, D, bs, max_ctx, max_group, max_prefix in [
            (50, 32, 8, 128, 16, 2512, 50, 2000), (8, 4, 4, 64, 32, 1372, 8, 672),
            (5, 8, 2, 128, 16, 9000, 1, 0), (56, 64, 16, 64, 32, 1005, 40, 640)]:
        units = S * Hkv * ((Hq // Hkv + 7) // 8)
        own = max(1, max_ctx - max_prefix)
        pt = own if own <= 1024 else part_tokens(units, own)
        pt = -(-pt // 64) * 64
        MP = max(1, -(-max_ctx // pt))
        PP = -(-max_prefix // (256 if D == 128 else 128))
        pre, own = S * Hq * PP, S * Hq * MP
        size = up(S * 4) + S * 4
        size = up(size) + pre * D * 4
        size = up(size) + pre * 2 * 4
        size = up(size) + own * D * 4
        size = up(up(size) + own * 2 * 4)
        got = pa.pa_decode_shared_prefix_workspace_size(S, Hq, Hkv, D, bs, pa.PA_KV_BF16, max_ctx,
                                                        max_group, max_prefix)
        assert got == size, (S, got, size)
    ws = lambda **k: pa.pa_decode_shared_prefix_workspace_size(  # noqa: E731
        **{**dict(S=4, Hq=8, Hkv=2, D=128, bs=16, kv_dtype=0, max_context_len=512,
                  max_group_size=4, max_prefix_len=256), **k})
    assert ws() > 0
    assert ws(kv_dtype=pa.PA_KV_INT8) == ws(kv_dtype=pa.PA_KV_FP8)
    assert ws(kv_dtype=pa.PA_KV_INT8, max_prefix_len=256) > ws(max_prefix_len=256)  # 128-token chunks
    assert ws(kv_dtype=pa.PA_KV_INT8, D=64) == ws(D=64)
    assert ws(kv_dtype=9) == 0                  # no such cache type
    assert ws(max_prefix_len=200) == 0          # not whole blocks
    assert ws(max_prefix_len=1024) == 0         # longer than any context
    assert ws(max_group_size=0) == 0
    assert ws(max_group_size=5) == 0            # more members than sequences

    fake = 1 << 20

    def call(S=2, kv=pa.PA_KV_BF16, n_groups=1, gs=fake, max_group=2, max_prefix=32, ws=fake,
             ws_bytes=1 << 30):
        return lib.pa_decode_shared_prefix(fake, fake, fake, fake, None, None, kv, fake, 4, fake, S,
                                           8, 2, 128, 16, 4, 0.1, 64, gs, fake, n_groups,
                                           max_group, max_prefix, ws, ws_bytes, None, None)

    assert call(kv=pa.PA_KV_FP8) == pa.PA_ERR_INVALID_ARG  # scales missing
    assert call(kv=6) == pa.PA_ERR_UNSUPPORTED
    assert call(gs=None) == pa.PA_ERR_INVALID_ARG
    assert call(n_groups=-1) == pa.PA_ERR_INVALID_ARG
    assert call(max_prefix=48 + 8) == pa.PA_ERR_INVALID_ARG
    assert call(ws_bytes=64) == pa.PA_ERR_INVALID_ARG
    assert call(ws=fake + 16) == pa.PA_ERR_INVALID_ARG  # not 256-byte aligned
    assert call(S=0) == pa.PA_OK


def test_multi_token_workspace_and_checks(lib):
    """Multi-token attention: 128 (token, head) columns per CTA, two CTAs per SM.  On
    the tcgen05 path with chunks of at least 64 columns (bf16 cache, head_dim 128,
    max_query_len * G >= 64) no partition unless the CTAs fill less than half the
    slots, then about one wave of partitions (multiples of 128 tokens, at least 512).  Otherwise no partition when the columns
    give 4 waves of 2 CTAs per SM and contexts are <= 4096 tokens, else the best of
    (last-wave fill) x (len / (len + 512)) over n balanced partitions of the longest
    context (ceil(ctx / n) rounded up to 64 tokens, 256..4096) with >= 2 waves (256 as
    the fallback).  Narrow chunks (at most 8 new tokens) of an 8-bit cache off the
    tcgen05 path run on the decode kernel, one CTA per (two new tokens, up to 8 query heads):
    the same rule with those CTAs as the units.  The workspace
    holds (D + 2) fp32 per query row, head and partition."""
    import math

    import paged_kv_cache_197_gb300 as pa

    def plan(S, Hq, Hkv, D, max_ctx, max_q, sms=152, kv=pa.PA_KV_BF16):
        G = Hq // Hkv
        cb = max(1, -(-max_q * G // 128))
        per_token = kv != pa.PA_KV_BF16 and not (D == 128 and max_q * G >= 64) and max_q <= 8
        rows = 2 if max_q >= 2 else 1  # new tokens per decode CTA
        units = S * Hkv * -(-G // 8) * -(-max_q // rows) if per_token else S * Hkv * cb
        ctx = max(max_ctx, 1)
        if D == 128 and max_q * G >= 64:
            if units < sms:
                want = math.ceil(2 * sms / units)
                return max(512, -(-(-(-ctx // want)) // 128) * 128)
            return -(-ctx // 64) * 64
        slots = 2 * sms
        if units >= 4 * slots and ctx <= 4096:
            return -(-ctx // 64) * 64
        best, best_p = -1.0, 256
        for n in range(1, (ctx + 255) // 256 + 1):
            cand = min(4096, max(256, -(-(-(-ctx // n)) // 64) * 64))
            parts = -(-ctx // cand)
            if parts != n:
                continue
            waves = units * parts / slots
            if waves < 2 and cand != 256:
                continue
            ln = min(cand, ctx)
            score = waves / math.ceil(waves) * ln / (ln + 512)
            if score > best + 1e-9:
                best, best_p = score, cand
        return best_p

    # the balanced rule's own properties, over a sweep of contexts, batch shapes and SM
    # counts: every partition is a multiple of 64 tokens in [256, 4096] (or the whole
    # context rounded up to 64), and the n partitions of the longest context leave less
    # than 64 tokens of slack each (no ragged last partition) unless they are of the
    # shortest length, 256 tokens
    for sms in (132, 148, 152):
        for ctx in (1, 63, 255, 256, 257, 1000, 2100, 4095, 4097, 8000, 12345, 32768):
            for S, Hkv, max_q, G in ((1, 1, 1, 1), (4, 8, 4, 8), (20, 8, 4, 8), (64, 8, 2, 4),
                                     (256, 8, 1, 4)):
                for kv in (pa.PA_KV_BF16, pa.PA_KV_FP8):
                    pt = plan(S, Hkv * G, Hkv, 64, ctx, max_q, sms=sms, kv=kv)
                    n = -(-ctx // pt)
                    assert pt % 64 == 0, (sms, ctx, S, pt)
                    if n > 1:
                        assert 256 <= pt <= 4096, (sms, ctx, S, pt)
                        assert n * pt - ctx < 64 * n or pt == 256, (sms, ctx, S, pt)
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for S, T, Hq, Hkv, D, max_ctx, max_q in [(20, 80, 64, 8, 128, 8000, 4), (4, 2048, 32, 8, 128, 4096, 512),
                                             (9, 72, 16, 2, 64, 12345, 8), (3, 12, 8, 8, 64, 4097, 4),
                                             (64, 128, 32, 8, 64, 3000, 2), (1, 1, 8, 1, 64, 32768, 1),
                                             (7, 40, 16, 2, 64, 2100, 8), (600, 600, 32, 32, 128, 1000, 1),
                                             (1, 128, 32, 8, 128, 32768, 128), (2, 300, 16, 2, 128, 9000, 150)]:
        for kv in (pa.PA_KV_BF16, pa.PA_KV_INT8, pa.PA_KV_FP8):
            if kv != pa.PA_KV_BF16 and D == 128 and max_q * Hq // Hkv >= 64:
                continue  # the dequantising pass adds its pool (below)
            pt = plan(S, Hq, Hkv, D, max_ctx, max_q, kv=kv)
            parts = -(-max_ctx // pt)
            rows = T * Hq * parts
            expect = 0 if parts == 1 else up(up(rows * D * 4) + rows * 2 * 4)
            got = pa.pa_multi_token_workspace_size(S, T, Hq, Hkv, D, 16, kv, max_ctx, max_q)
            assert got == expect, (S, T, kv, got, expect)
    ws = lambda **k: pa.pa_multi_token_workspace_size(  # noqa: E731
        **{**dict(S=4, T=64, Hq=8, Hkv=2, D=128, bs=16, kv_dtype=0, max_context_len=8000,
                  max_query_len=8), **k})
    assert ws() > 0
    # 8 new tokens x 4 heads, 8-bit caches: per-token CTAs, more of them, shorter partitions
    assert ws(kv_dtype=pa.PA_KV_INT8) == ws(kv_dtype=pa.PA_KV_FP8) != ws()
    assert ws(kv_dtype=pa.PA_KV_INT8, max_query_len=9) == ws(max_query_len=9)  # past 8: mma.sync
    # 16 tokens x 4 heads: the tcgen05 path's plan for every cache type (16 CTAs of
    # columns fill less than half the SMs, so the contexts are split for one wave); an
    # 8-bit cache adds the table of pool slots [S][Mq], the sequences' pool offsets
    # [S + 1], and the bf16 pool of the attended blocks (K and V), at most S x Mq blocks
    Mq = -(-8000 // 16)
    block = 2 * 16 * 128 * 2
    table = up(4 * Mq * 4) + up(4 * 5)
    for dt in (pa.PA_KV_INT8, pa.PA_KV_FP8):
        assert ws(max_query_len=16, kv_dtype=dt) == ws(max_query_len=16) + table + 2 * 4 * Mq * block
        # sized for the tokens the batch holds: ceil(total / bs) + S blocks
        for total in (1, 5000, 16000, 32000):
            got = pa.pa_multi_token_workspace_size_for_tokens(4, 64, 8, 2, 128, 16, dt, 8000, 16, total)
            blocks = min(4 * Mq, -(-total // 16) + 4)
            assert got == ws(max_query_len=16) + table + 2 * blocks * block
        assert pa.pa_multi_token_workspace_size_for_tokens(4, 64, 8, 2, 128, 16, dt, 8000, 16, -1) == 0
    # bf16 caches and narrow chunks have no pool: the token count changes nothing
    assert pa.pa_multi_token_workspace_size_for_tokens(4, 64, 8, 2, 128, 16, 0, 8000, 16, 77) == ws(max_query_len=16)
    assert ws(max_query_len=16, D=64) != ws(max_query_len=16)  # head_dim 64: the mma.sync plan
    assert ws(kv_dtype=7) == 0
    assert ws(max_query_len=0) == 0
    assert ws(max_query_len=65) == 0  # more than T rows
    fake = 1 << 20

    def call(S=2, T=8, kv=pa.PA_KV_BF16, max_q=4, qs=fake, ws=fake, ws_bytes=1 << 30, max_ctx=64):
        return lib.pa_multi_token_attention(fake, fake, fake, fake, None, None, kv, fake, 4, fake, qs,
                                            S, T, 8, 2, 128, 16, 4, 0.1, max_ctx, max_q, ws, ws_bytes,
                                            None, None)

    assert call(kv=pa.PA_KV_FP8) == pa.PA_ERR_INVALID_ARG  # scales missing
    assert call(kv=5) == pa.PA_ERR_UNSUPPORTED
    assert call(qs=None) == pa.PA_ERR_INVALID_ARG
    assert call(max_q=9) == pa.PA_ERR_INVALID_ARG       # above T
    assert call(max_ctx=65) == pa.PA_ERR_OUT_OF_RANGE   # above M * bs
    assert call(T=0) == pa.PA_OK and call(S=0) == pa.PA_OK


def test_cache_host_checks(lib):
    import paged_kv_cache_197_gb300 as pa

    fake = 1 << 20
    assert lib.pa_reshape_and_cache(fake, fake, fake, fake, fake, 0, 8, 128, 16, 4, None, None) == pa.PA_OK
    assert lib.pa_reshape_and_cache(fake, fake, fake, fake, fake, 3, 8, 80, 16, 4, None, None) == pa.PA_ERR_UNSUPPORTED
    assert lib.pa_reshape_and_cache(fake, fake, fake, fake, fake, -1, 8, 128, 16, 4, None, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_quantize_kv(fake, fake, fake, fake, None, fake, fake, 2, 8, 128, 32, 4, None, None) == pa.PA_ERR_INVALID_ARG

    def copy(pairs, N=10, block_bytes=4096):
        t = torch.tensor(pairs, dtype=torch.int64).reshape(-1, 2).contiguous()
        return lib.pa_copy_blocks(fake, fake, None, None, t.data_ptr(), t.shape[0], N, block_bytes, 0, None)

    assert copy([[1, 2], [3, 2]]) == pa.PA_ERR_INVALID_ARG  # two pairs write block 2
    assert copy([[1, 2], [2, 3]]) == pa.PA_ERR_INVALID_ARG  # block 2 read and written
    assert copy([[1, 10]]) == pa.PA_ERR_OUT_OF_RANGE
    assert copy([[-1, 3]]) == pa.PA_ERR_OUT_OF_RANGE
    assert copy([[1, 2]], block_bytes=100) == pa.PA_ERR_INVALID_ARG


def test_binding_rejects_host_tensors(lib):
    import paged_kv_cache_197_gb300 as pa

    x = torch.zeros((2, 4, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pa.pa_decode(x, x, x, x, x, x, 0.1, 16)


def test_eight_bit_prefill_workspace_scales_with_tokens(lib):
    """A prefill-shaped 8-bit call over a 256-sequence batch with log-uniform lengths in
    [128, 32768]: sized for the tokens it holds, the workspace is under twice the bf16
    bytes of the blocks it attends, where sizing every sequence at the longest context
    would take over five times that."""
    import paged_kv_cache_197_gb300 as pa
    import workloads

    lens = workloads.int8_lengths(256, seed=4)
    S, Hq, Hkv, D, bs, max_q = 256, 32, 8, 128, 32, 16
    T = S * max_q
    total = sum(lens)
    attended = sum(-(-c // bs) for c in lens) * Hkv * bs * D * 2 * 2  # bf16 K and V
    tight = pa.pa_multi_token_workspace_size_for_tokens(S, T, Hq, Hkv, D, bs, pa.PA_KV_FP8, max(lens), max_q,
                                                         total)
    loose = pa.pa_multi_token_workspace_size(S, T, Hq, Hkv, D, bs, pa.PA_KV_FP8, max(lens), max_q)
    assert attended < tight <= 2 * attended
    assert loose > 5 * attended

