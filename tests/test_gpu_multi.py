"""GPU parity of multi-token paged attention (chunked prefill / draft verification)
against the CPU oracle: every new token of a sequence attends the cache up to its
own position."""
import numpy as np
import pytest
import torch

import helpers
import workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_kv_cache_197_gb300 as pa

    pa.load_library()


def _run(case, orc, expect_flag=0, **kw):
    got = helpers.gpu_multi_step(case, DEV, **kw)
    caches = helpers.oracle_caches(case, orc)
    if case.kv_dtype == "bf16":
        assert np.array_equal(helpers.bits(got["k_cache"]), caches[0])
        assert np.array_equal(helpers.bits(got["v_cache"]), caches[1])
    else:
        assert np.array_equal(got["k_cache"].cpu().numpy(), caches[0])
        assert np.array_equal(got["v_cache"].cpu().numpy(), caches[1])
        assert np.array_equal(got["k_scale"].cpu().numpy().view(np.uint32), caches[2].view(np.uint32))
    assert got["flag"] == expect_flag
    ref = helpers.oracle_multi_out(case, orc, caches)
    rows = helpers.covered_rows(case)
    other = np.setdiff1d(np.arange(case.q.shape[0]), rows)
    if other.size:  # rows of no sequence are not written
        assert torch.isnan(got["out"][torch.as_tensor(other, device=DEV)].float()).all()
    idx = torch.as_tensor(rows, device=DEV)
    return helpers.compare(got["out"][idx], ref[rows], case.kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8", "fp8"])
@pytest.mark.parametrize("D,bs,Hq,Hkv", [(128, 16, 32, 8), (64, 32, 8, 8), (128, 32, 16, 2),
                                          (64, 16, 20, 2), (128, 16, 64, 8)])
def test_draft_verification(oracle, D, bs, Hq, Hkv, kv_dtype):
    """A few new tokens per sequence on contexts from one token up, including a
    sequence whose whole context is new and one with a single new token."""
    lens = [1, 5, 17, 100, 513, 1300, 2100]
    qlen = [1, 5, 4, 8, 3, 1, 7]
    case = workloads.build_multi_case(f"verify-{D}-{bs}-{Hq}-{Hkv}", S=len(lens), Hq=Hq, Hkv=Hkv,
                                      D=D, bs=bs, context_lens=lens, query_lens=qlen,
                                      seed=3 * D + bs + Hq, row_offset=2, extra_rows=3,
                                      kv_dtype=kv_dtype)
    _run(case, oracle)


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8", "fp8"])
def test_prefill_chunks(oracle, kv_dtype):
    """Long chunks (several CTAs of columns per kv head): a prompt's first chunk, a
    later chunk on top of cached tokens and a chunk of one token."""
    lens = [300, 1000, 77]
    qlen = [300, 260, 1]
    case = workloads.build_multi_case("prefill", S=3, Hq=16, Hkv=4, D=128, bs=16, context_lens=lens,
                                      query_lens=qlen, seed=31, kv_dtype=kv_dtype)
    _run(case, oracle)


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8", "fp8"])
def test_long_context_partitions(oracle, kv_dtype):
    """Few sequences with long contexts: the context is split into partitions that a
    second kernel merges; columns of one chunk straddle partition boundaries."""
    lens = [9000, 4097, 6000]
    qlen = [4, 64, 2]
    case = workloads.build_multi_case("long", S=3, Hq=8, Hkv=2, D=128, bs=16, context_lens=lens,
                                      query_lens=qlen, seed=32, kv_dtype=kv_dtype)
    _run(case, oracle)


@pytest.mark.parametrize("kv_dtype", ["int8", "fp8"])
@pytest.mark.parametrize("D,bs,Hq,Hkv", [(128, 32, 8, 2), (64, 16, 24, 2)])
def test_eight_bit_verification_long_contexts(oracle, kv_dtype, D, bs, Hq, Hkv):
    """Narrow chunks of an 8-bit cache on the decode kernel's per-token mode: long
    contexts split into partitions whose boundaries fall between one new token's causal
    limit and the next's, a chunk of one token on a one-token context, and 12 query
    heads per kv head (a full and a partial chunk of 8 heads)."""
    lens = [9000, 4097, 6000, 1, 2049]
    qlen = [4, 8, 2, 1, 3]
    case = workloads.build_multi_case(f"long8-{kv_dtype}-{D}-{Hq}", S=len(lens), Hq=Hq, Hkv=Hkv, D=D,
                                      bs=bs, context_lens=lens, query_lens=qlen, seed=D + Hq + 5,
                                      row_offset=1, extra_rows=2, kv_dtype=kv_dtype)
    _run(case, oracle)


def test_one_token_matches_decode(oracle):
    """With one new token per sequence the step is the decode step."""
    import paged_kv_cache_197_gb300 as pa

    lens = [1, 16, 33, 700, 5000]
    case = workloads.build_multi_case("one", S=5, Hq=16, Hkv=4, D=128, bs=16, context_lens=lens,
                                      query_lens=[1] * 5, seed=33)
    got = helpers.gpu_multi_step(case, DEV)
    c = case.to(DEV)
    dec = torch.empty_like(c.q)
    ws = pa.decode_workspace(c.q, got["k_cache"], max(lens))
    pa.pa_decode(dec, c.q, got["k_cache"], got["v_cache"], c.block_tables, c.context_lens,
                 case.scale, max(lens), workspace=ws)
    torch.cuda.synchronize()
    ref = helpers.oracle_multi_out(case, oracle, helpers.oracle_caches(case, oracle))
    helpers.compare(got["out"], ref, "bf16")
    helpers.compare(dec, ref, "bf16")


@pytest.mark.parametrize("kv_dtype,D", [("bf16", 64), ("int8", 64), ("fp8", 128)])
def test_bad_offsets_are_skipped(oracle, kv_dtype, D):
    """A sequence with more new tokens than max_query_len is skipped (QUERY flag, rows
    untouched); an empty chunk writes nothing; the others are exact.  8-bit caches: the
    decode kernel's per-token mode."""
    import paged_kv_cache_197_gb300 as pa

    lens = [50, 400, 90]
    qlen = [3, 9, 0]
    case = workloads.build_multi_case(f"bad-{kv_dtype}", S=3, Hq=8, Hkv=2, D=D, bs=16, context_lens=lens,
                                      query_lens=qlen, seed=34, kv_dtype=kv_dtype)
    got = helpers.gpu_multi_step(case, DEV, max_query_len=4)
    assert got["flag"] == pa.PA_FLAG_QUERY_OUT_OF_RANGE
    caches = helpers.oracle_caches(case, oracle)
    ref = helpers.oracle_multi_out(case, oracle, caches)
    assert torch.isnan(got["out"][3:12].float()).all()
    helpers.compare(got["out"][0:3], ref[0:3], kv_dtype)


def test_rejects_unsupported():
    import paged_kv_cache_197_gb300 as pa

    case = workloads.build_multi_case("rej", S=2, Hq=4, Hkv=4, D=64, bs=16, context_lens=[40, 40],
                                      query_lens=[2, 2], seed=35).to(DEV)
    out = torch.empty_like(case.q)
    i8 = torch.zeros(case.k_pool.shape, dtype=torch.int8, device=DEV)
    with pytest.raises(ValueError):  # an int8 cache without its scales
        pa.pa_multi_token_attention(out, case.q, i8, i8, case.block_tables, case.context_lens,
                                    case.query_start, case.scale, 40, 2)
    with pytest.raises(pa.PagedAttentionError):  # max_query_len above the context bound
        pa.pa_multi_token_attention(out, case.q, case.k_pool, case.v_pool, case.block_tables,
                                    case.context_lens, case.query_start, case.scale, 40, 41)
    torch.cuda.synchronize()


def test_block_permutation_bit_identical():
    """The result depends on logical order only: moving blocks changes no bit."""
    case = workloads.build_multi_case("perm", S=4, Hq=16, Hkv=4, D=128, bs=16,
                                      context_lens=[40, 700, 1300, 90], query_lens=[3, 8, 140, 1],
                                      seed=36, poison=False)
    a = helpers.gpu_multi_step(case, DEV)["out"]
    pi = torch.randperm(case.N, generator=torch.Generator().manual_seed(5))
    moved = workloads.PagedCase(**{**case.__dict__})
    moved.k_pool = torch.empty_like(case.k_pool)
    moved.v_pool = torch.empty_like(case.v_pool)
    moved.k_pool[pi] = case.k_pool
    moved.v_pool[pi] = case.v_pool
    moved.block_tables = pi[case.block_tables.long()].to(torch.int32)
    slots = case.slot_mapping.clone()
    ok = slots >= 0
    moved.slot_mapping = torch.where(ok, pi[(slots // case.bs).clamp(min=0)] * case.bs + slots % case.bs, slots)
    b = helpers.gpu_multi_step(moved, DEV)["out"]
    assert torch.equal(a, b)


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8", "fp8"])
def test_error_flags(kv_dtype):
    """A block id beyond the pool is skipped (read as zeros) and flagged; a context past
    max_context_len is clamped and flagged."""
    import paged_kv_cache_197_gb300 as pa

    case = workloads.build_multi_case(f"flags-{kv_dtype}", S=2, Hq=8, Hkv=2, D=64, bs=16,
                                      context_lens=[90, 300], query_lens=[4, 5], seed=37, poison=False,
                                      kv_dtype=kv_dtype)
    cached = helpers.gpu_multi_step(case, DEV)
    assert cached["flag"] == 0
    case = case.to(DEV)
    k, v = cached["k_cache"], cached["v_cache"]
    sc = dict(k_scale=cached["k_scale"], v_scale=cached["v_scale"])
    out = torch.empty_like(case.q)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    tables = case.block_tables.clone()
    tables[1, 2] = case.N + 7
    pa.pa_multi_token_attention(out, case.q, k, v, tables, case.context_lens,
                                case.query_start, case.scale, 300, 5, err_flag=flag, **sc)
    torch.cuda.synchronize()
    assert flag.item() == pa.PA_FLAG_BLOCK_OUT_OF_RANGE
    assert torch.isfinite(out.float()).all()
    flag.zero_()
    pa.pa_multi_token_attention(out, case.q, k, v, case.block_tables,
                                case.context_lens, case.query_start, case.scale, 200, 5, err_flag=flag, **sc)
    torch.cuda.synchronize()
    assert flag.item() == pa.PA_FLAG_CONTEXT_OUT_OF_RANGE


def test_graph_capture_replays():
    """The call captured in a CUDA graph (with its merge launched as a programmatic
    dependent) replays to the same bits as the eager call."""
    import paged_kv_cache_197_gb300 as pa

    case = workloads.build_multi_case("graph", S=3, Hq=16, Hkv=2, D=128, bs=16,
                                      context_lens=[5000, 9000, 300], query_lens=[4, 2, 150],
                                      seed=38, poison=False).to(DEV)
    max_ctx, max_q = 9000, 150
    n = pa.pa_multi_token_workspace_size(case.S, case.q.shape[0], case.Hq, case.Hkv, case.D, case.bs,
                                         pa.PA_KV_BF16, max_ctx, max_q)
    assert n > 0  # the contexts are split: the merge kernel is part of the call
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    eager = torch.empty_like(case.q)
    call = lambda out: pa.pa_multi_token_attention(  # noqa: E731
        out, case.q, case.k_pool, case.v_pool, case.block_tables, case.context_lens,
        case.query_start, case.scale, max_ctx, max_q, workspace=ws)
    call(eager)
    torch.cuda.synchronize()
    replay = torch.full_like(case.q, float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(replay)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager, replay)


@pytest.mark.parametrize("bs,Hq,Hkv,lens,qlen", [
    (32, 40, 8, [777, 2100, 64], [40, 300, 64]),  # G = 5, block 32, a chunk that is the whole context
    (16, 8, 8, [129, 1000], [129, 128]),         # G = 1
    (16, 64, 8, [5000, 17, 4200], [100, 17, 9]),  # G = 8, partitions, columns past one CTA
    (32, 16, 2, [40, 300], [33, 300]),           # G = 8, block 32, chunks shorter than a tile
])
def test_tensor_core_path(oracle, bs, Hq, Hkv, lens, qlen):
    """Shapes that run on the tcgen05 kernel (bf16 cache, head_dim 128, at least 64
    (token, head) columns per kv head): ragged chunks, groups that are not powers of
    two, block size 32, split contexts, and caches whose unused slots hold NaN."""
    case = workloads.build_multi_case(f"tc-{bs}-{Hq}-{Hkv}", S=len(lens), Hq=Hq, Hkv=Hkv, D=128,
                                      bs=bs, context_lens=lens, query_lens=qlen, seed=bs + Hq + len(lens),
                                      row_offset=1, extra_rows=2)
    _run(case, oracle)


def test_tensor_core_error_flags(oracle):
    """On the tcgen05 path too: a block id beyond the pool is read as zeros and
    flagged, and the rows stay finite; a context past max_context_len is clamped."""
    import paged_kv_cache_197_gb300 as pa

    case = workloads.build_multi_case("tc-flags", S=2, Hq=32, Hkv=4, D=128, bs=16,
                                      context_lens=[90, 700], query_lens=[20, 64], seed=39,
                                      poison=False).to(DEV)
    out = torch.empty_like(case.q)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    tables = case.block_tables.clone()
    tables[1, 5] = case.N + 3
    pa.pa_multi_token_attention(out, case.q, case.k_pool, case.v_pool, tables, case.context_lens,
                                case.query_start, case.scale, 700, 64, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == pa.PA_FLAG_BLOCK_OUT_OF_RANGE
    assert torch.isfinite(out.float()).all()
    flag.zero_()
    pa.pa_multi_token_attention(out, case.q, case.k_pool, case.v_pool, case.block_tables,
                                case.context_lens, case.query_start, case.scale, 600, 64, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == pa.PA_FLAG_CONTEXT_OUT_OF_RANGE


@pytest.mark.parametrize("kv_dtype", ["int8", "fp8"])
def test_eight_bit_prefill_pass_flags(oracle, kv_dtype):
    """8-bit prefill-shaped chunks go through the dequantising pass: a block id beyond
    the pool is flagged there and read as zeros, the other sequences stay exact, and
    the workspace includes the bf16 pool."""
    import paged_kv_cache_197_gb300 as pa

    lens, qlen = [300, 700], [100, 64]
    case = workloads.build_multi_case(f"q-flags-{kv_dtype}", S=2, Hq=16, Hkv=2, D=128, bs=16,
                                      context_lens=lens, query_lens=qlen, seed=40, kv_dtype=kv_dtype)
    base = pa.pa_multi_token_workspace_size(2, sum(qlen), 16, 2, 128, 16, pa.PA_KV_BF16, 700, 100)
    code = {"int8": pa.PA_KV_INT8, "fp8": pa.PA_KV_FP8}[kv_dtype]
    q8 = pa.pa_multi_token_workspace_size(2, sum(qlen), 16, 2, 128, 16, code, 700, 100)
    assert q8 > base  # the pool of dequantised blocks
    bad = workloads.PagedCase(**{**case.__dict__})
    bad.block_tables = case.block_tables.clone()
    bad.block_tables[1, 3] = case.N + 5
    got = helpers.gpu_multi_step(bad, DEV)
    assert got["flag"] == pa.PA_FLAG_BLOCK_OUT_OF_RANGE
    assert torch.isfinite(got["out"][torch.arange(sum(qlen), device=DEV)].float()).all()
    caches = helpers.oracle_caches(case, oracle)
    sub, rows = _sequences(case, [0])
    ref = helpers.oracle_multi_out(sub, oracle, caches)
    helpers.compare(got["out"][rows.to(DEV)], ref, kv_dtype)


def _sequences(case, seqs):
    """The case cut to the listed sequences (their query rows, tables and lengths)."""
    qs = case.query_start.cpu().tolist()
    rows = torch.cat([torch.arange(qs[s], qs[s + 1]) for s in seqs])
    sub = workloads.PagedCase(**{**case.__dict__})
    sub.q = case.q.cpu()[rows]
    sub.block_tables = case.block_tables.cpu()[seqs]
    sub.context_lens = case.context_lens.cpu()[seqs]
    starts = [0]
    for s in seqs:
        starts.append(starts[-1] + qs[s + 1] - qs[s])
    sub.query_start = torch.tensor(starts, dtype=torch.int32)
    sub.S = len(seqs)
    return sub, rows


@pytest.mark.slow
@pytest.mark.parametrize("name", ["verify70b", "prefill8b", "verify70b_fp8", "prefill8b_fp8"])
def test_full_size_sampled(oracle, name):
    """The full-size multi-token workloads in the launch configuration bench.py times
    (bf16 and fp8 caches: both kernels and the dequantising pass), checked on a sample
    of sequences."""
    case = workloads.CONFIGS[name](device="cpu", poison=True)
    got = helpers.gpu_multi_step(case, DEV)
    assert got["flag"] == 0
    caches = helpers.oracle_caches(case, oracle)
    seqs = [0, case.S - 1]
    sub, rows = _sequences(case, seqs)
    ref = helpers.oracle_multi_out(sub, oracle, caches)
    helpers.compare(got["out"][rows.to(DEV)], ref, case.kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["int8", "fp8"])
def test_eight_bit_pool_sized_for_tokens(oracle, kv_dtype):
    """Prefill-shaped 8-bit calls dequantise the attended blocks into a pool packed
    sequence after sequence: a workspace sized for the batch's tokens gives the same
    result as one sized for every sequence at the longest context; one whose pool is
    short by a block raises PA_FLAG_WORKSPACE_SHORT (the block left out is read as
    zeros; the attention kernel may flag its table entry as out of range too)."""
    import paged_kv_cache_197_gb300 as pa

    lens, qlen = [300, 1000, 77, 650], [300, 130, 1, 64]
    case = workloads.build_multi_case(f"pool-{kv_dtype}", S=4, Hq=16, Hkv=4, D=128, bs=16, context_lens=lens,
                                      query_lens=qlen, seed=35, kv_dtype=kv_dtype)
    T = case.q.shape[0]
    dt = pa.PA_KV_INT8 if kv_dtype == "int8" else pa.PA_KV_FP8
    tight = pa.pa_multi_token_workspace_size_for_tokens(4, T, 16, 4, 128, 16, dt, max(lens), max(qlen), sum(lens))
    loose = pa.pa_multi_token_workspace_size(4, T, 16, 4, 128, 16, dt, max(lens), max(qlen))
    assert tight < loose
    caches = helpers.oracle_caches(case, oracle)
    ref = helpers.oracle_multi_out(case, oracle, caches)
    rows = helpers.covered_rows(case)
    got = helpers.gpu_multi_step(case, DEV, workspace_bytes=tight)
    assert got["flag"] == 0
    helpers.compare(got["out"][torch.as_tensor(rows, device=DEV)], ref[rows], kv_dtype)
    # the exact need: every attended block, none to spare
    need = sum(-(-c // 16) for c in lens)
    block = 4 * 16 * 128 * 2
    short = tight - 2 * block * (-(-sum(lens) // 16) + 4 - need) - 2 * block
    got = helpers.gpu_multi_step(case, DEV, workspace_bytes=short)
    assert got["flag"] & pa.PA_FLAG_WORKSPACE_SHORT
    assert got["flag"] & ~(pa.PA_FLAG_WORKSPACE_SHORT | pa.PA_FLAG_BLOCK_OUT_OF_RANGE) == 0

