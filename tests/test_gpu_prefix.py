"""GPU parity of the prefix-aware decode (pa_decode_shared_prefix) against the CPU
oracle's paged attention: the same result as pa_decode for any grouping of the batch,
including groups whose members break the shared-prefix preconditions (decoded on their
own, flag raised)."""
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


def _share(case, members, plen):
    """Point the first plen // bs table entries of every member at the first member's
    blocks (what prefix caching does to a table); both sides read through the tables."""
    nb = plen // case.bs
    lead = members[0]
    for s in members[1:]:
        case.block_tables[s, :nb] = case.block_tables[lead, :nb]


def _run(case, orc, groups, expect_flag=0):
    got = helpers.gpu_step(case, DEV, groups=groups)
    caches = helpers.oracle_caches(case, orc)
    if case.kv_dtype == "bf16":
        assert np.array_equal(helpers.bits(got["k_cache"]), caches[0])
        assert np.array_equal(helpers.bits(got["v_cache"]), caches[1])
    assert got["flag"] == expect_flag
    ref = helpers.oracle_out(case, orc, caches)
    return helpers.compare(got["out"], ref, case.kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8", "fp8"])
@pytest.mark.parametrize("D,bs,Hq,Hkv", [(128, 16, 32, 8), (64, 32, 4, 4), (128, 32, 16, 2),
                                          (64, 16, 20, 2), (128, 16, 64, 8)])
def test_one_group_with_cow(oracle, D, bs, Hq, Hkv, kv_dtype):
    """Every sequence shares one prefix (several 128-token chunks and a ragged last
    chunk); each sequence's last block is a copy-on-write target."""
    prefix = 21 * 32  # 672 tokens: five chunks of 128 and one of 32
    own = [1, 2, 15, 16, 17, 100, 333, 700]
    lens = [prefix + o for o in own]
    case = workloads.build_case(f"pfx-{D}-{bs}-{Hq}-{Hkv}", S=len(lens), Hq=Hq, Hkv=Hkv, D=D,
                                bs=bs, context_lens=lens, seed=7 * D + bs + Hq,
                                prefix_tokens=prefix, cow=True, kv_dtype=kv_dtype)
    _run(case, oracle, ([0, case.S], [prefix], case.S, prefix))


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8", "fp8"])
def test_mixed_groups(oracle, kv_dtype):
    """Several groups with different prefixes, a one-member group, an empty group,
    sequences in no group, a member whose whole context is the prefix, and a prefix
    whose last chunk is ragged (208 = 128 + 80 tokens)."""
    lens = [300, 290, 1000, 129, 50, 208, 400, 209, 3000, 77, 1, 2500]
    case = workloads.build_case("pfx-mixed", S=len(lens), Hq=32, Hkv=8, D=128, bs=16,
                                context_lens=lens, seed=11, kv_dtype=kv_dtype)
    _share(case, [0, 1, 2, 3], 128)
    _share(case, [5, 6, 7, 8], 208)
    # groups: [0,4) 128 tokens, [4,5) 48 tokens, [5,5) empty, [5,9) 208 tokens; 9.. alone
    groups = ([0, 4, 5, 5, 9], [128, 48, 0, 208], 4, 256)
    _run(case, oracle, groups)


@pytest.mark.parametrize("D", [64, 128])
def test_groups_wider_than_one_cta(oracle, D):
    """A group with more (member, head) columns (160) than one CTA takes (128), beside a
    smaller one (head_dim 128: the tcgen05 kernel in group mode, two column blocks)."""
    lens = [700 + 13 * i for i in range(40)] + [900 + 7 * i for i in range(16)]
    case = workloads.build_case(f"pfx-wide-{D}", S=len(lens), Hq=64, Hkv=16, D=D, bs=32,
                                context_lens=lens, seed=12 + D)
    _share(case, list(range(40)), 512)
    _share(case, list(range(40, 56)), 640)
    _run(case, oracle, ([0, 40, 56], [512, 640], 40, 640))


def test_mismatch_falls_back(oracle):
    """A member whose table differs inside the prefix, a group whose first member is
    shorter than the prefix and a group whose prefix is not whole blocks are all
    decoded on their own: same result, PREFIX_MISMATCH raised."""
    import paged_kv_cache_197_gb300 as pa

    lens = [600, 700, 800, 100, 500, 600, 400, 410]
    case = workloads.build_case("pfx-bad", S=len(lens), Hq=16, Hkv=4, D=128, bs=16,
                                context_lens=lens, seed=13)
    _share(case, [0, 1, 2], 256)
    case.block_tables[2, 5] = case.block_tables[2, 20]  # member 2 breaks the prefix
    _share(case, [3, 4, 5], 96)                          # lead holds 100 tokens only
    _share(case, [6, 7], 256)
    groups = ([0, 3, 6, 8], [256, 160, 200], 3, 256)     # 160 > lead's 100; 200 % 16 != 0
    _run(case, oracle, groups, expect_flag=pa.PA_FLAG_PREFIX_MISMATCH)


def test_no_groups_matches_decode(oracle):
    """With no group the path is the ordinary decode of every sequence."""
    lens = [1, 17, 500, 4100, 9000]
    case = workloads.build_case("pfx-none", S=len(lens), Hq=8, Hkv=2, D=128, bs=16,
                                context_lens=lens, seed=14)
    _run(case, oracle, ([0], [], 1, 0))


def test_rejects_unsupported():
    """Host-side checks: an 8-bit cache without scales, prefix bounds that are not whole
    blocks, and a short workspace are refused before anything is queued."""
    import paged_kv_cache_197_gb300 as pa

    case = workloads.build_case("pfx-rej", S=2, Hq=4, Hkv=4, D=64, bs=16, context_lens=[40, 40],
                                seed=15).to(DEV)
    out = torch.empty_like(case.q)
    gs = torch.tensor([0, 2], dtype=torch.int32, device=DEV)
    gp = torch.tensor([32], dtype=torch.int32, device=DEV)
    i8 = torch.zeros(case.k_pool.shape, dtype=torch.int8, device=DEV)
    with pytest.raises(ValueError):  # an int8 cache without its scales
        pa.pa_decode_shared_prefix(out, case.q, i8, i8, case.block_tables, case.context_lens,
                                   case.scale, 40, gs, gp, 2, 32)
    with pytest.raises(pa.PagedAttentionError):
        pa.pa_decode_shared_prefix(out, case.q, case.k_pool, case.v_pool, case.block_tables,
                                   case.context_lens, case.scale, 40, gs, gp, 2, 24)
    small = torch.empty(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(pa.PagedAttentionError):
        pa.pa_decode_shared_prefix(out, case.q, case.k_pool, case.v_pool, case.block_tables,
                                   case.context_lens, case.scale, 40, gs, gp, 2, 32,
                                   workspace=small)
    torch.cuda.synchronize()


@pytest.mark.slow
def test_full_prefix_workload_sampled(oracle):
    """The 50-sequence, 2000-token shared-prompt workload at full size through the
    prefix path, every sequence's output checked on a sample of sequences."""
    case = workloads.prefix(device="cpu", poison=True)
    prefix = case.meta["prefix_tokens"]
    got = helpers.gpu_step(case, DEV, groups=([0, case.S], [prefix], case.S, prefix))
    assert got["flag"] == 0
    caches = helpers.oracle_caches(case, oracle)
    seqs = [0, 7, 23, 49]
    ref = helpers.oracle_out(case, oracle, caches, seqs)
    helpers.compare(got["out"][torch.as_tensor(seqs, device=DEV)], ref, "bf16")


def test_graph_capture_replays():
    """The shared-prefix call captured in a CUDA graph -- its side-stream fork and join
    become graph edges -- replays to the same bits as the eager call."""
    import paged_kv_cache_197_gb300 as pa

    prefix = 21 * 32
    lens = [prefix + o for o in (3, 40, 300, 900)]
    case = workloads.build_case("pfx-graph", S=4, Hq=32, Hkv=8, D=128, bs=16, context_lens=lens,
                                seed=16, prefix_tokens=prefix, poison=False).to(DEV)
    gs = torch.tensor([0, 4], dtype=torch.int32, device=DEV)
    gp = torch.tensor([prefix], dtype=torch.int32, device=DEV)
    max_ctx = max(lens)
    n = pa.pa_decode_shared_prefix_workspace_size(4, 32, 8, 128, 16, pa.PA_KV_BF16, max_ctx, 4, prefix)
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    call = lambda out: pa.pa_decode_shared_prefix(  # noqa: E731
        out, case.q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, case.scale,
        max_ctx, gs, gp, 4, prefix, workspace=ws)
    eager = torch.empty_like(case.q)
    call(eager)  # the first call on a device creates the side stream, outside the capture
    torch.cuda.synchronize()
    replay = torch.full_like(case.q, float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(replay)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager, replay)
