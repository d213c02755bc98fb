"""GPU parity: the CUDA library, called through its C ABI, against the CPU oracle on the
same seeded inputs.  Append, quantise-append and copy are compared bit for bit; decode
output element by element within the stated tolerances (helpers.py)."""
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


def _check_case(case, orc, seqs=None):
    got = helpers.gpu_step(case, DEV)
    caches = helpers.oracle_caches(case, orc)
    kc, vc, ks, vs = caches
    # append / quantise / COW copy: bit-exact
    if case.kv_dtype == "bf16":
        assert np.array_equal(helpers.bits(got["k_cache"]), kc)
        assert np.array_equal(helpers.bits(got["v_cache"]), vc)
    else:
        assert np.array_equal(got["k_cache"].cpu().numpy(), kc)
        assert np.array_equal(got["v_cache"].cpu().numpy(), vc)
        assert np.array_equal(got["k_scale"].cpu().numpy().view(np.uint32), ks.view(np.uint32))
        assert np.array_equal(got["v_scale"].cpu().numpy().view(np.uint32), vs.view(np.uint32))
    assert got["flag"] == 0
    ref = helpers.oracle_out(case, orc, caches, seqs)
    out = got["out"] if seqs is None else got["out"][torch.as_tensor(seqs, device=DEV)]
    return helpers.compare(out, ref, case.kv_dtype)


def test_tiny(oracle):
    _check_case(workloads.tiny(), oracle)


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8", "fp8"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (16, 2), (20, 2), (32, 2)])
def test_shapes(oracle, kv_dtype, D, bs, Hq, Hkv):
    """Several tiles, split partitions and ragged tails; G = 1, 4, 8, 10 and 16."""
    lens = [1, 15, 16, 17, 100, 511, 512, 513, 1300, 2100]
    case = workloads.build_case(f"shape-{kv_dtype}-{D}-{bs}-{Hq}-{Hkv}", S=len(lens), Hq=Hq,
                                Hkv=Hkv, D=D, bs=bs, context_lens=lens, seed=D + bs + Hq,
                                kv_dtype=kv_dtype, pool_blocks=None)
    _check_case(case, oracle)


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8", "fp8"])
def test_prefix_and_cow(oracle, kv_dtype):
    """Sequences sharing a prefix's physical blocks, each with a copy-on-write last block."""
    own = [64, 65, 80, 130, 511, 512]
    lens = [640 + o for o in own]
    case = workloads.build_case(f"prefix-small-{kv_dtype}", S=len(lens), Hq=16, Hkv=4, D=128,
                                bs=16 if kv_dtype == "bf16" else 32, context_lens=lens, seed=31,
                                kv_dtype=kv_dtype, prefix_tokens=640, cow=True)
    _check_case(case, oracle)


def test_empty_and_single_token(oracle):
    """Context 0 gives zeros; context 1 gives the appended value row (rounded to bf16)."""
    case = workloads.build_case("edge", S=4, Hq=8, Hkv=8, D=128, bs=16, context_lens=[0, 1, 0, 2],
                                seed=5)
    got = helpers.gpu_step(case, DEV)
    out = got["out"].float().cpu()
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    assert torch.equal(got["out"][1].cpu(), case.new_value[1])
    _check_case(case, oracle)


def test_block_permutation_bit_identical():
    """The GPU result depends on logical order only: moving blocks changes no bit."""
    case = workloads.build_case("perm", S=6, Hq=16, Hkv=2, D=128, bs=16,
                                context_lens=[33, 600, 1024, 7, 1500, 260], seed=12, poison=False)
    a = helpers.gpu_step(case, DEV)["out"]
    pi = torch.randperm(case.N, generator=torch.Generator().manual_seed(3))
    moved = workloads.PagedCase(**{**case.__dict__})
    moved.k_pool = torch.empty_like(case.k_pool)
    moved.v_pool = torch.empty_like(case.v_pool)
    moved.k_pool[pi] = case.k_pool
    moved.v_pool[pi] = case.v_pool
    moved.block_tables = pi[case.block_tables.long()].to(torch.int32)
    slots = case.slot_mapping.clone()
    blk = slots // case.bs
    moved.slot_mapping = pi[blk] * case.bs + slots % case.bs
    b = helpers.gpu_step(moved, DEV)["out"]
    assert torch.equal(a, b)


def test_error_flags_and_skips():
    """Out-of-range slots, block ids and context lengths are skipped and flagged, never
    read or written."""
    import paged_kv_cache_197_gb300 as pa

    case = workloads.build_case("flags", S=3, Hq=4, Hkv=4, D=128, bs=16, context_lens=[40, 40, 40],
                                seed=8, poison=False).to(DEV)
    k, v = case.k_pool.clone(), case.v_pool.clone()
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    bad_slots = torch.tensor([case.N * 16 + 5, -1, 3], dtype=torch.int64, device=DEV)
    pa.pa_reshape_and_cache(case.new_key, case.new_value, k, v, bad_slots, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == pa.PA_FLAG_SLOT_OUT_OF_RANGE
    expect = case.k_pool.clone()
    expect[0, :, 3, :] = case.new_key[2]
    assert torch.equal(k, expect)
    # a block id beyond the pool: that block is skipped, the rest still attended
    tables = case.block_tables.clone()
    tables[1, 1] = case.N + 100
    out = torch.empty_like(case.q)
    ws = pa.decode_workspace(case.q, k, 40)
    flag.zero_()
    pa.pa_decode(out, case.q, k, v, tables, case.context_lens, case.scale, 40, workspace=ws,
                 err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == pa.PA_FLAG_BLOCK_OUT_OF_RANGE
    assert torch.isfinite(out.float()).all()
    # a context longer than max_context_len is clamped and flagged
    flag.zero_()
    pa.pa_decode(out, case.q, k, v, case.block_tables, case.context_lens, case.scale, 33,
                 workspace=ws, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == pa.PA_FLAG_CONTEXT_OUT_OF_RANGE


def test_block_manager_plan_on_gpu(oracle):
    """A prefix reuse, a fork and a copy-on-write planned by the host block manager and
    executed by the CUDA library match the oracle executing the same plan."""
    import paged_kv_cache_197_gb300 as pa

    rng = np.random.default_rng(5)
    bs, Hkv, Hq, D, N = 16, 4, 16, 128, 96
    bm = pa.BlockManager(N, bs)
    kc_h = np.zeros((N, Hkv, bs, D), dtype=np.uint16)
    vc_h = np.zeros_like(kc_h)
    kc = torch.zeros((N, Hkv, bs, D), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)

    def write(sid, n, tokens=None):
        slots, pairs = bm.append(sid, n=n, tokens=tokens)
        if pairs:
            oracle.copy_blocks(kc_h, vc_h, np.array(pairs, dtype=np.int64))
            pa.pa_copy_blocks(kc, vc, pairs)
        k = helpers.bits(torch.randn((n, Hkv, D)).to(torch.bfloat16))
        v = helpers.bits(torch.randn((n, Hkv, D)).to(torch.bfloat16))
        sl = np.array(slots, dtype=np.int64)
        oracle.reshape_and_cache(k, v, kc_h, vc_h, sl, bs)
        kt = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).to(DEV)
        vt = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).to(DEV)
        pa.pa_reshape_and_cache(kt, vt, kc, vc, torch.from_numpy(sl).to(DEV))

    prompt = list(range(600))
    bm.add_sequence(0, prompt)
    write(0, 600, prompt)
    write(0, 9)
    assert bm.add_sequence(1, prompt) == 592
    write(1, 20)
    bm.fork(0, 2)
    write(2, 30)
    write(0, 1)
    tables = [bm.block_table(s) for s in (0, 1, 2)]
    M = max(len(t) for t, _ in tables)
    tab = np.zeros((3, M), dtype=np.int32)
    for i, (t, _) in enumerate(tables):
        tab[i, :len(t)] = t
    lens = np.array([n for _, n in tables], dtype=np.int32)
    q = helpers.bits(torch.randn((3, Hq, D)).to(torch.bfloat16))
    torch.cuda.synchronize()
    assert np.array_equal(helpers.bits(kc), kc_h) and np.array_equal(helpers.bits(vc), vc_h)
    ref = oracle.paged_attention(q, kc_h, vc_h, tab, lens, 0.088)
    qt = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(DEV)
    out = torch.empty_like(qt)
    tab_t, lens_t = torch.from_numpy(tab).to(DEV), torch.from_numpy(lens).to(DEV)
    max_ctx = int(lens.max())
    ws = pa.decode_workspace(qt, kc, max_ctx)
    pa.pa_decode(out, qt, kc, vc, tab_t, lens_t, 0.088, max_ctx, workspace=ws)
    torch.cuda.synchronize()
    helpers.compare(out, ref, "bf16")
    del rng


def test_copy_blocks_rejects_overlap():
    import paged_kv_cache_197_gb300 as pa

    k = torch.zeros((8, 2, 16, 64), dtype=torch.bfloat16, device=DEV)
    v = torch.zeros_like(k)
    with pytest.raises(pa.PagedAttentionError):
        pa.pa_copy_blocks(k, v, [[1, 2], [2, 3]])
    with pytest.raises(pa.PagedAttentionError):
        pa.pa_copy_blocks(k, v, [[1, 2], [3, 2]])
    with pytest.raises(pa.PagedAttentionError):
        pa.pa_copy_blocks(k, v, [[1, 8]])


# ------------------------------------------------------------------ full-size configs
FULL = {
    "mha13b": (workloads.mha13b, [0, 1, 17, 42, 63]),
    "gqa70b": (workloads.gqa70b, [0, 7, 19]),
    "prefix": (workloads.prefix, [0, 1, 25, 49]),
    "int8": (workloads.int8, [0, 3, 100, 200, 255]),
    "fp8": (workloads.fp8, [0, 5, 128, 255]),
}


@pytest.mark.slow
@pytest.mark.parametrize("name", list(FULL))
def test_full_size_sampled(oracle, name):
    """The benchmark workloads at full size, in the launch configuration the benchmark
    times; the oracle checks a sample of sequences (all their heads), and append, copy
    and quantisation are compared over the whole pool."""
    make, seqs = FULL[name]
    case = make(device=DEV, poison=(name not in ("int8", "fp8")))
    # the sample always holds the longest and the shortest sequence
    lens = case.context_lens.cpu()
    seqs = sorted(set(seqs) | {int(lens.argmax()), int(lens.argmin())})
    _check_case(case, oracle, seqs)
