"""Host-side bookkeeping of the seeded workloads: tables, slots, sharing, COW pairs and
byte accounting."""
import numpy as np
import pytest
import torch

import workloads


def test_slots_follow_tables(oracle):
    case = workloads.build_case("w", S=5, Hq=4, Hkv=2, D=64, bs=16, context_lens=[1, 16, 17, 90, 0],
                                seed=1)
    tabs = case.block_tables.numpy()
    for s in range(case.S):
        c = int(case.context_lens[s])
        if c == 0:
            assert case.slot_mapping[s] == -1
        else:
            assert int(case.slot_mapping[s]) == oracle.slot(tabs[s], c - 1, case.bs)


def test_tiny_shape():
    case = workloads.tiny()
    assert case.context_lens.tolist() == [1, 17, 40, 100]
    assert (case.S, case.Hq, case.Hkv, case.D, case.bs, case.N) == (4, 2, 2, 64, 16, 32)
    used = [int(case.block_tables[s, j]) for s in range(4)
            for j in range(workloads.blocks_needed(int(case.context_lens[s]), 16))]
    assert len(used) == 13 and len(set(used)) == 13 and max(used) < 32


def test_prefix_sharing_and_cow():
    case = workloads.build_case("p", S=6, Hq=8, Hkv=2, D=64, bs=16, context_lens=[200 + i for i in range(6)],
                                seed=2, prefix_tokens=160, cow=True)
    tabs = case.block_tables
    content = case.meta["content_tables"]
    assert torch.equal(tabs[:, :10], tabs[:1, :10].expand(6, 10))  # shared prefix blocks
    pairs = case.cow_pairs.tolist()
    assert len(pairs) == 6 and len({d for _, d in pairs}) == 6
    srcs = {s for s, _ in pairs}
    for s, (src, dst) in enumerate(pairs):
        last = workloads.blocks_needed(int(case.context_lens[s]), 16) - 1
        assert int(tabs[s, last]) == dst and int(content[s, last]) == src
        assert dst not in srcs
    # private blocks are not shared
    private = [int(content[s, j]) for s in range(6)
               for j in range(10, workloads.blocks_needed(int(case.context_lens[s]), 16))]
    assert len(private) == len(set(private))


def test_poison_marks_only_unused_slots():
    case = workloads.build_case("q", S=3, Hq=2, Hkv=2, D=64, bs=16, context_lens=[5, 33, 16], seed=3)
    valid = workloads.valid_slot_mask(case.block_tables, case.context_lens - 1, 16, case.N)
    assert int(valid.sum()) == 4 + 32 + 15
    pool = case.k_pool.permute(0, 2, 1, 3)
    assert torch.isnan(pool[~valid].float()).all()
    assert torch.isfinite(pool[valid].float()).all()


def test_int8_lengths_distribution():
    lens = np.array(workloads.int8_lengths(256, 4))
    assert lens.min() >= 128 and lens.max() <= 32768
    assert 1500 < np.exp(np.log(lens).mean()) < 2800  # geometric mean near sqrt(128*32768) = 2048


def test_byte_accounting():
    case = workloads.build_case("b", S=2, Hq=4, Hkv=2, D=64, bs=16, context_lens=[10, 20], seed=4)
    kv = 30 * 2 * 64 * 2 * 2
    qo = 2 * 2 * 4 * 64 * 2
    tables = (1 + 2) * 4 + 2 * 4
    assert workloads.decode_algorithmic_bytes(case) == kv + qo + tables
    shared = workloads.build_case("s", S=3, Hq=4, Hkv=2, D=64, bs=16, context_lens=[40, 40, 40],
                                  seed=5, prefix_tokens=32)
    logical = workloads.decode_algorithmic_bytes(shared)
    unique = workloads.decode_algorithmic_bytes(shared, unique_blocks=True)
    assert logical - unique == 2 * 32 * (2 * 64 * 2 * 2)


@pytest.mark.parametrize("make", [workloads.mha13b, workloads.prefix])
def test_paged_waste_below_page_claim(make):
    """Paging wastes under 4% of the reserved slots (ia-vox-magazine, "PagedAttention : la
    revolution de l'allocation memoire"; gotburnout.io block-table figure caption), while a
    contiguous max-length reservation wastes a large share."""
    case = make(poison=False)
    f = workloads.fragmentation(case, max_len=2048 if case.name == "mha13b" else 4096)
    assert f["paged_waste"] < 0.04
    assert f["contiguous_waste"] > 0.3
