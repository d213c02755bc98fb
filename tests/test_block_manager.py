"""Host block manager (include/pa_blocks.h): pool, block tables, copy-on-write, prefix
cache, LRU eviction.  Checked against a small Python model of the documented policy
on random operation sequences, against what the pages state, and end to end through
the CPU oracle."""
from __future__ import annotations

import random
from collections import OrderedDict

import numpy as np
import pytest

import pins


@pytest.fixture(scope="module")
def pa():
    from paged_kv_cache_197_gb300 import _build

    _build.build()
    import paged_kv_cache_197_gb300 as pa_mod

    return pa_mod


# ------------------------------------------------------------ reference model
class BlockModel:
    """The policy of pa_blocks.h in plain Python: LIFO free list, LRU of released
    registered blocks, registry keyed by (parent node, block token ids)."""

    def __init__(self, N: int, bs: int):
        self.N, self.bs = N, bs
        self.free = list(range(N - 1, -1, -1))
        self.ref = [0] * N
        self.fill = [0] * N
        self.node = [0] * N
        self.key = [None] * N
        self.lru = OrderedDict()
        self.registry = {}
        self.seqs = {}
        self.next_node = 1
        self.cow = self.lookups = self.hits = self.evictions = 0

    def available(self):
        return len(self.free) + len(self.lru)

    def take(self):
        if self.free:
            b = self.free.pop()
        else:
            b, _ = self.lru.popitem(last=False)
            if self.node[b]:
                if self.registry.get(self.key[b]) == b:
                    del self.registry[self.key[b]]
                self.node[b], self.key[b] = 0, None
            self.evictions += 1
        self.ref[b], self.fill[b] = 1, 0
        return b

    def hold(self, b):
        self.lru.pop(b, None)
        self.ref[b] += 1

    def release(self, b):
        self.ref[b] -= 1
        if self.ref[b] == 0:
            if self.node[b]:
                self.lru[b] = True
            else:
                self.free.append(b)

    def register_full(self, s):
        b = s["blocks"][-1]
        k = (s["chain"], tuple(s["pending"]))
        if k in self.registry:
            s["chain"] = self.node[self.registry[k]]
        elif self.node[b] == 0:
            self.node[b], self.key[b] = self.next_node, k
            self.next_node += 1
            self.registry[k] = b
            s["chain"] = self.node[b]
        else:
            s["chain"] = self.node[b]
        s["pending"] = []

    def add_sequence(self, sid, prompt=None):
        s = {"blocks": [], "len": 0, "chain": 0, "ids": True, "pending": []}
        prompt = prompt or []
        for i in range(0, len(prompt) - self.bs + 1, self.bs):
            self.lookups += 1
            b = self.registry.get((s["chain"], tuple(prompt[i:i + self.bs])))
            if b is None:
                break
            self.hold(b)
            s["blocks"].append(b)
            s["len"] += self.bs
            s["chain"] = self.node[b]
            self.hits += 1
        self.seqs[sid] = s
        return s["len"]

    def append(self, sid, n=None, tokens=None):
        s = self.seqs[sid]
        if tokens is not None:
            n = len(tokens)
        bs = self.bs
        need_cow = s["len"] % bs != 0 and self.ref[s["blocks"][-1]] > 1
        first_new = 0 if s["len"] % bs == 0 else bs - s["len"] % bs
        crossings = -(-(n - first_new) // bs) if n > first_new else 0
        if crossings + need_cow > self.available():
            raise MemoryError
        pairs = []
        if need_cow:
            src = s["blocks"][-1]
            dst = self.take()
            self.fill[dst] = s["len"] % bs
            self.release(src)
            s["blocks"][-1] = dst
            pairs.append((src, dst))
            self.cow += 1
        if tokens is None:
            s["ids"] = False
        slots = []
        for i in range(n):
            off = s["len"] % bs
            if off == 0:
                s["blocks"].append(self.take())
            b = s["blocks"][-1]
            slots.append(b * bs + off)
            self.fill[b] = max(self.fill[b], off + 1)
            s["len"] += 1
            if s["ids"]:
                s["pending"].append(tokens[i])
                if s["len"] % bs == 0:
                    self.register_full(s)
        return slots, pairs

    def fork(self, parent, child):
        p = self.seqs[parent]
        self.seqs[child] = {"blocks": list(p["blocks"]), "len": p["len"], "chain": p["chain"],
                            "ids": p["ids"], "pending": list(p["pending"])}
        for b in p["blocks"]:
            self.hold(b)

    def free_seq(self, sid):
        for b in reversed(self.seqs[sid]["blocks"]):
            self.release(b)
        del self.seqs[sid]

    def stats(self):
        used = [b for b in range(self.N) if self.ref[b] > 0]
        return {"num_blocks": self.N, "free_blocks": len(self.free), "cached_blocks": len(self.lru),
                "used_blocks": len(used), "used_slots": sum(self.fill[b] for b in used),
                "cow_copies": self.cow, "prefix_lookup_blocks": self.lookups,
                "prefix_hit_blocks": self.hits, "evictions": self.evictions}


# ------------------------------------------------------------------ random model
@pytest.mark.parametrize("seed", range(6))
def test_matches_reference_model(pa, seed):
    rng = random.Random(seed)
    N, bs = rng.choice([(24, 4), (64, 16), (40, 8)])
    bm, model = pa.BlockManager(N, bs), BlockModel(N, bs)
    vocab = [rng.randrange(3) for _ in range(8)]  # few distinct prompts -> cache hits
    live, next_id = [], 0
    for _ in range(400):
        op = rng.random()
        if op < 0.25 or not live:
            prompt = [vocab[(i * 7 + rng.randrange(2)) % len(vocab)] for i in range(rng.randrange(0, 3 * bs))]
            got, want = bm.add_sequence(next_id, prompt), model.add_sequence(next_id, prompt)
            assert got == want
            live.append(next_id)
            next_id += 1
        elif op < 0.65:
            sid = rng.choice(live)
            n = rng.randrange(1, 2 * bs)
            toks = [rng.randrange(3) for _ in range(n)] if rng.random() < 0.8 else None
            try:
                want = model.append(sid, n=n, tokens=toks)
            except MemoryError:
                with pytest.raises(pa.PagedAttentionError) as e:
                    bm.append(sid, n=n, tokens=toks)
                assert e.value.status == pa.PA_ERR_NO_SPACE
                continue
            assert bm.append(sid, n=n, tokens=toks) == want
        elif op < 0.75:
            parent = rng.choice(live)
            bm.fork(parent, next_id)
            model.fork(parent, next_id)
            live.append(next_id)
            next_id += 1
        else:
            sid = live.pop(rng.randrange(len(live)))
            bm.free(sid)
            model.free_seq(sid)
        for sid in live:
            assert bm.block_table(sid) == (model.seqs[sid]["blocks"], model.seqs[sid]["len"])
        assert bm.stats() == model.stats()
    for sid in live:
        bm.free(sid)
    st = bm.stats()
    assert st["used_blocks"] == 0 and st["free_blocks"] + st["cached_blocks"] == N


# -------------------------------------------------------- what the pages state
def test_figure_mapping(pa, oracle):
    """gotburnout.io block-table figure: a request whose logical blocks 0, 1, 2 land in
    physical blocks 7, 2 and 11; its tokens' slots follow the table."""
    import json

    fig = json.loads((pins.GOLDEN / "block_table_figure.json").read_text())
    bs = fig["block_size"]
    bm = pa.BlockManager(12, bs)
    for sid in range(12):  # one block each: sequence i holds physical block i
        bm.add_sequence(sid)
        bm.append(sid, n=bs)
        assert bm.block_table(sid) == ([sid], bs)
    for sid in (11, 2, 7):  # released in this order, block 7 is reused first
        bm.free(sid)
    bm.add_sequence(99)
    slots, _ = bm.append(99, n=48)
    table, n = bm.block_table(99)
    assert table == fig["block_table"] and n == 48
    t = np.array(table, dtype=np.int32)
    assert slots == [oracle.slot(t, p, bs) for p in range(48)]
    for j, (lo, hi) in enumerate(fig["logical_token_ranges"]):
        assert {slots[p] // bs for p in range(lo, hi + 1)} == {fig["block_table"][j]}


def test_free_on_cancel_returns_every_block(pa):
    """gotburnout.io section 4: a cancelled request must give its pages back at once."""
    bm = pa.BlockManager(64, 16)
    for sid in range(5):
        bm.add_sequence(sid)
        bm.append(sid, n=50 + 37 * sid)
    bm.fork(3, 9)
    bm.append(9, n=5)
    assert bm.stats()["free_blocks"] < 64
    for sid in (0, 1, 2, 3, 4, 9):
        bm.free(sid)
    st = bm.stats()
    assert st["free_blocks"] == 64 and st["used_blocks"] == 0 and st["cached_blocks"] == 0


def test_copy_on_write_on_first_own_write(pa):
    """gotburnout.io section 3.01: shared pages are copied only when a sequence starts
    writing its own tokens; the other holder keeps the original."""
    bm = pa.BlockManager(32, 16)
    bm.add_sequence(0)
    bm.append(0, n=20)  # blocks [0, 1], block 1 half full
    bm.fork(0, 1)
    t0, _ = bm.block_table(0)
    slots, pairs = bm.append(1, n=1)
    t1, n1 = bm.block_table(1)
    assert pairs == [(t0[1], t1[1])] and t1[0] == t0[0] and t1[1] != t0[1] and n1 == 21
    assert slots == [t1[1] * 16 + 4]
    _, pairs0 = bm.append(0, n=1)  # the parent now holds block 1 alone: no copy
    assert pairs0 == [] and bm.block_table(0)[0] == t0
    # a full last block is never copied: the next token opens a new block
    bm.add_sequence(2)
    bm.append(2, n=32)
    bm.fork(2, 3)
    _, pairs = bm.append(3, n=1)
    assert pairs == []


def test_branching_saves_three_quarters(pa):
    """gotburnout.io section 3.02: four branches of one context keep a single copy of
    it, saving up to 75% against four separate caches."""
    bs, ctx = 16, 4000
    bm = pa.BlockManager(2000, bs)
    bm.add_sequence(0)
    bm.append(0, n=ctx)
    for b in range(1, 4):
        bm.fork(0, b)
    for b in range(4):
        bm.append(b, n=16)
    shared = bm.stats()["used_blocks"]
    separate = 4 * ((ctx + 16 + bs - 1) // bs)
    saving = 1 - shared / separate
    assert 0.74 < saving <= 0.75


def test_shared_prompt_stored_once(pa):
    """ia-vox-magazine, "PagedAttention": two requests sharing a 2000-token system prompt
    store it only once; prefix caching finds it by exact token match (fabienvernieres,
    "le prefix caching")."""
    rng = random.Random(1)
    prompt = [rng.randrange(32000) for _ in range(2000)]
    bm = pa.BlockManager(400, 16)
    assert bm.add_sequence(0, prompt) == 0
    bm.append(0, tokens=prompt)
    used_one = bm.stats()["used_blocks"]
    assert bm.add_sequence(1, prompt) == 2000  # 125 full blocks found
    assert bm.stats()["used_blocks"] == used_one
    t0, _ = bm.block_table(0)
    t1, n1 = bm.block_table(1)
    assert t1 == t0 and n1 == 2000
    # one token different at position 1000: only the first 62 full blocks match
    other = list(prompt)
    other[1000] += 1
    assert bm.add_sequence(2, other) == 62 * 16
    st = bm.stats()
    assert st["prefix_hit_blocks"] == 125 + 62


def test_cached_prefix_survives_until_evicted(pa):
    """fabienvernieres, "Faire de la place : l'eviction": released prefix blocks stay
    reusable and are reclaimed least-recently-used first, tail blocks before heads."""
    bs = 4
    bm = pa.BlockManager(6, bs)
    p = list(range(12))  # 3 full blocks
    bm.add_sequence(0, p)
    bm.append(0, tokens=p)
    bm.free(0)
    st = bm.stats()
    assert st["cached_blocks"] == 3 and st["free_blocks"] == 3
    assert bm.add_sequence(1, p) == 12
    bm.free(1)
    bm.add_sequence(2)
    bm.append(2, n=4 * bs)  # needs 4 blocks: 3 free + evicts the oldest cached one
    assert bm.stats()["evictions"] == 1
    assert bm.add_sequence(3, p) == 8  # the tail block went first; the head two remain


def test_paged_waste_under_four_percent(pa):
    """ia-vox-magazine: paging brings KV waste down to about 4% (from 60-80%)."""
    rng = random.Random(3)
    lens = [rng.randrange(200, 2049) for _ in range(64)]
    bm = pa.BlockManager(sum((n + 15) // 16 for n in lens), 16)
    for sid, n in enumerate(lens):
        bm.add_sequence(sid)
        bm.append(sid, n=n)
    st = bm.stats()
    waste = 1 - st["used_slots"] / (st["used_blocks"] * 16)
    assert waste < 0.04
    assert 1 - sum(lens) / (64 * 2048) > 0.4  # contiguous max-length reservation


def test_errors_leave_state_unchanged(pa):
    bm = pa.BlockManager(4, 16)
    bm.add_sequence(0)
    bm.append(0, n=60)
    before = bm.stats(), bm.block_table(0)
    with pytest.raises(pa.PagedAttentionError) as e:
        bm.append(0, n=10)  # needs a 5th block
    assert e.value.status == pa.PA_ERR_NO_SPACE
    assert (bm.stats(), bm.block_table(0)) == before
    with pytest.raises(pa.PagedAttentionError):
        bm.add_sequence(0)
    with pytest.raises(pa.PagedAttentionError):
        bm.append(7, n=1)
    with pytest.raises(pa.PagedAttentionError):
        bm.fork(7, 8)


# ------------------------------------------------------- end to end, on the CPU
def test_manager_tables_drive_the_oracle(pa, oracle):
    """Prefix reuse, a fork and copy-on-write planned by the manager, executed by the
    oracle's append and block copy: every sequence's paged attention equals attention
    over its own logical token rows."""
    rng = np.random.default_rng(0)
    bs, Hkv, Hq, D, N = 16, 2, 4, 16, 64
    bm = pa.BlockManager(N, bs)
    kc = np.zeros((N, Hkv, bs, D), dtype=np.uint16)
    vc = np.zeros_like(kc)
    rows = {}  # sequence -> list of (k_row, v_row) in logical order

    def write(sid, n, tokens=None):
        slots, pairs = bm.append(sid, n=n, tokens=tokens)
        if pairs:
            oracle.copy_blocks(kc, vc, np.array(pairs, dtype=np.int64))
        k = pins.to_bf16_bits(rng.standard_normal((n, Hkv, D)))
        v = pins.to_bf16_bits(rng.standard_normal((n, Hkv, D)))
        assert oracle.reshape_and_cache(k, v, kc, vc, np.array(slots, dtype=np.int64), bs) == 0
        rows.setdefault(sid, []).extend(zip(k, v))

    prompt = list(range(48))
    bm.add_sequence(0, prompt)
    write(0, 48, prompt)
    write(0, 5)
    cached = bm.add_sequence(1, prompt)  # reuses the 3 prompt blocks
    assert cached == 48
    rows[1] = list(rows[0][:48])
    write(1, 7)
    bm.fork(0, 2)  # shares 0's partial last block
    rows[2] = list(rows[0])
    write(2, 3)  # copy-on-write
    write(0, 2)
    sids = [0, 1, 2]
    tables = [bm.block_table(s) for s in sids]
    M = max(len(t) for t, _ in tables)
    tab = np.zeros((3, M), dtype=np.int32)
    for i, (t, _) in enumerate(tables):
        tab[i, :len(t)] = t
    lens = np.array([n for _, n in tables], dtype=np.int32)
    q = pins.to_bf16_bits(rng.standard_normal((3, Hq, D)))
    out = oracle.paged_attention(q, kc, vc, tab, lens, 0.25)
    G = Hq // Hkv
    for i, sid in enumerate(sids):
        assert lens[i] == len(rows[sid])
        for h in range(Hq):
            K = np.array([pins.bf16_bits_to_f64(r[0][h // G]) for r in rows[sid]])
            V = np.array([pins.bf16_bits_to_f64(r[1][h // G]) for r in rows[sid]])
            sc = 0.25 * (K @ pins.bf16_bits_to_f64(q[i, h]))
            w = np.exp(sc - sc.max())
            w /= w.sum()
            assert np.allclose(out[i, h], w @ V, rtol=1e-12, atol=1e-13)
