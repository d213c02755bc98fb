"""Seeded synthetic inputs for the paged KV-cache decode path.

Both the GPU library (through the tests and the benchmark) and the CPU oracle
consume what this module makes; it holds none of the method's arithmetic.  It
draws random numbers and lays out the caller-side bookkeeping a block manager
would hold: context lengths, a random placement of each sequence's logical blocks
in the physical pool, block tables, the slot of each new token, and the
copy-on-write pairs.

Workloads (shapes and distributions of the benchmark configurations):
  tiny    4 sequences, context lengths {1, 17, 40, 100}, 2 query / 2 kv heads,
          head_dim 64, block size 16, pool of 32 blocks, scale 1/8.
  mha13b  Llama-2-13B-shaped layer: 64 sequences, 40 / 40 heads, head_dim 128,
          block size 16, context lengths uniform in [200, 2048].
  gqa70b  Llama-3-70B-shaped layer: 20 sequences of 8000 tokens, 64 / 8 heads,
          head_dim 128, block size 16.
  prefix  50 sequences sharing one 2000-token prefix (the same 125 physical blocks)
          plus 64..512 own tokens each, 32 / 8 heads, head_dim 128, block size 16,
          one copy-on-write block pair per sequence.
  int8    Llama-3-8B-shaped layer with an int8 cache: 256 sequences, 32 / 8 heads,
          head_dim 128, block size 32, context lengths log-uniform in [128, 32768].
  fp8     the int8 workload's shape with an fp8 (e4m3) cache.
All values (queries, cached keys and values, the new token's key and value) are
N(0, 1) rounded to bf16.  context_lens count the token appended in this step: the
new token sits at position context_len - 1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BF16_NAN_BITS = 0x7FC0


@dataclass
class PagedCase:
    name: str
    S: int
    Hq: int
    Hkv: int
    D: int
    bs: int
    N: int
    M: int
    kv_dtype: str  # "bf16", "int8" or "fp8"
    scale: float
    q: torch.Tensor  # [S][Hq][D] bf16
    k_pool: torch.Tensor  # [N][Hkv][bs][D] bf16 (int8 workloads: the bf16 source to quantise)
    v_pool: torch.Tensor
    block_tables: torch.Tensor  # [S][M] int32 (table used by this step's decode)
    context_lens: torch.Tensor  # [S] int32, including the new token
    new_key: torch.Tensor  # [S][Hkv][D] bf16, the token at position context_len - 1
    new_value: torch.Tensor
    slot_mapping: torch.Tensor  # [S] int64, slot of the new token
    cow_pairs: torch.Tensor  # [n][2] int64 (src, dst) physical blocks; n may be 0
    shared_prefix_blocks: int = 0
    meta: dict = field(default_factory=dict)
    # multi-token steps: [S + 1] int32 row offsets of each sequence's new tokens in q,
    # new_key, new_value and slot_mapping (then [T] rows instead of [S]); None = decode
    query_start: torch.Tensor | None = None

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def to(self, device) -> "PagedCase":
        moved = {}
        for k, v in self.__dict__.items():
            moved[k] = v.to(device) if isinstance(v, torch.Tensor) else v
        return PagedCase(**moved)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, gen, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def blocks_needed(ctx: int, bs: int) -> int:
    return (ctx + bs - 1) // bs


def build_case(name: str, S: int, Hq: int, Hkv: int, D: int, bs: int, context_lens,
               seed: int, kv_dtype: str = "bf16", pool_blocks: int | None = None,
               prefix_tokens: int = 0, cow: bool = False, poison: bool = True,
               device="cpu", scale: float | None = None) -> PagedCase:
    """Make one seeded paged-decode case.

    Physical blocks are drawn from a random permutation of the pool; with
    ``prefix_tokens`` > 0 the first prefix_tokens // bs logical blocks of every
    sequence point at the same physical blocks.  With ``cow`` each sequence's
    last logical block gets a (src, dst) copy-on-write pair: the cache content is
    written into src, the decode table already points at dst.  With ``poison``
    every slot of a bf16 pool that holds no valid token is filled with bf16 NaN, so a
    kernel that reads past a context shows up in the results (int8 pools are quantised
    from a finite source; the tests poison their scales instead).
    """
    meta_gen = _gen(seed)  # small metadata always on the CPU generator
    ctx = torch.as_tensor(context_lens, dtype=torch.int64).clone()
    assert ctx.numel() == S and int(ctx.min()) >= 0
    if prefix_tokens:
        assert prefix_tokens % bs == 0 and int(ctx.min()) > prefix_tokens
    n_shared = prefix_tokens // bs
    nblk = [blocks_needed(int(c), bs) for c in ctx]
    M = max(1, max(nblk))
    private = [nb - n_shared for nb in nblk]
    n_cow = S if cow else 0
    used = n_shared + sum(private) + n_cow
    N = pool_blocks if pool_blocks is not None else used
    assert N >= used, f"pool of {N} blocks cannot hold {used}"
    perm = torch.randperm(N, generator=meta_gen).tolist()
    nxt = 0
    shared_ids = perm[nxt:nxt + n_shared]
    nxt += n_shared
    tables = torch.zeros((S, M), dtype=torch.int32)  # padding entries: block 0
    content_tables = torch.zeros((S, M), dtype=torch.int32)
    cow_pairs = []
    for s in range(S):
        own = perm[nxt:nxt + private[s]]
        nxt += private[s]
        row = shared_ids + own
        if row:
            tables[s, : len(row)] = torch.tensor(row, dtype=torch.int32)
            content_tables[s, : len(row)] = torch.tensor(row, dtype=torch.int32)
        if cow and nblk[s] > 0:
            dst = perm[nxt]
            nxt += 1
            src = row[-1]
            cow_pairs.append((src, dst))
            tables[s, nblk[s] - 1] = dst
    cow_t = torch.tensor(cow_pairs, dtype=torch.int64).reshape(-1, 2)

    big = _gen(seed + 1, device)
    q = _randn_bf16((S, Hq, D), big, device)
    k_pool = _randn_bf16((N, Hkv, bs, D), big, device)
    v_pool = _randn_bf16((N, Hkv, bs, D), big, device)
    new_key = _randn_bf16((S, Hkv, D), big, device)
    new_value = _randn_bf16((S, Hkv, D), big, device)

    # slot of the new token (position ctx - 1) through the decode-time table
    slots = torch.full((S,), -1, dtype=torch.int64)
    for s in range(S):
        c = int(ctx[s])
        if c > 0:
            pos = c - 1
            slots[s] = int(tables[s, pos // bs]) * bs + pos % bs

    if poison and kv_dtype == "bf16":  # quantised sources stay finite: tests poison their scales
        valid = valid_slot_mask(content_tables, ctx - 1, bs, N)  # tokens present before the append
        bad = ~valid.to(device)
        nan = torch.tensor(BF16_NAN_BITS, dtype=torch.int16).view(torch.bfloat16).item()
        for pool in (k_pool, v_pool):
            view = pool.permute(0, 2, 1, 3)  # [N][bs][Hkv][D]
            view[bad] = nan
    return PagedCase(name=name, S=S, Hq=Hq, Hkv=Hkv, D=D, bs=bs, N=N, M=M, kv_dtype=kv_dtype,
                     scale=scale if scale is not None else 1.0 / math.sqrt(D),
                     q=q, k_pool=k_pool, v_pool=v_pool, block_tables=tables.to(device),
                     context_lens=ctx.to(torch.int32).to(device), new_key=new_key,
                     new_value=new_value, slot_mapping=slots.to(device),
                     cow_pairs=cow_t.to(device), shared_prefix_blocks=n_shared,
                     meta={"seed": seed, "content_tables": content_tables,
                           "prefix_tokens": prefix_tokens})


def valid_slot_mask(tables: torch.Tensor, lengths: torch.Tensor, bs: int, N: int) -> torch.Tensor:
    """Boolean [N][bs]: True where a slot holds one of the first lengths[s] tokens of some
    sequence s, reached through tables[s]."""
    mask = torch.zeros((N, bs), dtype=torch.bool)
    for s in range(tables.shape[0]):
        n = int(lengths[s])
        if n <= 0:
            continue
        pos = torch.arange(n)
        blocks = tables[s, pos // bs].long()
        mask[blocks, pos % bs] = True
    return mask


def build_multi_case(name: str, S: int, Hq: int, Hkv: int, D: int, bs: int, context_lens,
                     query_lens, seed: int, pool_blocks: int | None = None, poison: bool = True,
                     device="cpu", row_offset: int = 0, extra_rows: int = 0,
                     kv_dtype: str = "bf16") -> PagedCase:
    """A multi-token step: sequence s brings query_lens[s] new tokens at positions
    context_lens[s] - query_lens[s] .. context_lens[s] - 1 (context_lens count them).
    q, new_key, new_value and slot_mapping hold T rows, sequence s owning rows
    query_start[s] .. query_start[s + 1] - 1; row_offset rows before the first
    sequence and extra_rows after the last belong to no sequence (their slots are -1).
    With ``poison`` every slot not holding one of the tokens before the new ones is
    bf16 NaN."""
    L = [int(x) for x in query_lens]
    ctx = [int(c) for c in context_lens]
    assert len(L) == S and all(0 <= l <= c for l, c in zip(L, ctx))
    case = build_case(name, S=S, Hq=Hq, Hkv=Hkv, D=D, bs=bs, context_lens=ctx, seed=seed,
                      pool_blocks=pool_blocks, poison=False, device=device, kv_dtype=kv_dtype)
    qs = [row_offset]
    for l in L:
        qs.append(qs[-1] + l)
    T = qs[-1] + extra_rows
    big = _gen(seed + 2, device)
    q = _randn_bf16((T, Hq, D), big, device)
    new_key = _randn_bf16((T, Hkv, D), big, device)
    new_value = _randn_bf16((T, Hkv, D), big, device)
    tables = case.block_tables.cpu()
    slots = torch.full((T,), -1, dtype=torch.int64)
    for s_ in range(S):
        for i in range(L[s_]):
            pos = ctx[s_] - L[s_] + i
            slots[qs[s_] + i] = int(tables[s_, pos // bs]) * bs + pos % bs
    if poison and kv_dtype == "bf16":  # quantised sources stay finite: tests poison their scales
        before = torch.tensor([c - l for c, l in zip(ctx, L)], dtype=torch.int64)
        bad = ~valid_slot_mask(case.meta["content_tables"], before, bs, case.N).to(device)
        nan = torch.tensor(BF16_NAN_BITS, dtype=torch.int16).view(torch.bfloat16).item()
        for pool in (case.k_pool, case.v_pool):
            pool.permute(0, 2, 1, 3)[bad] = nan
    case.q, case.new_key, case.new_value = q, new_key, new_value
    case.slot_mapping = slots.to(device)
    case.query_start = torch.tensor(qs, dtype=torch.int32, device=device)
    case.meta["query_lens"] = L
    return case


def widen_scales(case: PagedCase, lo: float, hi: float, seed: int, outlier_channels: int = 3,
                 outlier_factor: float = 20.0) -> PagedCase:
    """Give every cached and new K/V row (one token of one kv head) its own magnitude:
    a few fixed channels per kv head are made outliers (x outlier_factor), then each row
    is rescaled so that its largest |value| is 10^u, u uniform in [log10 lo, log10 hi],
    and rounded to bf16.  With an 8-bit cache the per-token scales then span the same
    decades (the dynamic per-token scale of the pages' quantised caches).  NaN poison
    in unused slots stays NaN.  Modifies and returns the case."""
    gen = _gen(seed + 7)
    D, Hkv = case.D, case.Hkv
    chan = torch.ones((Hkv, D), dtype=torch.float32)
    for h in range(Hkv):
        idx = torch.randperm(D, generator=gen)[:outlier_channels]
        chan[h, idx] = outlier_factor

    def rescale(rows: torch.Tensor, head_axis: int) -> torch.Tensor:
        x = rows.float()
        shape = [1] * x.dim()
        shape[head_axis] = Hkv
        shape[-1] = D
        x = x * chan.reshape(shape)
        amax = torch.nan_to_num(x.abs(), nan=0.0).amax(dim=-1, keepdim=True)
        u = torch.rand(amax.shape, generator=gen, dtype=torch.float64)
        target = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))).float()
        return (x * torch.where(amax > 0, target / amax, torch.zeros_like(amax))).to(torch.bfloat16)

    dev = case.k_pool.device
    case.k_pool = rescale(case.k_pool.cpu(), 1).to(dev)
    case.v_pool = rescale(case.v_pool.cpu(), 1).to(dev)
    case.new_key = rescale(case.new_key.cpu(), 1).to(dev)
    case.new_value = rescale(case.new_value.cpu(), 1).to(dev)
    case.meta["scale_range"] = (lo, hi)
    return case


# --------------------------------------------------------------------------- configs
def tiny(seed: int = 0, device="cpu", poison=True) -> PagedCase:
    return build_case("tiny", S=4, Hq=2, Hkv=2, D=64, bs=16, context_lens=[1, 17, 40, 100],
                      seed=seed, pool_blocks=32, poison=poison, device=device, scale=1.0 / 8.0)


def mha13b(seed: int = 1, device="cpu", poison=False) -> PagedCase:
    lens = torch.randint(200, 2049, (64,), generator=_gen(seed + 100)).tolist()
    return build_case("mha13b", S=64, Hq=40, Hkv=40, D=128, bs=16, context_lens=lens,
                      seed=seed, poison=poison, device=device)


def gqa70b(seed: int = 2, device="cpu", poison=False) -> PagedCase:
    return build_case("gqa70b", S=20, Hq=64, Hkv=8, D=128, bs=16, context_lens=[8000] * 20,
                      seed=seed, pool_blocks=10000, poison=poison, device=device)


def prefix(seed: int = 3, device="cpu", poison=False, kv_dtype="bf16") -> PagedCase:
    own = torch.randint(64, 513, (50,), generator=_gen(seed + 100))
    lens = (2000 + own).tolist()
    return build_case("prefix", S=50, Hq=32, Hkv=8, D=128, bs=16, context_lens=lens, seed=seed,
                      prefix_tokens=2000, cow=True, poison=poison, device=device, kv_dtype=kv_dtype)


def prefix_fp8(seed: int = 3, device="cpu", poison=False) -> PagedCase:
    """The shared-prompt workload with an fp8 (e4m3) cache."""
    return prefix(seed, device, poison, kv_dtype="fp8")


def int8_lengths(S: int, seed: int, lo: int = 128, hi: int = 32768) -> list[int]:
    u = torch.rand((S,), generator=_gen(seed + 100), dtype=torch.float64)
    lens = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))).round().long()
    return lens.clamp(lo, hi).tolist()


def int8(seed: int = 4, device="cpu", poison=False) -> PagedCase:
    return build_case("int8", S=256, Hq=32, Hkv=8, D=128, bs=32, context_lens=int8_lengths(256, seed),
                      seed=seed, kv_dtype="int8", poison=poison, device=device)


def fp8(seed: int = 5, device="cpu", poison=False) -> PagedCase:
    """The int8 workload's shape with an fp8 (e4m3) cache."""
    return build_case("fp8", S=256, Hq=32, Hkv=8, D=128, bs=32, context_lens=int8_lengths(256, seed),
                      seed=seed, kv_dtype="fp8", poison=poison, device=device)


def verify70b(seed: int = 6, device="cpu", poison=False, kv_dtype="bf16") -> PagedCase:
    """Draft verification on the 70B-shaped GQA batch: 4 new tokens per sequence on
    8000-token contexts (the 4 included)."""
    return build_multi_case("verify70b", S=20, Hq=64, Hkv=8, D=128, bs=16, context_lens=[8000] * 20,
                            query_lens=[4] * 20, seed=seed, pool_blocks=10000, poison=poison,
                            device=device, kv_dtype=kv_dtype)


def prefill8b(seed: int = 7, device="cpu", poison=False, kv_dtype="bf16") -> PagedCase:
    """Chunked prefill, Llama-3-8B shape: 4 sequences each attending a 512-token chunk
    on top of 3584 cached tokens."""
    return build_multi_case("prefill8b", S=4, Hq=32, Hkv=8, D=128, bs=16, context_lens=[4096] * 4,
                            query_lens=[512] * 4, seed=seed, poison=poison, device=device,
                            kv_dtype=kv_dtype)


def verify70b_fp8(seed: int = 6, device="cpu", poison=False) -> PagedCase:
    """The draft-verification workload with an fp8 (e4m3) cache."""
    return verify70b(seed, device, poison, kv_dtype="fp8")


def prefill8b_fp8(seed: int = 7, device="cpu", poison=False) -> PagedCase:
    """The chunked-prefill workload with an fp8 (e4m3) cache."""
    return prefill8b(seed, device, poison, kv_dtype="fp8")


CONFIGS = {"tiny": tiny, "mha13b": mha13b, "gqa70b": gqa70b, "prefix": prefix, "int8": int8, "fp8": fp8,
           "verify70b": verify70b, "prefill8b": prefill8b, "verify70b_fp8": verify70b_fp8,
           "prefill8b_fp8": prefill8b_fp8, "prefix_fp8": prefix_fp8}


# ------------------------------------------------------------------ byte accounting
def kv_cache_bytes(layers: int, heads: int, head_dim: int, tokens: int, batch: int,
                   bytes_per_value: float) -> float:
    """KV-cache size: 2 (K and V) x layers x heads x head_dim x tokens x batch x bytes
    (ia-vox-magazine KV-cache article, "Pourquoi le KV cache domine la consommation
    memoire" and its FAQ)."""
    return 2.0 * layers * heads * head_dim * tokens * batch * bytes_per_value


def decode_algorithmic_bytes(case: PagedCase, unique_blocks: bool = False) -> int:
    """Bytes one decode call must move at minimum: every cached K and V element of every
    sequence's context once (int8: plus one fp32 scale per token, kv head and K/V), the
    queries, the outputs, the block-table entries and the context lengths.  With
    ``unique_blocks`` a physical block shared by several tables counts once."""
    quant = case.kv_dtype in ("int8", "fp8")
    e = 1 if quant else 2
    ctx = case.context_lens.long().cpu()
    per_token = case.Hkv * case.D * e * 2 + (case.Hkv * 2 * 4 if quant else 0)
    if unique_blocks:
        seen = {}
        tabs = case.block_tables.cpu()
        for s in range(case.S):
            n = int(ctx[s])
            nb = blocks_needed(n, case.bs)
            for j in range(nb):
                b = int(tabs[s, j])
                fill = min(case.bs, n - j * case.bs)
                seen[b] = max(seen.get(b, 0), fill)
        kv = sum(seen.values()) * per_token
    else:
        kv = int(ctx.sum()) * per_token
    qo = 2 * case.q.shape[0] * case.Hq * case.D * 2  # query rows: S, or T new tokens
    tables = sum(blocks_needed(int(c), case.bs) for c in ctx) * 4 + case.S * 4
    if case.query_start is not None:
        tables += (case.S + 1) * 4
    return int(kv + qo + tables)


def multi_token_flops(case: PagedCase) -> int:
    """Multiply-adds x 2 of a multi-token step: each new token and query head takes a
    D-long dot product with, and a D-long weighted sum of, every position it sees."""
    qs = case.query_start.cpu().tolist()
    ctx = case.context_lens.cpu().tolist()
    seen = 0
    for s in range(case.S):
        L = qs[s + 1] - qs[s]
        base = ctx[s] - L
        seen += L * base + L * (L + 1) // 2
    return 4 * seen * case.Hq * case.D


def append_algorithmic_bytes(case: PagedCase) -> int:
    """Bytes of one append of the step's new tokens (one per sequence, or T): read K and
    V rows, write them (int8: codes and one fp32 scale per row), plus the slot numbers."""
    T = case.new_key.shape[0]
    rows = T * case.Hkv
    if case.kv_dtype in ("int8", "fp8"):
        return rows * 2 * (case.D * 2 + case.D + 4) + T * 8
    return rows * 2 * case.D * 2 * 2 + T * 8


def fragmentation(case: PagedCase, max_len: int) -> dict:
    """Wasted KV capacity under contiguous max-length reservation versus paging (the pages'
    internal-fragmentation comparison): the fraction of reserved token slots that hold no
    token."""
    ctx = case.context_lens.long().cpu()
    used = int(ctx.sum())
    contiguous = case.S * max_len
    paged = sum(blocks_needed(int(c), case.bs) for c in ctx) * case.bs
    return {"contiguous_waste": 1.0 - used / contiguous, "paged_waste": 1.0 - used / paged}
