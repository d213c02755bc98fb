"""Pins for the CPU oracle: checks against what the source pages and mathematics fix.

Each ``pin_*`` function takes a loaded oracle and raises AssertionError when the
oracle disagrees with its pin.  ``test_oracle_pins.py`` runs them against the real
oracle; ``test_oracle_mutants.py`` runs them against deliberately broken copies of
the oracle and requires every planted mistake to be caught by at least one pin.

None of these recomputes the oracle's formula with the oracle's code path:
  - the block-table figure of the gotburnout.io glossary fixes where tokens live;
  - brute force in 40-digit arithmetic (mpmath) on tiny, contiguous (unpaged)
    inputs fixes the attention result;
  - closed forms (one token, equal keys, zero query, one dominant key), invariants
    (block permutation, shared versus copied prefix, weights summing to one) and
    hand-computed quantiser values fix the rest.
"""
from __future__ import annotations

import json
import math
from pathlib import Path

import mpmath
import numpy as np
import torch

GOLDEN = Path(__file__).resolve().parent / "golden"


# ----------------------------------------------------------------------- helpers
def to_bf16_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def scatter_pool(logical: list[np.ndarray], tables: np.ndarray, N: int, bs: int) -> np.ndarray:
    """Place each sequence's logical rows [ctx][Hkv][D] into a [N][Hkv][bs][D] pool.

    Written as a flat slot view ([N*bs][Hkv][D]) so that it shares no indexing code
    with the oracle's gather.  Unused slots hold bf16 NaN."""
    Hkv, D = logical[0].shape[1:]
    pool = np.full((N, Hkv, bs, D), 0x7FC0, dtype=logical[0].dtype)
    flat = pool.transpose(0, 2, 1, 3)  # [N][bs][Hkv][D], a view
    for s, rows in enumerate(logical):
        for t in range(rows.shape[0]):
            blk, off = divmod(t, bs)
            flat[tables[s][blk], off] = rows[t]
    return pool


def brute_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Softmax attention of one query over contiguous K, V [ctx][D], 40 digits."""
    mpmath.mp.dps = 40
    ctx = K.shape[0]
    if ctx == 0:
        return np.zeros(q.shape[0])
    scores = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(float(a)) * mpmath.mpf(float(b))
                                              for a, b in zip(q, K[t])) for t in range(ctx)]
    mx = max(scores)
    e = [mpmath.exp(s - mx) for s in scores]
    z = mpmath.fsum(e)
    out = [mpmath.fsum(e[t] * mpmath.mpf(float(V[t][d])) for t in range(ctx)) / z
           for d in range(q.shape[0])]
    return np.array([float(v) for v in out])


def _tiny_random_case(rng, S, Hq, Hkv, D, bs, ctx, N):
    """Random bf16 logical K/V per sequence, placed through random block tables."""
    M = max(1, max((c + bs - 1) // bs for c in ctx))
    perm = rng.permutation(N)
    tables = np.zeros((S, M), dtype=np.int32)
    k = 0
    for s, c in enumerate(ctx):
        nb = (c + bs - 1) // bs
        tables[s, :nb] = perm[k:k + nb]
        k += nb
    logical_k = [to_bf16_bits(rng.standard_normal((c, Hkv, D))) for c in ctx]
    logical_v = [to_bf16_bits(rng.standard_normal((c, Hkv, D))) for c in ctx]
    q = to_bf16_bits(rng.standard_normal((S, Hq, D)))
    k_pool = scatter_pool(logical_k, tables, N, bs)
    v_pool = scatter_pool(logical_v, tables, N, bs)
    return q, logical_k, logical_v, k_pool, v_pool, tables, np.array(ctx, dtype=np.int32)


# ---------------------------------------------------------------------- the pins
def pin_slot_figure(orc):
    """gotburnout.io block-table figure: logical blocks 0,1,2 (tokens 0-15, 16-31, 32-47)
    live in physical blocks 7, 2, 11."""
    fig = json.loads((GOLDEN / "block_table_figure.json").read_text())
    bs = fig["block_size"]
    table = np.array(fig["block_table"], dtype=np.int32)
    for j, (lo, hi) in enumerate(fig["logical_token_ranges"]):
        for pos in range(lo, hi + 1):
            slot = orc.slot(table, pos, bs)
            assert slot // bs == fig["block_table"][j], (pos, slot)
            assert slot % bs == pos - lo, (pos, slot)


def pin_append_places_rows(orc):
    """Each new token's K/V rows land exactly in the slot (physical block, offset) the
    figure's table gives, and nothing else in the cache changes."""
    rng = np.random.default_rng(11)
    N, Hkv, bs, D, T = 16, 3, 16, 8, 5
    table = np.array([7, 2, 11], dtype=np.int32)
    positions = [0, 15, 16, 33, 47]
    slots = np.array([7 * 16 + 0, 7 * 16 + 15, 2 * 16 + 0, 11 * 16 + 1, 11 * 16 + 15], dtype=np.int64)
    slots_pad = slots.copy()
    slots_pad[2] = -1  # a padding token is not written
    key = to_bf16_bits(rng.standard_normal((T, Hkv, D)))
    val = to_bf16_bits(rng.standard_normal((T, Hkv, D)))
    k_cache = to_bf16_bits(rng.standard_normal((N, Hkv, bs, D)))
    v_cache = to_bf16_bits(rng.standard_normal((N, Hkv, bs, D)))
    k0, v0 = k_cache.copy(), v_cache.copy()
    bad = orc.reshape_and_cache(key, val, k_cache, v_cache, slots_pad, bs)
    assert bad == 0
    expect_k, expect_v = k0.copy(), v0.copy()
    for t, pos in enumerate(positions):
        if slots_pad[t] < 0:
            continue
        blk = int(table[pos // 16])
        expect_k[blk, :, pos % 16, :] = key[t]
        expect_v[blk, :, pos % 16, :] = val[t]
    assert np.array_equal(k_cache, expect_k)
    assert np.array_equal(v_cache, expect_v)
    # an out-of-range slot is counted and leaves the cache untouched
    k1 = k_cache.copy()
    assert orc.reshape_and_cache(key[:1], val[:1], k_cache, v_cache,
                                 np.array([N * bs], dtype=np.int64), bs) == 1
    assert np.array_equal(k_cache, k1)


def pin_brute_force_bf16(orc):
    """Paged oracle output equals 40-digit softmax attention on the contiguous (unpaged)
    logical K/V; query head h reads kv head h // (Hq/Hkv)."""
    rng = np.random.default_rng(5)
    S, Hq, Hkv, D, bs, N = 3, 4, 2, 8, 4, 16
    ctx = [5, 11, 1]
    q, lk, lv, kp, vp, tables, lens = _tiny_random_case(rng, S, Hq, Hkv, D, bs, ctx, N)
    scale = 0.37
    out = orc.paged_attention(q, kp, vp, tables, lens, scale)
    G = Hq // Hkv
    qf = bf16_bits_to_f64(q)
    for s in range(S):
        for h in range(Hq):
            K = bf16_bits_to_f64(lk[s][:, h // G, :])
            V = bf16_bits_to_f64(lv[s][:, h // G, :])
            ref = brute_attention(qf[s, h], K, V, scale)
            assert np.allclose(out[s, h], ref, rtol=1e-12, atol=1e-13), (s, h)


def pin_brute_force_int8(orc):
    """int8 cache: the oracle attends over code x scale (per token and kv head), checked
    against 40-digit attention on those dequantised values."""
    rng = np.random.default_rng(7)
    S, Hq, Hkv, D, bs, N = 2, 4, 2, 8, 4, 8
    ctx = [6, 9]
    M = 3
    tables = np.array([[3, 0, 0], [5, 1, 6]], dtype=np.int32)
    codes_k = rng.integers(-127, 128, size=(N, Hkv, bs, D), dtype=np.int8)
    codes_v = rng.integers(-127, 128, size=(N, Hkv, bs, D), dtype=np.int8)
    sk = rng.uniform(0.005, 0.05, size=(N, Hkv, bs)).astype(np.float32)
    sv = rng.uniform(0.005, 0.05, size=(N, Hkv, bs)).astype(np.float32)
    q = to_bf16_bits(rng.standard_normal((S, Hq, D)))
    lens = np.array(ctx, dtype=np.int32)
    out = orc.paged_attention(q, codes_k, codes_v, tables, lens, 0.5, k_scale=sk, v_scale=sv)
    G = Hq // Hkv
    qf = bf16_bits_to_f64(q)
    for s in range(S):
        for h in range(Hq):
            hk = h // G
            K = np.array([[codes_k[tables[s][t // bs], hk, t % bs, d] * float(sk[tables[s][t // bs], hk, t % bs])
                           for d in range(D)] for t in range(ctx[s])])
            V = np.array([[codes_v[tables[s][t // bs], hk, t % bs, d] * float(sv[tables[s][t // bs], hk, t % bs])
                           for d in range(D)] for t in range(ctx[s])])
            ref = brute_attention(qf[s, h], K, V, 0.5)
            assert np.allclose(out[s, h], ref, rtol=1e-12, atol=1e-13), (s, h)
    assert M == tables.shape[1]


def pin_closed_forms(orc):
    """One token: output = its value row exactly.  Equal keys, or a zero query: output =
    mean of the values.  One key far ahead of the rest: output = that key's value."""
    rng = np.random.default_rng(3)
    Hkv, D, bs, N = 1, 16, 16, 8
    # single token
    q = to_bf16_bits(rng.standard_normal((1, 1, D)))
    kv = to_bf16_bits(rng.standard_normal((N, Hkv, bs, D)))
    vv = to_bf16_bits(rng.standard_normal((N, Hkv, bs, D)))
    tables = np.array([[5]], dtype=np.int32)
    out = orc.paged_attention(q, kv, vv, tables, np.array([1], dtype=np.int32), 0.25)
    assert np.array_equal(out[0, 0], bf16_bits_to_f64(vv[5, 0, 0]))
    # equal keys -> uniform weights
    ctx = 37
    tables = np.array([[6, 1, 3]], dtype=np.int32)
    k_eq = np.repeat(to_bf16_bits(rng.standard_normal((1, 1, 1, D))), bs, axis=2)
    k_eq = np.ascontiguousarray(np.repeat(k_eq, N, axis=0))
    vals = bf16_bits_to_f64(vv)
    mean = np.mean([vals[tables[0][t // bs], 0, t % bs] for t in range(ctx)], axis=0)
    out = orc.paged_attention(q, k_eq, vv, tables, np.array([ctx], dtype=np.int32), 0.9)
    assert np.allclose(out[0, 0], mean, rtol=1e-12, atol=1e-13)
    # zero query -> uniform weights
    q0 = np.zeros((1, 1, D), dtype=np.uint16)
    out = orc.paged_attention(q0, kv, vv, tables, np.array([ctx], dtype=np.int32), 0.9)
    assert np.allclose(out[0, 0], mean, rtol=1e-12, atol=1e-13)
    # one dominant key (token 20): weight -> 1 within exp(-large)
    qd = to_bf16_bits(np.full((1, 1, D), 1.0))
    kd = np.zeros((N, Hkv, bs, D), dtype=np.uint16)
    kd[tables[0][20 // bs], 0, 20 % bs] = to_bf16_bits(np.full(D, 8.0))
    out = orc.paged_attention(qd, kd, vv, tables, np.array([ctx], dtype=np.int32), 1.0)
    assert np.allclose(out[0, 0], vals[tables[0][20 // bs], 0, 20 % bs], rtol=0, atol=1e-40 + 1e-12)
    # empty context -> zeros
    out = orc.paged_attention(q, kv, vv, tables, np.array([0], dtype=np.int32), 1.0)
    assert np.array_equal(out, np.zeros_like(out))


def pin_block_permutation_invariance(orc):
    """Moving blocks to other physical places (and updating the tables) changes nothing:
    the result is bit-identical, since it depends on logical order only."""
    rng = np.random.default_rng(9)
    S, Hq, Hkv, D, bs, N = 3, 6, 3, 16, 16, 24
    q, lk, lv, kp, vp, tables, lens = _tiny_random_case(rng, S, Hq, Hkv, D, bs, [30, 64, 7], N)
    out = orc.paged_attention(q, kp, vp, tables, lens, 0.2)
    pi = rng.permutation(N)  # physical block b moves to pi[b]
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[pi] = kp
    vp2[pi] = vp
    tables2 = pi[tables].astype(np.int32)
    out2 = orc.paged_attention(q, kp2, vp2, tables2, lens, 0.2)
    assert np.array_equal(out, out2)


def pin_prefix_shared_equals_copied(orc):
    """Sequences pointing at the same physical prefix blocks give the same output as
    sequences holding private copies of that prefix (prefix caching does not change a
    request's output)."""
    rng = np.random.default_rng(13)
    Hq, Hkv, D, bs = 4, 2, 16, 16
    prefix_blocks, S = 3, 4
    own = [5, 17, 16, 1]
    N = prefix_blocks * (S + 1) + sum((o + bs - 1) // bs for o in own)
    kp = to_bf16_bits(rng.standard_normal((N, Hkv, bs, D)))
    vp = to_bf16_bits(rng.standard_normal((N, Hkv, bs, D)))
    q = to_bf16_bits(rng.standard_normal((S, Hq, D)))
    M = prefix_blocks + 2
    shared = np.zeros((S, M), dtype=np.int32)
    copied = np.zeros((S, M), dtype=np.int32)
    nxt = prefix_blocks
    for s in range(S):
        shared[s, :prefix_blocks] = np.arange(prefix_blocks)
        for j in range(prefix_blocks):  # private copy of the prefix
            kp[nxt] = kp[j]
            vp[nxt] = vp[j]
            copied[s, j] = nxt
            nxt += 1
    for s in range(S):
        nb = (own[s] + bs - 1) // bs
        for j in range(nb):
            shared[s, prefix_blocks + j] = nxt
            copied[s, prefix_blocks + j] = nxt
            nxt += 1
    lens = np.array([prefix_blocks * bs + o for o in own], dtype=np.int32)
    a = orc.paged_attention(q, kp, vp, shared, lens, 0.3)
    b = orc.paged_attention(q, kp, vp, copied, lens, 0.3)
    assert np.array_equal(a, b)


def pin_softmax_weights(orc):
    """Softmax weights are non-negative, sum to one, and are proportional to the exp of
    the scores computed by brute force."""
    rng = np.random.default_rng(21)
    S, Hq, Hkv, D, bs, N = 2, 4, 2, 8, 4, 16
    q, lk, lv, kp, vp, tables, lens = _tiny_random_case(rng, S, Hq, Hkv, D, bs, [13, 6], N)
    G = Hq // Hkv
    qf = bf16_bits_to_f64(q)
    for s in range(S):
        for h in range(Hq):
            w = orc.attention_weights(q, kp, vp, tables, lens, 0.7, s, h)
            assert w.shape == (lens[s],)
            assert np.all(w >= 0)
            assert abs(w.sum() - 1.0) < 1e-12
            K = bf16_bits_to_f64(lk[s][:, h // G, :])
            sc = 0.7 * (K @ qf[s, h])
            ref = np.exp(sc - sc.max())
            ref /= ref.sum()
            assert np.allclose(w, ref, rtol=1e-10, atol=1e-14)


def pin_quantizer_hand_values(orc):
    """Hand-computed int8 codes: absmax 127 gives scale exactly 1; x/scale is rounded half
    to even (62.5 -> 62, 0.5 -> 0, 1.5 -> 2, -63.5 -> -64); an all-zero row gets scale 1
    and zero codes; the absmax element always maps to +-127; every element is within half
    a step of its dequantised value."""
    D, bs, Hkv, N = 8, 4, 1, 2
    row = np.array([127.0, -63.5, 62.5, 0.5, -0.5, 1.5, 0.0, -127.0], dtype=np.float32)
    key = to_bf16_bits(row.reshape(1, 1, D))
    assert np.array_equal(bf16_bits_to_f64(key).ravel(), row.astype(np.float64))
    val = np.zeros((1, 1, D), dtype=np.uint16)
    kc = np.zeros((N, Hkv, bs, D), dtype=np.int8)
    vc = np.zeros((N, Hkv, bs, D), dtype=np.int8)
    ks = np.zeros((N, Hkv, bs), dtype=np.float32)
    vs = np.zeros((N, Hkv, bs), dtype=np.float32)
    slot = np.array([1 * bs + 2], dtype=np.int64)
    assert orc.quantize_kv(key, val, kc, vc, ks, vs, slot, bs) == 0
    assert ks[1, 0, 2] == np.float32(1.0)
    assert kc[1, 0, 2].tolist() == [127, -64, 62, 0, 0, 2, 0, -127]
    assert vs[1, 0, 2] == np.float32(1.0)
    assert vc[1, 0, 2].tolist() == [0] * D
    assert np.count_nonzero(kc[0]) == 0 and np.count_nonzero(kc[1, 0, :2]) == 0
    rng = np.random.default_rng(2)
    src = to_bf16_bits(rng.standard_normal((64, 128)) * rng.uniform(0.01, 100, size=(64, 1)))
    codes, scales = orc.quantize_pool(src)
    x = bf16_bits_to_f64(src)
    amax = np.abs(x).max(axis=1)
    assert np.all(scales == (amax.astype(np.float32) / np.float32(127.0)))
    idx = np.abs(x).argmax(axis=1)
    assert np.all(np.abs(codes[np.arange(64), idx]) == 127)
    err = np.abs(x - codes.astype(np.float64) * scales[:, None].astype(np.float64))
    # half a step, plus the fp32 division's own rounding of x/scale (<= 128 ulp of 1)
    assert np.all(err <= scales[:, None] * (0.5 + 128 * 2.0 ** -23))


def pin_copy_blocks(orc):
    """Copy-on-write: after the copy every byte of the destination block (K, V and
    scales) equals the source block; all other blocks are untouched."""
    rng = np.random.default_rng(4)
    N, Hkv, bs, D = 10, 2, 4, 8
    kc = rng.integers(-127, 128, size=(N, Hkv, bs, D), dtype=np.int8)
    vc = rng.integers(-127, 128, size=(N, Hkv, bs, D), dtype=np.int8)
    ks = rng.random((N, Hkv, bs), dtype=np.float32)
    vs = rng.random((N, Hkv, bs), dtype=np.float32)
    before = [a.copy() for a in (kc, vc, ks, vs)]
    pairs = np.array([[1, 7], [4, 2], [1, 9]], dtype=np.int64)
    orc.copy_blocks(kc, vc, pairs, k_scale=ks, v_scale=vs)
    for arr, old in zip((kc, vc, ks, vs), before):
        expect = old.copy()
        for src, dst in pairs:
            expect[dst] = old[src]
        assert np.array_equal(arr, expect)


def _e4m3_value(code: int) -> float:
    """Value of an e4m3 code from the format's definition: sign bit, 4-bit exponent with
    bias 7 (field 0: subnormal m * 2^-9), 3-bit mantissa."""
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 15, code & 7
    return sign * (m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))


def pin_fp8_hand_values(orc):
    """e4m3 by hand: 1 -> 0x38, 448 (largest) -> 0x7e, -2 -> 0xc0, 2^-4 -> 0x18, 2^-9
    (smallest subnormal) -> 0x01; ties go to the even mantissa (1 + 1/16 -> 1.0,
    1 + 3/16 -> 1.25, 232 -> 224, 3 * 2^-10 -> 2^-8, 2^-10 -> 0); beyond 448
    saturates."""
    cases = {1.0: 0x38, 448.0: 0x7E, -2.0: 0xC0, 0.0625: 0x18, 2.0 ** -9: 0x01,
             1.0625: 0x38, 1.1875: 0x3A, 232.0: 0x76, 3 * 2.0 ** -10: 0x02, 2.0 ** -10: 0x00,
             464.0: 0x7E, 1e9: 0x7E, -1e9: 0xFE, 0.0: 0x00, 7.5 * 2.0 ** -9: 0x08}
    for x, code in cases.items():
        assert orc.fp8_encode(x) == code, (x, hex(orc.fp8_encode(x)), hex(code))


def pin_fp8_round_trip_and_ties(orc):
    """Every finite code decodes to its format value and encodes back to itself; the
    midpoint of two neighbours goes to the one with the even mantissa, and anything
    off the midpoint to the nearer one."""
    finite = [c for c in range(256) if (c & 0x7F) != 0x7F]
    for c in finite:
        assert orc.fp8_decode(c) == _e4m3_value(c), hex(c)
        assert orc.fp8_encode(_e4m3_value(c)) == c, hex(c)
    pos = sorted((_e4m3_value(c), c) for c in finite if c < 0x80)
    for (v0, c0), (v1, c1) in zip(pos, pos[1:]):
        mid = (v0 + v1) / 2
        assert orc.fp8_encode(mid) == (c0 if c0 % 2 == 0 else c1), (v0, v1)
        assert orc.fp8_encode(v0 + (v1 - v0) * 0.49) == c0
        assert orc.fp8_encode(v0 + (v1 - v0) * 0.51) == c1


def pin_fp8_quantizer(orc):
    """fp8 rows: scale = absmax / 448, so the absmax element maps to +-448 exactly; an
    all-zero row gets scale 1."""
    rng = np.random.default_rng(8)
    src = to_bf16_bits(rng.standard_normal((32, 64)) * rng.uniform(0.01, 100, size=(32, 1)))
    codes, scales = orc.quantize_pool(src, fp8=True)
    x = bf16_bits_to_f64(src)
    idx = np.abs(x).argmax(axis=1)
    assert np.all((codes[np.arange(32), idx] & 0x7F) == 0x7E)
    dq = np.vectorize(_e4m3_value)(codes) * scales[:, None]
    # relative error of e4m3 (3 mantissa bits) is at most 2^-4, subnormals aside
    big = np.abs(x) > 2.0 ** -6 * scales[:, None]
    assert np.all(np.abs(dq - x)[big] <= 2.0 ** -4 * np.abs(x)[big] + 1e-12)
    zero = np.zeros((1, 1, 8), dtype=np.uint16)
    kc = np.zeros((1, 1, 4, 8), dtype=np.uint8)
    ks = np.zeros((1, 1, 4), dtype=np.float32)
    assert orc.quantize_kv_fp8(zero, zero, kc, kc.copy(), ks, ks.copy(), np.array([1], dtype=np.int64), 4) == 0
    assert ks[0, 0, 1] == 1.0 and not kc.any()


def pin_fp8_divisor_by_hand(orc):
    """The fp8 scale divisor is exactly 448, the largest finite e4m3 value: a row whose
    absmax is 448 gets scale 1.0 exactly and its codes are e4m3 of the values
    themselves, worked out by hand (448 -> 0x7e, -224 -> 0xf6, 3 -> 0x44, 2^-9 ->
    0x01); a row whose absmax is 448 * 2^-5 gets scale 2^-5 exactly.  Two ties pin the
    division's direction as well: 232 lies halfway between 224 and 240 and goes to 224
    (even mantissa), 1.1875 halfway between 1.125 and 1.25 goes to 1.25 -- a divisor
    slightly above 448 pushes 232 past the midpoint (-> 240), one slightly below pulls
    1.1875 under it (-> 1.125)."""
    D, bs = 8, 2
    row = np.array([448.0, -224.0, 3.0, 2.0 ** -9, 232.0, 1.1875, 0.0, -448.0])
    expect = [0x7E, 0xF6, 0x44, 0x01, 0x76, 0x3A, 0x00, 0xFE]
    for shift, want_scale in ((0, 1.0), (-5, 2.0 ** -5)):
        key = to_bf16_bits((row * 2.0 ** shift).reshape(1, 1, D))
        assert np.array_equal(bf16_bits_to_f64(key).ravel(), row * 2.0 ** shift)
        kc = np.zeros((1, 1, bs, D), dtype=np.uint8)
        vc = np.zeros_like(kc)
        ks = np.zeros((1, 1, bs), dtype=np.float32)
        vs = np.zeros_like(ks)
        assert orc.quantize_kv_fp8(key, key, kc, vc, ks, vs, np.array([1], dtype=np.int64), bs) == 0
        assert ks[0, 0, 1] == np.float32(want_scale), ks[0, 0, 1]
        assert kc[0, 0, 1].tolist() == expect, [hex(c) for c in kc[0, 0, 1]]
        assert np.array_equal(kc, vc) and np.array_equal(ks, vs)
    # and the division is IEEE fp32 (correctly rounded), not a multiply by 1/448: on rows
    # of random magnitude every scale equals numpy's float32 quotient absmax / 448
    rng = np.random.default_rng(9)
    src = to_bf16_bits(rng.standard_normal((256, 16)) * rng.uniform(0.01, 100, size=(256, 1)))
    _, scales = orc.quantize_pool(src, fp8=True)
    amax = np.abs(bf16_bits_to_f64(src)).max(axis=1).astype(np.float32)
    assert np.array_equal(scales, amax / np.float32(448.0))


def pin_brute_force_fp8(orc):
    """fp8 cache: attention over e4m3 value x scale, against 40-digit brute force."""
    rng = np.random.default_rng(17)
    S, Hq, Hkv, D, bs, N = 2, 4, 2, 8, 4, 8
    ctx = [5, 10]
    tables = np.array([[6, 2, 0], [1, 7, 4]], dtype=np.int32)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    ck = rng.choice(finite, size=(N, Hkv, bs, D)).astype(np.uint8)
    cv = rng.choice(finite, size=(N, Hkv, bs, D)).astype(np.uint8)
    sk = rng.uniform(0.001, 0.01, size=(N, Hkv, bs)).astype(np.float32)
    sv = rng.uniform(0.001, 0.01, size=(N, Hkv, bs)).astype(np.float32)
    q = to_bf16_bits(rng.standard_normal((S, Hq, D)))
    out = orc.paged_attention(q, ck, cv, tables, np.array(ctx, dtype=np.int32), 0.3, k_scale=sk, v_scale=sv)
    G = Hq // Hkv
    qf = bf16_bits_to_f64(q)
    for s in range(S):
        for h in range(Hq):
            hk = h // G
            rows = [(tables[s][t // bs], t % bs) for t in range(ctx[s])]
            K = np.array([[_e4m3_value(int(ck[b, hk, o, d])) * float(sk[b, hk, o]) for d in range(D)] for b, o in rows])
            V = np.array([[_e4m3_value(int(cv[b, hk, o, d])) * float(sv[b, hk, o]) for d in range(D)] for b, o in rows])
            ref = brute_attention(qf[s, h], K, V, 0.3)
            assert np.allclose(out[s, h], ref, rtol=1e-12, atol=1e-13), (s, h)


def _prefill_case(rng):
    """Three sequences with new-token chunks of 3, 1 and 3 (the last one's whole
    context is its chunk), query rows packed from row 1 on; rows 0 and 8 belong to
    no sequence."""
    S, Hq, Hkv, D, bs, N = 3, 4, 2, 8, 4, 16
    ctx = [7, 12, 3]
    qs = np.array([1, 4, 5, 8], dtype=np.int32)
    T = 9
    _, lk, lv, kp, vp, tables, lens = _tiny_random_case(rng, S, Hq, Hkv, D, bs, ctx, N)
    q = to_bf16_bits(rng.standard_normal((T, Hq, D)))
    return q, lk, lv, kp, vp, tables, lens, qs, Hq // Hkv


def pin_brute_force_prefill(orc):
    """Multi-token attention: new token i of sequence s (row query_start[s] + i) equals
    40-digit softmax attention over the unpaged logical K/V up to and including its
    own position ctx_s - L_s + i; rows of no sequence are zero."""
    rng = np.random.default_rng(21)
    q, lk, lv, kp, vp, tables, lens, qs, G = _prefill_case(rng)
    scale = 0.41
    out = orc.paged_prefill(q, kp, vp, tables, lens, qs, scale)
    qf = bf16_bits_to_f64(q)
    covered = set()
    for s in range(len(lens)):
        L = qs[s + 1] - qs[s]
        for i in range(L):
            row, pos = qs[s] + i, lens[s] - L + i
            covered.add(row)
            for h in range(q.shape[1]):
                K = bf16_bits_to_f64(lk[s][: pos + 1, h // G, :])
                V = bf16_bits_to_f64(lv[s][: pos + 1, h // G, :])
                ref = brute_attention(qf[row, h], K, V, scale)
                assert np.allclose(out[row, h], ref, rtol=1e-12, atol=1e-13), (s, i, h)
    for row in range(q.shape[0]):
        if row not in covered:
            assert np.array_equal(out[row], np.zeros_like(out[row]))


def pin_prefill_causality(orc):
    """A new token never reads a later position: NaN written into every slot after
    token i's position leaves row i bit-identical (and finite).  The first token of a
    chunk that is the whole context sees one token: its output is that value row."""
    rng = np.random.default_rng(22)
    q, lk, lv, kp, vp, tables, lens, qs, G = _prefill_case(rng)
    bs = kp.shape[2]
    base = orc.paged_prefill(q, kp, vp, tables, lens, qs, 0.8)
    for s in range(len(lens)):
        L = qs[s + 1] - qs[s]
        for i in range(L):
            pos = lens[s] - L + i
            kq, vq = kp.copy(), vp.copy()
            for t in range(pos + 1, lens[s]):
                kq[tables[s][t // bs], :, t % bs, :] = 0x7FC0
                vq[tables[s][t // bs], :, t % bs, :] = 0x7FC0
            out = orc.paged_prefill(q, kq, vq, tables, lens, qs, 0.8)
            row = qs[s] + i
            assert np.all(np.isfinite(out[row])) and np.array_equal(out[row], base[row]), (s, i)
    s = 2  # context == chunk: the first new token attends itself only
    for h in range(q.shape[1]):
        assert np.array_equal(base[qs[s], h], bf16_bits_to_f64(lv[s][0, h // G, :]))


ALL_PINS = [pin_slot_figure, pin_append_places_rows, pin_brute_force_bf16, pin_brute_force_int8,
            pin_closed_forms, pin_block_permutation_invariance, pin_prefix_shared_equals_copied,
            pin_softmax_weights, pin_quantizer_hand_values, pin_copy_blocks, pin_fp8_hand_values,
            pin_fp8_round_trip_and_ties, pin_fp8_quantizer, pin_fp8_divisor_by_hand, pin_brute_force_fp8,
            pin_brute_force_prefill, pin_prefill_causality]


def run_all(orc) -> list[str]:
    """Names of the pins that fail (or crash) for this oracle."""
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except Exception:  # noqa: BLE001 - any failure counts
            failed.append(pin.__name__)
    return failed


def kv_size_claims():
    return json.loads((GOLDEN / "kv_size_claims.json").read_text())


def isclose(a, b, rel=1e-9):
    return math.isclose(a, b, rel_tol=rel)
