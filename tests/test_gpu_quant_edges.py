"""GPU parity of the two quantisers on rows designed to sit on their decisions.

pa_quantize_kv and pa_quantize_kv_fp8 turn a floating-point quotient x / scale into an
integer code, so the GPU and the CPU oracle must take every rounding decision the same
way.  N(0, 1) rows never land on those decisions; the rows here do:
  - an all-zero row (scale 1, codes 0);
  - exact half-step ties of the int8 rule (x / scale = k + 1/2 for every k in
    [-127, 126]: round half to even);
  - e4m3 values, the midpoints between neighbouring e4m3 values (ties to the even
    mantissa), subnormal codes and their midpoints;
  - the absmax element at different lanes, with either sign and repeated, which must
    map to +-127 (int8) or +-448 (fp8);
  - rows whose magnitude runs over bf16's whole exponent range, subnormal bf16 values
    included, so that the scale itself is huge, tiny or an fp32 subnormal.
The scale of a row is absmax / 127 (int8) or absmax / 448 (fp8) in IEEE fp32
(ia-vox-magazine, "Quantization du KV cache": a dynamic scale recomputed for every
token; blog.fabienvernieres.com, "Reduire le poids par token": int8 or fp8 entries).
Codes and scale bits are compared bit for bit with the oracle.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_kv_cache_197_gb300 as pa

    pa.load_library()


def _bf16_exact(values) -> np.ndarray:
    """bf16 bits of values that bf16 holds exactly (checked)."""
    x = np.asarray(values, dtype=np.float64)
    bits = torch.as_tensor(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    bits = bits.view(np.uint16).copy()
    back = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(back, x), "a designed value is not a bf16 value"
    return bits


def _rows_of(values, absmax, D, rng):
    """Rows of D values: each row starts with +-absmax at a random lane, then as many of
    `values` as fit, the rest zeros."""
    values = list(values)
    rows = []
    per = D - 1
    for i in range(0, len(values), per):
        chunk = values[i:i + per]
        row = chunk + [0.0] * (per - len(chunk))
        lane = int(rng.integers(0, D))
        row.insert(lane, absmax if (i // per) % 2 == 0 else -absmax)
        rows.append(row)
    return rows


def _e4m3_positive() -> list[float]:
    """Every finite positive e4m3 value, from the format (bias 7, 3 mantissa bits)."""
    out = []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue  # the NaN code
            out.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return sorted(set(out))


def int8_rows(D, rng) -> np.ndarray:
    rows = [[0.0] * D]
    # every half-step tie at scale 1 (absmax 127), and the same row scaled by powers of
    # two (the scale is then 2^k exactly and the quotients are the same ties)
    ties = [k + 0.5 for k in range(-127, 127)]
    for shift in (0, -20, 7, 60, -100):
        rows += [[v * 2.0 ** shift for v in r] for r in _rows_of(ties, 127.0, D, rng)]
    rows.append([127.0, -63.5, 62.5, 0.5, -0.5, 1.5, 0.0, -127.0] + [0.0] * (D - 8))
    # every integer code at scale 1, and values a quarter step off the ties (|x| < 64,
    # where bf16 holds them exactly)
    rows += _rows_of([float(k) for k in range(-126, 127)], 127.0, D, rng)
    rows += _rows_of([k + 0.25 for k in range(-64, 63)] + [k + 0.75 for k in range(-64, 63)],
                     127.0, D, rng)
    return np.array(rows)


def fp8_rows(D, rng) -> np.ndarray:
    pos = _e4m3_positive()
    mids = [(a + b) / 2 for a, b in zip(pos, pos[1:])]
    vals = pos + mids + [-v for v in pos + mids]
    rows = [[0.0] * D]
    for shift in (0, -30, 9, 70, -110):  # absmax 448 * 2^shift: scale 2^shift exactly
        rows += [[v * 2.0 ** shift for v in r] for r in _rows_of(vals, 448.0, D, rng)]
    return np.array(rows)


def absmax_and_range_rows(D, rng, n=96) -> np.ndarray:
    """Random rows of magnitude 2^e, e over bf16's exponent range (subnormals included),
    with the absmax element repeated with both signs at random lanes in some rows."""
    rows = []
    for i in range(n):
        e = float(rng.uniform(-133, 124))
        row = rng.standard_normal(D) * 2.0 ** e
        row = torch.as_tensor(row.astype(np.float32)).to(torch.bfloat16).float().double().numpy()
        if i % 3 == 0:
            a = np.abs(row).max()
            for lane in rng.choice(D, size=3, replace=False):
                row[lane] = a if rng.integers(0, 2) else -a
        rows.append(row)
    for lane in (0, 31, 32, D - 1):  # a single non-zero element at an edge lane
        row = np.zeros(D)
        row[lane] = -3.0
        rows.append(row)
    return np.array(rows)


def _run(kind, rows: np.ndarray, D: int, orc):
    """Quantise `rows` (as K; the reversed rows as V) on the GPU and in the oracle, with
    Hkv = 2 and a random slot per token; compare codes and scale bits."""
    import paged_kv_cache_197_gb300 as pa

    Hkv, bs = 2, 16
    if len(rows) % Hkv:
        rows = np.concatenate([rows, np.zeros((1, D))])
    T = len(rows) // Hkv
    key = _bf16_exact(rows).reshape(T, Hkv, D)
    value = _bf16_exact(rows[::-1].copy()).reshape(T, Hkv, D)
    N = (T + bs - 1) // bs + 1
    slots = np.random.default_rng(T).permutation(N * bs)[:T].astype(np.int64)
    fp8 = kind == "fp8"
    code_t = np.uint8 if fp8 else np.int8
    kc = np.zeros((N, Hkv, bs, D), dtype=code_t)
    vc = np.zeros_like(kc)
    ks = np.zeros((N, Hkv, bs), dtype=np.float32)
    vs = np.zeros_like(ks)
    quant_o = orc.quantize_kv_fp8 if fp8 else orc.quantize_kv
    assert quant_o(key, value, kc, vc, ks, vs, slots, bs) == 0

    to_dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(DEV)  # noqa: E731
    gk = torch.zeros((N, Hkv, bs, D), dtype=torch.uint8 if fp8 else torch.int8, device=DEV)
    gv = torch.zeros_like(gk)
    gks = torch.zeros((N, Hkv, bs), dtype=torch.float32, device=DEV)
    gvs = torch.zeros_like(gks)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    quant_g = pa.pa_quantize_kv_fp8 if fp8 else pa.pa_quantize_kv
    quant_g(to_dev(key), to_dev(value), gk, gv, gks, gvs, torch.from_numpy(slots).to(DEV),
            err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    for got, ref, what in ((gk, kc, "K codes"), (gv, vc, "V codes")):
        g = got.cpu().numpy()
        bad = np.argwhere(g != ref)
        assert bad.size == 0, f"{what}: {len(bad)} codes differ, first at {bad[0].tolist()}"
    for got, ref, what in ((gks, ks, "K scales"), (gvs, vs, "V scales")):
        g = got.cpu().numpy().view(np.uint32)
        assert np.array_equal(g, ref.view(np.uint32)), f"{what} differ"
    # flat (block, kv head, offset) rows that received a token
    blk, off = slots // bs, slots % bs
    written = np.concatenate([(blk * Hkv + h) * bs + off for h in range(Hkv)])
    return kc, ks, written


@pytest.mark.parametrize("D", [64, 128])
def test_int8_ties_and_codes(oracle, D):
    rng = np.random.default_rng(D)
    kc, ks, _ = _run("int8", int8_rows(D, rng), D, oracle)
    # the hand row's codes (ties to even) as a direct check of the designed decisions
    hand = [127, -64, 62, 0, 0, 2, 0, -127]
    assert any(kc[b, h, o, :8].tolist() == hand for b, h, o in np.ndindex(ks.shape))


@pytest.mark.parametrize("D", [64, 128])
def test_fp8_ties_subnormals_and_saturation(oracle, D):
    rng = np.random.default_rng(100 + D)
    _run("fp8", fp8_rows(D, rng), D, oracle)


@pytest.mark.parametrize("kind", ["int8", "fp8"])
@pytest.mark.parametrize("D", [64, 128])
def test_absmax_lanes_and_extreme_scales(oracle, kind, D):
    rng = np.random.default_rng(7 * D + (kind == "fp8"))
    rows = absmax_and_range_rows(D, rng)
    kc, ks, written = _run(kind, rows, D, oracle)
    # every non-zero row has an element at +-127 (int8) or +-448 (fp8: code 0x7e / 0xfe)
    top = 127 if kind == "int8" else 0x7E
    codes = kc.reshape(-1, D)[written]
    nz = np.abs(codes.astype(np.int32)).max(axis=1) > 0 if kind == "int8" else (codes & 0x7F).max(axis=1) > 0
    if kind == "int8":
        assert np.all(np.abs(codes[nz].astype(np.int32)).max(axis=1) == top)
    else:
        assert np.all((codes[nz] & 0x7F).max(axis=1) == top)
    scales = ks.reshape(-1)[written]
    assert np.all(np.isfinite(scales)) and np.all(scales > 0)
