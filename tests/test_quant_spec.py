"""Pins for the oracle's FP8 (E4M3) and FP4 (E2M1) quantisers and for the two
read-copy tile formats, against the OCP format specifications and against
brute force (nearest representable value, ties to the even code)."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ocp_fp8_fp4_values.txt")


def _golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                fmt, code, val = line.split()
                rows.append((fmt, int(code, 16), float(val)))
    return rows


def _table(fmt):
    """All finite (code, value) pairs of a format, from the bit layout of the
    specs: E4M3 = 1 sign, 4 exponent (bias 7), 3 mantissa, S.1111.111 = NaN;
    E2M1 = 1 sign, 2 exponent (bias 1), 1 mantissa."""
    out = []
    if fmt == "e4m3":
        for c in range(256):
            s, e, m = c >> 7, (c >> 3) & 15, c & 7
            if e == 15 and m == 7:
                continue
            mag = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
            out.append((c, -mag if s else mag))
    else:
        for c in range(16):
            s, e, m = c >> 3, (c >> 1) & 3, c & 1
            mag = m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1)
            out.append((c, -mag if s else mag))
    return out


@pytest.mark.parametrize("row", _golden(), ids=lambda r: f"{r[0]}-{r[1]:#x}")
def test_decode_matches_spec_table(row):
    fmt, code, val = row
    got = (oracle.e4m3_decode if fmt == "e4m3" else oracle.e2m1_decode)([code])[0]
    if np.isnan(val):
        assert np.isnan(got)
    else:
        assert got == val and np.signbit(got) == np.signbit(val)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_every_finite_value_round_trips(fmt):
    enc = oracle.e4m3_encode if fmt == "e4m3" else oracle.e2m1_encode
    tab = _table(fmt)
    codes = enc(np.array([v for _, v in tab], np.float32))
    for (c, v), got in zip(tab, codes):
        if v == 0:
            assert got == c  # signed zeros keep their sign
        else:
            assert got == c, (fmt, hex(c), v, hex(got))


def _brute_nearest(fmt, x):
    """Nearest finite value; ties go to the code with an even mantissa; values
    beyond the largest finite magnitude saturate (satfinite)."""
    tab = [(c, v) for c, v in _table(fmt) if not (v == 0 and c & (0x80 if fmt == "e4m3" else 8))]
    vals = np.array([v for _, v in tab])
    codes = np.array([c for c, _ in tab])
    vmax = vals.max()
    out = []
    for xi in x:
        if abs(xi) >= vmax:  # satfinite
            out.append(int(codes[np.argmax(vals)]) | ((0x80 if fmt == "e4m3" else 8) if xi < 0 else 0))
            continue
        d = np.abs(vals - xi)
        best = np.flatnonzero(d == d.min())
        if len(best) > 1:
            best = [b for b in best if codes[b] % 2 == 0]
        c = int(codes[best[0]])
        v = vals[best[0]]
        if v == 0 and np.signbit(xi):
            c |= 0x80 if fmt == "e4m3" else 8
        out.append(c)
    return np.array(out, np.uint8)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_encode_is_nearest_with_ties_to_even(fmt):
    enc = oracle.e4m3_encode if fmt == "e4m3" else oracle.e2m1_encode
    vmax = 448.0 if fmt == "e4m3" else 6.0
    pos = sorted(v for _, v in _table(fmt) if v >= 0)
    mids = [(a + b) / 2 for a, b in zip(pos, pos[1:])]          # exact ties
    rng = np.random.default_rng(0)
    rand = np.concatenate([rng.uniform(-vmax * 1.2, vmax * 1.2, 4000),
                           rng.standard_normal(2000) * 2.0 ** rng.integers(-12, 3, 2000)])
    x = np.concatenate([mids, -np.array(mids), rand, [vmax * 3, -vmax * 3, 1e30]])
    x = x.astype(np.float32)
    np.testing.assert_array_equal(enc(x), _brute_nearest(fmt, x.astype(np.float64)))


def test_e4m3_spec_extremes():
    enc = oracle.e4m3_encode(np.array([448, 464, 1e9, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10,
                                       0.875 * 2 ** -6, 2.0 ** -6], np.float32))
    assert list(enc) == [0x7E, 0x7E, 0x7E, 0x01, 0x00, 0x02, 0x07, 0x08]


# ---------------------------------------------------------------------------
# tile formats
# ---------------------------------------------------------------------------
def test_fp8_tile_scale_and_bound():
    rng = np.random.default_rng(1)
    t = (rng.standard_normal((5, 8, 64)) * 10.0 ** rng.integers(-3, 3, (5, 1, 1))).astype(np.float32)
    codes, s = oracle.quant_fp8(t)
    amax = np.abs(t).reshape(5, -1).max(1)
    np.testing.assert_array_equal(s, (amax / np.float32(448)).astype(np.float32))
    # the largest element lands on +-448
    for i in range(5):
        j = np.argmax(np.abs(t[i]))
        assert codes[i].ravel()[j] & 0x7F == 0x7E
    deq = oracle.dequant_fp8(codes, s)
    err = np.abs(deq - t)
    # half an ulp of a 3-bit mantissa (normal range) or of 2^-9 (subnormal), times s
    bound = np.maximum(np.abs(t) * 2.0 ** -4, 2.0 ** -10 * s[:, None, None])
    assert np.all(err <= bound * (1 + 1e-6))


def test_fp8_zero_tile():
    codes, s = oracle.quant_fp8(np.zeros((1, 4, 16), np.float32))
    assert s[0] == 0 and not codes.any()


def _nvfp4_representable(rng, rows, cols):
    """A tile whose every block is exactly representable: block values are
    E2M1 values times an E4M3 block scale times s_t = 2^-10, and one block
    reaches the tile maximum 6 * 448 * s_t."""
    st = 2.0 ** -10
    e2 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    e4 = np.array([v for _, v in _table("e4m3") if 0 < v <= 448])
    t = np.zeros((rows, cols))
    for r in range(rows):
        for j in range(cols // 16):
            bs = rng.choice(e4)
            blk = rng.choice(e2, 16) * rng.choice([-1, 1], 16)
            blk[rng.integers(16)] = 6.0 * rng.choice([-1, 1])  # block max = 6 * bs
            t[r, j * 16:(j + 1) * 16] = blk * bs * st
    t[0, :16] = np.abs(t[0, :16]) / np.abs(t[0, :16]).max() * 6 * 448 * st
    t[0, :16] = np.round(t[0, :16] / (448 * st) * 2) / 2 * 448 * st  # back on the E2M1 grid
    t[0, 0] = 6 * 448 * st
    return t.astype(np.float32)


def test_nvfp4_representable_tile_round_trips():
    rng = np.random.default_rng(2)
    t = np.stack([_nvfp4_representable(rng, 4, 64) for _ in range(3)])
    codes, bsc, ts = oracle.quant_nvfp4(t)
    assert np.all(ts == np.float32(2.0 ** -10))
    np.testing.assert_array_equal(oracle.dequant_nvfp4(codes, bsc, ts), t.astype(np.float64))


def test_nvfp4_packing_low_nibble_first():
    t = np.zeros((1, 1, 16), np.float32)
    t[0, 0, :4] = [6.0, 1.0, -0.5, 3.0]
    codes, bsc, ts = oracle.quant_nvfp4(t)
    # amax 6 -> s_t = 6/2688, block scale = E4M3(6 / (6 s_t)) = 448 (code 0x7E)
    assert bsc[0, 0, 0] == 0x7E
    assert codes[0, 0, 0] == (0x7 | (0x2 << 4))   # elements 0 (6.0) and 1 (1.0)
    assert codes[0, 0, 1] == (0x9 | (0x5 << 4))   # elements 2 (-0.5) and 3 (3.0)


def test_nvfp4_bound_and_zero_blocks():
    rng = np.random.default_rng(3)
    t = (rng.standard_normal((4, 8, 64)) * 0.1).astype(np.float32)
    t[1, 2, 16:32] = 0.0
    codes, bsc, ts = oracle.quant_nvfp4(t)
    assert bsc[1, 2, 1] == 0
    deq = oracle.dequant_nvfp4(codes, bsc, ts)
    amax_blk = np.abs(t).reshape(4, 8, 4, 16).max(-1, keepdims=True)
    err = np.abs(deq - t).reshape(4, 8, 4, 16)
    assert np.all(err <= amax_blk * 17.0 / 96.0 + 1e-30)
    np.testing.assert_array_equal(deq[1, 2, 16:32], 0.0)
