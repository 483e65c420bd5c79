"""Pins of the read-copy rounding oracle (oracle/readcopy.py) against what the
formats' definitions fix: ties to even at the halfway points, the largest
finite values and overflow, the smallest subnormals, signed zero, the bit
layouts, numpy's own IEEE binary16 conversion, an independent integer route
for bfloat16, and brute force over every e4m3 code."""
import numpy as np
import pytest

from oracle import readcopy as rc


def f32(v):
    return np.asarray(v, np.float32)


# ----------------------------------------------------------------------------- bfloat16

def test_bf16_ties_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: the even neighbour is 1
    assert rc.to_bf16(f32(1 + 2 ** -8)) == 1.0
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert rc.to_bf16(f32(1 + 3 * 2 ** -8)) == 1 + 2 ** -6
    # just above the halfway point rounds up
    assert rc.to_bf16(f32(1 + 2 ** -8 + 2 ** -20)) == 1 + 2 ** -7
    assert rc.to_bf16(f32(-(1 + 2 ** -8 + 2 ** -20))) == -(1 + 2 ** -7)


def test_bf16_range_ends_and_codes():
    top = (2 - 2 ** -7) * 2.0 ** 127
    assert rc.to_bf16(f32(top)) == top
    assert np.isposinf(rc.to_bf16(f32(3.4e38)))              # beyond top + half a spacing
    assert rc.to_bf16(f32(2.0 ** -133)) == 2.0 ** -133         # smallest bf16 subnormal
    assert rc.to_bf16(f32(2.0 ** -134)) == 0.0                 # halfway to 0: even neighbour 0
    z = rc.to_bf16(f32(-0.0))
    assert z == 0 and np.signbit(z)
    assert rc.bf16_bits([1.0, -2.0, 0.0, -0.0, np.inf]).tolist() == [0x3F80, 0xC000, 0, 0x8000, 0x7F80]


def test_bf16_against_integer_route():
    """An independent derivation: RNE on the binary32 bit pattern (add
    0x7FFF plus the lowest kept bit, drop 16 bits)."""
    g = np.random.default_rng(3)
    x = np.concatenate([g.standard_normal(20000) * 10.0 ** g.uniform(-40, 38, 20000),
                        g.standard_normal(2000) * 1e-39]).astype(np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    want = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    got = rc.bf16_bits(rc.to_bf16(x))
    np.testing.assert_array_equal(got, want)


# ----------------------------------------------------------------------------- fp16

def test_fp16_ties_overflow_subnormals():
    assert rc.to_fp16(f32(1 + 2 ** -11)) == 1.0
    assert rc.to_fp16(f32(1 + 3 * 2 ** -11)) == 1 + 2 ** -9
    assert rc.to_fp16(f32(65519.0)) == 65504.0          # below the halfway point 65520
    assert np.isposinf(rc.to_fp16(f32(65520.0)))        # halfway, the even neighbour is 2^16: overflow
    assert rc.to_fp16(f32(2.0 ** -24)) == 2.0 ** -24    # smallest subnormal
    assert rc.to_fp16(f32(2.0 ** -25)) == 0.0           # halfway to 0
    assert rc.to_fp16(f32(3 * 2.0 ** -26)) == 2.0 ** -24
    assert rc.fp16_bits([1.0, -2.0, 65504.0, 2.0 ** -24]).tolist() == [0x3C00, 0xC000, 0x7BFF, 0x0001]


def test_fp16_against_numpy_binary16():
    """numpy's float32 -> float16 cast is IEEE round-to-nearest-even."""
    g = np.random.default_rng(4)
    x = np.concatenate([g.standard_normal(20000) * 10.0 ** g.uniform(-9, 5.5, 20000),
                        (np.arange(-3000, 3000) * 2.0 ** -26)]).astype(np.float32)
    want = x.astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(rc.to_fp16(x), want)


# ----------------------------------------------------------------------------- e4m3

def all_e4m3():
    """Every finite e4m3 code and its value, decoded from the bit layout."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = []
    for c in codes.tolist():
        s = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 7
        vals.append(s * (m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)))
    return codes, np.array(vals)


def test_e4m3_codes_and_values():
    codes, vals = all_e4m3()
    np.testing.assert_array_equal(rc.e4m3_value(codes), vals)
    np.testing.assert_array_equal(rc.e4m3_bits(vals[vals != 0]), codes[vals != 0])
    assert rc.e4m3_bits([448.0, -448.0, 1.0, 2.0 ** -9, 0.0, -0.0]).tolist() == [0x7E, 0xFE, 0x38, 0x01, 0x00, 0x80]
    assert np.isnan(rc.e4m3_value(0x7F)) and np.isnan(rc.e4m3_value(0xFF))


def test_e4m3_ties_saturation_subnormals():
    assert rc.to_e4m3(1 + 2 ** -4) == 1.0            # tie between 1 and 1.125: even
    assert rc.to_e4m3(1 + 3 * 2 ** -4) == 1.25       # tie between 1.125 and 1.25: even
    assert rc.to_e4m3(464.0) == 448.0                # beyond the largest value: saturates
    assert rc.to_e4m3(-1e9) == -448.0
    assert rc.to_e4m3(2.0 ** -10) == 0.0             # halfway to the smallest subnormal
    assert rc.to_e4m3(1.5 * 2.0 ** -10) == 2.0 ** -9


def test_e4m3_brute_force_nearest():
    """Every value's code is the nearest finite e4m3 value, ties to the even
    code, anything beyond 448 saturating."""
    codes, vals = all_e4m3()
    pos = vals[(vals > 0)]
    g = np.random.default_rng(5)
    mids = (np.sort(pos)[1:] + np.sort(pos)[:-1]) / 2           # every tie
    x = np.concatenate([g.uniform(-500, 500, 5000), g.standard_normal(5000) * 2.0 ** -8, mids, -mids])
    got = rc.to_e4m3(x)
    for xi, gi in zip(x, got):
        if abs(xi) > 448:
            assert gi == np.copysign(448.0, xi)
            continue
        d = np.abs(vals - xi)
        best = vals[d == d.min()]
        if len(set(best.tolist())) > 1:      # a tie: the code with the even trailing bit
            cand = [v for v in set(best.tolist()) if (int(rc.e4m3_bits(v)) & 1) == 0]
            assert gi == cand[0], xi
        else:
            assert gi == best[0], xi


def test_e4m3_rows_scaling():
    """A row's scale is max|row| / 448 and its values map its largest element
    to 448; a zero row gives scale 0."""
    x = np.zeros((2, 128), np.float32)
    x[0, :4] = [2.0, -1.0, 0.5, 2.0 ** -20]
    codes, scales = rc.e4m3_rows(x)
    assert scales[0] == np.float32(2.0) / np.float32(448.0) and scales[1] == 0.0
    # 2 -> 448 (0x7E); -1 -> -224 = -1.75 * 2^7 (0xF6); 0.5 -> 112 = 1.75 * 2^6 (0x6E); tiny -> 0
    assert codes[0, :4].tolist() == [0x7E, 0xF6, 0x6E, 0x00]
    assert not codes[1].any()
    back = rc.e4m3_rows_value(codes, scales)
    assert back[0, 0] == np.float32(448.0) * np.float64(scales[0])


def test_e4m3_rows_error_bound():
    """Read back through its row scale, every element is within half an e4m3
    spacing of the row-scaled value: relative 2^-4 for the normals."""
    g = np.random.default_rng(6)
    x = (g.standard_normal((64, 128)) * 10.0 ** g.uniform(-3, 3, (64, 1))).astype(np.float32)
    codes, scales = rc.e4m3_rows(x)
    back = rc.e4m3_rows_value(codes, scales)
    sub = np.abs(x) < 2.0 ** -6 * scales[:, None]
    rel = np.abs(back - x) / np.abs(x)
    assert (rel[~sub] <= 2.0 ** -4 * (1 + 1e-6)).all()
    assert (np.abs(back - x)[sub] <= 2.0 ** -10 * np.broadcast_to(scales[:, None], x.shape)[sub] * (1 + 1e-6)).all()


@pytest.mark.parametrize("fmt", ["bf16", "fp16"])
def test_rounding_is_idempotent_and_monotone(fmt):
    f = rc.to_bf16 if fmt == "bf16" else rc.to_fp16
    g = np.random.default_rng(7)
    x = np.sort(g.standard_normal(5000).astype(np.float32) * 100)
    r = f(x)
    np.testing.assert_array_equal(f(r.astype(np.float32)), r)
    assert (np.diff(r) >= 0).all()


# ----------------------------------------------------------------------------- emulated read precisions

def test_emulated_bf16_fp16_are_the_read_copies():
    """Emulated without a scale, bf16 and fp16 read exactly what the stored
    read copies hold (within range: the emulated formats saturate)."""
    g = np.random.default_rng(8)
    h = (g.standard_normal((2, 64, 128)) * 0.1).astype(np.float32)
    np.testing.assert_array_equal(rc.emulate_read(h, "bf16", "none"), rc.to_bf16(h))
    np.testing.assert_array_equal(rc.emulate_read(h, "fp16", "none"), rc.to_fp16(h))
    assert rc.emulate_read(np.float32([1e6]), "fp16", "none")[0] == 65504.0   # saturates


def test_emulated_e4m3_row_scale_is_the_fp8_read_copy():
    g = np.random.default_rng(9)
    h = (g.standard_normal((3, 64, 128)) * 10.0 ** g.uniform(-3, 1, (3, 64, 1))).astype(np.float32)
    h[0, 5] = 0.0
    codes, scales = rc.e4m3_rows(h)
    want = (rc.e4m3_value(codes).astype(np.float32) * scales[..., None]).astype(np.float32)
    np.testing.assert_array_equal(rc.emulate_read(h, "e4m3", "row"), want.astype(np.float64))


def test_emulated_tile_scale_groups_64_rows():
    """One scale per 64-row block: scaling one block leaves the other's reads
    unchanged, and each block's largest element reads back exactly."""
    g = np.random.default_rng(10)
    h = (g.standard_normal((128, 128)) * 0.1).astype(np.float32)
    r1 = rc.emulate_read(h, "int8", "tile64")
    h2 = h.copy()
    h2[64:] *= 8
    r2 = rc.emulate_read(h2, "int8", "tile64")
    np.testing.assert_array_equal(r1[:64], r2[:64])
    h3 = h.copy()
    h3[32:64] *= 8                        # same block as rows 0..31: their scale grows with it
    assert not np.array_equal(rc.emulate_read(h3, "int8", "tile64")[:32], r1[:32])
    for blk in (h[:64], h[64:]):
        i = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
        assert rc.emulate_read(blk, "int8", "tile64")[i] == pytest.approx(float(blk[i]), rel=1e-6)


def test_emulated_int8_closed_form():
    """A row with max 127/128 has scale 1/128 and reciprocal 128 (both exact):
    the codes are 128 v rounded half to even -- 2^-8 -> 0.5 -> 0,
    1.5/128 -> 2, -2.5/128 -> -2, 100.5/128 -> 100 -- and read back as
    code / 128; the largest element reads back exactly."""
    row = np.zeros((1, 128), np.float32)
    row[0, :5] = [127 / 128, 2.0 ** -8, 1.5 / 128, -2.5 / 128, 100.5 / 128]
    r = rc.emulate_read(row, "int8", "row")[0, :5]
    np.testing.assert_array_equal(r, [127 / 128, 0.0, 2 / 128, -2 / 128, 100 / 128])
    assert np.all(rc.emulate_read(row, "int8", "row")[0, 5:] == 0)


@pytest.mark.parametrize("fmt,scale,bound", [("bf16", "none", 2.0 ** -8), ("fp16", "none", 2.0 ** -11),
                                             ("e4m3", "row", 2.0 ** -4), ("e5m2", "row", 2.0 ** -3),
                                             ("e4m3", "tile64", 2.0 ** -4)])
def test_emulated_error_bounds(fmt, scale, bound):
    """Relative error of an emulated read of normal-range values is at most
    half a spacing of the format: 2^-p."""
    g = np.random.default_rng(11)
    h = (g.standard_normal((2, 64, 128)) * 0.1).astype(np.float32)
    r = rc.emulate_read(h, fmt, scale)
    big = np.abs(h) > 0.05 * np.abs(h).max()
    rel = np.abs(r - h)[big] / np.abs(h)[big]
    assert rel.max() <= bound * (1 + 1e-6)
    e, n = rc.emulation_error(h, fmt, scale)
    assert 0 < e < (bound ** 2) * n


def test_emulated_formats_need_their_scales():
    h = np.ones((64, 128), np.float32)
    for fmt in ("e4m3", "e5m2", "int8"):
        with pytest.raises(ValueError):
            rc.emulate_read(h, fmt, "none")
    for fmt in ("bf16", "fp16"):
        with pytest.raises(ValueError):
            rc.emulate_read(h, fmt, "row")
