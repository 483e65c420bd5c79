"""Rounding of the fp32 checkpoint to its low-precision read copies (oracle;
test-only).

"ReplaySSM" (the paper's code repository), introduction, "Separate state
precisions": non-flush steps read a low-precision copy of the checkpoint,
flushes update the high-precision one, and the copy's rounding never enters
the recurrence. The pages name no format or rounding rule. The readings
taken: the copy is the fp32 checkpoint rounded to nearest, ties to even, in
one of three formats --

* bfloat16: 8 significant bits, the exponent range of binary32;
* IEEE binary16 (fp16): 11 significant bits, normal exponents -14..15,
  subnormals down to 2^-24, overflow to infinity;
* OCP FP8 E4M3: 4 significant bits, normal exponents -6..8, subnormals down
  to 2^-9, no infinities, largest finite value 448 (the code S.1111.111 is
  NaN); a copy in it saturates at +-448 -- together with one fp32 scale per
  state row of 128 values: scale = max|row| / 448 and each value stored as
  RNE(value * (448 / max|row|)), both quotients and the product taken in
  fp32 (IEEE single: a quantised code is decided in the precision the copy is
  built in).

Rounding is written from the definition: x lies between two neighbours of
the format's grid; the nearer one is taken, the one with an even last
significand bit on a tie. For a binary format with p significant bits and
smallest normal exponent emin, the grid spacing around x is
2^(max(e, emin) - p + 1) with e = floor(log2 |x|), so x / spacing is exact
in fp64 and numpy's round (half to even) picks the neighbour.

Encodings (for comparing the GPU's bytes bit for bit) follow the formats'
bit layouts: sign, biased exponent, trailing significand.

Everything works on numpy arrays; values come back as fp64 (exact: every
value of these formats is an fp64 number).
"""
import numpy as np

# (significant bits p, smallest normal exponent emin, largest finite value)
BF16 = (8, -126, (2.0 - 2.0 ** -7) * 2.0 ** 127)
FP16 = (11, -14, 65504.0)
E4M3 = (4, -6, 448.0)
E4M3_MAX = 448.0


def round_rne(x, fmt, saturate=False):
    """x (any real array) rounded to nearest, ties to even, on the grid of
    format fmt = (p, emin, max_finite). Beyond the largest finite value the
    result is +-inf (IEEE overflow), or +-max_finite when ``saturate``.
    Signed zeros keep their sign; NaN stays NaN."""
    p, emin, vmax = fmt
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    fin = np.isfinite(x) & (a > 0)            # zeros, infinities and NaN are settled below
    a1 = np.where(fin, a, 1.0)
    e = np.floor(np.log2(a1))
    # log2 of a value just below a power of two can round up to the exponent;
    # settle e so that 2^e <= a < 2^(e + 1) holds exactly
    e = np.where(np.ldexp(1.0, e.astype(np.int64)) > a1, e - 1, e)
    e = np.where(np.ldexp(1.0, (e + 1).astype(np.int64)) <= a1, e + 1, e)
    spacing_exp = (np.maximum(e, emin) - p + 1).astype(np.int64)
    q = np.round(np.ldexp(np.where(fin, x, 0.0), -spacing_exp))   # exact scaling; half to even
    r = np.ldexp(q, spacing_exp)
    over = np.abs(r) > vmax
    if saturate:
        r = np.where(over, np.copysign(vmax, x), r)
    else:
        r = np.where(over, np.copysign(np.inf, x), r)
    r = np.where(a == 0, x, r)                        # +-0 kept as given
    r = np.where(np.isnan(x), np.nan, r)
    r = np.where(np.isinf(x), x if not saturate else np.copysign(vmax, x), r)
    return r


def to_bf16(x):
    """fp32 values -> their bfloat16 read copy (values, fp64)."""
    return round_rne(np.asarray(x, np.float32).astype(np.float64), BF16)


def to_fp16(x):
    """fp32 values -> their fp16 read copy (values, fp64)."""
    return round_rne(np.asarray(x, np.float32).astype(np.float64), FP16)


def to_e4m3(x):
    """Real values -> e4m3 (values, fp64), saturating at +-448."""
    return round_rne(x, E4M3, saturate=True)


def bf16_bits(v):
    """bfloat16 values -> uint16 codes: the upper half of the value's binary32
    encoding (a bfloat16 value is a binary32 value whose lower 16 bits are 0)."""
    u = np.asarray(v, np.float64).astype(np.float32).view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("not a bfloat16 value")
    return (u >> 16).astype(np.uint16)


def fp16_bits(v):
    """fp16 values -> uint16 codes (binary16 layout: 1 sign, 5 exponent bits
    biased by 15, 10 trailing significand bits)."""
    v = np.asarray(v, np.float64)
    h = v.astype(np.float16)
    if not np.array_equal(h.astype(np.float64), v, equal_nan=True):
        raise ValueError("not an fp16 value")
    return h.view(np.uint16)


def e4m3_bits(v):
    """e4m3 values -> uint8 codes: 1 sign bit, 4 exponent bits biased by 7,
    3 trailing significand bits; exponent field 0 holds the subnormals
    m * 2^-9."""
    v = np.asarray(v, np.float64)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    a = np.abs(v)
    code = np.zeros(a.shape, np.uint8)
    sub = a < 2.0 ** -6
    m_sub = a / 2.0 ** -9
    with np.errstate(divide="ignore", invalid="ignore"):
        e = np.floor(np.log2(np.where(sub, 1.0, a)))
    frac = np.where(sub, 0.0, a / np.ldexp(1.0, e.astype(np.int64)) - 1.0) * 8
    ok = np.where(sub, m_sub == np.round(m_sub), frac == np.round(frac)) & (a <= E4M3_MAX)
    if not ok.all():
        raise ValueError("not an e4m3 value")
    code = np.where(sub, m_sub, ((e + 7).astype(np.int64) << 3) + frac).astype(np.uint8)
    return code | sign


def e4m3_value(codes):
    """uint8 e4m3 codes -> values (fp64); the two NaN codes give NaN."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ef, mf = (c >> 3) & 0xF, c & 0x7
    v = np.where(ef == 0, mf * 2.0 ** -9, (1.0 + mf / 8.0) * np.ldexp(1.0, ef - 7))
    v = np.where((ef == 0xF) & (mf == 0x7), np.nan, v)
    return s * v


def e4m3_rows(x):
    """The fp8 read copy of fp32 rows x [..., n]: (codes uint8 [..., n], scales
    fp32 [...]). Per row m = max|x| (fp32); scale = m / 448 and every value is
    stored as RNE_e4m3(x * (448 / m)), saturating, with the quotients and the
    product in fp32; a row of zeros has scale 0 and codes 0."""
    x = np.asarray(x, np.float32)
    m = np.max(np.abs(x), axis=-1, keepdims=True)
    c448 = np.float32(E4M3_MAX)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.where(m > 0, c448 / m, np.float32(0)).astype(np.float32)
    t = (x * inv).astype(np.float32)                  # fp32 product
    codes = e4m3_bits(to_e4m3(t.astype(np.float64)))
    scales = (m / c448).astype(np.float32)[..., 0]
    return codes, scales


def e4m3_rows_value(codes, scales):
    """Values an fp8 read copy stands for: e4m3 value * its row's scale."""
    return e4m3_value(codes) * np.asarray(scales, np.float64)[..., None]


# ----------------------------------------------------------------------------- emulated read precisions

# "ReplaySSM" (the paper's code repository), introduction: the emulation
# kernels implement separate read and recurrence precision and expose their
# quantization behavior. Reading taken: the non-flush read of the fp32
# checkpoint goes through a quantise-dequantise in a chosen format (nothing
# low-precision is stored), flushes read the fp32 checkpoint exactly, and
# the call reports the quantisation error of what it read.
#
# Formats: (significant bits p, smallest normal exponent emin, largest finite
# value); every format saturates at its largest value. INT8 is symmetric
# 8-bit fixed point: RNE to an integer, clamped to [-127, 127].
EMU_FORMATS = {
    "bf16": BF16,
    "fp16": FP16,
    "e4m3": E4M3,
    "e5m2": (3, -14, 57344.0),
    "int8": None,
}
# Scaled formats (a scale per state row of dstate values, or per 64-row tile)
# store value / s with s = max|group| / qmax; bf16 and fp16 take no scale.
EMU_QMAX = {"e4m3": 448.0, "e5m2": 57344.0, "int8": 127.0}


def emulate_quantise(t, fmt):
    """t (already divided by its scale) rounded into format fmt, saturating."""
    t = np.asarray(t, np.float64)
    if fmt == "int8":
        return np.clip(np.round(t), -127.0, 127.0)     # half to even
    return round_rne(t, EMU_FORMATS[fmt], saturate=True)


def emulate_read(h, fmt, scale):
    """The emulated read of fp32 checkpoint rows h [..., rows, n]: the value
    each element reads as. scale: "none", "row" (one scale per row of n
    values) or "tile64" (one per 64-row block of a (sequence, head) tile).
    The scale s = max|group| / qmax and its reciprocal qmax / max|group| are
    fp32 divisions, the scaled value x * (qmax / max|group|) an fp32 product
    (a code is decided in the precision the kernel computes in), and the read
    value code * s an fp32 product; a group of zeros reads as zeros."""
    h = np.asarray(h, np.float32)
    if scale == "none":
        if fmt not in ("bf16", "fp16"):
            raise ValueError("e4m3, e5m2 and int8 are emulated with a scale")
        return emulate_quantise(h.astype(np.float64), fmt)
    if fmt not in EMU_QMAX:
        raise ValueError("bf16 and fp16 are emulated without a scale")
    qmax = np.float32(EMU_QMAX[fmt])
    if scale == "row":
        m = np.max(np.abs(h), axis=-1, keepdims=True)
    elif scale == "tile64":
        rows = h.shape[-2]
        blocks = h.reshape(h.shape[:-2] + (rows // 64, 64, h.shape[-1]))
        m = np.max(np.abs(blocks), axis=(-2, -1), keepdims=True)
        m = np.broadcast_to(m, blocks.shape[:-1] + (1,)).reshape(h.shape[:-1] + (1,))
    else:
        raise ValueError(scale)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.where(m > 0, qmax / m, np.float32(0)).astype(np.float32)
    s = (m / qmax).astype(np.float32)
    t = (h * inv).astype(np.float32)
    q = emulate_quantise(t.astype(np.float64), fmt).astype(np.float32)
    return (q * s).astype(np.float32).astype(np.float64)


def emulation_error(h, fmt, scale):
    """The quantisation behaviour of one emulated read: (sum of squared
    errors, sum of squares of the exact values) over h."""
    h64 = np.asarray(h, np.float32).astype(np.float64)
    d = emulate_read(h, fmt, scale) - h64
    return float(np.sum(d * d)), float(np.sum(h64 * h64))
