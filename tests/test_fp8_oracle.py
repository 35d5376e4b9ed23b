"""Pins of the oracle's 8-bit (E4M3) pool format: closed-form code values,
the format's defining counts, round-to-nearest-even ties worked by hand,
saturation, agreement with PyTorch's float8_e4m3fn conversions (a library
routine), and attention over a pool whose codes are exactly its bf16 values.
Planted mistakes (wrong bias, truncation, overflow to NaN) must fail them."""
import numpy as np
import pytest

from oracle import bf16, fp8, paged


def _bits(values):
    return bf16.from_f64(np.asarray(values, dtype=np.float64))


def check_decode_closed_forms(dec):
    v = dec(np.arange(256, dtype=np.uint8))
    assert v[0x38] == 1.0 and v[0xB8] == -1.0          # exponent field 7 = bias
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0      # largest finite: 1.75 * 2^8
    assert v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9   # subnormals m * 2^-9
    assert v[0x08] == 2.0 ** -6                        # smallest normal
    assert v[0x39] == 1.125 and v[0x3F] == 1.875 and v[0x40] == 2.0
    assert v[0x00] == 0.0 and np.signbit(v[0x80])
    nan = np.isnan(v)
    assert np.array_equal(np.nonzero(nan)[0], [0x7F, 0xFF])   # exactly two NaN codes, no infinities
    assert np.all(np.isfinite(v[~nan]))
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                    # codes 0..126 in increasing order


def check_encode_ties_and_saturation(enc):
    # exact values map to their codes
    assert list(enc([1.0, -1.0, 448.0, 2.0 ** -9, 0.0])) == [0x38, 0xB8, 0x7E, 0x01, 0x00]
    # halfway cases go to the even code (mantissa lsb 0)
    assert enc([1.0625])[0] == 0x38       # between 1.0 (0x38) and 1.125 (0x39)
    assert enc([1.1875])[0] == 0x3A       # between 1.125 (0x39) and 1.25 (0x3A)
    assert enc([-1.1875])[0] == 0xBA
    assert enc([1.5 * 2.0 ** -9])[0] == 0x02   # subnormal tie between 1 and 2 units
    assert enc([0.5 * 2.0 ** -9])[0] == 0x00   # tie between 0 and the smallest subnormal
    assert enc([1.9375])[0] == 0x40       # between 1.875 (0x3F) and 2.0 (0x40): even is 0x40
    # just off the halfway point
    assert enc([1.0625 + 2 ** -20])[0] == 0x39 and enc([1.0625 - 2 ** -20])[0] == 0x38
    # saturation: finite values never become NaN
    assert list(enc([447.9, 460.0, 464.0, 1e6, -1e6])) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
    assert enc([np.nan])[0] & 0x7F == 0x7F


def test_decode_closed_forms():
    check_decode_closed_forms(fp8.decode)


def test_encode_ties_and_saturation():
    check_encode_ties_and_saturation(fp8.encode)


def test_decode_and_encode_match_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.decode(codes)
    fin = ~np.isnan(got)
    assert np.array_equal(np.isnan(want), ~fin) and np.array_equal(got[fin], want[fin])
    # every finite code round-trips
    assert np.array_equal(fp8.encode(got[fin]), codes[fin])
    # float32 values inside the finite range: torch's round-to-nearest-even conversion
    x = (np.random.default_rng(3).standard_normal(200000) * np.exp2(np.random.default_rng(4).integers(-12, 8, 200000)))
    x = x.astype(np.float32).astype(np.float64)
    x = x[np.abs(x) < 448.0]
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.encode(x), t)


def test_quantize_is_one_float32_division_then_rne():
    # 3 / fl32(0.1) in float32 differs from the float64 quotient; the code follows float32
    q = np.float32(3.0) / np.float32(0.1)
    assert fp8.quantize(_bits([3.0]), 0.1)[0] == fp8.encode([float(q)])[0]
    assert fp8.quantize(_bits([1.0]), 1.0)[0] == 0x38
    assert fp8.quantize(_bits([2.0]), 0.5)[0] == 0x48      # 4.0
    assert fp8.quantize(_bits([-600.0]), 1.0)[0] == 0xFE   # saturates


def test_attention_over_codes_equals_bf16_attention_of_their_values():
    """A pool whose codes decode (scale 1) to bf16-exact values gives the same
    attention as the bf16 pool holding those values."""
    rng = np.random.default_rng(5)
    hkv, hq, d, npages = 2, 8, 64, 3
    codes_k = rng.integers(0x20, 0x48, size=(hkv, npages * 64, d)).astype(np.uint8) | \
        (rng.integers(0, 2, size=(hkv, npages * 64, d)).astype(np.uint8) << 7)
    codes_v = rng.integers(0x20, 0x48, size=(hkv, npages * 64, d)).astype(np.uint8)
    kb, vb = _bits(fp8.decode(codes_k)), _bits(fp8.decode(codes_v))
    assert np.array_equal(bf16.to_f64(kb), fp8.decode(codes_k))  # bf16-exact
    table = np.array([[2, 0, 1]], dtype=np.int32)
    q = _bits(rng.standard_normal((hq, d)))
    for pos in (0, 63, 100, 191):
        a = fp8.attention_at(q, 0, pos, table, codes_k, codes_v, 1.0, 1.0, 0)
        b = paged.attention_at(q, 0, pos, table, kb, vb, 0)
        assert np.allclose(a, b, rtol=0, atol=1e-12)
    # and scales multiply the values
    a = fp8.attention_at(q, 0, 150, table, codes_k, codes_v, 1.0, 0.25, 0)
    b = paged.attention_at(q, 0, 150, table, kb, vb, 0)
    assert np.allclose(a, 0.25 * b, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- mutations ----

def _decode_bias8(codes):
    return fp8.decode(codes) / 2.0


def _encode_truncating(x):
    x = np.asarray(x, dtype=np.float64)
    mags = fp8._finite_values()
    a = np.minimum(np.abs(np.nan_to_num(x)), fp8.MAX_FINITE)
    code = np.searchsorted(mags, a, side="right") - 1
    return (code.astype(np.uint8) | (np.signbit(x).astype(np.uint8) << 7)).astype(np.uint8)


def _encode_overflow_nan(x):
    out = fp8.encode(x)
    big = np.abs(np.asarray(x, dtype=np.float64)) > fp8.MAX_FINITE
    return np.where(big, out | 0x7F, out).astype(np.uint8)


@pytest.mark.parametrize("check, wrong", [
    (check_decode_closed_forms, _decode_bias8),
    (check_encode_ties_and_saturation, _encode_truncating),
    (check_encode_ties_and_saturation, _encode_overflow_nan),
])
def test_pins_catch_planted_mistakes(check, wrong):
    with pytest.raises(AssertionError):
        check(wrong)
