"""FP8 (E4M3) page pools for the oracle (test infrastructure only).

The pages define the pool as bf16; an 8-bit pool is a variant this library
adds (it halves the bytes of an HBM-bound path).  The readings taken, each
stated once here and in the design notes:

  * Format: the OCP 8-bit E4M3 ("E4M3FN") encoding: 1 sign bit, 4 exponent
    bits with bias 7, 3 mantissa bits; exponent field 0 holds subnormals
    (m * 2^-9); no infinities; S.1111.111 is NaN, so the largest finite
    magnitude is 1.75 * 2^8 = 448.
  * Scales: one float32 scale per pool (k_scale for K, v_scale for V); a code
    c stands for decode(c) * scale.
  * Quantizer: a stored element is first the bf16 value the bf16 pool would
    hold (the rotated, rounded K; the V input), then
        code = RNE_e4m3(fl32(value / scale))
    with one IEEE float32 division and round-to-nearest-even to E4M3,
    saturating to +-448 (a finite value never becomes NaN; NaN stays NaN).
  * Attention over an 8-bit pool is the exact attention of the dequantized
    keys and values.
"""
import numpy as np

from . import bf16
from . import paged

MAX_FINITE = 448.0
NAN_CODES = (0x7F, 0xFF)


def decode(codes) -> np.ndarray:
    """Value of each E4M3 code (float64; NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def _finite_values() -> np.ndarray:
    """The 127 non-negative finite E4M3 magnitudes in increasing order (codes 0x00..0x7E)."""
    return decode(np.arange(0x7F, dtype=np.uint8))


def encode(x) -> np.ndarray:
    """Round each value (float64 holding a float32) to the nearest E4M3 code,
    ties to the even code, magnitudes of 448 or more saturating to 448; NaN
    gives the NaN code."""
    x = np.asarray(x, dtype=np.float64)
    mags = _finite_values()                    # ascending; the code of mags[i] is i
    a = np.abs(x)
    nan, sat = np.isnan(a), a >= MAX_FINITE
    ac = np.where(nan | sat, 0.0, a)
    hi = np.minimum(np.searchsorted(mags, ac, side="left"), 0x7E)  # first magnitude >= value
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = ac - mags[lo], mags[hi] - ac
    take_lo = (dlo < dhi) | ((dlo == dhi) & (lo % 2 == 0))
    code = np.where(mags[hi] == ac, hi, np.where(take_lo, lo, hi))
    code = np.where(sat, 0x7E, np.where(nan, 0x7F, code)).astype(np.uint8)
    sign = (np.signbit(x) & ~nan).astype(np.uint8) << 7
    return code | sign


def quantize(bits, scale: float) -> np.ndarray:
    """Codes of bf16 values `bits` for a pool with float32 `scale`."""
    q = bf16.to_f64(bits).astype(np.float32) / np.float32(scale)  # one IEEE float32 division
    return encode(q.astype(np.float64))


def dequantize(codes, scale: float) -> np.ndarray:
    return decode(codes) * float(np.float32(scale))


def append_rope(q, k, v, positions, rows, table, k_codes, v_codes, inv, k_scale, v_scale,
                slots=None, gamma_q=None, gamma_k=None, eps=1e-6):
    """The bf16 append (oracle.paged.append_rope) followed by the quantizer on
    the slots it writes.  Returns (q_out, k_codes', v_codes')."""
    shape = k_codes.shape
    scratch = np.zeros(shape, dtype=np.uint16)
    q_out, kb, vb = paged.append_rope(q, k, v, positions, rows, table, scratch, scratch, inv,
                                      slots=slots, gamma_q=gamma_q, gamma_k=gamma_k, eps=eps)
    k_codes = np.array(k_codes, dtype=np.uint8, copy=True)
    v_codes = np.array(v_codes, dtype=np.uint8, copy=True)
    for t in range(q.shape[0]):
        p = int(positions[t])
        if p < 0:
            continue
        s = int(slots[t]) if slots is not None else paged.slot_of(table, int(rows[t]), p)
        k_codes[:, s, :] = quantize(kb[:, s, :], k_scale)
        v_codes[:, s, :] = quantize(vb[:, s, :], v_scale)
    return q_out, k_codes, v_codes


def attention_at(q_bits, row, position, table, k_codes, v_codes, k_scale, v_scale, window, scale=None):
    """Output of one token over its row's visible keys of 8-bit pools: exact
    attention of the dequantized keys and values.  Returns float64 [Hq, D]."""
    hq, d = q_bits.shape
    hkv = k_codes.shape[0]
    group = hq // hkv
    if scale is None:
        scale = paged.default_scale(d)
    out = np.zeros((hq, d), dtype=np.float64)
    if position < 0:
        return out
    lo, hi = paged.visible_range(position, window)
    slots = paged.row_slots(table, row, lo, hi)
    qf = bf16.to_f64(q_bits)
    for kvh in range(hkv):
        heads = [h for h in range(hq) if paged.kv_head_of(h, group, hkv) == kvh]
        keys = dequantize(k_codes[kvh, slots, :], k_scale)
        values = dequantize(v_codes[kvh, slots, :], v_scale)
        out[heads] = paged.attend(qf[heads], keys, values, scale)
    return out


def decode_attention(q_out, positions, table, k_codes, v_codes, k_scale, v_scale, window, scale=None):
    """Decode rows (row b uses table row b) over 8-bit pools."""
    return np.stack([attention_at(q_out[b], b, int(positions[b]), table, k_codes, v_codes, k_scale,
                                  v_scale, window, scale) for b in range(q_out.shape[0])])
