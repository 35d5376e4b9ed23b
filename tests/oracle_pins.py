"""Pins for the CPU oracle: facts fixed by the pages or by the mathematics.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
the fact it checks.  ``test_oracle_pins.py`` runs them all;
``test_oracle_mutations.py`` plants plausible mistakes in the oracle and checks
that some pin fails for each.
"""
import json
import math
from pathlib import Path

import numpy as np

from oracle import bf16, paged, rope

GOLDEN = json.loads((Path(__file__).parent / "golden" / "pages_facts.json").read_text())


def _rand_bits(rng, shape, scale=1.0):
    return bf16.from_f64(rng.standard_normal(shape) * scale)


# ---------------------------------------------------------------- bf16 ----

def pin_bf16_rounding():
    """Direct float64 -> bf16 rounding: agrees with torch's float32 -> bf16 cast
    (round to nearest even) on float32 inputs, and rounds once from float64."""
    import torch
    rng = np.random.default_rng(0)
    x32 = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    t = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16.from_f64(x32.astype(np.float64)), t)
    # ties go to even; a float64 just above a tie rounds up (no double rounding)
    one = 1.0
    cases = {one + 2.0 ** -8: one, one + 3 * 2.0 ** -8: one + 2.0 ** -6,
             one + 2.0 ** -8 + 2.0 ** -30: one + 2.0 ** -7, -(one + 2.0 ** -8): -one}
    for x, want in cases.items():
        assert bf16.to_f64(bf16.from_f64(np.array([x])))[0] == want, x
    # round trip is exact
    b = _rand_bits(rng, 1000)
    assert np.array_equal(bf16.from_f64(bf16.to_f64(b)), b)


# ---------------------------------------------------------------- tables ----

def pin_inv_freq_exact():
    """The float32 table is within 1e-6 relative of theta**(-2i/D) (exact)."""
    import mpmath
    mpmath.mp.dps = 40
    for theta, d in [(10000.0, 96), (1e6, 128), (5e5, 128), (10000.0, 64)]:
        inv = rope.inv_freq_plain(theta, d).astype(np.float64)
        exact = np.array([float(mpmath.power(theta, -mpmath.mpf(2 * i) / d)) for i in range(d // 2)])
        assert inv[0] == 1.0
        assert np.max(np.abs(inv - exact) / exact) < 1e-6
        assert np.all(np.diff(inv) < 0)


def pin_inv_freq_float32_agreement():
    """The llama3-scaled table agrees with the same three-band rule evaluated in
    float32 library ops (torch.pow / where) to the level the Llama page reports."""
    import torch
    g = GOLDEN["llama3_table"]
    ours = rope.inv_freq(g["theta"], g["head_dim"], (g["factor"], g["low_freq_factor"],
                                                    g["high_freq_factor"], g["original_max_position"]))
    d = g["head_dim"]
    base = 1.0 / torch.pow(torch.tensor(g["theta"], dtype=torch.float32),
                           torch.arange(0, d, 2, dtype=torch.float32) / d)
    wl = 2 * math.pi / base
    lo_wl = g["original_max_position"] / g["low_freq_factor"]
    hi_wl = g["original_max_position"] / g["high_freq_factor"]
    smooth = (g["original_max_position"] / wl - g["low_freq_factor"]) / (g["high_freq_factor"] - g["low_freq_factor"])
    blend = (1 - smooth) * base / g["factor"] + smooth * base
    ref = torch.where(wl > lo_wl, base / g["factor"], torch.where(wl < hi_wl, base, blend))
    worst = float(np.max(np.abs(ours.astype(np.float64) - ref.numpy().astype(np.float64))))
    # the page prints the agreement to three significant digits
    assert float(f"{worst:.3g}") <= g["table_agreement_abs"], worst


def pin_llama3_band():
    """Only frequencies 29..34 of 64 are blended; the rest are unchanged or divided by 8."""
    g = GOLDEN["llama3_table"]
    base = rope.inv_freq_plain(g["theta"], g["head_dim"])
    sc = rope.inv_freq(g["theta"], g["head_dim"], (g["factor"], g["low_freq_factor"],
                                                  g["high_freq_factor"], g["original_max_position"]))
    assert len(sc) == g["num_frequencies"]
    ratio = base.astype(np.float64) / sc.astype(np.float64)
    band = [i for i in range(len(sc)) if 1.0 < ratio[i] < g["factor"]]
    assert band == list(range(g["blend_band_first_index"], g["blend_band_last_index"] + 1))
    assert np.array_equal(sc[:band[0]], base[:band[0]])
    assert np.array_equal(sc[band[-1] + 1:] * np.float32(g["factor"]), base[band[-1] + 1:])
    # blended values lie strictly between the two neighbouring bands' rules
    for i in band:
        assert base[i] / g["factor"] < sc[i] < base[i]


def pin_llama3_continuity():
    """At wavelen == 2048 the blend gives the unscaled frequency (smooth = 1);
    at wavelen == 8192 it gives the divided one: the rule is continuous."""
    g = GOLDEN["llama3_table"]
    args = (g["factor"], g["low_freq_factor"], g["high_freq_factor"], g["original_max_position"])
    for wl, want_div in [(g["high_freq_wavelen"], 1.0), (g["low_freq_wavelen"], g["factor"])]:
        inv = 2 * math.pi / wl
        got = rope.llama3_scale_one(inv, *args)
        assert abs(got - inv / want_div) <= 1e-15 * inv, (wl, got, inv / want_div)
    # just inside and just outside each edge the two rules meet
    eps = 1e-9
    for wl, inside_sign in [(g["high_freq_wavelen"], +1), (g["low_freq_wavelen"], -1)]:
        inside = rope.llama3_scale_one(2 * math.pi / (wl * (1 + inside_sign * eps)), *args)
        outside = rope.llama3_scale_one(2 * math.pi / (wl * (1 - inside_sign * eps)), *args)
        assert abs(inside - outside) < 1e-7 * (2 * math.pi / wl)


def pin_llama3_periods():
    """Periods after scaling run from a few tokens (2*pi) to about 2e7 tokens."""
    g = GOLDEN["llama3_table"]
    sc = rope.inv_freq(g["theta"], g["head_dim"], (g["factor"], g["low_freq_factor"],
                                                  g["high_freq_factor"], g["original_max_position"]))
    longest = 2 * math.pi / float(sc.min())
    assert 0.5 * g["longest_period_tokens_order"] < longest < 2 * g["longest_period_tokens_order"]
    assert abs(2 * math.pi / float(sc.max()) - 2 * math.pi) < 1e-6


# ---------------------------------------------------------------- rope ----

def pin_rope_identity():
    """Position 0 leaves every vector unchanged."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 128))
    inv = rope.inv_freq_plain(10000.0, 128)
    assert np.array_equal(rope.rotate(x, rope.angles(0, inv)), x)


def pin_rope_basis():
    """Element i pairs with i + D/2, turning towards it: e_i -> cos e_i + sin e_{i+D/2}."""
    d, h = 8, 4
    inv = rope.inv_freq_plain(10000.0, d)
    ang = rope.angles(1, inv).astype(np.float64)
    for i in range(h):
        e = np.zeros(d)
        e[i] = 1.0
        want = np.zeros(d)
        want[i], want[i + h] = math.cos(ang[i]), math.sin(ang[i])
        assert np.allclose(rope.rotate(e, ang), want, atol=1e-15, rtol=0)
        e = np.zeros(d)
        e[i + h] = 1.0
        want = np.zeros(d)
        want[i], want[i + h] = -math.sin(ang[i]), math.cos(ang[i])
        assert np.allclose(rope.rotate(e, ang), want, atol=1e-15, rtol=0)


def pin_rope_norm():
    """Each (i, i + D/2) pair keeps its Euclidean norm."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal((7, 96))
    inv = rope.inv_freq_plain(10000.0, 96)
    for pos in [1, 17, 4095, 131071]:
        y = rope.rotate(x, rope.angles(pos, inv))
        n0 = x[:, :48] ** 2 + x[:, 48:] ** 2
        n1 = y[:, :48] ** 2 + y[:, 48:] ** 2
        assert np.allclose(n0, n1, rtol=1e-13, atol=0)


def pin_rope_relative():
    """<rope(q, m), rope(k, n)> depends on m - n only (up to float32 angle rounding)."""
    rng = np.random.default_rng(3)
    inv = rope.inv_freq_plain(10000.0, 64)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    scale = np.linalg.norm(q) * np.linalg.norm(k)
    for m, n, shift in [(5, 2, 40), (30, 30, 17), (3, 60, 1)]:
        a = rope.rotate(q, rope.angles(m, inv)) @ rope.rotate(k, rope.angles(n, inv))
        b = rope.rotate(q, rope.angles(m + shift, inv)) @ rope.rotate(k, rope.angles(n + shift, inv))
        assert abs(a - b) < 1e-4 * scale


# ---------------------------------------------------------------- qk-norm ----

def pin_qknorm_rms():
    """With gamma = 1 each head's output has mean square ms / (ms + eps)."""
    rng = np.random.default_rng(4)
    eps = 1e-6
    x = rng.standard_normal((6, 128)) * np.array([1e-4, 1e-3, 1e-2, 1.0, 3.0, 1e-3])[:, None]
    y = rope.qk_norm(x, np.ones(128), eps)
    ms = np.mean(x * x, axis=-1)
    assert np.allclose(np.mean(y * y, axis=-1), ms / (ms + eps), rtol=1e-12, atol=0)


def pin_qknorm_per_head():
    """Scaling one head's input leaves the other heads' outputs unchanged."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 128))
    gamma = 1.0 + 0.1 * rng.standard_normal(128)
    y = rope.qk_norm(x, gamma, 1e-6)
    x2 = x.copy()
    x2[1] *= 1000.0
    y2 = rope.qk_norm(x2, gamma, 1e-6)
    assert np.array_equal(y2[[0, 2, 3]], y[[0, 2, 3]])
    assert np.allclose(y2[1], y[1], rtol=1e-5)
    # and gamma multiplies elementwise after the normalisation
    y1 = rope.qk_norm(x, np.ones(128), 1e-6)
    assert np.allclose(y, y1 * gamma, rtol=1e-14, atol=0)


def pin_qknorm_before_rope():
    """The append normalises each head (QK-norm, gamma included) before it rotates
    ("Qwen3-4B", model description: the norm follows the head split and precedes
    the rotation).  A rotation keeps the norm of every (i, i + D/2) pair, so with
    the norm first the pair norms of a token's rotated q and k are the same at
    every position as at position 0, where the rotation is the identity.  With a
    gamma of 2 on the first half and 0.5 on the second, rotating first would mix
    the two halves before gamma weighs them, and the pair norms would change with
    the position."""
    rng = np.random.default_rng(14)
    d, h = 16, 8
    x_q = _rand_bits(rng, (1, 2, d))
    x_k = _rand_bits(rng, (1, 1, d))
    gamma = bf16.from_f64(np.concatenate([np.full(h, 2.0), np.full(h, 0.5)]))
    positions = np.array([0, 1, 3, 100, 4097, 70001])
    T = len(positions)
    q = np.repeat(x_q, T, axis=0)
    k = np.repeat(x_k, T, axis=0)
    v = _rand_bits(rng, (T, 1, d))
    pool = np.zeros((1, 64, d), dtype=np.uint16)
    inv = rope.inv_freq_plain(10000.0, d)
    q_out, kp, _ = paged.append_rope(q, k, v, positions, np.zeros(T, dtype=np.int64), None, pool, pool,
                                     inv, slots=np.arange(T), gamma_q=gamma, gamma_k=gamma, eps=1e-6)

    def pair_norms(bits):
        y = bf16.to_f64(bits)
        return np.sqrt(y[..., :h] ** 2 + y[..., h:] ** 2)

    for got in (pair_norms(q_out), pair_norms(kp[0, :T][:, None, :])):
        # each side is rounded to bf16 once (relative 2^-9 per element)
        assert np.allclose(got[1:], got[:1], rtol=2.0 ** -7, atol=0), got
    # the gamma above does separate the orders: rotating first changes the norms
    ang = rope.angles(1, inv)
    g = bf16.to_f64(gamma)
    xq = bf16.to_f64(x_q[0, 0])
    wrong = rope.qk_norm(rope.rotate(xq, ang), g, 1e-6)
    assert not np.allclose(pair_norms(bf16.from_f64(wrong)), pair_norms(q_out[0, 0]), rtol=2.0 ** -5, atol=0)


# ---------------------------------------------------------------- attention ----

def _identity_pool(values_k, values_v):
    """Compact pool for one row whose positions are laid out page by page."""
    n = values_k.shape[1]
    pages = (n + 63) // 64
    pad = pages * 64 - n
    kp = np.pad(values_k, ((0, 0), (0, pad), (0, 0)))
    vp = np.pad(values_v, ((0, 0), (0, pad), (0, 0)))
    table = np.arange(pages, dtype=np.int32)[None, :]
    return kp, vp, table


def pin_attention_uniform():
    """A zero query weighs every visible key equally: the output is the mean of
    the visible values, which fixes the visible range (window included)."""
    w = GOLDEN["window"]["window"]
    n = 5200
    j = np.arange(n)
    v = np.zeros((1, n, 4))
    v[0, :, 0] = j // 64          # exact in bf16 (< 256)
    v[0, :, 1] = j % 64
    kp, vp, table = _identity_pool(bf16.from_f64(np.ones((1, n, 4))), bf16.from_f64(v + 0.0))
    q = bf16.from_f64(np.zeros((1, 4)))
    for p, window in [(5000, w), (100, w), (w - 1, w), (w, w), (5000, 0), (0, w), (64, 64)]:
        out = paged.attention_at(q, 0, p, table, kp, vp, window)
        mean_pos = 64 * out[0, 0] + out[0, 1]
        lo = max(0, p - window + 1) if window else 0
        assert abs(mean_pos - (lo + p) / 2) < 1e-9, (p, window, mean_pos)
        if window and p >= window:
            count = p - (2 * mean_pos - p) + 1
            assert abs(count - window) < 1e-6
            if window == w:  # the query plus the 2046 positions before it
                assert count - 1 == GOLDEN["window"]["positions_before_query"]


def pin_attention_single_and_constant():
    """One visible key gives its value exactly; constant values give that value."""
    rng = np.random.default_rng(6)
    kp = _rand_bits(rng, (2, 128, 16))
    vp = _rand_bits(rng, (2, 128, 16))
    table = np.array([[1, 0]], dtype=np.int32)
    q = _rand_bits(rng, (4, 16))
    out = paged.attention_at(q, 0, 0, table, kp, vp, 0)
    slot = 1 * 64
    for h in range(4):
        assert np.array_equal(out[h], bf16.to_f64(vp[h // 2, slot]))
    vc = np.broadcast_to(bf16.from_f64(np.full((1, 1, 16), 0.375)), (2, 128, 16)).copy()
    out = paged.attention_at(q, 0, 100, table, kp, vc, 0)
    assert np.allclose(out, 0.375, rtol=0, atol=1e-15)


def pin_attention_two_keys():
    """Two keys: the weights are a logistic function of the scaled score gap,
    with scale 1/sqrt(head_dim)."""
    d = 4
    k = np.zeros((1, 64, d))
    k[0, 0, 0] = 2.0
    v = np.zeros((1, 64, d))
    v[0, 0, 1] = 1.0
    v[0, 1, 2] = 1.0
    kp, vp = bf16.from_f64(k), bf16.from_f64(v)
    table = np.array([[0]], dtype=np.int32)
    for c in [0.5, 1.0, 3.0]:
        q = bf16.from_f64(np.array([[c, 0, 0, 0]]))
        out = paged.attention_at(q, 0, 1, table, kp, vp, 0)
        gap = 2.0 * c / math.sqrt(d)
        w1 = 1.0 / (1.0 + math.exp(-gap))
        assert abs(out[0, 1] - w1) < 1e-15 and abs(out[0, 2] - (1 - w1)) < 1e-15


def pin_attention_gqa_groups():
    """Query head h reads kv head h // (Hq / Hkv)."""
    hq, hkv, d = 8, 2, 8
    rng = np.random.default_rng(7)
    kp = _rand_bits(rng, (hkv, 64, d))
    vp = np.stack([np.full((64, d), c + 1.0) for c in range(hkv)])
    vp = bf16.from_f64(vp)
    q = _rand_bits(rng, (hq, d))
    out = paged.attention_at(q, 0, 30, np.array([[0]], dtype=np.int32), kp, vp, 0)
    for h in range(hq):
        assert np.allclose(out[h], h // (hq // hkv) + 1.0, atol=1e-14)


def pin_attention_bruteforce():
    """Tiny inputs against a 50-digit evaluation of softmax attention, including
    scores large enough to overflow a naive exp."""
    import mpmath
    mpmath.mp.dps = 50
    rng = np.random.default_rng(8)
    hq, hkv, d, n = 4, 2, 8, 10
    kp = _rand_bits(rng, (hkv, 64, d), 4.0)
    vp = _rand_bits(rng, (hkv, 64, d))
    perm = np.array([[0]], dtype=np.int32)
    for qscale in [1.0, 300.0]:
        q = _rand_bits(rng, (hq, d), qscale)
        out = paged.attention_at(q, 0, n - 1, perm, kp, vp, 0)
        qf, kf, vf = bf16.to_f64(q), bf16.to_f64(kp), bf16.to_f64(vp)
        for h in range(hq):
            c = h // (hq // hkv)
            s = [mpmath.fsum(mpmath.mpf(qf[h, i]) * mpmath.mpf(kf[c, j, i]) for i in range(d))
                 / mpmath.sqrt(d) for j in range(n)]
            w = [mpmath.exp(x) for x in s]
            tot = mpmath.fsum(w)
            for i in range(d):
                want = mpmath.fsum(w[j] * mpmath.mpf(vf[c, j, i]) for j in range(n)) / tot
                assert abs(out[h, i] - float(want)) <= 1e-12 * (1 + abs(float(want))), (qscale, h, i)


def pin_window_short_is_causal():
    """A row at or under the window sees plain causal attention."""
    rng = np.random.default_rng(9)
    kp = _rand_bits(rng, (2, 40 * 64, 8))
    vp = _rand_bits(rng, (2, 40 * 64, 8))
    table = rng.permutation(40).astype(np.int32).reshape(1, 40)
    q = _rand_bits(rng, (2, 8))
    for p in [0, 5, 700, 2046]:
        a = paged.attention_at(q, 0, p, table, kp, vp, 2047)
        b = paged.attention_at(q, 0, p, table, kp, vp, 0)
        assert np.array_equal(a, b)
    a = paged.attention_at(q, 0, 2047, table, kp, vp, 2047)
    b = paged.attention_at(q, 0, 2047, table, kp, vp, 0)
    assert not np.array_equal(a, b)


def pin_paging_invariance():
    """Moving pages around the pool (and the table with them) changes nothing,
    and a paged row equals the same row stored contiguously."""
    rng = np.random.default_rng(10)
    npg, d = 24, 16
    kp = _rand_bits(rng, (2, npg * 64, d))
    vp = _rand_bits(rng, (2, npg * 64, d))
    table = rng.permutation(npg).astype(np.int32).reshape(3, 8)
    q = _rand_bits(rng, (3, 4, d))
    pos = np.array([511, 64, 300])
    base = paged.decode_attention(q, pos, table, kp, vp, 0)
    pi = rng.permutation(npg)
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    for p in range(npg):
        kp2[:, pi[p] * 64:(pi[p] + 1) * 64] = kp[:, p * 64:(p + 1) * 64]
        vp2[:, pi[p] * 64:(pi[p] + 1) * 64] = vp[:, p * 64:(p + 1) * 64]
    moved = paged.decode_attention(q, pos, pi[table].astype(np.int32), kp2, vp2, 0)
    assert np.array_equal(base, moved)
    for b in range(3):
        kc = np.concatenate([kp[:, table[b, j] * 64:(table[b, j] + 1) * 64] for j in range(8)], axis=1)
        vc = np.concatenate([vp[:, table[b, j] * 64:(table[b, j] + 1) * 64] for j in range(8)], axis=1)
        ident = np.arange(8, dtype=np.int32)[None, :]
        contig = paged.attention_at(q[b], 0, int(pos[b]), ident, kc, vc, 0)
        assert np.array_equal(contig, base[b])


# ---------------------------------------------------------------- append / chunks ----

def _small_step(rng, hq=4, hkv=2, d=16, chunk_lens=(70, 5, 130), window=0):
    npg = sum((n + 63) // 64 for n in chunk_lens) + 2
    perm = rng.permutation(npg).astype(np.int32)
    width = max((n + 63) // 64 for n in chunk_lens)
    table = np.full((len(chunk_lens), width), -1, dtype=np.int32)
    at = 0
    rows, pos, seg = [], [], []
    for c, n in enumerate(chunk_lens):
        k = (n + 63) // 64
        table[c, :k] = perm[at:at + k]
        at += k
        rows += [c] * n
        pos += list(range(n))
        seg += [c] * n
    P = len(pos)
    q = _rand_bits(rng, (P, hq, d))
    k = _rand_bits(rng, (P, hkv, d))
    v = _rand_bits(rng, (P, hkv, d))
    kp = _rand_bits(rng, (hkv, npg * 64, d))
    vp = _rand_bits(rng, (hkv, npg * 64, d))
    return dict(q=q, k=k, v=v, rows=np.array(rows), pos=np.array(pos), seg=np.array(seg),
                table=table, kp=kp, vp=vp, dump=int(perm[at]))


def pin_append_placement():
    """Each token's rotated key and its value land at its logical position of its
    row (pages concatenated in table order), and nothing else in the pool moves."""
    rng = np.random.default_rng(11)
    s = _small_step(rng)
    inv = rope.inv_freq_plain(10000.0, 16)
    q_out, kp2, vp2 = paged.append_rope(s["q"], s["k"], s["v"], s["pos"], s["rows"], s["table"],
                                        s["kp"], s["vp"], inv)
    changed = np.any(kp2 != s["kp"], axis=(0, 2)) | np.any(vp2 != s["vp"], axis=(0, 2))
    assert changed.sum() <= len(s["pos"])
    written = np.zeros(kp2.shape[1], dtype=bool)
    for t in range(len(s["pos"])):
        r, p = int(s["rows"][t]), int(s["pos"][t])
        npages = int(np.sum(s["table"][r] >= 0))
        contig_k = np.concatenate([kp2[:, s["table"][r, j] * 64:(s["table"][r, j] + 1) * 64]
                                   for j in range(npages)], axis=1)
        contig_v = np.concatenate([vp2[:, s["table"][r, j] * 64:(s["table"][r, j] + 1) * 64]
                                   for j in range(npages)], axis=1)
        want_k = bf16.from_f64(rope.rotate(bf16.to_f64(s["k"][t]), rope.angles(p, inv)))
        assert np.array_equal(contig_k[:, p], want_k)
        assert np.array_equal(contig_v[:, p], s["v"][t])
        page = s["table"][r, p // 64]
        written[page * 64 + p % 64] = True
        assert np.array_equal(q_out[t], bf16.from_f64(rope.rotate(bf16.to_f64(s["q"][t]), rope.angles(p, inv))))
    assert not np.any(changed & ~written)
    # an explicit slot overrides the table; a negative position writes nothing
    slots = np.full(len(s["pos"]), s["dump"] * 64 + 7)
    pos = s["pos"].copy()
    pos[1:] = -1
    _, kp3, vp3 = paged.append_rope(s["q"], s["k"], s["v"], pos, s["rows"], s["table"],
                                    s["kp"], s["vp"], inv, slots=slots)
    diff = np.nonzero(np.any(vp3 != s["vp"], axis=(0, 2)))[0]
    assert list(diff) == [s["dump"] * 64 + 7]


def pin_chunks_match_packed_rule():
    """Prompts starting at position 0 in their own rows: attending over the row's
    pages equals the row-based packed rule (own segment, up to itself, window)."""
    rng = np.random.default_rng(12)
    s = _small_step(rng)
    inv = rope.inv_freq_plain(10000.0, 16)
    q_out, kp2, vp2 = paged.append_rope(s["q"], s["k"], s["v"], s["pos"], s["rows"], s["table"],
                                        s["kp"], s["vp"], inv)
    k_rot = np.stack([bf16.from_f64(rope.rotate(bf16.to_f64(s["k"][t]), rope.angles(int(s["pos"][t]), inv)))
                      for t in range(len(s["pos"]))])
    for window in [0, 50]:
        a = paged.chunk_attention(q_out, s["rows"], s["pos"], s["table"], kp2, vp2, window)
        b = paged.packed_attention(q_out, k_rot, s["v"], s["pos"], s["seg"], window)
        assert np.allclose(a, b, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- sizes ----

def pin_cache_size():
    """The pool layout [kv_heads, positions, head_dim] bf16, K and V, over the
    Llama layers reproduces the cache sizes the Llama page states."""
    g = GOLDEN["cache_size"]
    one = np.zeros((g["kv_heads"], 1, g["head_dim"]), dtype=np.uint16).nbytes
    per_pos = one * g["caches"] * g["layers"]
    assert per_pos * g["max_seq"] == g["gib"] * 2 ** 30
    assert per_pos * g["max_seq_long"] == g["gib_long"] * 2 ** 30
    assert paged.PAGE_SIZE == GOLDEN["page_size"]["page_size"]


def pin_decode_rows_is_identity_table():
    """Row-based decode over contiguous caches (each row its own MaxSeq positions)
    is paged decode with an identity table: row b's page j is page b * pages + j."""
    rng = np.random.default_rng(13)
    rows, pages, d = 3, 4, 16
    cache_k = _rand_bits(rng, (rows, 2, pages * 64, d))   # [Batch, Heads, MaxSeq, D]
    cache_v = _rand_bits(rng, (rows, 2, pages * 64, d))
    pos = np.array([200, 0, 255])
    q = _rand_bits(rng, (rows, 4, d))
    # the pool is the caches' rows laid end to end per head
    kp = np.concatenate([cache_k[b] for b in range(rows)], axis=1)
    vp = np.concatenate([cache_v[b] for b in range(rows)], axis=1)
    table = (np.arange(rows)[:, None] * pages + np.arange(pages)[None, :]).astype(np.int32)
    paged_out = paged.decode_attention(q, pos, table, kp, vp, 0)
    for b in range(rows):
        # decode_rows: row b attends over cache row b, positions 0..pos[b]
        ident = np.arange(pages, dtype=np.int32)[None, :]
        row_out = paged.attention_at(q[b], 0, int(pos[b]), ident, cache_k[b], cache_v[b], 0)
        assert np.array_equal(row_out, paged_out[b])


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
