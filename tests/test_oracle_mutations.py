"""Plant plausible mistakes in the oracle and check that the pins catch each one.

Every mutation replaces one oracle step (on the CPU, for the duration of one
test) with a wrong variant; the named pin must then fail.
"""
import math

import numpy as np
import pytest

import oracle_pins as pins
from oracle import paged, rope


def _rotate_interleaved(x, ang):
    x = np.asarray(x, dtype=np.float64)
    a = np.asarray(ang, dtype=np.float32).astype(np.float64)
    c, s = np.cos(a), np.sin(a)
    x1, x2 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x1 * c - x2 * s
    out[..., 1::2] = x2 * c + x1 * s
    return out


def _rotate_sign_flip(x, ang):
    x = np.asarray(x, dtype=np.float64)
    h = x.shape[-1] // 2
    a = np.asarray(ang, dtype=np.float32).astype(np.float64)
    c, s = np.cos(a), np.sin(a)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c - x1 * s], axis=-1)


def _qknorm_across_heads(x, gamma, eps):
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x)
    return x / np.sqrt(ms + eps) * gamma


def _qknorm_eps_outside(x, gamma, eps):
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / (np.sqrt(ms) + eps) * gamma


def _llama3_swapped(inv, factor, low, high, orig):
    wavelen = 2 * math.pi / inv
    if wavelen > orig / low:
        return inv / factor
    if wavelen < orig / high:
        return inv
    smooth = (orig / wavelen - low) / (high - low)
    return smooth * (inv / factor) + (1.0 - smooth) * inv


def _inv_freq_missing_two(theta, head_dim):
    return np.array([np.float32(math.exp(-(i / head_dim) * math.log(theta)))
                     for i in range(head_dim // 2)], dtype=np.float32)


def _attend_no_shift(q, keys, values, scale):
    with np.errstate(over="ignore", invalid="ignore"):
        w = np.exp((q @ keys.T) * scale)
        return (w @ values) / np.sum(w, axis=1, keepdims=True)


def _slot_offset_wrong(table, row, position):
    return int(table[row, position // 64]) * 64 + (position // 64) % 64


def _append_rotate_then_norm(q, k, v, positions, rows, table, k_pool, v_pool, inv,
                             slots=None, gamma_q=None, gamma_k=None, eps=1e-6):
    """The append with its two steps swapped: RoPE first, QK-norm second."""
    from oracle import bf16
    q_out = np.zeros_like(q, dtype=np.uint16)
    k_pool = np.array(k_pool, dtype=np.uint16, copy=True)
    v_pool = np.array(v_pool, dtype=np.uint16, copy=True)
    for t in range(q.shape[0]):
        p = int(positions[t])
        if p < 0:
            continue
        ang = rope.angles(p, inv)
        qf = rope.rotate(bf16.to_f64(q[t]), ang)
        kf = rope.rotate(bf16.to_f64(k[t]), ang)
        if gamma_q is not None:
            qf = rope.qk_norm(qf, bf16.to_f64(gamma_q), eps)
        if gamma_k is not None:
            kf = rope.qk_norm(kf, bf16.to_f64(gamma_k), eps)
        q_out[t] = bf16.from_f64(qf)
        s = int(slots[t]) if slots is not None else paged.slot_of(table, int(rows[t]), p)
        k_pool[:, s, :] = bf16.from_f64(kf)
        v_pool[:, s, :] = v[t]
    return q_out, k_pool, v_pool


MUTATIONS = [
    # (description, module, attribute, replacement, pin that must fail)
    ("query head reads kv head h % Hkv", paged, "kv_head_of",
     lambda h, g, hkv: h % hkv, pins.pin_attention_gqa_groups),
    ("window one position too wide", paged, "visible_range",
     lambda p, w: (max(0, p - w) if w > 0 else 0, p), pins.pin_attention_uniform),
    ("query does not see itself", paged, "visible_range",
     lambda p, w: (max(0, p - w + 1) if w > 0 else 0, p - 1), pins.pin_attention_single_and_constant),
    ("scale 1/D instead of 1/sqrt(D)", paged, "default_scale",
     lambda d: 1.0 / d, pins.pin_attention_two_keys),
    ("softmax without the max shift", paged, "attend",
     _attend_no_shift, pins.pin_attention_bruteforce),
    ("in-page offset taken from the page index", paged, "slot_of",
     _slot_offset_wrong, pins.pin_append_placement),
    ("rope pairs adjacent elements", rope, "rotate",
     _rotate_interleaved, pins.pin_rope_basis),
    ("rope sign flipped in the second half", rope, "rotate",
     _rotate_sign_flip, pins.pin_rope_norm),
    ("qk-norm over all heads at once", rope, "qk_norm",
     _qknorm_across_heads, pins.pin_qknorm_per_head),
    ("qk-norm eps outside the square root", rope, "qk_norm",
     _qknorm_eps_outside, pins.pin_qknorm_rms),
    ("rope before qk-norm", paged, "append_rope",
     _append_rotate_then_norm, pins.pin_qknorm_before_rope),
    ("llama3 blend weights swapped", rope, "llama3_scale_one",
     _llama3_swapped, pins.pin_llama3_continuity),
    ("frequency exponent missing the factor 2", rope, "inv_freq_plain",
     _inv_freq_missing_two, pins.pin_inv_freq_exact),
]


@pytest.mark.parametrize("desc,module,attr,bad,pin", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pin_catches_mutation(monkeypatch, desc, module, attr, bad, pin):
    monkeypatch.setattr(module, attr, bad)
    with pytest.raises((AssertionError, ValueError, FloatingPointError)):
        pin()
