"""Rotary positions and per-head QK-norm for the oracle (test infrastructure only).

Sources
  * "Phi-3 Mini 4K Instruct -- files", src/rope.linnet, ``tables``: the
    frequency table ``inv_freq[i] = exp(-(f32(i) * 2.0 / f32(D)) * log(theta))``
    in float32, angles ``f32(s) * inv_freq[i]`` in float32, and each frequency
    repeated for both halves of the head dimension.
  * "Llama 3.1 8B Instruct", the rope-scaling paragraph and Validation: the
    llama3 three-band rescale of each frequency by its wavelength.
  * "Qwen3-4B", model description: QK-norm, an RMS normalisation (eps 1e-6)
    of each head's head_dim slice of q and k, after the head split and before
    the rotation.

Readings where the pages are silent (each one is listed in the design notes):
  * The rotation pairs element i with element i + D/2 ("rotate half"), since
    the tables repeat each frequency for both halves.
  * cos/sin are evaluated in float64 from the float32 angle, and the rotation
    is exact (float64); the result is rounded to bf16 once, when stored.  The
    pages materialise tables at the model dtype; no table is materialised here.
  * The float32 log and exp of the frequency table are taken correctly
    rounded (evaluated in float64, rounded once to float32).
  * The llama3 blend weight is ``smooth = (orig / wavelen - low) / (high - low)``,
    affine in frequency: 1 at wavelen = orig/high (2048), 0 at orig/low (8192),
    matching the boundary condition the Llama page states.  The rescaled value
    is evaluated in float64 from the float32 base frequency and rounded once.
"""
import math

import numpy as np

TWO_PI = 2.0 * math.pi


def _f32(x) -> np.float32:
    return np.float32(x)


def inv_freq_plain(theta: float, head_dim: int) -> np.ndarray:
    """The plain-theta table, ``head_dim // 2`` float32 values, as the pages
    write it: every operation in float32, log and exp correctly rounded."""
    if head_dim % 2:
        raise ValueError("head_dim must be even")
    theta32 = _f32(theta)
    log_theta = _f32(math.log(float(theta32)))
    d32 = _f32(head_dim)
    out = np.empty(head_dim // 2, dtype=np.float32)
    for i in range(head_dim // 2):
        t = _f32(_f32(i) * _f32(2.0))        # f32(i) * 2.0
        t = _f32(t / d32)                    # ... / f32(D)
        e = _f32(_f32(-t) * log_theta)       # -(...) * log(theta)
        out[i] = _f32(math.exp(float(e)))    # exp(...)
    return out


def llama3_scale_one(inv: float, factor: float, low_freq_factor: float,
                     high_freq_factor: float, original_max_position: float) -> float:
    """Rescale one frequency by its wavelength (three bands), in float64."""
    wavelen = TWO_PI / inv
    low_freq_wavelen = original_max_position / low_freq_factor    # 8192 for Llama 3.1
    high_freq_wavelen = original_max_position / high_freq_factor  # 2048 for Llama 3.1
    if wavelen > low_freq_wavelen:
        return inv / factor
    if wavelen < high_freq_wavelen:
        return inv
    smooth = (original_max_position / wavelen - low_freq_factor) / (high_freq_factor - low_freq_factor)
    return (1.0 - smooth) * (inv / factor) + smooth * inv


def inv_freq_llama3(base: np.ndarray, factor: float, low_freq_factor: float,
                    high_freq_factor: float, original_max_position: float) -> np.ndarray:
    """llama3-scaled table: each float32 base frequency rescaled, rounded once."""
    out = np.empty_like(base, dtype=np.float32)
    for i, inv in enumerate(np.asarray(base, dtype=np.float32)):
        out[i] = _f32(llama3_scale_one(float(inv), factor, low_freq_factor,
                                       high_freq_factor, original_max_position))
    return out


def inv_freq(theta: float, head_dim: int, llama3=None) -> np.ndarray:
    """Frequency table of a model: plain, or llama3-rescaled when
    ``llama3 = (factor, low_freq_factor, high_freq_factor, original_max_position)``."""
    base = inv_freq_plain(theta, head_dim)
    if llama3 is None:
        return base
    return inv_freq_llama3(base, *llama3)


def angles(position: int, inv: np.ndarray) -> np.ndarray:
    """float32 angles ``f32(position) * inv[i]`` (one float32 multiply each)."""
    return (np.float32(position) * np.asarray(inv, dtype=np.float32)).astype(np.float32)


def rotate(x: np.ndarray, ang: np.ndarray) -> np.ndarray:
    """Rotate the last axis of ``x`` (float64, length D) by the angles (length D/2).

    Element i pairs with element i + D/2:
      out[i]       = x[i] cos(a_i) - x[i+D/2] sin(a_i)
      out[i+D/2]   = x[i+D/2] cos(a_i) + x[i] sin(a_i)
    """
    x = np.asarray(x, dtype=np.float64)
    h = x.shape[-1] // 2
    a = np.asarray(ang, dtype=np.float32).astype(np.float64)
    c, s = np.cos(a), np.sin(a)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def qk_norm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """RMS-normalise each head's vector over the last axis only, then scale by gamma.

    ``x``: float64 [..., heads, D]; ``gamma``: float64 [D].
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    r = 1.0 / np.sqrt(ms + eps)
    return x * r * np.asarray(gamma, dtype=np.float64)
