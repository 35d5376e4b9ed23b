"""Seeded synthetic inputs for the paged decode / step attention path.

This module is shared by both sides of every comparison (the CPU oracle and
the CUDA library), so it holds none of the attention arithmetic: only random
numbers, page tables and position lists.

Value generator
---------------
Every bf16 value is a pure function of (seed, stream, index), so any slice of a
tensor can be regenerated independently on the host or on the device (see
``synth/fill.cu`` for the device copy of the same definition):

* ``key(seed, stream) = mix64(mix64(seed) + (stream + 1) * GAMMA)``
* ``h_i = mix64(key + (i + 1) * GAMMA)`` (all arithmetic mod 2**64), i.e. the
  i-th output of SplitMix64 (Steele, Lea & Flood, OOPSLA 2014) started at
  ``key``; ``mix64`` is its output function.
* the four 16-bit fields u0..u3 of ``h_i`` are summed, centred and scaled:
  ``x = f32(u0+u1+u2+u3 - 131070) * f32(sqrt(3)/65535)`` (one IEEE f32
  multiply), then rounded to bf16 (round to nearest even).  ``x`` is an
  Irwin-Hall(4) sample rescaled to mean 0 and variance 1: a bounded
  (|x| <= 2*sqrt(3)) stand-in for N(0, 1) whose bits are reproducible exactly on
  any IEEE machine, with no transcendental functions involved.

Workloads
---------
``build(name, ...)`` returns a :class:`Workload`: shapes, positions, the page
table, the chunk tokens of a step, and the streams the tensors are drawn from.
The five named workloads follow the shapes of the models on the pages
(Phi-3 Mini 4K Instruct, Mistral 7B Instruct v0.3, Qwen3-4B,
Llama 3.1 8B Instruct); ``scale`` shrinks lengths and row counts for tests.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

PAGE_SIZE = 64

GAMMA = 0x9E3779B97F4A7C15
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1
# f32(sqrt(3) / 65535): evaluated in double, rounded once to float.
IH_SCALE = np.float32(1.7320508075688772 / 65535.0)

# Stream ids: one per synthetic tensor.
STREAM_K_POOL = 1
STREAM_V_POOL = 2
STREAM_Q = 3
STREAM_K_NEW = 4
STREAM_V_NEW = 5
STREAM_GAMMA_Q = 6
STREAM_GAMMA_K = 7


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _mix64_int(z: int) -> int:
    return int(mix64(np.array([z & _MASK64], dtype=np.uint64))[0])


def stream_key(seed: int, stream: int) -> int:
    """64-bit key of one synthetic tensor."""
    return _mix64_int((_mix64_int(seed) + (stream + 1) * GAMMA) & _MASK64)


def splitmix64(key: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of SplitMix64 started at ``key``."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = np.uint64(key) + idx * np.uint64(GAMMA)
    return mix64(state)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bf16 (nearest, ties to even); returns bits."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_f32(key: int, start: int, count: int) -> np.ndarray:
    """Unit-variance Irwin-Hall(4) values as float32 (before bf16 rounding)."""
    h = splitmix64(key, start, count)
    s = np.zeros(count, dtype=np.int64)
    for k in range(4):
        s += ((h >> np.uint64(16 * k)) & np.uint64(0xFFFF)).astype(np.int64)
    s -= 131070
    return s.astype(np.float32) * IH_SCALE


def normal_bf16(key: int, start: int, count: int) -> np.ndarray:
    """bf16 bits of ``count`` unit-variance values starting at ``start``."""
    return f32_to_bf16_bits(normal_f32(key, start, count))


def gauss_bf16(key: int, start: int, count: int) -> np.ndarray:
    """bf16 bits of ``count`` standard normal values with their tails (host only).

    Value i is Box-Muller (Box & Muller, 1958) on SplitMix64 outputs 2i and 2i+1
    started at ``key``: ``u1 = (h_2i >> 11) + 1`` and ``u2 = h_2i+1 >> 11``, both
    times 2^-53, ``z = sqrt(-2 ln u1) cos(2 pi u2)`` in float64, rounded to bf16
    through float32.  |z| reaches about 8.6, unlike the bounded Irwin-Hall values.
    """
    h = splitmix64(key, 2 * start, 2 * count).reshape(count, 2)
    u1 = ((h[:, 0] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    u2 = (h[:, 1] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return f32_to_bf16_bits(z.astype(np.float32))


def scale_bf16_pow2(bits: np.ndarray, factor: float) -> np.ndarray:
    """bf16 bits times a power of two (exact while the result stays normal and finite)."""
    m, e = math.frexp(float(factor))
    if factor <= 0 or m != 0.5:
        raise ValueError("factor must be a power of two")
    if factor == 1.0:
        return bits
    return f32_to_bf16_bits(bf16_bits_to_f32(bits) * np.float32(factor))


def e4m3_codes(key: int, start: int, count: int) -> np.ndarray:
    """Bytes for a prefilled 8-bit (E4M3) pool: from SplitMix64 output i, the
    sign is bit 63, the exponent field 4 + (bits 8.. mod 6) and the mantissa
    bits 16..18, so every code is finite with magnitude in [2^-3, 2^3)."""
    h = splitmix64(key, start, count)
    sign = (h >> np.uint64(63)) & np.uint64(1)
    e = np.uint64(4) + ((h >> np.uint64(8)) % np.uint64(6))
    m = (h >> np.uint64(16)) & np.uint64(7)
    return ((sign << np.uint64(7)) | (e << np.uint64(3)) | m).astype(np.uint8)


# every finite E4M3 code (all but the two NaN codes, S.1111.111)
E4M3_FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def e4m3_codes_all(key: int, start: int, count: int) -> np.ndarray:
    """Bytes for a prefilled 8-bit pool drawn from every finite E4M3 code
    (subnormals, zeros and the saturated +-448 included): byte i is finite code
    number (SplitMix64 output i) mod 254 (host only)."""
    h = splitmix64(key, start, count)
    return E4M3_FINITE[(h % np.uint64(len(E4M3_FINITE))).astype(np.int64)]


def tensor_bf16(seed: int, stream: int, shape) -> np.ndarray:
    n = int(np.prod(shape)) if len(shape) else 1
    return normal_bf16(stream_key(seed, stream), 0, n).reshape(shape)


def gamma_bf16(seed: int, stream: int, dim: int) -> np.ndarray:
    """QK-norm weights ~ 1 + 0.1 * z, as bf16 bits (two separate f32 ops)."""
    z = normal_f32(stream_key(seed, stream), 0, dim)
    g = np.float32(1.0) + z * np.float32(0.1)
    return f32_to_bf16_bits(g.astype(np.float32))


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------


@dataclasses.dataclass
class Workload:
    """One synthetic layer step.

    Decode row ``b`` (``b < B``) uses table row ``b`` and position
    ``dec_positions[b]``.  Chunk token ``t`` (``t < P``) is position
    ``ch_positions[t]`` of prompt ``ch_segments[t]`` in table row
    ``ch_rows[t]``.  A step's tokens are the ``P`` chunk tokens followed by the
    ``B`` decode rows.  The whole pool is filled from the generator; the step
    then overwrites its own tokens' slots.
    """

    name: str
    seed: int
    hq: int
    hkv: int
    head_dim: int
    theta: float
    llama3: Optional[tuple]  # (factor, low_freq_factor, high_freq_factor, original_max_position)
    window: int  # 0: no window
    qk_norm: bool
    num_pages: int
    table: np.ndarray  # int32 [num_rows, pages_per_row], -1 = unused
    dec_positions: np.ndarray  # int32 [B]
    ch_rows: np.ndarray  # int32 [P]
    ch_positions: np.ndarray  # int32 [P]
    ch_segments: np.ndarray  # int32 [P]
    dump_page: int = -1
    norm_eps: float = 1e-6
    # input shaping for edge cases (no attention arithmetic):
    dist: str = "ih"            # "ih": Irwin-Hall values (host and device); "gauss": Box-Muller (host only)
    q_scale: float = 1.0        # power of two multiplying the step's queries
    k_page_scale: Optional[dict] = None  # physical page -> power of two multiplying its K values
    gamma_halves: Optional[tuple] = None  # QK-norm gamma (a, b): a on the first half of D, b on the second
    e4m3_all: bool = False      # 8-bit pools drawn from every finite code (host only)

    @property
    def B(self) -> int:
        return int(self.dec_positions.shape[0])

    @property
    def P(self) -> int:
        return int(self.ch_positions.shape[0])

    @property
    def T(self) -> int:
        return self.P + self.B

    @property
    def num_rows(self) -> int:
        return int(self.table.shape[0])

    @property
    def pages_per_row(self) -> int:
        return int(self.table.shape[1])

    @property
    def pool_positions(self) -> int:
        return self.num_pages * PAGE_SIZE

    def token_positions(self) -> np.ndarray:
        return np.concatenate([self.ch_positions, self.dec_positions]).astype(np.int32)

    def token_rows(self) -> np.ndarray:
        return np.concatenate([self.ch_rows, np.arange(self.B, dtype=np.int32)]).astype(np.int32)

    # -- tensors -----------------------------------------------------------
    @property
    def device_fillable(self) -> bool:
        """The pool can be filled on the device (``synth/fill.cu``): Irwin-Hall
        values with no page scaling."""
        return self.dist == "ih" and not self.k_page_scale and not self.e4m3_all

    def _values(self, key: int, start: int, count: int) -> np.ndarray:
        if self.dist == "gauss":
            return gauss_bf16(key, start, count)
        return normal_bf16(key, start, count)

    def _tensor(self, stream: int, shape) -> np.ndarray:
        n = int(np.prod(shape)) if len(shape) else 1
        return self._values(stream_key(self.seed, stream), 0, n).reshape(shape)

    def step_q(self) -> np.ndarray:
        return scale_bf16_pow2(self._tensor(STREAM_Q, (self.T, self.hq, self.head_dim)), self.q_scale)

    def step_k(self) -> np.ndarray:
        return self._tensor(STREAM_K_NEW, (self.T, self.hkv, self.head_dim))

    def step_v(self) -> np.ndarray:
        return self._tensor(STREAM_V_NEW, (self.T, self.hkv, self.head_dim))

    def _gamma(self, stream: int) -> Optional[np.ndarray]:
        if not self.qk_norm:
            return None
        if self.gamma_halves is not None:
            a, b = self.gamma_halves
            h = self.head_dim // 2
            return f32_to_bf16_bits(np.array([a] * h + [b] * h, dtype=np.float32))
        return gamma_bf16(self.seed, stream, self.head_dim)

    def gamma_q(self) -> Optional[np.ndarray]:
        return self._gamma(STREAM_GAMMA_Q)

    def gamma_k(self) -> Optional[np.ndarray]:
        return self._gamma(STREAM_GAMMA_K)

    def pool_key(self, which: str) -> int:
        return stream_key(self.seed, STREAM_K_POOL if which == "k" else STREAM_V_POOL)

    def pool(self, which: str) -> np.ndarray:
        """The whole initial pool ``[Hkv, num_pages*64, D]`` (small workloads only)."""
        n = self.hkv * self.pool_positions * self.head_dim
        out = self._values(self.pool_key(which), 0, n).reshape(
            self.hkv, self.pool_positions, self.head_dim)
        if which == "k" and self.k_page_scale:
            for pg, f in self.k_page_scale.items():
                sl = slice(int(pg) * PAGE_SIZE, (int(pg) + 1) * PAGE_SIZE)
                out[:, sl] = scale_bf16_pow2(out[:, sl], f)
        return out

    def _codes(self, key: int, start: int, count: int) -> np.ndarray:
        return (e4m3_codes_all if self.e4m3_all else e4m3_codes)(key, start, count)

    def pool_e4m3(self, which: str) -> np.ndarray:
        """The whole 8-bit pool [Hkv][num_pages * 64][D] of codes (prefilled context)."""
        n = self.hkv * self.pool_positions * self.head_dim
        return self._codes(self.pool_key(which), 0, n).reshape(self.hkv, self.pool_positions, self.head_dim)

    def pool_pages_e4m3(self, which: str, kv_head: int, pages: np.ndarray) -> np.ndarray:
        """Codes of the listed pages of one kv head, [len(pages)][64][D]."""
        per_head = self.pool_positions * self.head_dim
        out = np.empty((len(pages), PAGE_SIZE, self.head_dim), dtype=np.uint8)
        for i, pg in enumerate(np.asarray(pages).tolist()):
            start = kv_head * per_head + int(pg) * PAGE_SIZE * self.head_dim
            out[i] = self._codes(self.pool_key(which), start, PAGE_SIZE * self.head_dim).reshape(PAGE_SIZE, self.head_dim)
        return out

    def pool_pages(self, which: str, kv_head: int, pages: np.ndarray) -> np.ndarray:
        """Initial content of the given physical pages of one kv head: ``[n, 64, D]``."""
        key = self.pool_key(which)
        per_page = PAGE_SIZE * self.head_dim
        out = np.empty((len(pages), PAGE_SIZE, self.head_dim), dtype=np.uint16)
        for i, pg in enumerate(np.asarray(pages, dtype=np.int64)):
            start = (kv_head * self.pool_positions + int(pg) * PAGE_SIZE) * self.head_dim
            out[i] = self._values(key, start, per_page).reshape(PAGE_SIZE, self.head_dim)
            if which == "k" and self.k_page_scale and int(pg) in self.k_page_scale:
                out[i] = scale_bf16_pow2(out[i], self.k_page_scale[int(pg)])
        return out

    def visible_keys(self) -> int:
        """Total (row, key) pairs the decode rows attend to."""
        lens = self.dec_positions.astype(np.int64) + 1
        if self.window > 0:
            lens = np.minimum(lens, self.window)
        return int(np.sum(np.where(self.dec_positions >= 0, lens, 0)))


def _assign_pages(rng: np.random.Generator, need: list[int], extra_pages: int = 1):
    """Give row r ``need[r]`` private pages from a shuffled pool; one spare dump page."""
    total = int(sum(need)) + extra_pages
    perm = rng.permutation(total).astype(np.int32)
    width = max(max(need), 1)
    table = np.full((len(need), width), -1, dtype=np.int32)
    at = 0
    for r, n in enumerate(need):
        table[r, :n] = perm[at:at + n]
        at += n
    dump = int(perm[at]) if extra_pages else -1
    return table, total, dump


def _pages_for(last_position: int) -> int:
    return last_position // PAGE_SIZE + 1


# workload name -> index (the default seed of workload k is 1000 + k)
WORKLOADS = {"phi3_tiny": 1, "mistral": 2, "phi3_window": 3, "qwen3": 4, "llama_step": 5,
             "llama_prefill": 6}


def build(name: str, seed: Optional[int] = None, scale: float = 1.0,
          rows: Optional[int] = None) -> Workload:
    """Build one of the five named workloads.

    ``scale`` (<= 1) shrinks context lengths (and chunk offsets) for small
    parity cases; ``rows`` overrides the number of decode rows.
    """
    idx = WORKLOADS[name]
    if seed is None:
        seed = 1000 + idx
    rng = np.random.default_rng(seed)
    empty = np.zeros(0, dtype=np.int32)

    def scaled(v: int, lo: int = 1) -> int:
        return max(lo, int(round(v * scale)))

    if name == "phi3_tiny":
        B = rows or 4
        pos = rng.integers(1, scaled(300, 2) + 1, size=B).astype(np.int32)
        num_pages = 64 if B <= 4 else 16 * B
        perm = rng.permutation(num_pages).astype(np.int32)
        table = perm.reshape(B, num_pages // B)
        return Workload(name, seed, 32, 32, 96, 10000.0, None, 2047, False, num_pages, table,
                        pos, empty, empty, empty, dump_page=-1)

    if name in ("mistral", "phi3_window"):
        if name == "mistral":
            B = rows or 64
            lo, hi = scaled(512, 2), scaled(8192, 3)
            hq, hkv, d, theta, window = 32, 8, 128, 1e6, 0
        else:
            B = rows or 32
            lo, hi = scaled(1000, 2), scaled(4096, 3)
            hq, hkv, d, theta, window = 32, 32, 96, 10000.0, 2047
        L = rng.integers(lo, hi + 1, size=B)
        pos = (L - 1).astype(np.int32)
        table, num_pages, dump = _assign_pages(rng, [_pages_for(int(p)) for p in pos])
        return Workload(name, seed, hq, hkv, d, theta, None, window, False, num_pages, table,
                        pos, empty, empty, empty, dump_page=dump)

    if name == "qwen3":
        B = rows or 256
        lo, hi = scaled(128, 2), scaled(16384, 3)
        L = np.floor(np.exp(rng.uniform(math.log(lo), math.log(hi), size=B))).astype(np.int64)
        L = np.clip(L, lo, hi)
        pos = (L - 1).astype(np.int32)
        group = 16
        share_max = 8
        need = []
        shared_n = []
        for b in range(B):
            s = min(share_max, int(pos[b]) // PAGE_SIZE)  # the page a row writes stays private
            shared_n.append(s)
            need.append(_pages_for(int(pos[b])) - s)
        n_groups = (B + group - 1) // group
        total = int(sum(need)) + n_groups * share_max + 1
        perm = rng.permutation(total).astype(np.int32)
        width = max(_pages_for(int(p)) for p in pos)
        table = np.full((B, width), -1, dtype=np.int32)
        at = 0
        shared_pages = []
        for g in range(n_groups):
            shared_pages.append(perm[at:at + share_max])
            at += share_max
        for b in range(B):
            s = shared_n[b]
            table[b, :s] = shared_pages[b // group][:s]
            n = need[b]
            table[b, s:s + n] = perm[at:at + n]
            at += n
        dump = int(perm[at])
        return Workload(name, seed, 32, 8, 128, 1e6, None, 0, True, total, table, pos,
                        empty, empty, empty, dump_page=dump)

    if name in ("llama_step", "llama_prefill"):
        # llama_step: 128 decode rows plus 4 chunks of 512 tokens;
        # llama_prefill: prefill alone, 4 chunks of 1024 tokens (4096 tokens)
        step = name == "llama_step"
        B = rows if rows is not None else (128 if step else 0)
        L = rng.integers(scaled(1024, 2), scaled(131072, 3) + 1, size=B)
        pos = (L - 1).astype(np.int32)
        full = 512 if step else 1024
        n_chunks, chunk = 4, (full if scale >= 1.0 else max(8, scaled(full, 8)))
        offsets = rng.integers(0, scaled(16384, 1) + 1, size=n_chunks)
        need = [_pages_for(int(p)) for p in pos]
        need += [_pages_for(int(o) + chunk - 1) for o in offsets]
        table, num_pages, dump = _assign_pages(rng, need)
        ch_rows = np.repeat(np.arange(B, B + n_chunks, dtype=np.int32), chunk)
        ch_pos = np.concatenate([np.arange(o, o + chunk) for o in offsets]).astype(np.int32)
        ch_seg = np.repeat(np.arange(n_chunks, dtype=np.int32), chunk)
        return Workload(name, seed, 32, 8, 128, 500000.0, (8.0, 1.0, 4.0, 8192), 0, False,
                        num_pages, table, pos, ch_rows, ch_pos, ch_seg, dump_page=dump)

    raise KeyError(name)


def custom(seed: int, hq: int, hkv: int, head_dim: int, dec_lengths, chunks=(),
           window: int = 0, theta: float = 10000.0, llama3=None, qk_norm: bool = False,
           inactive=(), spare_pages: int = 3) -> Workload:
    """A small workload with explicit lengths.

    ``dec_lengths[b]`` keys for decode row b (position = length - 1);
    ``chunks`` is a list of ``(offset, n_tokens)``: each chunk gets its own
    table row after the decode rows and positions ``offset .. offset+n-1``.
    Rows listed in ``inactive`` get position -1.
    """
    rng = np.random.default_rng(seed)
    pos = np.asarray(dec_lengths, dtype=np.int64) - 1
    need = [_pages_for(max(int(p), 0)) for p in pos]
    need += [_pages_for(int(o) + int(n) - 1) for o, n in chunks]
    table, num_pages, dump = _assign_pages(rng, need, extra_pages=spare_pages)
    pos = pos.astype(np.int32)
    for r in inactive:
        pos[r] = -1
    B = len(pos)
    ch_rows, ch_pos, ch_seg = [], [], []
    for c, (o, n) in enumerate(chunks):
        ch_rows += [B + c] * n
        ch_pos += list(range(o, o + n))
        ch_seg += [c] * n
    as32 = lambda a: np.asarray(a, dtype=np.int32)
    return Workload("custom", seed, hq, hkv, head_dim, theta, llama3, window, qk_norm,
                    num_pages, table, pos, as32(ch_rows), as32(ch_pos), as32(ch_seg),
                    dump_page=dump)
