"""Paged pool, append and attention for the oracle (test infrastructure only).

Sources
  * "Phi-3 Mini 4K Instruct -- files", src/attention.linnet:
    - ``decode_rows``: each row's new key/value is written at its position,
      and its query attends over that row up to and including it;
    - ``prefill_packed`` / ``step_packed``: packed prompt tokens, each with a
      row, a position and a segment; a token attends to its own prompt's
      tokens up to itself; a step is the prompts followed by one token per row;
    - ``window_mask`` and the masks of every entry: key j is visible to a
      query at position p iff ``j <= p`` and ``j > p - WINDOW`` (the query
      itself and the WINDOW - 1 positions before it);
    - the attention scale ``rsqrt(head_dim)``.
  * "Mistral 7B Instruct v0.3", Entries table (``prefill_paged``,
    ``decode_paged``, ``step_paged``): the caches' one row is a pool of
    positions in pages of 64, row b's positions lie in the pages ``table[b]``
    lists, and each token is written at its place in the pool and attends over
    its row's pages up to its position.
  * "Phi-3 Mini 4K Instruct -- files", src/lib.linnet, ``prefill_packed``:
    padding tokens write where no request reads.

Readings where the pages are silent (each one is listed in the design notes):
  * Pool layout ``[kv_heads, num_pages * 64, head_dim]`` (the caches'
    ``[Batch=1, Heads, MaxSeq, D]`` with MaxSeq = num_pages * 64); logical
    position j of row r is pool slot ``table[r][j // 64] * 64 + j % 64``.
  * Query head h reads kv head ``h // (Hq / Hkv)`` (contiguous groups).
  * A packed chunk token attends over its own row's pages, so it sees that
    row's earlier cached context as well as its own chunk up to itself; tokens
    of other prompts live in other rows and are never seen.
  * Decode row b uses table row b.  A negative position marks an inactive
    token: nothing is written and its output is zero.
"""
import numpy as np

from . import bf16
from . import rope

PAGE_SIZE = 64


def slot_of(table: np.ndarray, row: int, position: int) -> int:
    """Pool slot of logical position ``position`` of table row ``row``."""
    page = int(table[row, position // PAGE_SIZE])
    return page * PAGE_SIZE + position % PAGE_SIZE


def kv_head_of(q_head: int, group: int, num_kv_heads: int) -> int:
    """kv head read by query head ``q_head`` (groups of ``group`` consecutive heads)."""
    return q_head // group


def default_scale(head_dim: int) -> float:
    """Attention scale ``rsqrt(head_dim)``."""
    return 1.0 / np.sqrt(head_dim)


def visible_range(position: int, window: int):
    """Inclusive key range ``(lo, hi)`` a query at ``position`` attends to."""
    lo = max(0, position - window + 1) if window > 0 else 0
    return lo, position


def append_rope(q, k, v, positions, rows, table, k_pool, v_pool, inv,
                slots=None, gamma_q=None, gamma_k=None, eps=1e-6):
    """Rotate (after optional QK-norm) each token's q and k, write k and v.

    q: bf16 [T, Hq, D]; k, v: bf16 [T, Hkv, D]; positions, rows: int [T];
    pools: bf16 [Hkv, S, D] (not modified); ``slots[t]`` overrides the slot
    token t writes.  Returns ``(q_out, k_pool', v_pool')`` as bf16 arrays.
    """
    T = q.shape[0]
    q_out = np.zeros_like(q, dtype=np.uint16)
    k_pool = np.array(k_pool, dtype=np.uint16, copy=True)
    v_pool = np.array(v_pool, dtype=np.uint16, copy=True)
    gq = None if gamma_q is None else bf16.to_f64(gamma_q)
    gk = None if gamma_k is None else bf16.to_f64(gamma_k)
    for t in range(T):
        p = int(positions[t])
        if p < 0:
            continue
        ang = rope.angles(p, inv)
        qf = bf16.to_f64(q[t])
        kf = bf16.to_f64(k[t])
        if gq is not None:
            qf = rope.qk_norm(qf, gq, eps)
        if gk is not None:
            kf = rope.qk_norm(kf, gk, eps)
        q_out[t] = bf16.from_f64(rope.rotate(qf, ang))
        k_rot = bf16.from_f64(rope.rotate(kf, ang))
        s = int(slots[t]) if slots is not None else slot_of(table, int(rows[t]), p)
        k_pool[:, s, :] = k_rot
        v_pool[:, s, :] = v[t]
    return q_out, k_pool, v_pool


def attend(q: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float) -> np.ndarray:
    """softmax(q keys^T * scale) values, float64.  q: [G, D]; keys, values: [n, D]."""
    s = (q @ keys.T) * scale
    m = np.max(s, axis=1, keepdims=True)
    w = np.exp(s - m)
    return (w @ values) / np.sum(w, axis=1, keepdims=True)


def row_slots(table: np.ndarray, row: int, lo: int, hi: int) -> np.ndarray:
    j = np.arange(lo, hi + 1, dtype=np.int64)
    return table[row, j // PAGE_SIZE].astype(np.int64) * PAGE_SIZE + j % PAGE_SIZE


def attention_at(q_bits, row, position, table, k_pool, v_pool, window, scale=None):
    """Output of one token (all its query heads) over its row's visible keys.

    q_bits: bf16 [Hq, D] (already rotated); returns float64 [Hq, D].
    """
    hq, d = q_bits.shape
    hkv = k_pool.shape[0]
    group = hq // hkv
    if scale is None:
        scale = default_scale(d)
    out = np.zeros((hq, d), dtype=np.float64)
    if position < 0:
        return out
    lo, hi = visible_range(position, window)
    slots = row_slots(table, row, lo, hi)
    qf = bf16.to_f64(q_bits)
    for kvh in range(hkv):
        heads = [h for h in range(hq) if kv_head_of(h, group, hkv) == kvh]
        if not heads:
            continue
        keys = bf16.to_f64(k_pool[kvh, slots, :])
        values = bf16.to_f64(v_pool[kvh, slots, :])
        out[heads] = attend(qf[heads], keys, values, scale)
    return out


def decode_attention(q_out, positions, table, k_pool, v_pool, window, scale=None):
    """One token per decode row b, over table row b.  Returns float64 [B, Hq, D]."""
    B = q_out.shape[0]
    out = np.zeros(q_out.shape, dtype=np.float64)
    for b in range(B):
        out[b] = attention_at(q_out[b], b, int(positions[b]), table, k_pool, v_pool, window, scale)
    return out


def chunk_attention(q_out, rows, positions, table, k_pool, v_pool, window, scale=None):
    """Packed prompt tokens, each over its own row's pages.  Returns float64 [P, Hq, D]."""
    P = q_out.shape[0]
    out = np.zeros(q_out.shape, dtype=np.float64)
    for t in range(P):
        out[t] = attention_at(q_out[t], int(rows[t]), int(positions[t]), table,
                              k_pool, v_pool, window, scale)
    return out


def step_attention(q_out, rows, positions, step_positions, table, k_pool, v_pool,
                   window, scale=None):
    """``P`` chunk tokens followed by ``B`` decode rows (row b = table row b)."""
    P = len(positions)
    a = chunk_attention(q_out[:P], rows, positions, table, k_pool, v_pool, window, scale)
    b = decode_attention(q_out[P:], step_positions, table, k_pool, v_pool, window, scale)
    return np.concatenate([a, b], axis=0)


def packed_attention(q_bits, k_bits, v_bits, positions, segments, window, scale=None):
    """The row-based packed-prompt rule over the pack's own keys and values.

    Token i attends to pack tokens j with ``segments[j] == segments[i]``,
    ``positions[j] <= positions[i]`` and ``positions[j] > positions[i] - WINDOW``.
    q_bits: bf16 [P, Hq, D]; k_bits, v_bits: bf16 [P, Hkv, D] (k already rotated).
    """
    P, hq, d = q_bits.shape
    hkv = k_bits.shape[1]
    group = hq // hkv
    if scale is None:
        scale = default_scale(d)
    positions = np.asarray(positions)
    segments = np.asarray(segments)
    out = np.zeros((P, hq, d), dtype=np.float64)
    qf, kf, vf = bf16.to_f64(q_bits), bf16.to_f64(k_bits), bf16.to_f64(v_bits)
    for i in range(P):
        own = (segments == segments[i]) & (positions <= positions[i])
        if window > 0:
            own &= positions > positions[i] - window
        js = np.nonzero(own)[0]
        js = js[np.argsort(positions[js], kind="stable")]
        for h in range(hq):
            kvh = kv_head_of(h, group, hkv)
            out[i, h] = attend(qf[i, h][None], kf[js, kvh], vf[js, kvh], scale)[0]
    return out
