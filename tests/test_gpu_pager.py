"""Rows that share a prompt prefix, driven by the library's page allocator.

Row 0 is prefilled with a 150-token prompt (prefill_paged); rows 1 and 2
fork it at 150 tokens and row 3 at 100, so that the pages of the prefix are
mapped by several rows, the partial last pages included.  Then every row
decodes 70 tokens.  The first write of a row into a shared page moves it onto
a private copy (lnk_paged_copy_pages), later pages are fresh.  The library's
allocator must match the oracle's model call by call, and every row's
outputs must match the oracle's attention over that row's own contiguous
history (its prefix followed by its own tokens).
"""
import numpy as np
import pytest

import synth
from harness import assert_attention_close, assert_ulp_close, to_bits
from oracle import paged as opaged
from oracle import pager as opager
from oracle import rope as orope

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

HQ, HKV, D = 8, 2, 128
NUM_PAGES, NUM_ROWS, PPR = 24, 4, 5
THETA = 10000.0
PROMPT, FORK3, STEPS = 150, 100, 70
SEED = 4242


def _d16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def _d32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


class _History:
    """The oracle's view: each row's keys and values in its own contiguous
    pool (identity page table), written by the oracle's append."""

    def __init__(self):
        self.inv = orope.inv_freq(THETA, D, None)
        self.ident = np.arange(PPR, dtype=np.int32)[None, :]
        self.k = {r: np.zeros((HKV, PPR * 64, D), np.uint16) for r in range(NUM_ROWS)}
        self.v = {r: np.zeros((HKV, PPR * 64, D), np.uint16) for r in range(NUM_ROWS)}

    def append(self, row, pos, q, k, v):
        q_out, self.k[row], self.v[row] = opaged.append_rope(
            q[None], k[None], v[None], np.array([pos]), np.array([0]), self.ident, self.k[row], self.v[row],
            self.inv)
        return q_out[0]

    def fork(self, src, dst):
        # positions past the fork point are overwritten by dst before it sees them
        self.k[dst], self.v[dst] = self.k[src].copy(), self.v[src].copy()

    def attention(self, row, pos, q_bits):
        return opaged.attention_at(q_bits, 0, pos, self.ident, self.k[row], self.v[row], 0)


def test_forked_rows_decode_through_the_pager():
    import paged_kv_gqa_row_gb300 as lnk
    pg = lnk.Pager(NUM_PAGES, NUM_ROWS, PPR)
    model = opager.Pager(NUM_PAGES, NUM_ROWS, PPR)
    hist = _History()
    desc = lnk.attn_desc(HQ, HKV, D, NUM_PAGES, NUM_ROWS, PPR)
    rd = lnk.rope_desc(THETA)
    # the pool starts with stale data everywhere
    k_pool = _d16(synth.tensor_bf16(SEED, 1, (HKV, NUM_PAGES * 64, D)))
    v_pool = _d16(synth.tensor_bf16(SEED, 2, (HKV, NUM_PAGES * 64, D)))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws_bytes = lnk.lnk_paged_workspace_size(desc, NUM_ROWS)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")

    def append(rows, positions, q, k, v):
        copies = pg.prepare_append(rows, positions)
        assert copies == model.prepare_append(rows, positions)
        if copies:
            lnk.lnk_paged_copy_pages(desc, k_pool, v_pool, _d32([c[0] for c in copies]),
                                     _d32([c[1] for c in copies]), len(copies), status)
        table = pg.table()
        assert np.array_equal(table, np.asarray(model.table(), dtype=np.int32))
        dt = _d32(table)
        q_out = torch.zeros((len(rows), HQ, D), dtype=torch.int16, device="cuda")
        lnk.lnk_paged_append_rope(desc, rd, _d16(q), _d16(k), _d16(v), _d32(positions), _d32(rows), None, dt,
                                  None, None, 1e-6, k_pool, v_pool, q_out, len(rows), status)
        q_want = np.stack([hist.append(r, p, q[i], k[i], v[i]) for i, (r, p) in enumerate(zip(rows, positions))])
        assert_ulp_close(to_bits(q_out), q_want, "q_out")
        return dt, q_out, q_want

    # ---- prefill of row 0 ----
    q = synth.tensor_bf16(SEED, 10, (PROMPT, HQ, D))
    k = synth.tensor_bf16(SEED, 11, (PROMPT, HKV, D))
    v = synth.tensor_bf16(SEED, 12, (PROMPT, HKV, D))
    rows, pos = [0] * PROMPT, list(range(PROMPT))
    dt, q_out, q_want = append(rows, pos, q, k, v)
    out = torch.zeros_like(q_out)
    lnk.lnk_paged_step_attn(desc, q_out, _d32(rows), _d32(pos), _d32([0] * PROMPT), None, dt, k_pool, v_pool,
                            out, None, None, PROMPT, 0, 0, ws, ws_bytes, status)
    got = to_bits(out)
    for t in (0, 1, 63, 64, 127, 128, 149):
        assert_attention_close(got[t], hist.attention(0, t, q_want[t]), f"prompt token {t}")

    # ---- forks ----
    for dst, n in ((1, PROMPT), (2, PROMPT), (3, FORK3)):
        pg.fork(0, dst, n)
        model.fork(0, dst, n)
        hist.fork(0, dst)
    assert [pg.refcount(p) for p in range(3)] == [4, 4, 3]

    # ---- decode ----
    check = {0, 1, 27, 28, 29, 41, 42, 43, STEPS - 1}
    for s in range(STEPS):
        rows = [0, 1, 2, 3]
        positions = [PROMPT + s, PROMPT + s, PROMPT + s, FORK3 + s]
        q = synth.tensor_bf16(SEED, 100 + 3 * s, (4, HQ, D))
        k = synth.tensor_bf16(SEED, 101 + 3 * s, (4, HKV, D))
        v = synth.tensor_bf16(SEED, 102 + 3 * s, (4, HKV, D))
        dt, q_out, q_want = append(rows, positions, q, k, v)
        out = torch.zeros_like(q_out)
        lnk.lnk_paged_decode_attn(desc, q_out, _d32(positions), dt, k_pool, v_pool, out, 4, ws, ws_bytes,
                                  status)
        if s in check:
            got = to_bits(out)
            for r in rows:
                assert_attention_close(got[r], hist.attention(r, positions[r], q_want[r]), f"step {s} row {r}")
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # every row now owns private pages for what it wrote; the prefix pages stay shared
    t = pg.table()
    assert len({int(t[r, 2]) for r in range(4)}) == 4
    for r in range(NUM_ROWS):
        pg.release(r)
    assert pg.free_pages() == NUM_PAGES


def test_copy_pages_moves_whole_pages():
    import paged_kv_gqa_row_gb300 as lnk
    desc = lnk.attn_desc(HQ, HKV, 96, 10, 1, 10)
    k0 = synth.tensor_bf16(SEED, 50, (HKV, 10 * 64, 96))
    v0 = synth.tensor_bf16(SEED, 51, (HKV, 10 * 64, 96))
    k_pool, v_pool = _d16(k0), _d16(v0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lnk.lnk_paged_copy_pages(desc, k_pool, v_pool, _d32([3, 7, 12]), _d32([5, 0, 1]), 3, status)
    torch.cuda.synchronize()
    kw, vw = k0.copy(), v0.copy()
    for s, d in ((3, 5), (7, 0)):
        kw[:, d * 64:(d + 1) * 64] = k0[:, s * 64:(s + 1) * 64]
        vw[:, d * 64:(d + 1) * 64] = v0[:, s * 64:(s + 1) * 64]
    assert np.array_equal(to_bits(k_pool), kw) and np.array_equal(to_bits(v_pool), vw)
    assert int(status.item()) == lnk.binding.DEV_BAD_PAGE  # the pair with page 12 was skipped
