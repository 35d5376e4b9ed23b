"""8-bit (E4M3) pools through the C ABI against the oracle (oracle/fp8.py).

The append's codes are integers decided from one float32 division and a
round-to-nearest-even on both sides, so they must match bit for bit; the
attention outputs match the exact attention of the dequantized pool within
the same bounds as the bf16 path.
"""
import zlib

import numpy as np
import pytest

import synth
from harness import ATT_MAX_ABS, ATT_MEAN_ABS, assert_attention_close, assert_ulp_close, to_bits
from oracle import fp8 as ofp8
from oracle import paged as opaged
from oracle import rope as orope

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

K_SCALE, V_SCALE = 0.25, 0.5


def _d16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def _d8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def _d32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _u8(t):
    return t.detach().cpu().numpy().astype(np.uint8)


class F8Step:
    """Device buffers of one workload step over 8-bit pools."""

    def __init__(self, w, fill="host", k_scale=K_SCALE, v_scale=V_SCALE):
        import paged_kv_gqa_row_gb300 as lnk
        self.w, self.lnk = w, lnk
        shape = (w.hkv, w.pool_positions, w.head_dim)
        if fill == "host":
            self.k_pool, self.v_pool = _d8(w.pool_e4m3("k")), _d8(w.pool_e4m3("v"))
        else:
            from synth import device as sdev
            self.k_pool = torch.empty(shape, dtype=torch.uint8, device="cuda")
            self.v_pool = torch.empty(shape, dtype=torch.uint8, device="cuda")
            sdev.fill_e4m3(self.k_pool, w.pool_key("k"))
            sdev.fill_e4m3(self.v_pool, w.pool_key("v"))
        self.q, self.k, self.v = _d16(w.step_q()), _d16(w.step_k()), _d16(w.step_v())
        self.positions, self.rows, self.table = _d32(w.token_positions()), _d32(w.token_rows()), _d32(w.table)
        gq, gk = w.gamma_q(), w.gamma_k()
        self.gamma_q = None if gq is None else _d16(gq)
        self.gamma_k = None if gk is None else _d16(gk)
        self.q_out = torch.zeros((w.T, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
        self.out = torch.zeros_like(self.q_out)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.desc = lnk.attn_desc(w.hq, w.hkv, w.head_dim, w.num_pages, w.num_rows, w.pages_per_row,
                                  window=w.window, kv_dtype=lnk.KV_E4M3, k_scale=k_scale, v_scale=v_scale)
        self.rope = lnk.rope_desc(w.theta, w.llama3)
        self.ws_bytes = max(lnk.lnk_paged_workspace_size(self.desc, max(w.B, 1)), 256)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device="cuda")
        self.dec_positions = _d32(w.dec_positions)

    def append(self):
        w = self.w
        self.lnk.lnk_paged_append_rope(self.desc, self.rope, self.q, self.k, self.v, self.positions, self.rows,
                                       None, self.table, self.gamma_q, self.gamma_k, w.norm_eps, self.k_pool,
                                       self.v_pool, self.q_out, w.T, self.status)

    def decode(self):
        w = self.w
        self.lnk.lnk_paged_decode_attn(self.desc, self.q_out[w.P:], self.dec_positions, self.table, self.k_pool,
                                       self.v_pool, self.out[w.P:], w.B, self.ws, self.ws_bytes, self.status)


def _oracle_full(w, k_scale=K_SCALE, v_scale=V_SCALE):
    inv = orope.inv_freq(w.theta, w.head_dim, w.llama3)
    q_out, kc, vc = ofp8.append_rope(w.step_q(), w.step_k(), w.step_v(), w.token_positions(), w.token_rows(),
                                     w.table, w.pool_e4m3("k"), w.pool_e4m3("v"), inv, k_scale, v_scale,
                                     gamma_q=w.gamma_q(), gamma_k=w.gamma_k(), eps=w.norm_eps)
    out = ofp8.decode_attention(q_out[w.P:], w.dec_positions, w.table, kc, vc, k_scale, v_scale, w.window)
    return q_out, kc, vc, out


def _check_full(w, poison=False, k_scale=K_SCALE, v_scale=V_SCALE):
    dev = F8Step(w, k_scale=k_scale, v_scale=v_scale)
    if poison:
        _poison(w, dev)
    dev.append()
    dev.decode()
    torch.cuda.synchronize()
    q_want, kc, vc, out_want = _oracle_full(w, k_scale, v_scale)
    assert_ulp_close(to_bits(dev.q_out), q_want, "q_out")
    kg, vg = _u8(dev.k_pool), _u8(dev.v_pool)
    if poison:  # the oracle's pool has finite codes where the device pool was poisoned
        m = np.broadcast_to(dev.poison_mask[None, :, None], kg.shape)
        kc, vc = np.where(m, kg, kc), np.where(m, vg, vc)
    assert np.array_equal(kg, kc), f"K codes: {int(np.sum(kg != kc))} differ"
    assert np.array_equal(vg, vc), f"V codes: {int(np.sum(vg != vc))} differ"
    got = to_bits(dev.out)[w.P:]
    for b in range(w.B):
        assert_attention_close(got[b], out_want[b], f"{w.name} row {b}")
    assert int(dev.status.item()) == 0


def _poison(w, dev):
    """NaN codes in every slot after each token's position in its last page."""
    mask = np.zeros(w.pool_positions, dtype=bool)
    for p, r in zip(w.token_positions(), w.token_rows()):
        if p >= 0:
            pg = int(w.table[r, p // 64])
            mask[pg * 64 + p % 64 + 1: pg * 64 + 64] = True
    for p, r in zip(w.token_positions(), w.token_rows()):
        if p >= 0:
            mask[int(w.table[r, p // 64]) * 64 + p % 64] = False
    idx = torch.from_numpy(np.nonzero(mask)[0]).cuda()
    dev.k_pool[:, idx, :] = 0x7F
    dev.v_pool[:, idx, :] = 0xFF
    dev.poison_mask = mask


DECODE_CASES = [
    ("mha64-edges", 4, 4, 64, [1, 2, 63, 64, 65, 130], 0, ()),
    ("gqa4-ragged", 8, 2, 128, [1000, 5, 64, 128, 2000, 777], 0, ()),
    ("gqa8", 16, 2, 128, [3000, 10, 4096], 0, ()),
    ("gqa2-window2047", 8, 4, 96, [300, 2047, 2048, 2049, 2100, 5000], 2047, ()),
    ("mha96-window100", 6, 6, 96, [50, 129, 700, 101, 100], 100, ()),
    ("inactive-rows", 8, 2, 128, [100, 1, 257, 64], 0, (1, 3)),
    ("many-short-rows", 32, 8, 128, [17] * 40 + [65] * 9, 0, ()),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=[c[0] for c in DECODE_CASES])
def test_e4m3_append_and_decode_match_oracle(case):
    name, hq, hkv, d, lengths, window, inactive = case
    w = synth.custom(seed=zlib.crc32(("e4m3" + name).encode()) % 10000, hq=hq, hkv=hkv, head_dim=d,
                     dec_lengths=lengths, window=window, inactive=inactive)
    _check_full(w)


def test_e4m3_decode_ignores_nan_codes_in_unread_slots():
    w = synth.custom(seed=77, hq=8, hkv=2, head_dim=128, dec_lengths=[5, 64, 130, 300])
    _check_full(w, poison=True)


@pytest.mark.parametrize("hq,hkv,d,window", [(8, 2, 128, 0), (6, 6, 96, 100), (16, 2, 64, 0)],
                         ids=["gqa4-128", "mha96-window100", "gqa8-64"])
def test_e4m3_every_finite_code_in_the_pools(hq, hkv, d, window):
    """Prefilled pools drawn from all 254 finite codes: subnormals, zeros, the
    smallest and the saturated +-448 are all read by the decode kernel.  Small
    pool scales (K x 2^-6, V x 2^-7) keep the outputs at unit scale."""
    w = synth.custom(seed=zlib.crc32(f"e4m3-all-{hq}-{d}".encode()) % 10000, hq=hq, hkv=hkv, head_dim=d,
                     dec_lengths=[1, 64, 65, 700, 2000, 3000], window=window)
    w.e4m3_all = True
    codes = w.pool_e4m3("k")
    assert len(np.unique(codes)) == 254  # every finite code occurs
    _check_full(w, k_scale=2.0 ** -6, v_scale=2.0 ** -7)


@pytest.mark.parametrize("name, scale, rows", [("mistral", 0.06, 12), ("qwen3", 0.05, 40), ("phi3_window", 0.6, 8)])
def test_e4m3_workloads_scaled_down(name, scale, rows):
    _check_full(synth.build(name, scale=scale, rows=rows))


def _oracle_token_e4m3(w, t):
    """One decode token's output on a compact 8-bit pool of the pages it reads."""
    tp, tr = w.token_positions(), w.token_rows()
    p, row = int(tp[t]), int(tr[t])
    lo, hi = opaged.visible_range(p, w.window)
    lps = np.arange(lo // 64, hi // 64 + 1)
    pages = w.table[row, lps]
    index = {int(pg): i for i, pg in enumerate(pages)}
    kc = np.stack([w.pool_pages_e4m3("k", h, pages).reshape(-1, w.head_dim) for h in range(w.hkv)])
    vc = np.stack([w.pool_pages_e4m3("v", h, pages).reshape(-1, w.head_dim) for h in range(w.hkv)])
    writers, slots = [], []
    for u in range(w.T):
        pu = int(tp[u])
        if pu >= 0 and int(w.table[int(tr[u]), pu // 64]) in index:
            writers.append(u)
            slots.append(index[int(w.table[int(tr[u]), pu // 64])] * 64 + pu % 64)
    wi = np.array(writers)
    inv = orope.inv_freq(w.theta, w.head_dim, w.llama3)
    gq, gk = w.gamma_q(), w.gamma_k()
    q_out, kc, vc = ofp8.append_rope(w.step_q()[wi], w.step_k()[wi], w.step_v()[wi], tp[wi], tr[wi], None, kc, vc,
                                     inv, K_SCALE, V_SCALE, slots=np.array(slots), gamma_q=gq, gamma_k=gk,
                                     eps=w.norm_eps)
    ctable = np.full((1, lps[-1] + 1), -1, dtype=np.int32)
    ctable[0, lps] = np.arange(len(lps), dtype=np.int32)
    return ofp8.attention_at(q_out[writers.index(t)], 0, p, ctable, kc, vc, K_SCALE, V_SCALE, w.window)


@pytest.mark.parametrize("name", ["mistral", "qwen3"])
def test_e4m3_workload_full_size_sampled(name):
    w = synth.build(name)
    dev = F8Step(w, fill="device")
    dev.append()
    dev.decode()
    torch.cuda.synchronize()
    assert int(dev.status.item()) == 0
    out = to_bits(dev.out)
    order = np.argsort(w.dec_positions)
    for b in sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1]), 0, w.B - 1}):
        assert_attention_close(out[w.P + b], _oracle_token_e4m3(w, w.P + b), f"{name} row {b}")


def test_e4m3_step_rejects_chunks_and_serves_decode_rows():
    import paged_kv_gqa_row_gb300 as lnk
    w = synth.custom(seed=5, hq=8, hkv=2, head_dim=128, dec_lengths=[100, 200], chunks=[(0, 40)])
    dev = F8Step(w)
    dev.append()
    with pytest.raises(lnk.LnkError) as e:
        lnk.lnk_paged_step_attn(dev.desc, dev.q_out, _d32(w.ch_rows), _d32(w.ch_positions), None,
                                dev.dec_positions, dev.table, dev.k_pool, dev.v_pool, dev.out, None, None,
                                w.P, w.B, 0, dev.ws, dev.ws_bytes, dev.status)
    assert e.value.status == 4  # LNK_EUNSUPPORTED
    # decode rows alone through step_attn
    lnk.lnk_paged_step_attn(dev.desc, dev.q_out[w.P:], None, None, None, dev.dec_positions, dev.table,
                            dev.k_pool, dev.v_pool, dev.out[w.P:], None, None, 0, w.B, 0, dev.ws, dev.ws_bytes,
                            dev.status)
    torch.cuda.synchronize()
    q_want, kc, vc, out_want = _oracle_full(w)
    got = to_bits(dev.out)[w.P:]
    for b in range(w.B):
        assert_attention_close(got[b], out_want[b], f"row {b}")


def test_e4m3_copy_pages_and_argument_errors():
    import paged_kv_gqa_row_gb300 as lnk
    d = lnk.attn_desc(4, 2, 96, 6, 1, 6, kv_dtype=lnk.KV_E4M3, k_scale=1.0, v_scale=1.0)
    k0 = synth.e4m3_codes(11, 0, 2 * 6 * 64 * 96).reshape(2, 6 * 64, 96)
    v0 = synth.e4m3_codes(12, 0, 2 * 6 * 64 * 96).reshape(2, 6 * 64, 96)
    kp, vp = _d8(k0), _d8(v0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lnk.lnk_paged_copy_pages(d, kp, vp, _d32([4, 1]), _d32([0, 5]), 2, status)
    torch.cuda.synchronize()
    kw, vw = k0.copy(), v0.copy()
    for s, t in ((4, 0), (1, 5)):
        kw[:, t * 64:(t + 1) * 64] = k0[:, s * 64:(s + 1) * 64]
        vw[:, t * 64:(t + 1) * 64] = v0[:, s * 64:(s + 1) * 64]
    assert np.array_equal(_u8(kp), kw) and np.array_equal(_u8(vp), vw) and int(status.item()) == 0
    # bad descriptors are refused on the host
    q = torch.zeros((1, 4, 96), dtype=torch.int16, device="cuda")
    pos = _d32([3])
    tab = _d32(np.zeros((1, 6)))
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    for bad, code in ((dict(kv_dtype=2), 4), (dict(kv_dtype=lnk.KV_E4M3, k_scale=0.0), 1),
                      (dict(kv_dtype=lnk.KV_E4M3, v_scale=float("nan")), 1),
                      (dict(kv_dtype=lnk.KV_E4M3, k_scale=float("inf")), 1)):
        args = dict(kv_dtype=lnk.KV_BF16, k_scale=1.0, v_scale=1.0)
        args.update(bad)
        bd = lnk.attn_desc(4, 2, 96, 6, 1, 6, **args)
        with pytest.raises(lnk.LnkError) as e:
            lnk.lnk_paged_decode_attn(bd, q, pos, tab, kp, vp, q, 1, ws, ws.numel(), status)
        assert e.value.status == code
