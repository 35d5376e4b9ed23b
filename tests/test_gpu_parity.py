"""CUDA path (through the C ABI) against the CPU oracle on the same seeded inputs."""
import zlib

import numpy as np
import pytest

import synth
from harness import (DeviceStep, assert_attention_close, assert_ulp_close, oracle_full,
                     oracle_tokens, to_bits)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _sync():
    torch.cuda.synchronize()


def _check_full(w, dev=None, nan_tails=False):
    """Run the workload on the GPU and compare everything against the whole-pool oracle."""
    dev = dev or DeviceStep(w, fill="host")
    if nan_tails:
        _poison_tails(w, dev)
    k0 = to_bits(dev.k_pool)
    dev.step()
    _sync()
    q_want, kp_want, vp_want, out_want = oracle_full(w)
    assert_ulp_close(to_bits(dev.q_out), q_want, "q_out")
    kp_got, vp_got = to_bits(dev.k_pool), to_bits(dev.v_pool)
    if nan_tails:  # the oracle pool has finite values where the device pool was poisoned
        mask = to_bits_mask(w)
        kp_want = np.where(mask, kp_got, kp_want)
        vp_want = np.where(mask, vp_got, vp_want)
    assert_ulp_close(kp_got, kp_want, "k_pool")
    assert np.array_equal(vp_got, vp_want), "v_pool"
    changed = np.any(kp_got != k0, axis=(0, 2))
    assert changed.sum() <= w.T
    mx, mean = assert_attention_close(to_bits(dev.out), out_want, w.name)
    assert int(dev.status.item()) == 0
    return mx, mean


_POISON = {}


def _poison_tails(w, dev):
    """Write NaN into every slot after each token's position in the last page it reads
    (never visible to anyone), so that masked keys must not leak into P.V."""
    mask = np.zeros((w.pool_positions,), dtype=bool)
    for p, r in zip(w.token_positions(), w.token_rows()):
        if p < 0:
            continue
        pg = int(w.table[r, p // 64])
        mask[pg * 64 + p % 64 + 1: pg * 64 + 64] = True
    # slots written by the step itself stay as they are
    for p, r in zip(w.token_positions(), w.token_rows()):
        if p >= 0:
            mask[int(w.table[r, p // 64]) * 64 + p % 64] = False
    idx = torch.from_numpy(np.nonzero(mask)[0]).cuda()
    nan = torch.tensor(0x7FC0, dtype=torch.int16, device="cuda")
    dev.k_pool[:, idx, :] = nan
    dev.v_pool[:, idx, :] = nan
    _POISON[id(w)] = mask


def to_bits_mask(w):
    m = _POISON[id(w)]
    return np.broadcast_to(m[None, :, None], (w.hkv, w.pool_positions, w.head_dim))


# ------------------------------------------------------------------ decode ----

DECODE_CASES = [
    # id, hq, hkv, D, lengths, window, inactive rows
    ("mha64-edges", 4, 4, 64, [1, 2, 63, 64, 65, 130], 0, ()),
    ("gqa4-ragged", 8, 2, 128, [1000, 5, 64, 128, 2000, 777], 0, ()),
    ("gqa8", 16, 2, 128, [3000, 10, 4096], 0, ()),
    ("gqa2-window2047", 8, 4, 96, [300, 2047, 2048, 2049, 2100, 5000], 2047, ()),
    ("mha96-window100", 6, 6, 96, [50, 129, 700, 101, 100], 100, ()),
    ("inactive-rows", 8, 2, 128, [100, 1, 257, 64], 0, (1, 3)),
    ("many-short-rows", 32, 8, 128, [17] * 40 + [65] * 9, 0, ()),
    ("one-row-long", 32, 8, 128, [40000], 0, ()),
    ("window-1-sees-itself", 8, 2, 64, [1, 2, 64, 65, 300], 1, ()),
    ("all-inactive", 8, 2, 128, [5, 6, 7], 0, (0, 1, 2)),
    # enough (row, kv head) pairs for the two-CTAs-per-SM variant (B * Hkv >= 4 * SMs)
    ("many-pairs", 32, 8, 128, [1 + (37 * i) % 700 for i in range(80)], 0, ()),
    ("many-pairs-mha96-window", 16, 16, 96, [1 + (53 * i) % 900 for i in range(40)], 300, ()),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=[c[0] for c in DECODE_CASES])
def test_decode_matches_oracle(case):
    name, hq, hkv, d, lengths, window, inactive = case
    w = synth.custom(seed=zlib.crc32(name.encode()) % 10000, hq=hq, hkv=hkv, head_dim=d, dec_lengths=lengths,
                     window=window, inactive=inactive)
    _check_full(w)


def test_decode_ignores_garbage_beyond_positions():
    w = synth.custom(seed=5, hq=8, hkv=2, head_dim=128, dec_lengths=[70, 5, 200, 64, 1], window=0)
    _check_full(w, nan_tails=True)


def test_decode_window_garbage_before_window():
    w = synth.custom(seed=6, hq=8, hkv=8, head_dim=96, dec_lengths=[3000, 2500], window=2047)
    dev = DeviceStep(w, fill="host")
    # NaN in the part of each row's first visible page that lies before the window
    for b, p in enumerate(w.dec_positions):
        lo = int(p) - 2047 + 1
        pg = int(w.table[b, lo // 64])
        dev.k_pool[:, pg * 64: pg * 64 + lo % 64, :] = torch.tensor(0x7FC0, dtype=torch.int16, device="cuda")
        dev.v_pool[:, pg * 64: pg * 64 + lo % 64, :] = torch.tensor(0x7FC0, dtype=torch.int16, device="cuda")
    dev.step()
    _sync()
    _, kp, vp, out = oracle_full(w)
    assert_attention_close(to_bits(dev.out), out, "window garbage")


# -------------------------------------------------------------------- step ----

STEP_CASES = [
    # id, hq, hkv, D, decode lengths, chunks (offset, tokens), window
    ("step-gqa4", 8, 2, 128, [300, 1200], [(0, 70), (100, 5), (1000, 130)], 0),
    ("prefill-only-mha64", 8, 8, 64, [], [(0, 200), (37, 60)], 0),
    ("step-window-gqa2", 8, 4, 96, [3000], [(2500, 300), (0, 40)], 2047),
    ("step-gqa8-window100", 16, 2, 128, [64], [(63, 20), (640, 64)], 100),
    ("tiny-chunks", 8, 2, 128, [5, 9], [(0, 1), (3, 2), (7, 3), (64, 1), (100, 9)], 0),
]


@pytest.mark.parametrize("case", STEP_CASES, ids=[c[0] for c in STEP_CASES])
def test_step_matches_oracle(case):
    name, hq, hkv, d, lengths, chunks, window = case
    w = synth.custom(seed=zlib.crc32(name.encode()) % 10000, hq=hq, hkv=hkv, head_dim=d, dec_lengths=lengths,
                     chunks=chunks, window=window)
    _check_full(w)


def test_step_with_garbage_tails():
    w = synth.custom(seed=9, hq=8, hkv=2, head_dim=128, dec_lengths=[90], chunks=[(10, 50), (0, 7)])
    _check_full(w, nan_tails=True)


def test_step_last_gather():
    w = synth.custom(seed=10, hq=8, hkv=2, head_dim=128, dec_lengths=[300], chunks=[(0, 40), (64, 30)])
    dev = DeviceStep(w, fill="host")
    last = torch.tensor([39, 69, 0], dtype=torch.int32, device="cuda")
    last_out = torch.zeros((3, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
    dev.append()
    dev.attend(last=last, last_out=last_out)
    _sync()
    got = to_bits(dev.out)
    assert np.array_equal(to_bits(last_out), got[[39, 69, 0]])


# ----------------------------------------------------------- rope / append ----

APPEND_CASES = [
    # id, hq, hkv, D, theta, llama3, qk_norm
    ("plain-96", 8, 8, 96, 10000.0, None, False),
    ("qknorm-128", 8, 2, 128, 1e6, None, True),
    ("llama3-128", 8, 2, 128, 500000.0, (8.0, 1.0, 4.0, 8192), False),
    ("qknorm-64-gqa8", 16, 2, 64, 1e4, None, True),
]


@pytest.mark.parametrize("case", APPEND_CASES, ids=[c[0] for c in APPEND_CASES])
def test_append_rope_matches_oracle(case):
    name, hq, hkv, d, theta, llama3, qkn = case
    lengths = [1, 64, 65, 1000, 20000] + ([131072] if hkv <= 2 else [])
    w = synth.custom(seed=11, hq=hq, hkv=hkv, head_dim=d, dec_lengths=lengths, theta=theta,
                     llama3=llama3, qk_norm=qkn, chunks=[(5, 3)])
    _check_full(w)


@pytest.mark.parametrize("hq,hkv,d,qkn", [(32, 8, 128, True), (32, 32, 96, False)], ids=["qknorm-128", "mha-96"])
def test_append_wide_launch_matches_oracle(hq, hkv, d, qkn):
    # at least 4 tokens per SM: the append takes its 8-warps-per-token form
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = 4 * sms + 50
    w = synth.custom(seed=17, hq=hq, hkv=hkv, head_dim=d, dec_lengths=[300, 9000, 1], theta=1e6, qk_norm=qkn,
                     chunks=[(0, n // 2), (1000, n - n // 2)])
    assert w.T >= 4 * sms
    _check_full(w)


def test_append_explicit_slots_and_inactive():
    w = synth.custom(seed=12, hq=8, hkv=2, head_dim=128, dec_lengths=[100, 10, 300])
    dev = DeviceStep(w, fill="host")
    dump = w.dump_page * 64 + 5
    slots = torch.tensor([dump, int(w.table[1, 0]) * 64 + 9, dump], dtype=torch.int32, device="cuda")
    pos = w.token_positions().copy()
    pos[2] = -1
    dev.positions.copy_(torch.from_numpy(pos))
    k0, v0 = to_bits(dev.k_pool), to_bits(dev.v_pool)
    dev.append(slots=slots)
    _sync()
    k1, v1 = to_bits(dev.k_pool), to_bits(dev.v_pool)
    changed = sorted(set(np.nonzero(np.any(k1 != k0, axis=(0, 2)))[0]) |
                     set(np.nonzero(np.any(v1 != v0, axis=(0, 2)))[0]))
    assert changed == sorted([dump, int(w.table[1, 0]) * 64 + 9])
    assert np.array_equal(v1[:, dump], w.step_v()[0])
    assert not np.any(to_bits(dev.q_out)[2])  # inactive token: zero query output


def test_inv_freq_table_matches_oracle():
    import paged_kv_gqa_row_gb300 as lnk
    from oracle import rope
    for theta, d, l3 in [(1e4, 96, None), (1e6, 128, None), (5e5, 128, (8.0, 1.0, 4.0, 8192)), (1e4, 64, None)]:
        got = np.array(lnk.lnk_rope_inv_freq(lnk.rope_desc(theta, l3), d), dtype=np.float32)
        assert np.array_equal(got.view(np.uint32), rope.inv_freq(theta, d, l3).view(np.uint32))


# ------------------------------------------------------------- workloads ----

@pytest.mark.parametrize("name", ["phi3_tiny", "mistral", "phi3_window", "qwen3", "llama_step", "llama_prefill"])
def test_workload_scaled_down(name):
    scale = {"phi3_tiny": 1.0, "mistral": 0.06, "phi3_window": 0.6, "qwen3": 0.05, "llama_step": 0.02,
             "llama_prefill": 0.03}[name]
    rows = {"phi3_tiny": None, "mistral": 12, "phi3_window": 8, "qwen3": 40, "llama_step": 6,
            "llama_prefill": None}[name]
    w = synth.build(name, scale=scale, rows=rows)
    _check_full(w)


def _sample_tokens(w, n_dec=6, per_chunk=2):
    toks = []
    if w.B:
        order = np.argsort(w.dec_positions)
        picks = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])} |
                       {int(x) for x in np.linspace(0, w.B - 1, max(0, n_dec - 3)).astype(int)})
        toks = [w.P + b for b in picks]
    for c in np.unique(w.ch_segments):
        idx = np.nonzero(w.ch_segments == c)[0]
        # first, last, and (for long chunks) a token inside: a tile boundary and a ragged one
        extra = [int(idx[len(idx) // 2]), int(idx[min(len(idx) - 1, 130)])] if per_chunk > 2 else []
        toks += ([int(idx[0]), int(idx[-1])] + extra)[:per_chunk]
    return toks


@pytest.mark.parametrize("name", ["mistral", "phi3_window", "qwen3", "llama_step", "llama_prefill"])
def test_workload_full_size_sampled(name):
    """Full-size workloads in the bench's launch configuration, checked on sampled tokens."""
    w = synth.build(name)
    dev = DeviceStep(w, fill="device")
    dev.step()
    _sync()
    assert int(dev.status.item()) == 0
    out = to_bits(dev.out)
    from oracle import bf16
    assert np.all(np.isfinite(bf16.to_f64(out)))
    toks = _sample_tokens(w, per_chunk=4 if w.B == 0 else 2)
    want = oracle_tokens(w, toks)
    for t in toks:
        assert_attention_close(out[t], want[t], f"{name} token {t}")
    del dev
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ errors ----

def test_host_argument_errors():
    import paged_kv_gqa_row_gb300 as lnk
    w = synth.custom(seed=13, hq=8, hkv=2, head_dim=128, dec_lengths=[100, 200])
    dev = DeviceStep(w, fill="host")
    bad = [
        (lnk.attn_desc(8, 2, 80, w.num_pages, w.num_rows, w.pages_per_row), 4),   # head_dim
        (lnk.attn_desc(8, 3, 128, w.num_pages, w.num_rows, w.pages_per_row), 1),  # hq % hkv
        (lnk.attn_desc(32, 2, 128, w.num_pages, w.num_rows, w.pages_per_row), 4),  # group 16
        (lnk.attn_desc(8, 2, 128, w.num_pages, w.num_rows, w.pages_per_row, page_size=32), 4),
        (lnk.attn_desc(8, 2, 128, 0, w.num_rows, w.pages_per_row), 1),
    ]
    for desc, want in bad:
        with pytest.raises(lnk.LnkError) as e:
            lnk.lnk_paged_decode_attn(desc, dev.q_out, dev.dec_positions, dev.table, dev.k_pool,
                                      dev.v_pool, dev.out, w.B, dev.workspace, dev.ws_bytes)
        assert e.value.status == want
    with pytest.raises(lnk.LnkError) as e:  # workspace too small
        lnk.lnk_paged_decode_attn(dev.desc, dev.q_out, dev.dec_positions, dev.table, dev.k_pool,
                                  dev.v_pool, dev.out, w.B, dev.workspace, 16)
    assert e.value.status == 5
    with pytest.raises(lnk.LnkError) as e:  # B beyond the table's rows
        lnk.lnk_paged_decode_attn(dev.desc, dev.q_out, dev.dec_positions, dev.table, dev.k_pool,
                                  dev.v_pool, dev.out, w.num_rows + 1, dev.workspace, dev.ws_bytes)
    assert e.value.status == 1
    with pytest.raises(lnk.LnkError) as e:  # null pool
        lnk.lnk_paged_append_rope(dev.desc, dev.rope, dev.q, dev.k, dev.v, dev.positions, dev.rows,
                                  None, dev.table, None, None, 1e-6, None, dev.v_pool, dev.q_out, w.T)
    assert e.value.status == 1
    # empty calls enqueue nothing and succeed
    lnk.lnk_paged_append_rope(dev.desc, dev.rope, dev.q, dev.k, dev.v, dev.positions, dev.rows,
                              None, dev.table, None, None, 1e-6, dev.k_pool, dev.v_pool, dev.q_out, 0)
    lnk.lnk_paged_decode_attn(dev.desc, dev.q_out, dev.dec_positions, dev.table, dev.k_pool,
                              dev.v_pool, dev.out, 0, None, 0)
    lnk.lnk_paged_step_attn(dev.desc, dev.q_out, None, None, None, None, dev.table, dev.k_pool,
                            dev.v_pool, dev.out, None, None, 0, 0, 0, None, 0)


def test_device_status_bits():
    import paged_kv_gqa_row_gb300 as lnk
    w = synth.custom(seed=14, hq=8, hkv=2, head_dim=128, dec_lengths=[100, 200, 300],
                     chunks=[(0, 10)])
    dev = DeviceStep(w, fill="host")
    dev.append()
    _sync()
    # a table entry outside the pool on a page row 1 reads
    table = dev.table.clone()
    table[1, 1] = w.num_pages + 7
    dev.status.zero_()
    lnk.lnk_paged_decode_attn(dev.desc, dev.q_out[w.P:], dev.dec_positions, table, dev.k_pool,
                              dev.v_pool, dev.out, w.B, dev.workspace, dev.ws_bytes, dev.status)
    _sync()
    assert int(dev.status.item()) & lnk.binding.DEV_BAD_PAGE
    assert np.all(np.isfinite(torch.from_numpy(to_bits(dev.out).view(np.int16)).view(torch.bfloat16).float().numpy()))
    # a position past the table row
    pos = dev.dec_positions.clone()
    pos[0] = w.pages_per_row * 64
    dev.status.zero_()
    lnk.lnk_paged_decode_attn(dev.desc, dev.q_out[w.P:], pos, dev.table, dev.k_pool, dev.v_pool,
                              dev.out, w.B, dev.workspace, dev.ws_bytes, dev.status)
    _sync()
    assert int(dev.status.item()) & lnk.binding.DEV_BAD_POSITION
    assert not np.any(to_bits(dev.out)[0])
    # append: a bad row and a bad slot
    rows = dev.rows.clone()
    rows[0] = w.num_rows
    dev.status.zero_()
    lnk.lnk_paged_append_rope(dev.desc, dev.rope, dev.q, dev.k, dev.v, dev.positions, rows, None,
                              dev.table, None, None, 1e-6, dev.k_pool, dev.v_pool, dev.q_out, w.T,
                              dev.status)
    slots = torch.full((w.T,), w.num_pages * 64, dtype=torch.int32, device="cuda")
    lnk.lnk_paged_append_rope(dev.desc, dev.rope, dev.q, dev.k, dev.v, dev.positions, dev.rows, slots,
                              dev.table, None, None, 1e-6, dev.k_pool, dev.v_pool, dev.q_out, w.T,
                              dev.status)
    _sync()
    st = int(dev.status.item())
    assert st & lnk.binding.DEV_BAD_ROW and st & lnk.binding.DEV_BAD_SLOT
    # step: equal segments on two rows, and a bad `last`
    seg = torch.zeros(w.P, dtype=torch.int32, device="cuda")
    rows_c = dev.ch_rows.clone()
    rows_c[5:] = 0
    last = torch.tensor([w.P], dtype=torch.int32, device="cuda")
    last_out = torch.zeros((1, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
    dev.status.zero_()
    lnk.lnk_paged_step_attn(dev.desc, dev.q_out, rows_c, dev.ch_positions, seg, dev.dec_positions,
                            dev.table, dev.k_pool, dev.v_pool, dev.out, last, last_out, w.P, w.B, 1,
                            dev.workspace, dev.ws_bytes, dev.status)
    _sync()
    st = int(dev.status.item())
    assert st & lnk.binding.DEV_SEGMENT and st & lnk.binding.DEV_BAD_LAST
    # the context is still healthy
    dev.status.zero_()
    dev.step()
    _sync()
    assert int(dev.status.item()) == 0


def test_synth_device_fill_matches_host():
    from synth import device as sdev
    key = synth.stream_key(77, 3)
    t = torch.empty(1 << 20, dtype=torch.int16, device="cuda")
    sdev.fill_normal_bf16(t, key, start=12345)
    _sync()
    assert np.array_equal(to_bits(t), synth.normal_bf16(key, 12345, 1 << 20))


def test_repeatable():
    w = synth.custom(seed=15, hq=32, hkv=8, head_dim=128, dec_lengths=[5000, 300, 9000])
    dev = DeviceStep(w, fill="host")
    dev.step()
    _sync()
    a = to_bits(dev.out).copy()
    dev.step()
    _sync()
    assert np.array_equal(a, to_bits(dev.out))


def test_decode_rows_over_contiguous_caches():
    """decode_rows (contiguous cache rows of MaxSeq positions) through the paged
    call with an identity table, against the oracle's row-by-row attention."""
    import paged_kv_gqa_row_gb300 as lnk
    from oracle import bf16, paged, rope
    rng = np.random.default_rng(21)
    rows, max_seq, hq, hkv, d = 5, 1024, 8, 2, 128
    pages = max_seq // 64
    ck = bf16.from_f64(rng.standard_normal((rows, hkv, max_seq, d)))
    cv = bf16.from_f64(rng.standard_normal((rows, hkv, max_seq, d)))
    pos = np.array([1023, 0, 64, 500, 63], dtype=np.int32)
    q = bf16.from_f64(rng.standard_normal((rows, hq, d)))
    k = bf16.from_f64(rng.standard_normal((rows, hkv, d)))
    v = bf16.from_f64(rng.standard_normal((rows, hkv, d)))
    pool_k = np.concatenate([ck[b] for b in range(rows)], axis=1)
    pool_v = np.concatenate([cv[b] for b in range(rows)], axis=1)
    table = (np.arange(rows)[:, None] * pages + np.arange(pages)[None, :]).astype(np.int32)
    t16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    t32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    dk, dv = t16(pool_k), t16(pool_v)
    dq, dkk, dvv, dpos, dtab = t16(q), t16(k), t16(v), t32(pos), t32(table)
    q_out = torch.zeros_like(dq)
    out = torch.zeros_like(dq)
    desc = lnk.attn_desc(hq, hkv, d, rows * pages, rows, pages)
    rd = lnk.rope_desc(500000.0)
    ws_bytes = lnk.lnk_paged_workspace_size(desc, rows)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    lnk.lnk_paged_append_rope(desc, rd, dq, dkk, dvv, dpos, None, None, dtab, None, None, 1e-6, dk, dv, q_out, rows)
    lnk.lnk_paged_decode_attn(desc, q_out, dpos, dtab, dk, dv, out, rows, ws, ws_bytes)
    torch.cuda.synchronize()
    inv = rope.inv_freq(500000.0, d)
    ident = np.arange(pages, dtype=np.int32)[None, :]
    got = to_bits(out)
    for b in range(rows):
        qo, ck_b, cv_b = paged.append_rope(q[[b]], k[[b]], v[[b]], pos[[b]], [0], ident, ck[b], cv[b], inv)
        want = paged.attention_at(qo[0], 0, int(pos[b]), ident, ck_b, cv_b, 0)
        assert_attention_close(got[b], want, f"row {b}")


def test_decode_max_rows():
    """The largest decode batch (4096 rows, ragged short lengths): many pairs,
    claimed chunks, the workspace at its largest for the shape; one more row
    is refused."""
    import paged_kv_gqa_row_gb300 as lnk
    lengths = [1 + (97 * i) % 200 for i in range(4096)]
    w = synth.custom(seed=4096, hq=4, hkv=2, head_dim=64, dec_lengths=lengths)
    _check_full(w)
    d = lnk.attn_desc(4, 2, 64, w.num_pages, 4097, w.pages_per_row)
    dev = DeviceStep(w, fill="host")
    with pytest.raises(lnk.LnkError) as e:
        lnk.lnk_paged_decode_attn(d, dev.q_out, dev.dec_positions, dev.table, dev.k_pool, dev.v_pool, dev.out,
                                  4097, dev.workspace, dev.ws_bytes)
    assert e.value.status == 2  # LNK_ERANGE


def test_chunk_many_tiles_keep_token_order():
    """A prompt long enough for more tiles than the kernel orders by cost
    (17000 tokens at G = 8: 532 tiles of 32 tokens), checked on sampled tokens."""
    from harness import oracle_tokens
    w = synth.custom(seed=17000, hq=16, hkv=2, head_dim=64, dec_lengths=[], chunks=[(0, 17000)])
    dev = DeviceStep(w, fill="host")
    dev.step()
    _sync()
    assert int(dev.status.item()) == 0
    out = to_bits(dev.out)
    toks = [0, 31, 32, 8000, 16999]
    want = oracle_tokens(w, toks)
    for t in toks:
        assert_attention_close(out[t], want[t], f"token {t}")
