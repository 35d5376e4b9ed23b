"""lnk_paged_decode_step (append, then attention, one kernel for small
launches) through the C ABI against the CPU oracle on the same seeded inputs.

The one-kernel form must write exactly what lnk_paged_append_rope writes
(q_out and the pools, bit for bit: both use the same float-pair rotation) and
attend like lnk_paged_decode_attn, for every kind of decode row: windows,
inactive rows, QK-norm, head_dim 64 / 96 / 128, 8-bit pools.
"""
import zlib

import numpy as np
import pytest

import synth
from harness import (DeviceStep, assert_attention_close, assert_ulp_close, oracle_full, oracle_inv,
                     to_bits)
from oracle import paged as opaged

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FUSE_MAX_PAGES = 16  # the library's bound on a pair's pages for the one-kernel form


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _grid(kv8=False):
    return _sms() * (2 if kv8 else 1)


def _one_kernel(w, grid):
    """Whether the call takes the one-kernel form (the library's rule, restated)."""
    pairs = w.B * w.hkv
    pages = w.pages_per_row
    if w.window > 0:
        pages = min(pages, (w.window - 1) // 64 + 2)
    return pairs <= grid and 2 * pairs >= _sms() and pages <= FUSE_MAX_PAGES


def _decode_step(dev, stream=None):
    w = dev.w
    dev.lnk.lnk_paged_decode_step(dev.desc, dev.rope, dev.q, dev.k, dev.v, dev.positions, dev.table,
                                  dev.gamma_q, dev.gamma_k, w.norm_eps, dev.k_pool, dev.v_pool, dev.q_out,
                                  dev.out, w.B, dev.workspace, dev.ws_bytes, dev.status, stream)


def _rows_for(pairs_target, hkv):
    return max(1, pairs_target // hkv)


def _case_workload(name, hq, hkv, d, lengths, window, inactive, qk_norm):
    return synth.custom(seed=zlib.crc32(("step" + name).encode()) % 10000, hq=hq, hkv=hkv, head_dim=d,
                        dec_lengths=lengths, window=window, inactive=inactive, qk_norm=qk_norm)


def _lengths(n, lo, hi, salt):
    return [lo + (salt * 7919 + 104729 * i) % (hi - lo + 1) for i in range(n)]


# id, hq, hkv, D, rows as a fraction of the grid's pairs, length range, window, inactive rows, QK-norm
STEP_CASES = [
    ("mha96-phi3-shape", 32, 32, 96, 0.84, (1, 300), 0, (), False),
    ("gqa4-128", 32, 8, 128, 0.6, (1, 1000), 0, (), False),
    ("gqa4-window200", 32, 8, 128, 0.9, (100, 3000), 200, (), False),
    ("mha64-inactive", 16, 16, 64, 0.7, (1, 600), 0, (1, 4), False),
    ("gqa4-qknorm", 32, 8, 128, 0.55, (1, 900), 0, (), True),
    ("gqa8-96-window1", 16, 2, 96, 0.8, (1, 500), 1, (0,), False),
]


def _build_case(case, grid):
    name, hq, hkv, d, frac, (lo, hi), window, inactive, qkn = case
    rows = _rows_for(int(frac * grid), hkv)
    lengths = _lengths(rows, lo, hi, zlib.crc32(name.encode()) % 97)
    return _case_workload(name, hq, hkv, d, lengths, window, tuple(r for r in inactive if r < rows), qkn)


def _check_against_two_calls_and_oracle(w, launches):
    one = DeviceStep(w, fill="host")
    two = DeviceStep(w, fill="host")
    assert one.lnk.lnk_paged_decode_step_launches(one.desc, w.B) == launches
    _decode_step(one)
    two.step()
    torch.cuda.synchronize()
    # the append's results: identical to the two-call path, and to the oracle
    assert np.array_equal(to_bits(one.q_out), to_bits(two.q_out)), "q_out differs from lnk_paged_append_rope"
    assert np.array_equal(to_bits(one.k_pool), to_bits(two.k_pool)), "k_pool differs from lnk_paged_append_rope"
    assert np.array_equal(to_bits(one.v_pool), to_bits(two.v_pool)), "v_pool differs from lnk_paged_append_rope"
    q_want, kp_want, vp_want, out_want = oracle_full(w)
    assert_ulp_close(to_bits(one.q_out), q_want, "q_out")
    assert_ulp_close(to_bits(one.k_pool), kp_want, "k_pool")
    assert np.array_equal(to_bits(one.v_pool), vp_want), "v_pool"
    assert_attention_close(to_bits(one.out), out_want, w.name)
    assert int(one.status.item()) == 0


@pytest.mark.parametrize("case", STEP_CASES, ids=[c[0] for c in STEP_CASES])
def test_decode_step_one_kernel_matches_oracle(case):
    w = _build_case(case, _grid())
    assert _one_kernel(w, _grid()), "case outside the one-kernel form"
    _check_against_two_calls_and_oracle(w, 1)


@pytest.mark.parametrize("rows,lengths", [(2, [5, 4000]), (600, None)], ids=["few-pairs", "many-pairs"])
def test_decode_step_two_kernel_form_matches_oracle(rows, lengths):
    """Launches outside the one-kernel form (too few or too many pairs) run the
    append and the attention kernels; the results are the same."""
    lengths = lengths or _lengths(rows, 1, 400, 3)
    w = _case_workload(f"two-{rows}", 32, 8, 128, lengths, 0, (), False)
    assert not _one_kernel(w, _grid())
    _check_against_two_calls_and_oracle(w, 2)


def test_decode_step_phi3_tiny_workload():
    w = synth.build("phi3_tiny")
    assert _one_kernel(w, _grid())
    _check_against_two_calls_and_oracle(w, 1)


def test_decode_step_nan_tails_never_leak():
    """NaN in every slot after each row's position in its last page (never
    visible): the one-kernel form must mask them like the attention kernel."""
    grid = _grid()
    rows = _rows_for(int(0.8 * grid), 8)
    w = _case_workload("nan-tails", 32, 8, 128, _lengths(rows, 1, 700, 11), 0, (), False)
    assert _one_kernel(w, grid)
    dev = DeviceStep(w, fill="host")
    mask = np.zeros(w.pool_positions, dtype=bool)
    for p, r in zip(w.token_positions(), w.token_rows()):
        if p >= 0:
            pg = int(w.table[r, p // 64])
            mask[pg * 64 + p % 64 + 1: pg * 64 + 64] = True
    for p, r in zip(w.token_positions(), w.token_rows()):
        if p >= 0:
            mask[int(w.table[r, p // 64]) * 64 + p % 64] = False
    idx = torch.from_numpy(np.nonzero(mask)[0]).cuda()
    dev.k_pool[:, idx, :] = torch.tensor(0x7FC0, dtype=torch.int16, device="cuda")
    dev.v_pool[:, idx, :] = torch.tensor(0x7FC0, dtype=torch.int16, device="cuda")
    _decode_step(dev)
    torch.cuda.synchronize()
    _, _, _, out_want = oracle_full(w)
    assert_attention_close(to_bits(dev.out), out_want, "nan tails")
    assert int(dev.status.item()) == 0


def test_decode_step_two_steps_in_a_row():
    """Two one-kernel steps back to back on one stream: the second step's
    attention reads the key and value the first step wrote (its position is
    the next one in the same page), through the pool, after the first step's
    kernel has finished."""
    grid = _grid()
    rows = _rows_for(int(0.75 * grid), 8)
    lengths = [1 + ((37 * i) % 60) + 64 * (i % 9) for i in range(rows)]  # never the last slot of a page
    w1 = _case_workload("two-steps", 32, 8, 128, lengths, 0, (), False)
    w2 = _case_workload("two-steps", 32, 8, 128, [n + 1 for n in lengths], 0, (), False)
    assert np.array_equal(w1.table, w2.table)
    assert _one_kernel(w1, grid) and _one_kernel(w2, grid)
    dev = DeviceStep(w1, fill="host")
    pos2 = torch.from_numpy(w2.token_positions().astype(np.int32)).cuda()
    out1, out2 = dev.out, torch.zeros_like(dev.out)
    torch.cuda.synchronize()
    _decode_step(dev)  # nothing else on the stream between the two steps
    dev.positions, dev.out = pos2, out2
    _decode_step(dev)
    torch.cuda.synchronize()
    inv = oracle_inv(w1)
    rows_idx = w1.token_rows()
    q1, kp, vp = opaged.append_rope(w1.step_q(), w1.step_k(), w1.step_v(), w1.token_positions(), rows_idx,
                                    w1.table, w1.pool("k"), w1.pool("v"), inv)
    out1_want = opaged.decode_attention(q1, w1.token_positions(), w1.table, kp, vp, 0)
    q2, kp, vp = opaged.append_rope(w2.step_q(), w2.step_k(), w2.step_v(), w2.token_positions(), rows_idx,
                                    w1.table, kp, vp, inv)
    out2_want = opaged.decode_attention(q2, w2.token_positions(), w1.table, kp, vp, 0)
    assert_attention_close(to_bits(out1), out1_want, "step 1")
    assert_ulp_close(to_bits(dev.q_out), q2, "step 2 q_out")
    assert_ulp_close(to_bits(dev.k_pool), kp, "k_pool after two steps")
    assert np.array_equal(to_bits(dev.v_pool), vp), "v_pool after two steps"
    assert_attention_close(to_bits(dev.out), out2_want, "step 2")
    assert int(dev.status.item()) == 0


def test_decode_step_e4m3_pools():
    from test_gpu_fp8 import F8Step, _oracle_full
    rows = _rows_for(int(0.84 * _sms()), 32)  # the Phi-3 tiny shape: 4 rows x 32 kv heads on 152 SMs
    w = _case_workload("e4m3", 32, 32, 96, _lengths(rows, 1, 300, 5), 0, (), False)
    one, two = F8Step(w), F8Step(w)
    assert one.lnk.lnk_paged_decode_step_launches(one.desc, w.B) == 1
    one.lnk.lnk_paged_decode_step(one.desc, one.rope, one.q, one.k, one.v, one.positions, one.table, None, None,
                                  w.norm_eps, one.k_pool, one.v_pool, one.q_out, one.out, w.B, one.ws,
                                  one.ws_bytes, one.status)
    two.append()
    two.decode()
    torch.cuda.synchronize()
    assert np.array_equal(to_bits(one.q_out), to_bits(two.q_out))
    assert np.array_equal(one.k_pool.cpu().numpy(), two.k_pool.cpu().numpy())
    assert np.array_equal(one.v_pool.cpu().numpy(), two.v_pool.cpu().numpy())
    q_want, kc, vc, out_want = _oracle_full(w)
    assert np.array_equal(one.k_pool.cpu().numpy().astype(np.uint8), kc)
    got = to_bits(one.out)
    for b in range(w.B):
        assert_attention_close(got[b], out_want[b], f"e4m3 row {b}")
    assert int(one.status.item()) == 0


def test_decode_step_argument_errors_enqueue_nothing():
    import paged_kv_gqa_row_gb300 as lnk
    w = synth.build("phi3_tiny")
    dev = DeviceStep(w, fill="host")
    k0 = to_bits(dev.k_pool).copy()
    with pytest.raises(lnk.LnkError):  # workspace too small: nothing may have been appended
        dev.lnk.lnk_paged_decode_step(dev.desc, dev.rope, dev.q, dev.k, dev.v, dev.positions, dev.table, None,
                                      None, w.norm_eps, dev.k_pool, dev.v_pool, dev.q_out, dev.out, w.B,
                                      dev.workspace, 16, dev.status)
    with pytest.raises(lnk.LnkError):  # misaligned q_out
        dev.lnk.lnk_paged_decode_step(dev.desc, dev.rope, dev.q, dev.k, dev.v, dev.positions, dev.table, None,
                                      None, w.norm_eps, dev.k_pool, dev.v_pool, dev.q_out.view(-1)[1:], dev.out,
                                      w.B, dev.workspace, dev.ws_bytes, dev.status)
    torch.cuda.synchronize()
    assert np.array_equal(to_bits(dev.k_pool), k0)


def test_decode_step_one_kernel_bad_data_is_flagged():
    """Bad table data in the one-kernel form: the affected row skips its work
    and a status bit is set; the other rows are unaffected and the context
    stays healthy."""
    import paged_kv_gqa_row_gb300 as lnk
    grid = _grid()
    rows = _rows_for(int(0.8 * grid), 8)
    w = _case_workload("bad-data", 32, 8, 128, _lengths(rows, 70, 700, 17), 0, (), False)
    assert _one_kernel(w, grid)
    _, _, _, out_want = oracle_full(w)
    # the page that holds row 1's new token: outside the pool
    dev = DeviceStep(w, fill="host")
    p1 = int(w.token_positions()[1])
    dev.table[1, p1 // 64] = w.num_pages + 5
    _decode_step(dev)
    torch.cuda.synchronize()
    assert int(dev.status.item()) & lnk.binding.DEV_BAD_PAGE
    got = to_bits(dev.out)
    assert np.all(np.isfinite(torch.from_numpy(got.view(np.int16)).view(torch.bfloat16).float().numpy()))
    others = [b for b in range(w.B) if b != 1]
    assert_attention_close(got[others], out_want[others], "rows with valid pages")
    # a position past the table row: that row's output is zero
    dev = DeviceStep(w, fill="host")
    pos = dev.positions.clone()
    pos[0] = w.pages_per_row * 64
    dev.positions = pos
    _decode_step(dev)
    torch.cuda.synchronize()
    assert int(dev.status.item()) & lnk.binding.DEV_BAD_POSITION
    assert not np.any(to_bits(dev.out)[0])
    assert_attention_close(to_bits(dev.out)[1:], out_want[1:], "rows after the bad one")
    # the context is still healthy
    _check_against_two_calls_and_oracle(w, 1)
