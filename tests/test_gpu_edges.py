"""Softmax edge cases, through the C ABI, against the oracle on the same inputs.

* Peaked scores: queries scaled by 16 and 32 (a power of two, so the inputs
  stay exact bf16 values), so that one or a few keys carry almost all the
  weight and the running maximum moves by many units of log2 from page to page.
* A running maximum that jumps by far more than 2^8 (log2 units) on a later
  page: the keys of every page but a row's first two are scaled by 8 and the
  queries by 16.  This drives the chunk kernel's deferred rescale of O.
* Explicit attention scales (``lnk_attn_desc.scale``) of 0.05 and 0.3 instead of
  the default rsqrt(head_dim) ("Phi-3 Mini 4K Instruct -- files",
  src/attention.linnet, the scale of ``attention_rows``).
* Values with Gaussian tails (Box-Muller on the host, |x| up to about 8.6)
  instead of the bounded Irwin-Hall values, on a Mistral-shaped workload.
* A QK-norm gamma of 2 on the first half of head_dim and 0.5 on the second: the
  append must normalise before it rotates ("Qwen3-4B", model description).

The error bounds are the ones every parity test uses: max |err| <= 2e-2 and
mean |err| <= 2e-3 for attention outputs; stored K and q_out within one bf16
ulp, V bit-exact.
"""
import zlib

import numpy as np
import pytest

import synth
from harness import (DeviceStep, assert_attention_close, assert_ulp_close, oracle_full, to_bits)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _run(w, scale=0.0):
    dev = DeviceStep(w, fill="host", scale=scale)
    dev.step()
    torch.cuda.synchronize()
    q_want, kp_want, vp_want, out_want = oracle_full(w, scale if scale > 0 else None)
    assert_ulp_close(to_bits(dev.q_out), q_want, "q_out")
    assert_ulp_close(to_bits(dev.k_pool), kp_want, "k_pool")
    assert np.array_equal(to_bits(dev.v_pool), vp_want), "v_pool"
    mx, mean = assert_attention_close(to_bits(dev.out), out_want, w.name)
    assert int(dev.status.item()) == 0
    return mx, mean


def _custom(name, hq, hkv, d, lengths, chunks, window, **kw):
    w = synth.custom(seed=zlib.crc32(name.encode()) % 10000, hq=hq, hkv=hkv, head_dim=d, dec_lengths=lengths,
                     chunks=chunks, window=window)
    for k, v in kw.items():
        setattr(w, k, v)
    return w


CASES = [
    # id, hq, hkv, D, decode lengths, chunks (offset, tokens), window
    ("decode-gqa4-ragged", 8, 2, 128, [1000, 5, 64, 128, 2000, 777], [], 0),
    ("decode-mha64-edges", 4, 4, 64, [1, 2, 63, 64, 65, 130], [], 0),
    ("decode-window2047-gqa2", 8, 4, 96, [300, 2047, 2048, 2049, 2100, 5000], [], 2047),
    ("decode-many-pairs", 32, 8, 128, [1 + (37 * i) % 700 for i in range(80)], [], 0),
    ("step-gqa4", 8, 2, 128, [300, 1200], [(0, 70), (100, 5), (1000, 130)], 0),
    ("step-window-gqa2", 8, 4, 96, [3000], [(2500, 300), (0, 40)], 2047),
    ("prefill-gqa8", 16, 2, 128, [], [(0, 300), (4000, 200)], 0),
]


@pytest.mark.parametrize("q_scale", [16.0, 32.0], ids=["q16", "q32"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_peaked_scores(case, q_scale):
    w = _custom(*case, q_scale=q_scale)
    _run(w)


@pytest.mark.parametrize("scale", [0.05, 0.3])
@pytest.mark.parametrize("case", [CASES[0], CASES[2], CASES[4], CASES[6]], ids=lambda c: c[0])
def test_explicit_scale(case, scale):
    w = _custom(*case)
    _run(w, scale=scale)


def _jump_workload(name, hq, hkv, d, lengths, chunks, window):
    """Prefilled keys on every logical page from the third on scaled by 8,
    queries by 16.  (A chunk's own keys are the step's keys, written over the
    pool, so the chunks start past the second page: their rows' earlier
    context carries the jump.)"""
    w = _custom(name, hq, hkv, d, lengths, chunks, window, q_scale=16.0)
    scaled = {}
    for r in range(w.num_rows):
        for j in range(2, w.pages_per_row):
            if w.table[r, j] >= 0:
                scaled[int(w.table[r, j])] = 8.0
    w.k_page_scale = scaled
    return w


JUMP_CASES = [
    ("jump-prefill-gqa4", 8, 2, 128, [], [(700, 300), (200, 100)], 0),
    ("jump-step-gqa8", 16, 2, 128, [2000, 700], [(1000, 300)], 0),
    ("jump-step-window-mha96", 8, 8, 96, [3000], [(2100, 130)], 2047),
]


@pytest.mark.parametrize("case", JUMP_CASES, ids=[c[0] for c in JUMP_CASES])
def test_running_max_jumps_past_rescale_threshold(case):
    w = _jump_workload(*case)
    # the inputs do what the case is for: for the chunk tokens past the second
    # page, the largest score of a later page exceeds the largest of the first
    # page by more than 2^8 in log2 units (here the score is q.k / sqrt(D))
    from oracle import bf16
    kp = bf16.to_f64(w.pool("k"))
    q = bf16.to_f64(w.step_q())
    c = 1.0 / np.sqrt(w.head_dim) / np.log(2.0)
    t = int(np.nonzero(w.ch_positions >= 3 * 64)[0][0])
    row = int(w.ch_rows[t])
    first = kp[:, int(w.table[row, 0]) * 64:(int(w.table[row, 0]) + 1) * 64]
    later = kp[:, int(w.table[row, 2]) * 64:(int(w.table[row, 2]) + 1) * 64]
    g = w.hq // w.hkv
    qh = q[t].reshape(w.hkv, g, w.head_dim)
    s_first = np.einsum("hgd,hkd->hgk", qh, first).max() * c
    s_later = np.einsum("hgd,hkd->hgk", qh, later).max() * c
    assert s_later - s_first > 256.0, (s_first, s_later)
    _run(w)


@pytest.mark.parametrize("q_scale", [1.0, 16.0], ids=["q1", "q16"])
def test_gaussian_tails_mistral_shaped(q_scale):
    w = synth.build("mistral", scale=0.06, rows=12)
    w.dist = "gauss"
    w.q_scale = q_scale
    if q_scale == 1.0:
        # the pool does have tails beyond the Irwin-Hall bound 2 sqrt(3)
        from oracle import bf16
        assert np.abs(bf16.to_f64(w.pool("k"))).max() > 4.5
    _run(w)


def test_qknorm_gamma_halves_differ():
    w = synth.custom(seed=71, hq=32, hkv=8, head_dim=128, dec_lengths=[1, 64, 65, 900, 5000, 20000],
                     theta=1e6, qk_norm=True, chunks=[(100, 70)])
    w.gamma_halves = (2.0, 0.5)
    _run(w)
