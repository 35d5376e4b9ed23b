"""lnk_paged_decode_attn_static: decode attention for callers that cannot
allocate device memory when the step runs (a runtime that reserved all device
memory up front, a serving loop with a fixed footprint).  Its scratch is a
static device array inside the library; the call allocates nothing.

This file is collected last so that a run stopping at the first failure has
already run every other test.  It must pass alone in a fresh process too.
"""
import numpy as np
import pytest

import synth
from harness import ATT_MAX_ABS, ATT_MEAN_ABS, DeviceStep, to_bits
from oracle import bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_static_scratch_matches_workspace_entry_point_twice():
    import paged_kv_gqa_row_gb300 as lnk
    # rows long enough that pairs are cut across CTAs (partials and counters in use)
    w = synth.custom(seed=31, hq=32, hkv=8, head_dim=128,
                     dec_lengths=[4000, 300, 9000, 64, 1, 2500, 7000, 130], inactive=(3,))
    dev = DeviceStep(w, fill="host")
    dev.append()
    ref = torch.zeros_like(dev.out)
    lnk.lnk_paged_decode_attn(dev.desc, dev.q_out, dev.dec_positions, dev.table, dev.k_pool, dev.v_pool,
                              ref, w.B, dev.workspace, dev.ws_bytes, dev.status)
    torch.cuda.synchronize()
    want = bf16.to_f64(to_bits(ref))
    for call in range(2):
        out = torch.full_like(dev.out, 0x7FC0)  # NaN everywhere: every output must be written
        lnk.lnk_paged_decode_attn_static(dev.desc, dev.q_out, dev.dec_positions, dev.table, dev.k_pool,
                                         dev.v_pool, out, w.B, dev.status)
        torch.cuda.synchronize()
        got = bf16.to_f64(to_bits(out))
        err = np.abs(got - want)
        assert np.all(np.isfinite(got)), f"call {call}: non-finite output"
        assert err.max() <= ATT_MAX_ABS and err.mean() <= ATT_MEAN_ABS, f"call {call}: {err.max()} {err.mean()}"
    assert int(dev.status.item()) == 0


def test_static_scratch_rejects_sizes_beyond_its_maximum():
    import paged_kv_gqa_row_gb300 as lnk
    desc = lnk.attn_desc(32, 8, 128, num_pages=100, num_rows=4096, pages_per_row=4)
    with pytest.raises(lnk.LnkError) as e:
        lnk.lnk_paged_decode_attn_static(desc, 16, 16, 16, 16, 16, 16, 4096)
    assert e.value.status == 2  # LNK_ERANGE, nothing enqueued
