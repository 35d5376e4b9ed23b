"""lnk_paged_decode_attn_static: decode attention for callers that cannot
allocate device memory when the step runs (a runtime that reserved all device
memory up front, a serving loop with a fixed footprint).  Its scratch is a
static device array inside the library; the call allocates nothing.

Each call is checked against the oracle on the same inputs and against the
workspace entry point lnk_paged_decode_attn, within the bounds every parity
test uses.  Calls come in a row, so that each finds the array as the previous
call left it: twice with the same rows, then a smaller call with other lengths
after a larger one.

This file is collected last so that a run stopping at the first failure has
already run every other test.  It must pass alone in a fresh process too.
"""
import numpy as np
import pytest

import synth
from harness import ATT_MAX_ABS, ATT_MEAN_ABS, DeviceStep, assert_attention_close, oracle_full, to_bits
from oracle import bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _static_calls(w, calls):
    """Append, then `calls` static decode calls in a row; each output is checked
    against the oracle and against the workspace entry point's output."""
    import paged_kv_gqa_row_gb300 as lnk
    dev = DeviceStep(w, fill="host")
    dev.append()
    ref = torch.zeros_like(dev.out)
    lnk.lnk_paged_decode_attn(dev.desc, dev.q_out, dev.dec_positions, dev.table, dev.k_pool, dev.v_pool,
                              ref, w.B, dev.workspace, dev.ws_bytes, dev.status)
    torch.cuda.synchronize()
    _, _, _, oracle_out = oracle_full(w)
    want = bf16.to_f64(to_bits(ref))
    for call in range(calls):
        out = torch.full_like(dev.out, 0x7FC0)  # NaN everywhere: every output must be written
        lnk.lnk_paged_decode_attn_static(dev.desc, dev.q_out, dev.dec_positions, dev.table, dev.k_pool,
                                         dev.v_pool, out, w.B, dev.status)
        torch.cuda.synchronize()
        got_bits = to_bits(out)
        assert_attention_close(got_bits, oracle_out, f"call {call} vs oracle")
        err = np.abs(bf16.to_f64(got_bits) - want)
        assert err.max() <= ATT_MAX_ABS and err.mean() <= ATT_MEAN_ABS, f"call {call}: {err.max()} {err.mean()}"
    assert int(dev.status.item()) == 0


def test_static_scratch_matches_oracle_and_workspace_entry_point_twice():
    # rows long enough that pairs are cut across CTAs (partials and counters in use)
    w = synth.custom(seed=31, hq=32, hkv=8, head_dim=128,
                     dec_lengths=[4000, 300, 9000, 64, 1, 2500, 7000, 130], inactive=(3,))
    _static_calls(w, 2)


def test_static_scratch_smaller_call_after_larger_one():
    # a call over many rows (many pairs: claimed chunks, the two-CTAs-per-SM
    # form), then one over fewer rows with other lengths on the same array
    big = synth.custom(seed=32, hq=32, hkv=8, head_dim=128, dec_lengths=[1 + (37 * i) % 900 for i in range(160)])
    _static_calls(big, 1)
    small = synth.custom(seed=33, hq=32, hkv=8, head_dim=128, dec_lengths=[6000, 17, 3000])
    _static_calls(small, 1)


def test_static_scratch_rejects_sizes_beyond_its_maximum():
    import paged_kv_gqa_row_gb300 as lnk
    desc = lnk.attn_desc(32, 8, 128, num_pages=100, num_rows=4096, pages_per_row=4)
    with pytest.raises(lnk.LnkError) as e:
        lnk.lnk_paged_decode_attn_static(desc, 16, 16, 16, 16, 16, 16, 4096)
    assert e.value.status == 2  # LNK_ERANGE, nothing enqueued
