"""The bounded-wait path of the kernels, run on purpose without a fault.

lnk_selftest_wait_timeout launches one CTA whose two warps wait on pipeline
barriers that nothing arrives at, through the same wait routine the attention
kernels use.  The first warp gives up after a short limit; the second, whose
own limit is the kernels' two seconds, must stop through the CTA's abort flag.
The call must report LNK_DEV_TIMEOUT in the device status and take far less
than two seconds, and the context must stay usable: a decode step right
after it still matches the oracle.
"""
import time

import pytest

import synth
from harness import DeviceStep, assert_attention_close, oracle_full, to_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_wait_gives_up_reports_timeout_and_context_stays_usable():
    import paged_kv_gqa_row_gb300 as lnk
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    lnk.lnk_selftest_wait_timeout(status, 20_000_000)  # 20 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == lnk.DEV_TIMEOUT
    # the second warp left through the abort flag, not its own 2 s limit
    assert elapsed < 1.0, elapsed

    w = synth.custom(seed=5, hq=8, hkv=2, head_dim=128, dec_lengths=[300, 70])
    dev = DeviceStep(w, fill="host")
    dev.step()
    torch.cuda.synchronize()
    _, _, _, want = oracle_full(w)
    got = to_bits(dev.out)
    for t in range(w.T):
        assert_attention_close(got[t], want[t], f"token {t}")
    assert int(dev.status.item()) == 0
