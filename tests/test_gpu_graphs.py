"""The entry points under CUDA graph capture: a step (append + step_attn with
chunks and decode rows, bf16 pools) and a decode step on 8-bit pools are
captured once, replayed, and replayed again after the inputs were updated in
place; every replay must equal the eager calls on the same inputs bit for bit
(the kernels are deterministic), and the eager results equal the oracle."""
import numpy as np
import pytest

import synth
from harness import DeviceStep, assert_attention_close, oracle_full, to_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _graph_of(fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm-up outside capture (kernel attributes, first launches)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    return g


def test_step_replays_equal_eager_calls():
    w = synth.custom(seed=31, hq=8, hkv=2, head_dim=128, dec_lengths=[700, 65, 1300, 9],
                     chunks=[(0, 70), (130, 40)])
    dev = DeviceStep(w, fill="host")
    k0, v0 = dev.k_pool.clone(), dev.v_pool.clone()

    def eager(q_bits):
        dev.k_pool.copy_(k0)
        dev.v_pool.copy_(v0)
        dev.q.copy_(torch.from_numpy(q_bits.view(np.int16)).cuda())
        dev.step()
        torch.cuda.synchronize()
        return to_bits(dev.out).copy()

    q1 = w.step_q()
    want1 = eager(q1)
    # the eager path is the oracle's
    _, _, _, out_oracle = oracle_full(w)
    for t in range(w.T):
        assert_attention_close(want1[t], out_oracle[t], f"token {t}")
    q2 = synth.tensor_bf16(77, 3, q1.shape)
    want2 = eager(q2)

    dev.k_pool.copy_(k0)
    dev.v_pool.copy_(v0)
    dev.q.copy_(torch.from_numpy(q1.view(np.int16)).cuda())
    graph = _graph_of(dev.step)
    for q_bits, want in ((q1, want1), (q1, want1), (q2, want2)):
        dev.k_pool.copy_(k0)
        dev.v_pool.copy_(v0)
        dev.q.copy_(torch.from_numpy(q_bits.view(np.int16)).cuda())
        dev.out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(to_bits(dev.out), want)
    assert int(dev.status.item()) == 0


def test_e4m3_decode_replays_equal_eager_calls():
    import paged_kv_gqa_row_gb300 as lnk
    from test_gpu_fp8 import F8Step
    w = synth.custom(seed=41, hq=16, hkv=4, head_dim=128, dec_lengths=[900, 17, 256, 4000, 65])
    dev = F8Step(w)
    k0, v0 = dev.k_pool.clone(), dev.v_pool.clone()

    def run():
        dev.append()
        dev.decode()

    run()
    torch.cuda.synchronize()
    want = to_bits(dev.out).copy()
    dev.k_pool.copy_(k0)
    dev.v_pool.copy_(v0)
    graph = _graph_of(run)
    for _ in range(3):
        dev.k_pool.copy_(k0)
        dev.v_pool.copy_(v0)
        dev.out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(to_bits(dev.out), want)
    assert int(dev.status.item()) == 0
    assert dev.desc.kv_dtype == lnk.KV_E4M3


def test_one_kernel_decode_step_replays_equal_eager_calls():
    """The one-kernel decode step (lnk_paged_decode_step on a small launch)
    under capture: replays equal the eager call bit for bit, also after the
    positions were moved on by one in place (read again by every replay)."""
    w = synth.build("phi3_tiny")
    dev = DeviceStep(w, fill="host")
    assert dev.lnk.lnk_paged_decode_step_launches(dev.desc, w.B) == 1
    k0, v0 = dev.k_pool.clone(), dev.v_pool.clone()
    pos1 = dev.positions.clone()
    pos2 = pos1 + 1  # still inside each row's last page or the next one of its table row
    assert int(pos2.max().item()) < w.pages_per_row * 64

    def call():
        dev.lnk.lnk_paged_decode_step(dev.desc, dev.rope, dev.q, dev.k, dev.v, dev.positions, dev.table,
                                      dev.gamma_q, dev.gamma_k, w.norm_eps, dev.k_pool, dev.v_pool, dev.q_out,
                                      dev.out, w.B, dev.workspace, dev.ws_bytes, dev.status)

    def eager(pos):
        dev.k_pool.copy_(k0)
        dev.v_pool.copy_(v0)
        dev.positions.copy_(pos)
        call()
        torch.cuda.synchronize()
        return to_bits(dev.out).copy(), to_bits(dev.k_pool).copy()

    want1, kp1 = eager(pos1)
    _, _, _, out_oracle = oracle_full(w)
    assert_attention_close(want1, out_oracle, "phi3_tiny")
    want2, kp2 = eager(pos2)
    dev.positions.copy_(pos1)
    graph = _graph_of(call)
    for pos, want, kp in ((pos1, want1, kp1), (pos2, want2, kp2), (pos1, want1, kp1)):
        dev.k_pool.copy_(k0)
        dev.v_pool.copy_(v0)
        dev.positions.copy_(pos)
        dev.out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(to_bits(dev.out), want)
        assert np.array_equal(to_bits(dev.k_pool), kp)
    assert int(dev.status.item()) == 0
