"""Test harness: runs a synthetic workload through the C ABI and through the
CPU oracle on the same seeded inputs, and compares.

The CUDA side only ever sees device buffers filled from the generator; the
oracle side regenerates the same values on the host.  No expected value comes
from the CUDA path.
"""
from __future__ import annotations

import numpy as np

import synth
from oracle import bf16 as obf16
from oracle import paged as opaged
from oracle import rope as orope

# Tolerances: stored K and q_out within one bf16 unit in the last place
# (the append kernel rounds a double-precision result once, so in practice
# they are identical); attention outputs within the absolute error bounds
# stated for unit-scale inputs.
ATT_MAX_ABS = 2e-2
ATT_MEAN_ABS = 2e-3
KQ_MAX_ULP = 1


def _t(np_bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(np_bits).view(np.int16)).to(device)


def _i32(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def to_bits(t) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint16)


class DeviceStep:
    """Device buffers of one workload step and the library calls on them."""

    def __init__(self, w: synth.Workload, fill: str = "auto", device="cuda", scale: float = 0.0):
        import torch
        import paged_kv_gqa_row_gb300 as lnk
        self.w, self.lnk = w, lnk
        shape = (w.hkv, w.pool_positions, w.head_dim)
        n_pool = int(np.prod(shape))
        if fill == "auto":
            fill = "host" if (n_pool <= (1 << 26) or not w.device_fillable) else "device"
        if fill == "device" and not w.device_fillable:
            raise ValueError("this workload's pool can only be filled on the host")
        if fill == "host":
            self.k_pool = _t(w.pool("k"), device)
            self.v_pool = _t(w.pool("v"), device)
        else:
            from synth import device as sdev
            self.k_pool = torch.empty(shape, dtype=torch.int16, device=device)
            self.v_pool = torch.empty(shape, dtype=torch.int16, device=device)
            sdev.fill_normal_bf16(self.k_pool, w.pool_key("k"))
            sdev.fill_normal_bf16(self.v_pool, w.pool_key("v"))
        self.q = _t(w.step_q(), device)
        self.k = _t(w.step_k(), device)
        self.v = _t(w.step_v(), device)
        self.positions = _i32(w.token_positions(), device)
        self.rows = _i32(w.token_rows(), device)
        self.table = _i32(w.table, device)
        gq, gk = w.gamma_q(), w.gamma_k()
        self.gamma_q = None if gq is None else _t(gq, device)
        self.gamma_k = None if gk is None else _t(gk, device)
        self.q_out = torch.zeros((w.T, w.hq, w.head_dim), dtype=torch.int16, device=device)
        self.out = torch.zeros((w.T, w.hq, w.head_dim), dtype=torch.int16, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.desc = lnk.attn_desc(w.hq, w.hkv, w.head_dim, w.num_pages, w.num_rows,
                                  w.pages_per_row, window=w.window, scale=scale)
        self.rope = lnk.rope_desc(w.theta, w.llama3)
        self.ws_bytes = max(lnk.lnk_paged_workspace_size(self.desc, max(w.B, 1)), 256)
        self.workspace = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)
        self.dec_positions = _i32(w.dec_positions, device)
        if w.P:
            self.ch_rows = _i32(w.ch_rows, device)
            self.ch_positions = _i32(w.ch_positions, device)
            self.ch_segments = _i32(w.ch_segments, device)

    def append(self, stream=None, slots=None):
        w = self.w
        self.lnk.lnk_paged_append_rope(self.desc, self.rope, self.q, self.k, self.v, self.positions,
                                       self.rows, slots, self.table, self.gamma_q, self.gamma_k,
                                       w.norm_eps, self.k_pool, self.v_pool, self.q_out, w.T,
                                       self.status, stream)

    def attend(self, stream=None, last=None, last_out=None):
        w = self.w
        if w.P == 0:
            self.lnk.lnk_paged_decode_attn(self.desc, self.q_out, self.dec_positions, self.table,
                                           self.k_pool, self.v_pool, self.out, w.B, self.workspace,
                                           self.ws_bytes, self.status, stream)
        else:
            M = 0 if last is None else int(last.shape[0])
            self.lnk.lnk_paged_step_attn(self.desc, self.q_out, self.ch_rows, self.ch_positions,
                                         self.ch_segments, self.dec_positions, self.table,
                                         self.k_pool, self.v_pool, self.out, last, last_out,
                                         w.P, w.B, M, self.workspace, self.ws_bytes, self.status,
                                         stream)

    def step(self, stream=None):
        self.append(stream)
        self.attend(stream)


# ----------------------------------------------------------------- oracle ----

def oracle_inv(w: synth.Workload) -> np.ndarray:
    return orope.inv_freq(w.theta, w.head_dim, w.llama3)


def oracle_full(w: synth.Workload, scale=None):
    """Whole-pool oracle (small workloads): (q_out, k_pool, v_pool, out).
    ``scale``: the attention scale (None: the default rsqrt(head_dim))."""
    q_out, kp, vp = opaged.append_rope(w.step_q(), w.step_k(), w.step_v(), w.token_positions(),
                                       w.token_rows(), w.table, w.pool("k"), w.pool("v"),
                                       oracle_inv(w), gamma_q=w.gamma_q(), gamma_k=w.gamma_k(),
                                       eps=w.norm_eps)
    out = opaged.step_attention(q_out, w.ch_rows, w.ch_positions, w.dec_positions, w.table, kp, vp,
                                w.window, scale)
    return q_out, kp, vp, out


def oracle_tokens(w: synth.Workload, tokens, scale=None) -> dict:
    """Oracle outputs of selected step tokens (index into the P + B tokens),
    computed on a compact pool holding only the pages those tokens read."""
    tp, tr = w.token_positions(), w.token_rows()
    q_all, k_all, v_all = w.step_q(), w.step_k(), w.step_v()
    results = {}
    inv = oracle_inv(w)
    for t in tokens:
        p, row = int(tp[t]), int(tr[t])
        if p < 0:
            results[t] = np.zeros((w.hq, w.head_dim))
            continue
        lo, hi = opaged.visible_range(p, w.window)
        lps = np.arange(lo // 64, hi // 64 + 1)
        pages = w.table[row, lps]
        index = {int(pg): i for i, pg in enumerate(pages)}
        kp = np.stack([w.pool_pages("k", h, pages).reshape(-1, w.head_dim) for h in range(w.hkv)])
        vp = np.stack([w.pool_pages("v", h, pages).reshape(-1, w.head_dim) for h in range(w.hkv)])
        # step tokens whose slot lands in these pages (their appended k/v)
        writers, slots = [], []
        for u in range(w.T):
            pu = int(tp[u])
            if pu < 0:
                continue
            pg = int(w.table[int(tr[u]), pu // 64])
            if pg in index:
                writers.append(u)
                slots.append(index[pg] * 64 + pu % 64)
        assert t in writers  # a token's own slot is in the last page it reads
        wi = np.array(writers)
        q_out, kp2, vp2 = opaged.append_rope(q_all[wi], k_all[wi], v_all[wi], tp[wi], tr[wi], None,
                                             kp, vp, inv, slots=np.array(slots),
                                             gamma_q=w.gamma_q(), gamma_k=w.gamma_k(), eps=w.norm_eps)
        ctable = np.full((1, lps[-1] + 1), -1, dtype=np.int32)
        ctable[0, lps] = np.arange(len(lps), dtype=np.int32)
        q_t = q_out[writers.index(t)]
        results[t] = opaged.attention_at(q_t, 0, p, ctable, kp2, vp2, w.window, scale)
    return results


# ------------------------------------------------------------- comparison ----

def attention_errors(got_bits: np.ndarray, want: np.ndarray):
    got = obf16.to_f64(got_bits)
    err = np.abs(got - want)
    return float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0


def assert_attention_close(got_bits, want, what=""):
    mx, mean = attention_errors(got_bits, want)
    assert np.all(np.isfinite(obf16.to_f64(got_bits))), f"{what}: non-finite output"
    assert mx <= ATT_MAX_ABS and mean <= ATT_MEAN_ABS, f"{what}: max {mx:.3g} mean {mean:.3g}"
    return mx, mean


def assert_ulp_close(got_bits, want_bits, what=""):
    """Within one bf16 ulp everywhere, and bit-identical except in at most one
    element per million (the append kernel rounds a result accurate to about
    2^-46 once, so a difference needs the exact value within that of a tie)."""
    d = obf16.ulp_distance(got_bits, want_bits)
    assert d.max(initial=0) <= KQ_MAX_ULP, f"{what}: {int(d.max())} ulp"
    n = int(np.count_nonzero(d))
    assert n <= max(1, d.size // 1_000_000), f"{what}: {n} of {d.size} elements differ"
    return n
