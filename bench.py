"""Benchmark of the paged decode / step attention path on one or more GPUs.

Default workload: one Llama-3.1-8B-shaped step_paged layer, the largest
single-GPU configuration: 128 decode rows of context lengths uniform in
[1024, 131072] plus 4 packed prompt chunks of 512 tokens at offsets uniform in
[0, 16384], 32 q / 8 kv heads, head_dim 128, llama3 RoPE, pages of 64 shuffled
in a ~36 GB pool, bf16 synthetic data.  A step is one pass of the whole path:
append_rope over the step's tokens, then step_attn (chunks and decode rows), or
decode_attn for the decode-only workloads.

Metric: achieved HBM GB/s = algorithmic bytes of a step (the visible K/V
bytes, each page counted once, plus q in, q/k/v append traffic, outputs and
page-table entries) / step time; row-steps/s alongside.  The roofline object
covers the decode kernel (HBM); for steps with prompt chunks it also carries
the chunk kernel's tensor-core figure (TFLOP/s against the sustained bf16
peak).  With the default workload the same line also reports the
Mistral-7B-shaped decode step (64 rows, lengths U[512, 8192]), run in the same
process, under "mistral".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl lnk|reference]

With N > 1 (torchrun, one rank per GPU) every rank runs its own batch of
rows (weak scaling: rows are independent, no exchange in the path); the
timed region is bracketed by barriers and the max over ranks is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

CONFIGS = {
    "mistral": "Mistral-7B-v0.3-shaped layer, 64 decode rows, lengths U[512,8192]",
    "phi3_tiny": "Phi-3-mini-shaped tiny layer, 4 rows, MHA 32/32, head_dim 96",
    "phi3_window": "Phi-3-mini sliding-window layer, 32 rows, window 2047",
    "qwen3": "Qwen3-4B-shaped layer, 256 rows, QK-norm, shared prefix pages",
    "llama_step": "Llama-3.1-8B-shaped step_paged layer, 4x512 chunk tokens + 128 decode rows",
    "llama_prefill": "Llama-3.1-8B-shaped prefill_paged layer, 4x1024 chunk tokens at offsets U[0,16384]",
}
METRIC = "paged decode attention: achieved HBM GB/s (% of peak) and row-steps/sec per layer"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1700.0


L2_FALLBACK = 129 * 1024 * 1024  # GB300 L2, when the device does not report it
POOL_COPY_LIMIT = 8 << 30         # pools of this size and more are read whole each step (one copy)


def pool_copies(pool_bytes: int, read_per_step: int, l2_bytes: int, requested: int = 0) -> int:
    """Pool copies alternated step to step, so that a copy comes back only after
    the steps in between have read more than twice the L2 (at most
    POOL_COPY_LIMIT of pools in all)."""
    if requested:
        return requested
    if pool_bytes >= POOL_COPY_LIMIT:
        return 1
    need = 1 + -(-2 * l2_bytes // max(1, read_per_step))
    return max(2, min(need, POOL_COPY_LIMIT // pool_bytes))


def algorithmic_bytes(w, kv_bytes: int = 2) -> dict:
    """Bytes a step must move at least once, by part (kv_bytes: bytes per pool
    element, 2 for bf16 pools, 1 for 8-bit pools)."""
    d, hq, hkv = w.head_dim, w.hq, w.hkv
    # decode rows: visible K/V keys, a page shared by several rows counted once
    # (the covered in-page range of a shared page is the union of the rows' ranges)
    cover = {}
    table_entries = 0
    for b, p in enumerate(w.dec_positions):
        p = int(p)
        if p < 0:
            continue
        lo = max(0, p - w.window + 1) if w.window else 0
        lps = np.arange(lo // 64, p // 64 + 1)
        table_entries += len(lps)
        a = np.maximum(lo, lps * 64) - lps * 64
        z = np.minimum(p, lps * 64 + 63) - lps * 64
        for pg, aa, zz in zip(w.table[b, lps].tolist(), a.tolist(), z.tolist()):
            if pg in cover:
                c = cover[pg]
                cover[pg] = (min(c[0], aa), max(c[1], zz))
            else:
                cover[pg] = (aa, zz)
    kv_keys = sum(z - a + 1 for a, z in cover.values())
    dec_kv = 2 * hkv * kv_keys * d * kv_bytes
    dec_q_out = 2 * w.B * hq * d * 2                     # q read + out written
    dec_table = 4 * table_entries
    # chunk tokens: their rows' visible keys (each key once per row)
    ch_kv = 0
    if w.P:
        per_row = {}
        for r, p in zip(w.ch_rows, w.ch_positions):
            lo = max(0, int(p) - w.window + 1) if w.window else 0
            a, z = per_row.get(int(r), (lo, int(p)))
            per_row[int(r)] = (min(a, lo), max(z, int(p)))
        ch_kv = sum(2 * hkv * (z - a + 1) * d * kv_bytes for a, z in per_row.values())
    ch_q_out = 2 * w.P * hq * d * 2
    # reads q, k, v; writes q_out and the pool slots
    append = w.T * (hq + 2 * hkv) * d * 2 + w.T * hq * d * 2 + w.T * 2 * hkv * d * kv_bytes + 8 * w.T
    return {"decode_kv": dec_kv, "decode_q_out": dec_q_out, "decode_table": dec_table,
            "chunk_kv": ch_kv, "chunk_q_out": ch_q_out, "append": append,
            "decode_call": dec_kv + dec_q_out + dec_table,
            "step": dec_kv + dec_q_out + dec_table + ch_kv + ch_q_out + append}


def chunk_flops(w) -> int:
    """Algorithmic flops of the chunk tokens' attention: for each token and q
    head, a multiply-add per visible key and dimension for Q.K and for P.V."""
    tot = 0
    for p in w.ch_positions:
        p = int(p)
        lo = max(0, p - w.window + 1) if w.window else 0
        tot += 4 * (p - lo + 1) * w.hq * w.head_dim
    return tot


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return float(peaks["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def read_tensor_peak():
    """Dense bf16 TFLOP/s: the sustained figure (kernels here run inside long
    loops of steps)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return float(peaks["bf16_tflops_sustained"]), "measured (sustained)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback (sustained)"


def recorded_traffic(kernel_file: str, config: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current source of the kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        with open(os.path.join(ROOT, "paged_kv_gqa_row_gb300", "csrc", kernel_file), "rb") as f:
            src = f.read()
        entry = rec.get(config)
        if entry and entry.get("source_sha256") == hashlib.sha256(src).hexdigest():
            return float(entry["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_on = self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_on(self):
        self.t_on = time.time()

    def mark_off(self):
        self.t_off = time.time()

    def stop(self):
        if self.proc is not None:
            time.sleep(0.12)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        rows = [l for (t, l) in self.lines if self.t_on is not None and self.t_on - 0.06 <= t <= (self.t_off or t) + 0.06]
        if not rows:
            rows = [l for (_, l) in self.lines]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [x.strip() for x in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def sample_tokens(w, n):
    """A seeded sample of n step tokens: decode rows if the step has any, else
    chunk tokens."""
    rng = np.random.default_rng(0)
    if w.B:
        return sorted((w.P + rng.choice(w.B, size=min(w.B, n), replace=False)).tolist())
    return sorted(rng.choice(w.P, size=min(w.P, n), replace=False).tolist())


def sample_units(w, n_tokens):
    """(token, kv head) units of the oracle samples: every kv head of a seeded
    sample of step tokens."""
    return [(t, h) for t in sample_tokens(w, n_tokens) for h in range(w.hkv)]


K_SCALE_E4M3, V_SCALE_E4M3 = 0.25, 0.5  # scales of the 8-bit pools in the e4m3 runs


def prepare_oracle_sample(w, units, kv="bf16"):
    """Inputs of the oracle for each (token, kv head) unit: the pages the token
    reads of that kv head, and the step tokens that write into them (their q
    heads of the kv head's group, their k and v of the kv head)."""
    e4m3 = kv == "e4m3"
    tp, tr = w.token_positions(), w.token_rows()
    q_all, k_all, v_all = w.step_q(), w.step_k(), w.step_v()
    g = w.hq // w.hkv
    pool_pages = w.pool_pages_e4m3 if e4m3 else w.pool_pages
    prepared = []
    for t, h in units:
        p, row = int(tp[t]), int(tr[t])
        lo = max(0, p - w.window + 1) if w.window else 0
        lps = np.arange(lo // 64, p // 64 + 1)
        pages = w.table[row, lps]
        index = {int(pg): i for i, pg in enumerate(pages)}
        kp = pool_pages("k", h, pages).reshape(1, -1, w.head_dim)
        vp = pool_pages("v", h, pages).reshape(1, -1, w.head_dim)
        writers, slots = [], []
        for u in range(w.T):
            pu = int(tp[u])
            if pu < 0:
                continue
            pg = int(w.table[int(tr[u]), pu // 64])
            if pg in index:
                writers.append(u)
                slots.append(index[pg] * 64 + pu % 64)
        wi = np.array(writers)
        ctable = np.full((1, lps[-1] + 1), -1, dtype=np.int32)
        ctable[0, lps] = np.arange(len(lps), dtype=np.int32)
        prepared.append(dict(q=q_all[wi][:, h * g:(h + 1) * g], k=k_all[wi][:, h:h + 1], v=v_all[wi][:, h:h + 1],
                             pos=tp[wi], rows=tr[wi], slots=np.array(slots), me=writers.index(t), p=p,
                             kp=kp, vp=vp, ctable=ctable, nkeys=p - lo + 1))
    return prepared


def run_oracle_sample(w, prepared, kv="bf16"):
    """Run the oracle (as it stands) on prepared units: for each, the append of
    the step tokens that write into the pages it reads, then its attention.
    Returns (wall seconds, CPU seconds of the process, algorithmic bytes)."""
    from oracle import fp8, paged, rope
    e4m3 = kv == "e4m3"
    inv = rope.inv_freq(w.theta, w.head_dim, w.llama3)
    gq, gk = w.gamma_q(), w.gamma_k()
    g = w.hq // w.hkv
    c0, t0 = time.process_time(), time.perf_counter()
    nbytes = 0
    for u in prepared:
        if e4m3:
            q_out, kp2, vp2 = fp8.append_rope(u["q"], u["k"], u["v"], u["pos"], u["rows"], None, u["kp"], u["vp"],
                                              inv, K_SCALE_E4M3, V_SCALE_E4M3, slots=u["slots"], gamma_q=gq,
                                              gamma_k=gk, eps=w.norm_eps)
            fp8.attention_at(q_out[u["me"]], 0, u["p"], u["ctable"], kp2, vp2, K_SCALE_E4M3, V_SCALE_E4M3,
                             w.window)
        else:
            q_out, kp2, vp2 = paged.append_rope(u["q"], u["k"], u["v"], u["pos"], u["rows"], None, u["kp"], u["vp"],
                                                inv, slots=u["slots"], gamma_q=gq, gamma_k=gk, eps=w.norm_eps)
            paged.attention_at(q_out[u["me"]], 0, u["p"], u["ctable"], kp2, vp2, w.window)
        nbytes += 2 * u["nkeys"] * w.head_dim * (1 if e4m3 else 2) + 2 * g * w.head_dim * 2
    return time.perf_counter() - t0, time.process_time() - c0, nbytes


def run_reference(args, rank, world):
    """The oracle timed on the host cores: exactly `steps` timed steps, each a
    bounded sample of the workload's (token, kv head) units, sized so that the
    whole run takes about --ref-seconds."""
    import synth
    if rank != 0:
        return None
    w = synth.build(args.config, scale=args.scale, rows=args.rows)
    units = sample_units(w, args.ref_rows)
    prepared = prepare_oracle_sample(w, units, kv=args.kv)
    # warm-up: one unit per step; it also gives the time of one unit
    wsecs = []
    for i in range(max(0, args.warmup)):
        s, _, _ = run_oracle_sample(w, prepared[i % len(prepared):i % len(prepared) + 1], kv=args.kv)
        wsecs.append(s)
    per_unit = max(1e-4, statistics.median(wsecs)) if wsecs else 0.05
    n = int(max(1, min(len(prepared), args.ref_seconds / max(1, args.steps) / per_unit)))
    secs = cpu = 0.0
    nbytes = 0
    at = 0
    for _ in range(args.steps):
        chunk = [prepared[(at + i) % len(prepared)] for i in range(n)]
        at = (at + n) % len(prepared)
        s, c, nb = run_oracle_sample(w, chunk, kv=args.kv)
        secs += s
        cpu += c
        nbytes += nb
    value = nbytes / secs / 1e9
    cores = round(cpu / secs, 2)
    what = "decode rows" if w.B else "chunk tokens"
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "impl": "reference",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000 * secs / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.config, "description": CONFIGS[args.config], "kv_dtype": args.kv,
                   "sample_units_per_step": n},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} (token, kv head) units per step, cycling through all kv heads of "
                                   f"{len(prepared) // w.hkv} seeded {what} of the {args.config} workload; "
                                   f"cores = process CPU time / wall time"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


class GpuWorkload:
    """Device buffers of one workload and the library calls of its step."""

    def __init__(self, args, w, dev, kv):
        import torch

        import paged_kv_gqa_row_gb300 as lnk
        from synth import device as sdev
        self.torch, self.lnk, self.w, self.dev = torch, lnk, w, dev
        e4m3 = kv == "e4m3"
        if e4m3 and w.P:
            raise SystemExit("--kv e4m3: chunk attention runs on bf16 pools only; use a decode workload")
        self.e4m3 = e4m3
        self.kv_bytes = 1 if e4m3 else 2
        self.parts = algorithmic_bytes(w, self.kv_bytes)
        self.pool_bytes = 2 * w.hkv * w.pool_positions * w.head_dim * self.kv_bytes
        # (a small workload's pages would otherwise stay in L2 from one step to the next)
        self.l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or L2_FALLBACK)
        self.read_per_step = max(1, self.parts["decode_kv"] + self.parts["chunk_kv"])
        self.copies = pool_copies(self.pool_bytes, self.read_per_step, self.l2_bytes, args.pool_copies)

        def d16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)

        def d32(a):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

        shape = (w.hkv, w.pool_positions, w.head_dim)
        self.pools = []
        for _ in range(self.copies):
            kp = torch.empty(shape, dtype=torch.uint8 if e4m3 else torch.int16, device=dev)
            vp = torch.empty_like(kp)
            fill = sdev.fill_e4m3 if e4m3 else sdev.fill_normal_bf16
            fill(kp, w.pool_key("k"))
            fill(vp, w.pool_key("v"))
            self.pools.append((kp, vp))
        self.q, self.k, self.v = d16(w.step_q()), d16(w.step_k()), d16(w.step_v())
        self.pos, self.rows, self.table = d32(w.token_positions()), d32(w.token_rows()), d32(w.table)
        self.dec_pos = d32(w.dec_positions)
        self.ch = (d32(w.ch_rows), d32(w.ch_positions), d32(w.ch_segments)) if w.P else (None, None, None)
        self.gq = None if w.gamma_q() is None else d16(w.gamma_q())
        self.gk = None if w.gamma_k() is None else d16(w.gamma_k())
        self.q_out = torch.zeros_like(self.q)
        self.out = torch.zeros_like(self.q)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.desc = lnk.attn_desc(w.hq, w.hkv, w.head_dim, w.num_pages, w.num_rows, w.pages_per_row,
                                  window=w.window, kv_dtype=lnk.KV_E4M3 if e4m3 else lnk.KV_BF16,
                                  k_scale=K_SCALE_E4M3, v_scale=V_SCALE_E4M3)
        self.rd = lnk.rope_desc(w.theta, w.llama3)
        self.ws_bytes = lnk.lnk_paged_workspace_size(self.desc, max(1, w.B))
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.Stream(device=dev)
        self.s_handle = self.stream.cuda_stream
        self.inputs = (self.q, self.k, self.v, self.pos, self.table)
        if w.P == 0:  # lnk_paged_decode_step: one kernel or two
            self.launches_per_step = lnk.lnk_paged_decode_step_launches(self.desc, w.B)
        else:
            self.launches_per_step = 1 + 1 + (1 if w.B else 0)
        self.one_kernel = w.P == 0 and self.launches_per_step == 1

    def l2_note(self):
        """How the timed steps keep their K/V reads out of L2."""
        between = (self.copies - 1) * self.read_per_step
        if self.copies == 1:
            return (f"inputs larger than L2: one pool of {self.pool_bytes / 1e9:.2f} GB, "
                    f"{self.read_per_step / 1e9:.2f} GB of K/V read per step (L2 {self.l2_bytes / 1e6:.0f} MB)")
        return (f"inputs larger than L2: {self.copies} pool copies of {self.pool_bytes / 1e9:.3f} GB alternated "
                f"step to step; a copy comes back after {between / 1e6:.0f} MB of other steps' K/V reads "
                f"(L2 {self.l2_bytes / 1e6:.0f} MB)")

    def attend(self, kp, vp, q_src, out_dst, tab):
        w, lnk = self.w, self.lnk
        if w.P == 0:
            lnk.lnk_paged_decode_attn(self.desc, q_src, self.dec_pos, tab, kp, vp, out_dst, w.B, self.ws,
                                      self.ws_bytes, self.status, self.s_handle)
        else:
            lnk.lnk_paged_step_attn(self.desc, q_src, self.ch[0], self.ch[1], self.ch[2], self.dec_pos, tab, kp, vp,
                                    out_dst, None, None, w.P, w.B, 0, self.ws, self.ws_bytes, self.status,
                                    self.s_handle)

    def attend_part(self, kp, vp, part):
        """One kernel of the step's attention call on its own: the decode rows
        ("decode") or the prompt chunks ("chunk")."""
        w, lnk = self.w, self.lnk
        if part == "decode":
            lnk.lnk_paged_decode_attn(self.desc, self.q_out[w.P:], self.dec_pos, self.table, kp, vp,
                                      self.out[w.P:], w.B, self.ws, self.ws_bytes, self.status, self.s_handle)
        else:
            lnk.lnk_paged_step_attn(self.desc, self.q_out, self.ch[0], self.ch[1], self.ch[2], None, self.table,
                                    kp, vp, self.out, None, None, w.P, 0, 0, None, 0, self.status, self.s_handle)

    def step(self, i, inp, ev=None, out_dst=None):
        """One whole step.  Decode-only steps are one lnk_paged_decode_step call
        (append and attention, one kernel for small launches); steps with prompt
        chunks are lnk_paged_append_rope then lnk_paged_step_attn.  With `ev`,
        events around the attention call (two calls then, for decode-only steps:
        the append and lnk_paged_decode_attn)."""
        w = self.w
        qq, kk, vv, pp, tab = inp
        kp, vp = self.pools[i % self.copies]
        if w.P == 0 and ev is None:
            self.lnk.lnk_paged_decode_step(self.desc, self.rd, qq, kk, vv, pp, tab, self.gq, self.gk, w.norm_eps,
                                           kp, vp, self.q_out, self.out if out_dst is None else out_dst, w.B,
                                           self.ws, self.ws_bytes, self.status, self.s_handle)
            return
        self.lnk.lnk_paged_append_rope(self.desc, self.rd, qq, kk, vv, pp, self.rows, None, tab, self.gq, self.gk,
                                       w.norm_eps, kp, vp, self.q_out, w.T, self.status, self.s_handle)
        if ev is not None:
            ev[0].record(self.stream)
        self.attend(kp, vp, self.q_out, self.out if out_dst is None else out_dst, tab)
        if ev is not None:
            ev[1].record(self.stream)

    def check_status(self):
        st = int(self.status.item())
        assert st == 0, f"device status {st:#x}"

    def warm(self, n):
        """n untimed steps; their average time decides whether the timed steps
        run from a CUDA graph (steps under 50 us)."""
        torch = self.torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            for i in range(n):
                self.step(i, self.inputs)
            e1.record(self.stream)
        self.stream.synchronize()
        self.check_status()
        self.short_steps = n > 0 and e0.elapsed_time(e1) / n <= 0.05

    def timed(self, steps, dist=None, sampler=None):
        """Device time of `steps` whole steps, CUDA events on the launching stream.
        Steps under 50 us would time the host's calls (a call through the
        binding costs a few microseconds of Python): their calls are captured
        once in a CUDA graph before the timed region, which replays it, as a
        serving loop of short steps would run them."""
        torch = self.torch
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        graph = None
        if getattr(self, "short_steps", False):
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=self.stream):
                for i in range(steps):
                    self.step(i, self.inputs)
            graph.replay()  # (one untimed replay)
            self.stream.synchronize()
            self.check_status()
        self.loop = "CUDA graph of the timed steps, captured before the timed region" if graph else "host loop"
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        if sampler:
            sampler.mark_on()
        with torch.cuda.stream(self.stream):
            t_start.record(self.stream)
            if graph is not None:
                graph.replay()
            else:
                for i in range(steps):
                    self.step(i, self.inputs)
            t_end.record(self.stream)
        self.stream.synchronize()
        if sampler:
            sampler.mark_off()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        return t_start.elapsed_time(t_end)

    def kernel_times(self, n, step_ms=None):
        """Average device time of the step's kernels, timed on the launching
        stream with CUDA events around each call, over n calls on the same
        workload: the attention call ("attn"; for decode-only steps
        lnk_paged_decode_attn alone, call after call) and, for steps with both
        prompt chunks and decode rows, each of its two kernels alone.  A
        decode step that is one kernel (lnk_paged_decode_step's one-kernel
        form) is that kernel: its time is the timed region's time per step
        (step_ms), since events around calls that short would time the host.
        (Events between the append and the attention call would stop the
        attention kernel from overlapping the append kernel's tail, so the
        whole-step timing has none.)"""
        torch, w = self.torch, self.w

        def timed_calls(call):
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            with torch.cuda.stream(self.stream):
                for i in range(n):
                    ev[i][0].record(self.stream)
                    call(i)
                    ev[i][1].record(self.stream)
            self.stream.synchronize()
            return sum(a.elapsed_time(b) for a, b in ev) / n

        if self.one_kernel:
            times = {"attn": step_ms}
        elif w.P == 0:
            times = {"attn": timed_calls(lambda i: self.attend_part(*self.pools[i % self.copies], "decode"))}
        else:
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            with torch.cuda.stream(self.stream):
                for i in range(n):
                    self.step(i, self.inputs, ev[i])
            self.stream.synchronize()
            times = {"attn": sum(a.elapsed_time(b) for a, b in ev) / n}
            if w.B:
                for part in ("decode", "chunk"):
                    times[part] = timed_calls(lambda i: self.attend_part(*self.pools[i % self.copies], part))
        self.check_status()
        return times

    def roofline(self, times, config, kt_steps):
        """The roofline object: the decode kernel against the HBM peak (the
        step's dominant kernel whenever it has decode rows), or, for prefill
        alone, the chunk kernel against the tensor peak; for steps with both,
        the chunk kernel's tensor figure under "chunk"."""
        w, parts = self.w, self.parts
        peak, peak_kind = read_peaks()
        tpeak, tkind = read_tensor_peak()
        timing = (f"CUDA events around the call on its stream, average over {kt_steps} calls on the same "
                  "workload right after the timed region")
        if self.one_kernel:
            timing = "the timed region's device time per step (the step is this one kernel)"
        if w.B:
            dec_ms = times["decode"] if w.P else times["attn"]
            # (a one-kernel decode step: the kernel also reads the step's q/k/v and writes k/v and q_out)
            dec_bytes = parts["step"] if self.one_kernel else parts["decode_call"]
            achieved = dec_bytes / (dec_ms / 1e3) / 1e9
            name = ("decode_kernel (lnk_paged_decode_step in one kernel: append and attention)" if self.one_kernel
                    else "decode_kernel (lnk_paged_decode_attn over the step's decode rows)")
            r = {"bound": "hbm", "kernel": name,
                 "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                 "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                 "traffic": recorded_traffic("decode.cu", config + ("_e4m3" if self.e4m3 else "")),
                 "algorithmic_bytes": dec_bytes, "avg_launch_ms": round(dec_ms, 5), "timing": timing}
        if w.P:
            flops = chunk_flops(w)
            ch_ms = times["chunk"] if w.B else times["attn"]
            achieved = flops / (ch_ms / 1e3) / 1e12
            c = {"bound": "tensor", "kernel": "chunk_kernel (lnk_paged_step_attn over the step's prompt chunks)",
                 "achieved": round(achieved, 2), "peak": tpeak, "unit": "TFLOP/s",
                 "frac": round(achieved / tpeak, 4), "peak_source": tkind,
                 "traffic": recorded_traffic("chunk.cu", config), "algorithmic_flops": flops,
                 "avg_launch_ms": round(ch_ms, 5), "timing": timing}
            if not w.B:
                return c
            r["chunk"] = c
            step_bytes = parts["decode_call"] + parts["chunk_kv"] + parts["chunk_q_out"]
            r["step_attn"] = {"kernels": "chunk_kernel + decode_kernel (one lnk_paged_step_attn call)",
                              "achieved": round(step_bytes / (times["attn"] / 1e3) / 1e9, 2), "unit": "GB/s",
                              "frac": round(step_bytes / (times["attn"] / 1e3) / 1e9 / peak, 4),
                              "algorithmic_bytes": step_bytes, "avg_launch_ms": round(times["attn"], 5)}
        return r

    def e2e(self, steps, elapsed_ms, dist=None):
        """End to end through the C ABI: every step's inputs copied from pinned
        host memory (one packed buffer, one copy), the calls, and the result
        copied back to pinned host memory.  As a serving loop would, the two
        copy directions run on their own streams with double buffers, so that
        step i + 1's inputs and step i - 1's result move while the kernels of
        step i run.  Returns (ms, h2d bytes, d2h bytes, steps, how)."""
        torch, w, dev = self.torch, self.w, self.dev
        host_parts = [w.step_q().view(np.uint8).ravel(), w.step_k().view(np.uint8).ravel(),
                      w.step_v().view(np.uint8).ravel(), w.token_positions().astype(np.int32).view(np.uint8),
                      np.ascontiguousarray(w.table, dtype=np.int32).view(np.uint8).ravel()]
        offs = np.cumsum([0] + [((a.size + 255) // 256) * 256 for a in host_parts])
        h_in = torch.zeros(int(offs[-1]), dtype=torch.uint8).pin_memory()
        for a, o0 in zip(host_parts, offs[:-1]):
            h_in[int(o0):int(o0) + a.size] = torch.from_numpy(a.copy())
        d_in = [torch.empty_like(h_in, device=dev) for _ in range(2)]

        def views(sl):
            def view(i, dtype, shape):
                n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
                return d_in[sl][int(offs[i]):int(offs[i]) + n].view(dtype).view(shape)
            return (view(0, torch.int16, self.q.shape), view(1, torch.int16, self.k.shape),
                    view(2, torch.int16, self.v.shape), view(3, torch.int32, self.pos.shape),
                    view(4, torch.int32, self.table.shape))

        e_inputs = [views(0), views(1)]
        d_out = [torch.zeros_like(self.out) for _ in range(2)]
        h_out = [torch.empty(self.out.shape, dtype=torch.int16).pin_memory() for _ in range(2)]
        h2d = int(sum(a.size for a in host_parts))
        d2h = h_out[0].numel() * h_out[0].element_size()
        stream = self.stream
        up_stream, down_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of the slot copied in
        ev_done = [torch.cuda.Event() for _ in range(2)]  # the slot's step finished (inputs read, output written)
        ev_back = [torch.cuda.Event() for _ in range(2)]  # the slot's output copied back
        # Short steps would be bound by the host's calls: there all the steps'
        # copies and calls (the same streams and events) are captured once in a
        # CUDA graph and replayed, as a serving loop of short steps would run
        # them (the entry points allocate nothing and never synchronise).
        use_graph = elapsed_ms <= 0.05
        ev_fork = torch.cuda.Event()
        ev_join = [torch.cuda.Event() for _ in range(2)]

        def run(n, fork_join=False):
            if fork_join:  # bring the copy streams into the capture and back
                ev_fork.record(stream)
                up_stream.wait_event(ev_fork)
                down_stream.wait_event(ev_fork)
            for i in range(n):
                sl = i & 1
                with torch.cuda.stream(up_stream):
                    if i >= 2:
                        up_stream.wait_event(ev_done[sl])
                    d_in[sl].copy_(h_in, non_blocking=True)
                    ev_in[sl].record(up_stream)
                stream.wait_event(ev_in[sl])
                if i >= 2:
                    stream.wait_event(ev_back[sl])
                with torch.cuda.stream(stream):
                    self.step(i, e_inputs[sl], out_dst=d_out[sl])
                    ev_done[sl].record(stream)
                with torch.cuda.stream(down_stream):
                    down_stream.wait_event(ev_done[sl])
                    h_out[sl].copy_(d_out[sl], non_blocking=True)
                    ev_back[sl].record(down_stream)
            if fork_join:
                ev_join[0].record(up_stream)
                ev_join[1].record(down_stream)
                stream.wait_event(ev_join[0])
                stream.wait_event(ev_join[1])

        run(3)
        torch.cuda.synchronize()
        graph = None
        if use_graph:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                run(steps, fork_join=True)
            graph.replay()
            torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        if graph is not None:
            e0.record(stream)
            with torch.cuda.stream(stream):
                graph.replay()
            e1.record(stream)
        else:
            e0.record(up_stream)
            run(steps)
            e1.record(down_stream)
        torch.cuda.synchronize()
        self.check_status()
        last = (steps - 1) & 1
        assert np.array_equal(h_out[last].numpy(), self.out.cpu().numpy()), \
            "end-to-end result differs from the device result"
        how = ("every step: inputs host->device and result device->host (pinned), each direction on its own "
               "stream overlapping the kernels of the neighbouring steps (double buffers)")
        if use_graph:
            how += "; all the steps' copies and calls captured once in a CUDA graph and replayed"
        return e0.elapsed_time(e1), h2d, d2h, how


def run_gpu(args, rank, world, dist):
    import torch

    import synth

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    def rank_workload(name, scale, rows):
        seed = None if rank == 0 else 1000 + 97 * rank + synth.WORKLOADS[name]
        return synth.build(name, seed=seed, scale=scale, rows=rows)

    w = rank_workload(args.config, args.scale, args.rows)
    g = GpuWorkload(args, w, dev, args.kv)
    g.warm(args.warmup)

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    elapsed_ms = g.timed(args.steps, dist, sampler)
    kt_steps = max(1, min(args.steps, 500))
    times = g.kernel_times(kt_steps, elapsed_ms / args.steps)
    clocks = sampler.stop() if sampler else None
    e2e_steps = max(1, min(args.steps, 200))
    e2e_ms, h2d, d2h, e2e_how = g.e2e(e2e_steps, elapsed_ms / args.steps, dist)

    keys = ["elapsed", "e2e"] + sorted(times)
    vals = torch.tensor([elapsed_ms, e2e_ms] + [times[k] for k in sorted(times)], dtype=torch.float64, device=dev)
    if dist:
        dist.all_reduce(vals, op=dist.ReduceOp.MAX)
    got = dict(zip(keys, [float(x) for x in vals.tolist()]))
    elapsed_ms, e2e_ms = got["elapsed"], got["e2e"]
    times = {k: got[k] for k in times}

    # the Mistral-shaped decode step, in the same process, when the main
    # workload is the Llama step (the two long-context configurations)
    extra = None
    if args.config == "llama_step" and not args.no_extra and args.kv == "bf16":
        wm = rank_workload("mistral", 1.0, None)
        gm = GpuWorkload(args, wm, dev, "bf16")
        gm.warm(args.warmup)
        m_ms = gm.timed(args.steps, dist)
        m_times = gm.kernel_times(kt_steps)
        vals = torch.tensor([m_ms, m_times["attn"]], dtype=torch.float64, device=dev)
        if dist:
            dist.all_reduce(vals, op=dist.ReduceOp.MAX)
        m_ms, m_times["attn"] = [float(x) for x in vals.tolist()]
        m_step = gm.parts["step"]
        extra = {"workload": "mistral", "description": CONFIGS["mistral"],
                 "value": round(world * m_step * args.steps / (m_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                 "ms_per_step": round(m_ms / args.steps, 5),
                 "row_steps_per_s": round(world * wm.B * args.steps / (m_ms / 1e3), 1),
                 "algorithmic_bytes_per_step": m_step,
                 "l2": gm.l2_note(),
                 "roofline": gm.roofline(m_times, "mistral", kt_steps)}
        del gm

    if rank != 0:
        return None
    peak, _ = read_peaks()
    step_bytes = g.parts["step"]
    value = world * step_bytes * args.steps / (elapsed_ms / 1e3) / 1e9
    e2e_value = world * step_bytes * e2e_steps / (e2e_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if g.e4m3 else "bf16", "data": "synthetic",
        "config": {"workload": args.config, "description": CONFIGS[args.config], "kv_dtype": args.kv,
                   "scale": args.scale, "decode_rows": w.B, "chunk_tokens": w.P, "q_heads": w.hq, "kv_heads": w.hkv,
                   "head_dim": w.head_dim, "page_size": 64, "num_pages": w.num_pages,
                   "parallelism": f"rows x{world} (independent batches per GPU)",
                   "l2": g.l2_note(), "timed_loop": g.loop,
                   "algorithmic_bytes_per_step": step_bytes},
        "row_steps_per_s": round(world * w.B * args.steps / (elapsed_ms / 1e3), 1),
        "chunk_tokens_per_s": round(world * w.P * args.steps / (elapsed_ms / 1e3), 1),
        "pct_of_peak": round(100 * value / world / peak, 2),
        "roofline": g.roofline(times, args.config, kt_steps),
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps, "copies": e2e_how},
        "gpu_launches": g.launches_per_step * args.steps,
        "clocks": clocks,
    }
    if extra is not None:
        line["mistral"] = extra
    if not args.no_cpu_baseline:
        units = sample_units(w, args.ref_rows)
        prepared = prepare_oracle_sample(w, units, kv=args.kv)
        secs = cpu = 0.0
        nb, reps = 0, 0
        while secs < args.cpu_seconds and reps < 50:
            s, c, b = run_oracle_sample(w, prepared, kv=args.kv)
            secs += s
            cpu += c
            nb += b
            reps += 1
        what = "decode rows" if w.B else "chunk tokens"
        line["cpu_baseline"] = {"value": round(nb / secs / 1e9, 4), "unit": "GB/s", "cores": round(cpu / secs, 2),
                                "kind": "oracle",
                                "sample": f"all kv heads of {len(units) // w.hkv} seeded {what} x {reps} repeats "
                                          f"of the {args.config} workload ({secs:.1f} s); cores = process CPU "
                                          "time / wall time"}
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="llama_step", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="lnk", choices=["lnk", "reference"])
    ap.add_argument("--kv", default="bf16", choices=["bf16", "e4m3"],
                    help="pool element type (e4m3: 8-bit pools, decode workloads only)")
    ap.add_argument("--ref-rows", type=int, default=4, help="step tokens sampled for the oracle timings")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="reference arm: about this many seconds of oracle work over all timed steps")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the Mistral line of the default run")
    ap.add_argument("--pool-copies", type=int, default=0, help="pool copies alternated step to step (0: auto)")
    ap.add_argument("--scale", type=float, default=1.0, help="shrink context lengths (profiling runs only)")
    ap.add_argument("--rows", type=int, default=None, help="override the number of decode rows (profiling runs only)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group(backend)
        dist = tdist
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_gpu(args, rank, world, dist)
    if line is not None:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
