"""Benchmark of the paged decode / step attention path on one or more GPUs.

Default workload: one Mistral-7B-v0.3-shaped layer decode step (64 rows,
32 q / 8 kv heads, head_dim 128, context lengths uniform in [512, 8192],
pages of 64 shuffled in a pool sized to the total, bf16 synthetic data).
A step is one pass of the whole path: append_rope over the step's tokens,
then decode_attn (or step_attn for the Llama step workload).

Metric: achieved HBM GB/s = algorithmic bytes of a step (the visible K/V
bytes, each page counted once, plus q in, q/k/v append traffic, outputs and
page-table entries) / step time; row-steps/s alongside.

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


K_SCALE_E4M3, V_SCALE_E4M3 = 0.25, 0.5  # scales of the 8-bit pools in the e4m3 runs


def cpu_oracle_sample(w, tokens, repeats=1, kv="bf16"):
    """Time the oracle (as it stands) on a sample of step tokens: for each, the
    append of the step tokens that write into the pages it reads, then its
    attention; returns (seconds, algorithmic bytes of the sample)."""
    import synth  # noqa: F401
    from oracle import fp8, paged, rope
    e4m3 = kv == "e4m3"
    sample = []
    tp, tr = w.token_positions(), w.token_rows()
    inv = rope.inv_freq(w.theta, w.head_dim, w.llama3)
    q_all, k_all, v_all = w.step_q(), w.step_k(), w.step_v()
    gq, gk = w.gamma_q(), w.gamma_k()
    for t in tokens:
        p, row = int(tp[t]), int(tr[t])
        lo = max(0, p - w.window + 1) if w.window else 0
        lps = np.arange(lo // 64, p // 64 + 1)
        pages = w.table[row, lps]
        index = {int(pg): i for i, pg in enumerate(pages)}
        pool_pages = w.pool_pages_e4m3 if e4m3 else w.pool_pages
        kp = np.stack([pool_pages("k", h, pages).reshape(-1, w.head_dim) for h in range(w.hkv)])
        vp = np.stack([pool_pages("v", h, pages).reshape(-1, w.head_dim) for h in range(w.hkv)])
        writers, slots = [], []
        for u in range(w.T):
            pu = int(tp[u])
            if pu < 0:
                continue
            pg = int(w.table[int(tr[u]), pu // 64])
            if pg in index:
                writers.append(u)
                slots.append(index[pg] * 64 + pu % 64)
        ctable = np.full((1, lps[-1] + 1), -1, dtype=np.int32)
        ctable[0, lps] = np.arange(len(lps), dtype=np.int32)
        sample.append((np.array(writers), np.array(slots), writers.index(t), p, kp, vp, ctable, p - lo + 1))
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(repeats):
        for (wi, slots, me, p, kp, vp, ctable, nkeys) in sample:
            if e4m3:
                q_out, kp2, vp2 = fp8.append_rope(q_all[wi], k_all[wi], v_all[wi], tp[wi], tr[wi], None, kp, vp,
                                                  inv, K_SCALE_E4M3, V_SCALE_E4M3, slots=slots, gamma_q=gq,
                                                  gamma_k=gk, eps=w.norm_eps)
                fp8.attention_at(q_out[me], 0, p, ctable, kp2, vp2, K_SCALE_E4M3, V_SCALE_E4M3, w.window)
            else:
                q_out, kp2, vp2 = paged.append_rope(q_all[wi], k_all[wi], v_all[wi], tp[wi], tr[wi], None,
                                                    kp, vp, inv, slots=slots, gamma_q=gq,
                                                    gamma_k=gk, eps=w.norm_eps)
                paged.attention_at(q_out[me], 0, p, ctable, kp2, vp2, w.window)
            nbytes += 2 * w.hkv * nkeys * w.head_dim * (1 if e4m3 else 2) + 2 * w.hq * w.head_dim * 2
    return time.perf_counter() - t0, nbytes


def threads_used():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        return max([i.get("num_threads", 1) for i in info] + [1])
    except Exception:
        return os.cpu_count() or 1


def run_reference(args, rank, world):
    """The oracle timed on the host cores, each step a bounded sample of rows."""
    import synth
    if rank != 0:
        return None
    w = synth.build(args.config, scale=args.scale, rows=args.rows)
    rows = sample_tokens(w, args.ref_rows)
    for _ in range(max(0, args.warmup)):
        cpu_oracle_sample(w, rows[:1], kv=args.kv)
    secs, nbytes = 0.0, 0
    for _ in range(args.steps):
        s, nb = cpu_oracle_sample(w, rows, kv=args.kv)
        secs += s
        nbytes += nb
    value = nbytes / secs / 1e9
    cores = threads_used()
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "impl": "reference",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000 * secs / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.config, "description": CONFIGS[args.config], "kv_dtype": args.kv,
                   "sample_rows_per_step": len(rows)},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{len(rows)} {'decode rows' if w.B else 'chunk tokens'} of the "
                                   f"{args.config} workload per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def run_gpu(args, rank, world, dist):
    import torch

    import paged_kv_gqa_row_gb300 as lnk
    import synth
    from synth import device as sdev

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    seed = None if rank == 0 else 1000 + 97 * rank + synth.WORKLOADS[args.config]
    w = synth.build(args.config, seed=seed, scale=args.scale, rows=args.rows)
    e4m3 = args.kv == "e4m3"
    if e4m3 and w.P:
        raise SystemExit("--kv e4m3: chunk attention runs on bf16 pools only; use a decode workload")
    kv_bytes = 1 if e4m3 else 2
    parts = algorithmic_bytes(w, kv_bytes)
    pool_bytes = 2 * w.hkv * w.pool_positions * w.head_dim * kv_bytes
    copies = args.pool_copies or (2 if pool_bytes < (8 << 30) else 1)

    def d16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)

    def d32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    shape = (w.hkv, w.pool_positions, w.head_dim)
    pools = []
    for _ in range(copies):
        kp = torch.empty(shape, dtype=torch.uint8 if e4m3 else torch.int16, device=dev)
        vp = torch.empty_like(kp)
        fill = sdev.fill_e4m3 if e4m3 else sdev.fill_normal_bf16
        fill(kp, w.pool_key("k"))
        fill(vp, w.pool_key("v"))
        pools.append((kp, vp))
    q, k, v = d16(w.step_q()), d16(w.step_k()), d16(w.step_v())
    pos, rows, table = d32(w.token_positions()), d32(w.token_rows()), d32(w.table)
    dec_pos = d32(w.dec_positions)
    ch = (d32(w.ch_rows), d32(w.ch_positions), d32(w.ch_segments)) if w.P else (None, None, None)
    gq = None if w.gamma_q() is None else d16(w.gamma_q())
    gk = None if w.gamma_k() is None else d16(w.gamma_k())
    q_out = torch.zeros_like(q)
    out = torch.zeros_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    desc = lnk.attn_desc(w.hq, w.hkv, w.head_dim, w.num_pages, w.num_rows, w.pages_per_row, window=w.window,
                         kv_dtype=lnk.KV_E4M3 if e4m3 else lnk.KV_BF16, k_scale=K_SCALE_E4M3,
                         v_scale=V_SCALE_E4M3)
    rd = lnk.rope_desc(w.theta, w.llama3)
    ws_bytes = lnk.lnk_paged_workspace_size(desc, max(1, w.B))
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    s_handle = stream.cuda_stream
    row_elems = w.hq * w.head_dim

    def attend(kp, vp, q_src, out_dst, tab):
        if w.P == 0:
            lnk.lnk_paged_decode_attn(desc, q_src, dec_pos, tab, kp, vp, out_dst, w.B, ws, ws_bytes,
                                      status, s_handle)
        else:
            lnk.lnk_paged_step_attn(desc, q_src, ch[0], ch[1], ch[2], dec_pos, tab, kp, vp, out_dst,
                                    None, None, w.P, w.B, 0, ws, ws_bytes, status, s_handle)

    def step(i, inp, ev=None, out_dst=None):
        qq, kk, vv, pp, tab = inp
        kp, vp = pools[i % copies]
        lnk.lnk_paged_append_rope(desc, rd, qq, kk, vv, pp, rows, None, tab, gq, gk, w.norm_eps, kp, vp,
                                  q_out, w.T, status, s_handle)
        if ev is not None:
            ev[0].record(stream)
        attend(kp, vp, q_out, out if out_dst is None else out_dst, tab)
        if ev is not None:
            ev[1].record(stream)

    inputs = (q, k, v, pos, table)
    launches_per_step = 1 + (1 if w.P else 0) + (1 if w.B else 0)

    # warm-up
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i, inputs)
    stream.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item()):#x}"

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_on()
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for i in range(args.steps):
            step(i, inputs)
        t_end.record(stream)
    stream.synchronize()
    if sampler:
        sampler.mark_off()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    # Kernel time for the roofline: the same steps again, with events around the
    # attention call.  (Events between the append and the attention call would
    # stop the attention kernel from overlapping the append kernel's tail, so the
    # main timed region above has none.)
    kt_steps = max(1, min(args.steps, 500))
    dec_events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(kt_steps)]
    with torch.cuda.stream(stream):
        for i in range(kt_steps):
            step(i, inputs, dec_events[i])
    stream.synchronize()
    dec_ms = [a.elapsed_time(b) for a, b in dec_events]
    dec_avg_ms = sum(dec_ms) / len(dec_ms)
    clocks = sampler.stop() if sampler else None

    # ---- end to end: every step's inputs copied from pinned host memory (one
    # packed buffer, one copy), the C ABI calls, and the result copied back to
    # pinned host memory.  As a serving loop would, the two copy directions
    # run on their own streams with double buffers, so that step i + 1's inputs
    # and step i - 1's result move while the kernels of step i run. ----
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
        return (view(0, torch.int16, q.shape), view(1, torch.int16, k.shape), view(2, torch.int16, v.shape),
                view(3, torch.int32, pos.shape), view(4, torch.int32, table.shape))

    e_inputs = [views(0), views(1)]
    d_out = [torch.zeros_like(out) for _ in range(2)]
    h_out = [torch.empty(out.shape, dtype=torch.int16).pin_memory() for _ in range(2)]
    h2d = int(sum(a.size for a in host_parts))
    d2h = h_out[0].numel() * h_out[0].element_size()
    e2e_steps = max(1, min(args.steps, 200))
    up_stream, down_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of the slot copied in
    ev_done = [torch.cuda.Event() for _ in range(2)]  # the slot's step finished (inputs read, output written)
    ev_back = [torch.cuda.Event() for _ in range(2)]  # the slot's output copied back

    # Short steps are bound by the host's calls, not the copies: there the
    # plain loop (copies and kernels in order on one stream) is faster.
    pipelined = elapsed_ms / args.steps > 0.05

    def e2e_run(n):
        if not pipelined:
            with torch.cuda.stream(stream):
                for i in range(n):
                    d_in[0].copy_(h_in, non_blocking=True)
                    step(i, e_inputs[0], out_dst=d_out[0])
                    h_out[0].copy_(d_out[0], non_blocking=True)
            return
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
                step(i, e_inputs[sl], out_dst=d_out[sl])
                ev_done[sl].record(stream)
            with torch.cuda.stream(down_stream):
                down_stream.wait_event(ev_done[sl])
                h_out[sl].copy_(d_out[sl], non_blocking=True)
                ev_back[sl].record(down_stream)

    e2e_run(3)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    e0.record(up_stream if pipelined else stream)
    e2e_run(e2e_steps)
    e1.record(down_stream if pipelined else stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    assert int(status.item()) == 0, f"device status {int(status.item()):#x}"
    last = (e2e_steps - 1) & 1 if pipelined else 0
    assert np.array_equal(h_out[last].numpy(), out.cpu().numpy()), "end-to-end result differs from the device result"

    vals = torch.tensor([elapsed_ms, e2e_ms, dec_avg_ms], dtype=torch.float64, device=dev)
    if dist:
        dist.all_reduce(vals, op=dist.ReduceOp.MAX)
    elapsed_ms, e2e_ms, dec_avg_ms = [float(x) for x in vals.tolist()]

    if rank != 0:
        return None
    peak, peak_kind = read_peaks()
    step_bytes = parts["step"]
    value = world * step_bytes * args.steps / (elapsed_ms / 1e3) / 1e9
    e2e_value = world * step_bytes * e2e_steps / (e2e_ms / 1e3) / 1e9
    dec_bytes = parts["decode_call"] + (parts["chunk_kv"] + parts["chunk_q_out"] if w.P else 0)
    if w.B:  # decode rows dominate: HBM bound
        achieved = dec_bytes / (dec_avg_ms / 1e3) / 1e9
        roofline = {"bound": "hbm",
                    "kernel": ("lnk_paged_step_attn (chunk_kernel + decode_kernel)" if w.P
                               else "lnk_paged_decode_attn (decode_kernel)"),
                    "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                    "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                    "traffic": recorded_traffic("decode.cu", args.config + ("_e4m3" if e4m3 else "")),
                    "algorithmic_bytes": dec_bytes}
    else:  # prefill alone: the chunk kernel's contractions, tensor bound
        flops = chunk_flops(w)
        tpeak, tkind = read_tensor_peak()
        achieved = flops / (dec_avg_ms / 1e3) / 1e12
        roofline = {"bound": "tensor", "kernel": "lnk_paged_step_attn (chunk_kernel)",
                    "achieved": round(achieved, 2), "peak": tpeak, "unit": "TFLOP/s",
                    "frac": round(achieved / tpeak, 4), "peak_source": tkind,
                    "traffic": recorded_traffic("chunk.cu", args.config), "algorithmic_flops": flops}
    roofline["avg_launch_ms"] = round(dec_avg_ms, 5)
    roofline["timing"] = (f"CUDA events around the attention call on its stream, {kt_steps} steps "
                          "of the same workload right after the timed region")
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if e4m3 else "bf16", "data": "synthetic",
        "config": {"workload": args.config, "description": CONFIGS[args.config], "kv_dtype": args.kv,
                   "scale": args.scale, "decode_rows": w.B, "chunk_tokens": w.P, "q_heads": w.hq, "kv_heads": w.hkv,
                   "head_dim": w.head_dim, "page_size": 64, "num_pages": w.num_pages,
                   "parallelism": f"rows x{world} (independent batches per GPU)",
                   "l2": f"inputs larger than L2: {copies} pool copies of {pool_bytes / 1e9:.2f} GB, "
                         "alternated step to step",
                   "algorithmic_bytes_per_step": step_bytes},
        "row_steps_per_s": round(world * w.B * args.steps / (elapsed_ms / 1e3), 1),
        "chunk_tokens_per_s": round(world * w.P * args.steps / (elapsed_ms / 1e3), 1),
        "pct_of_peak": round(100 * value / world / peak, 2),
        "roofline": roofline,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "copies": ("every step: inputs host->device and result device->host (pinned), each direction "
                           "on its own stream overlapping the kernels of the neighbouring steps (double buffers)"
                           if pipelined else "every step: inputs host->device, the kernels and the result "
                           "device->host (pinned), in order on one stream")},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        rows_s = sample_tokens(w, args.ref_rows)
        secs, nb, reps = 0.0, 0, 0
        while secs < args.cpu_seconds and reps < 50:
            s, b = cpu_oracle_sample(w, rows_s, kv=args.kv)
            secs += s
            nb += b
            reps += 1
        line["cpu_baseline"] = {"value": round(nb / secs / 1e9, 4), "unit": "GB/s", "cores": threads_used(),
                                "kind": "oracle",
                                "sample": f"{len(rows_s)} {'decode rows' if w.B else 'chunk tokens'} x {reps} "
                                          f"repeats of the {args.config} workload ({secs:.1f} s)"}
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="mistral", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="lnk", choices=["lnk", "reference"])
    ap.add_argument("--kv", default="bf16", choices=["bf16", "e4m3"],
                    help="pool element type (e4m3: 8-bit pools, decode workloads only)")
    ap.add_argument("--ref-rows", type=int, default=4)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
        args.steps = min(args.steps, 10)
        line = run_reference(args, rank, world)
    else:
        line = run_gpu(args, rank, world, dist)
    if line is not None:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
