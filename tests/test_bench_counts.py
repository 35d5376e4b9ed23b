"""The bench's own arithmetic, on the CPU: the algorithmic bytes and flops that
its roofline figures divide by, checked against brute-force counts, and the
reference arm's JSON line (the oracle timed on the host cores)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

# scaled-down workloads of every config, so that shared prefix pages (Qwen3),
# windows (Phi-3) and chunks (Llama) all occur
SCALED = {"phi3_tiny": (1.0, None), "mistral": (0.06, 12), "phi3_window": (0.6, 8), "qwen3": (0.05, 40),
          "llama_step": (0.02, 6), "llama_prefill": (0.03, None)}


def _visible(p, window):
    lo = max(0, p - window + 1) if window else 0
    return range(lo, p + 1)


def _brute_decode_keys(w):
    """Distinct pool slots the decode rows read: each visible key through its row's table."""
    slots = set()
    entries = 0
    for b, p in enumerate(w.dec_positions):
        p = int(p)
        if p < 0:
            continue
        keys = _visible(p, w.window)
        entries += keys[-1] // 64 - keys[0] // 64 + 1
        for j in keys:
            slots.add(int(w.table[b, j // 64]) * 64 + j % 64)
    return len(slots), entries


@pytest.mark.parametrize("name", list(SCALED))
def test_algorithmic_bytes_by_brute_force(name):
    scale, rows = SCALED[name]
    w = synth.build(name, scale=scale, rows=rows)
    for kv_bytes in (2, 1):
        got = bench.algorithmic_bytes(w, kv_bytes)
        keys, entries = _brute_decode_keys(w)
        d, hq, hkv = w.head_dim, w.hq, w.hkv
        assert got["decode_kv"] == 2 * hkv * keys * d * kv_bytes
        assert got["decode_table"] == 4 * entries
        assert got["decode_q_out"] == 2 * w.B * hq * d * 2
        # chunk tokens: each row's visible keys once (a row's chunk tokens share them)
        per_row = {}
        for r, p in zip(w.ch_rows, w.ch_positions):
            per_row.setdefault(int(r), set()).update(_visible(int(p), w.window))
        assert got["chunk_kv"] == sum(2 * hkv * len(k) * d * kv_bytes for k in per_row.values())
        assert got["chunk_q_out"] == 2 * w.P * hq * d * 2
        append = (w.T * (hq + 2 * hkv) * d * 2      # q, k, v read
                  + w.T * hq * d * 2                 # q_out written
                  + w.T * 2 * hkv * d * kv_bytes     # k, v slots written
                  + 8 * w.T)                         # positions and rows (or table reads)
        assert got["append"] == append
        assert got["step"] == sum(got[k] for k in ("decode_kv", "decode_q_out", "decode_table", "chunk_kv",
                                                   "chunk_q_out", "append"))


def test_shared_prefix_pages_counted_once():
    # Qwen3-shaped rows share their first pages: the count must fall below the per-row sum
    w = synth.build("qwen3", scale=0.05, rows=40)
    per_row = sum(len(_visible(int(p), w.window)) for p in w.dec_positions if p >= 0)
    keys, _ = _brute_decode_keys(w)
    assert keys < per_row
    assert bench.algorithmic_bytes(w)["decode_kv"] == 2 * w.hkv * keys * w.head_dim * 2


@pytest.mark.parametrize("name", ["llama_step", "llama_prefill"])
def test_chunk_flops_by_brute_force(name):
    scale, rows = SCALED[name]
    w = synth.build(name, scale=scale, rows=rows)
    want = sum(4 * len(_visible(int(p), w.window)) * w.hq * w.head_dim for p in w.ch_positions)
    assert bench.chunk_flops(w) == want > 0


@pytest.mark.parametrize("config", ["mistral", "llama_prefill"])
def test_reference_arm_prints_one_json_line(config):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", config,
                        "--steps", "1", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == config
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert np.isfinite(d["ms_per_step"]) and d["ms_per_step"] > 0


@pytest.mark.parametrize("name", ["phi3_tiny", "mistral", "phi3_window", "qwen3", "llama_prefill"])
@pytest.mark.parametrize("kv_bytes", [2, 1])
def test_pool_copies_keep_reads_out_of_l2(name, kv_bytes):
    """The timed steps alternate pool copies so that a copy's pages were evicted
    before it comes back: the other copies' reads in between exceed twice the L2."""
    if kv_bytes == 1 and name == "llama_prefill":
        pytest.skip("chunk attention runs on bf16 pools only")
    w = synth.build(name)
    parts = bench.algorithmic_bytes(w, kv_bytes)
    pool = 2 * w.hkv * w.pool_positions * w.head_dim * kv_bytes
    read = parts["decode_kv"] + parts["chunk_kv"]
    for l2 in (bench.L2_FALLBACK, 136 * 10**6):
        c = bench.pool_copies(pool, read, l2)
        assert c >= 2 and c * pool <= max(bench.POOL_COPY_LIMIT, 2 * pool)
        assert (c - 1) * read > 2 * l2
    assert bench.pool_copies(pool, read, bench.L2_FALLBACK, requested=3) == 3


def test_pool_copies_large_pool_is_read_whole():
    w = synth.build("llama_step", scale=1.0)
    pool = 2 * w.hkv * w.pool_positions * w.head_dim * 2
    read = bench.algorithmic_bytes(w)["decode_kv"]
    assert pool >= bench.POOL_COPY_LIMIT and read > 2 * bench.L2_FALLBACK
    assert bench.pool_copies(pool, read, bench.L2_FALLBACK) == 1
