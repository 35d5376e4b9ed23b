"""Builds liblnk.so (this package's CUDA library) and synth/libsynth.so in-tree.

Each translation unit is compiled by its own nvcc process (in parallel) for
sm_103a only, then linked into a shared library next to its sources.  A
library is rebuilt when any of its sources or headers is newer than it.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
                     "-Xcompiler", "-fPIC,-ffp-contract=off", "-I", INCLUDE]

LIBS = {
    "lnk": {
        "sources": [os.path.join(CSRC, f) for f in ("api.cu", "append_rope.cu", "decode.cu", "chunk.cu", "decode_static.cu", "pages.cu", "selftest.cu", "pager.cpp")],
        "headers": [os.path.join(CSRC, f) for f in ("common.cuh", "ptx.cuh", "rope_math.cuh")] + [os.path.join(INCLUDE, "lnk.h")],
        "out": os.path.join(PKG, "liblnk.so"),
    },
    "synth": {
        "sources": [os.path.join(ROOT, "synth", "fill.cu")],
        "headers": [],
        "out": os.path.join(ROOT, "synth", "libsynth.so"),
    },
}


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(spec) -> bool:
    out = spec["out"]
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(f) > t for f in spec["sources"] + spec["headers"])


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed: " + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> list:
    """Compile whatever is out of date; returns the paths of the libraries."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    for name, spec in LIBS.items():
        if force or _stale(spec):
            for src in spec["sources"]:
                obj = os.path.join(BUILD_DIR, name + "_" + os.path.basename(src) + ".o")
                jobs.append((name, [nvcc, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj], obj))
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        outs = list(ex.map(lambda j: _run(j[1]), jobs))
    if verbose:
        for o in outs:
            if o.strip():
                sys.stdout.write(o)
    for name in {j[0] for j in jobs}:
        objs = [j[2] for j in jobs if j[0] == name]
        _run([nvcc, *ARCH, "-shared", "-o", LIBS[name]["out"], *objs])
    return [spec["out"] for spec in LIBS.values()]


if __name__ == "__main__":
    force = "--force" in sys.argv
    for path in build(force=force, verbose="-v" in sys.argv):
        print(path)
