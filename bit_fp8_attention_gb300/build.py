"""Build the sm_103a library in-tree: csrc/*.cu -> _build/libvc_attn.so (nvcc, one -gencode).

Each translation unit is compiled in parallel; the link step produces one shared library with
the C ABI of include/vc_attn.h. The FP8 tensor-core rate probe that the benchmark uses for its
roofline (probe/fp8_mma_peak.cu) is built beside it as _build/libvc_probe.so; it is measurement
support, not part of the attention library. Run as `python -m bit_fp8_attention_gb300.build`.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libvc_attn.so")
PROBE_SRC = os.path.join(PKG, "probe", "fp8_mma_peak.cu")
PROBE_LIB = os.path.join(OUT, "libvc_probe.so")
NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", f"-I{os.path.join(ROOT, 'include')}"]


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                     [os.path.join(ROOT, "include", "vc_attn.h")])
    objs = []
    jobs = []
    probe_deps = [PROBE_SRC, os.path.join(CSRC, "vc_device.cuh")]
    if force or _stale(PROBE_LIB, probe_deps):
        jobs.append([NVCC, *ARCH, *FLAGS, "-shared", PROBE_SRC, "-o", PROBE_LIB])
    for src in sources:
        obj = os.path.join(OUT, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            cmd = [NVCC, *ARCH, *FLAGS, "-c", src, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
        for cmd, r in zip(jobs, results):
            if verbose or r.returncode:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode:
                raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run([NVCC, *ARCH, "-shared", "-o", tmp, *objs], check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
