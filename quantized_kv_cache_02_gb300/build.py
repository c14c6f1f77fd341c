"""Build libkvq.so (and the input generator's libkvqgen.so) for sm_103a with nvcc.

Translation units compile in parallel; objects go to ``_build/`` beside the
sources.  ``python -m quantized_kv_cache_02_gb300.build`` runs it.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc") if os.path.exists(os.path.join(CUDA_HOME, "bin", "nvcc")) else "nvcc"
CFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", os.path.join(ROOT, "include")]
LDFLAGS = ARCH + ["-shared", "-cudart", "shared", f"-Xlinker=-rpath={CUDA_HOME}/lib64"]

SOURCES = ["kvq_host.cu", "kvq_append.cu", "kvq_decode_simt.cu", "kvq_decode_mma.cu", "kvq_decode_mma_b2.cu",
           "kvq_decode_mma_b4.cu", "kvq_decode_mma_b8.cu", "kvq_decode_tc.cu", "kvq_restore.cu",
           "kvq_segment.cu"]


def _run(cmd):
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + proc.stdout + proc.stderr)
    return proc.stdout + proc.stderr


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, extra_flags=()) -> list[str]:
    """Compile what is out of date; returns the paths of the shared libraries."""
    os.makedirs(OBJ, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(ROOT, "include", "kvq.h"))
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OBJ, src.replace(".cu", ".o"))
        objs.append(o)
        if _stale(o, [s] + headers) or extra_flags:
            jobs.append([NVCC, *CFLAGS, *extra_flags, "-c", s, "-o", o])
    gen_src = os.path.join(ROOT, "kvq_inputs", "csrc", "kvq_gen.cu")
    gen_lib = os.path.join(ROOT, "kvq_inputs", "libkvqgen.so")
    gen_job = None
    if _stale(gen_lib, [gen_src]):
        gen_job = [NVCC, *CFLAGS, *LDFLAGS, gen_src, "-o", gen_lib]
    all_jobs = jobs + ([gen_job] if gen_job else [])
    with ThreadPoolExecutor(max_workers=max(1, min(len(all_jobs), os.cpu_count() or 4))) as ex:
        for out in ex.map(_run, all_jobs):
            if verbose and out.strip():
                print(out)
    lib = os.path.join(PKG, "libkvq.so")
    if jobs or _stale(lib, objs):
        tmp = lib + ".tmp"
        _run([NVCC, *LDFLAGS, *objs, "-o", tmp])
        shutil.move(tmp, lib)
    return [lib, gen_lib]


if __name__ == "__main__":
    flags = [a for a in sys.argv[1:] if a.startswith("-")]
    for p in build(verbose=True, extra_flags=flags):
        print(p)
