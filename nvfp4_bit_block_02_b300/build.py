"""Build libnvfp4.so (the C-ABI library) in-tree for sm_103a with nvcc.

    python -m nvfp4_bit_block_02_b300.build [--force]
"""
from __future__ import annotations

import os
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libnvfp4.so")
SOURCES = ["api.cu", "quantize.cu", "repack.cu", "gemm.cu", "w4a16.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "nvfp4.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, extra_flags=(), out: str | None = None, verbose: bool = False) -> str:
    """Compile every source to an object in parallel, then link one shared
    library with the static CUDA runtime (no libcuda link dependency: the
    driver entry point for tensor maps is fetched at run time)."""
    out = out or LIB
    if not force and out == LIB and not extra_flags and not _stale():
        return out
    with tempfile.TemporaryDirectory() as tmp:
        procs = []
        objs = []
        for src in SOURCES:
            obj = os.path.join(tmp, src.replace(".cu", ".o"))
            cmd = [nvcc(), *ARCH, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
            objs.append(obj)
        failed = []
        for src, p in procs:
            log, _ = p.communicate()
            if p.returncode != 0:
                failed.append(f"--- {src}\n{log}")
            elif verbose:
                sys.stdout.write(log)
        if failed:
            raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
        tmp_out = out + f".tmp{os.getpid()}"
        link = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp_out, *objs, "-ldl", "-lpthread", "-lrt"]
        p = subprocess.run(link, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError("link failed:\n" + p.stdout + p.stderr)
        os.replace(tmp_out, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
