"""Builds libsyn.so in-tree from csrc/*.cu (and the host-only gguf.cpp) for sm_103a (nvcc, one
process per source file).

    python -m gguf_block_quantized_gb300.build [--force] [--variant debug|stall]

Two checking variants build the same sources into libraries of their own (never loaded by
the product path; the tests load them beside libsyn.so):
  debug  libsyn_debug.so  -DSYN_DEBUG: every kernel checks its indices and copy windows
         against the buffers before each access, records SYN_DEVERR_BOUNDS and skips the
         access (syn_device_status then returns SYN_ERR_BOUNDS).
  stall  libsyn_stall.so  -DSYN_TEST_STALL and a 20,000,000-cycle wait bound: the decode and
         prefill kernels never receive their activations, so their bounded waits run out
         (syn_device_status then returns SYN_ERR_TIMEOUT); the timeout tests use it.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsyn.so")
INCLUDE = os.path.join(ROOT, "include")

SOURCES = ["api.cu", "quant.cu", "gemv.cu", "gemv_f16.cu", "gemm.cu", "noalloc.cu", "gguf.cpp"]
HEADERS = ["common.cuh", "quant_dev.cuh", "kernels.h"]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         f"-I{INCLUDE}", f"-I{CSRC}"]


def _mtime(p: str) -> float:
    return os.path.getmtime(p) if os.path.exists(p) else -1.0


VARIANTS = {
    None: ("_build", "libsyn.so", []),
    "debug": ("_build_debug", "libsyn_debug.so", ["-DSYN_DEBUG"]),
    "stall": ("_build_stall", "libsyn_stall.so", ["-DSYN_TEST_STALL", "-DSYN_WAIT_CYCLES=20000000ll"]),
}


def build(force: bool = False, verbose: bool = False, variant: str | None = None) -> str:
    obj_dir, lib_name, defines = VARIANTS[variant]
    obj_root = os.path.join(HERE, obj_dir)
    lib = os.path.join(HERE, lib_name)
    os.makedirs(obj_root, exist_ok=True)
    deps = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "syn.h")]
    newest_dep = max(_mtime(d) for d in deps)
    procs, objs = [], []
    for src in SOURCES:
        sp = os.path.join(CSRC, src)
        op = os.path.join(obj_root, os.path.splitext(src)[0] + ".o")
        objs.append(op)
        if force or _mtime(op) < max(_mtime(sp), newest_dep):
            cmd = [NVCC, *ARCH, *FLAGS, *defines, "-c", sp, "-o", op]
            if verbose:
                print(" ".join(cmd), flush=True)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"))
    if failed:
        msg = "\n".join(f"--- {s}\n{o}" for s, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    if force or procs or _mtime(lib) < max(_mtime(o) for o in objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [NVCC, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    v = sys.argv[sys.argv.index("--variant") + 1] if "--variant" in sys.argv else None
    build(force="--force" in sys.argv, verbose=True, variant=v)
