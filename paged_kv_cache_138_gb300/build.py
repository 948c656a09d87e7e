"""Builds libpagedkv.so in-tree: nvcc for sm_103a, one process per translation unit.

    python -m paged_kv_cache_138_gb300.build [--force] [--verbose]

The library lands next to this file; ``_build/`` holds the object files.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpagedkv.so")

SOURCES = ["attention_bs16.cu", "attention_bs8.cu", "attention_bs32.cu", "attention_bs64.cu",
           "paged_attention.cu", "cache_ops.cu", "synthetic.cu", "block_manager.cpp",
           "scheduler.cpp", "api.cpp"]
HEADERS = [os.path.join(CSRC, "pkv_device.cuh"), os.path.join(CSRC, "attention_kernel.cuh"),
           os.path.join(INCLUDE, "pagedkv.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    objs, procs = [], []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        if not force and not _stale(obj, [path] + HEADERS + [__file__]):
            continue
        cmd = [nvcc(), *ARCH, "-O3", "-std=c++17", "-lineinfo", "-I", INCLUDE, "-I", CSRC,
               "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall", "-c", path, "-o", obj]
        if src.endswith(".cu"):
            cmd[1:1] = ["-Xptxas", "-v"] if verbose else []
        procs.append((src, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                  stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, cmd, p in procs:
        out, _ = p.communicate()
        if verbose and out:
            sys.stdout.write(out)
        if p.returncode != 0:
            failed.append((src, " ".join(cmd), out))
    if failed:
        msg = "\n".join("%s failed:\n%s\n%s" % f for f in failed)
        raise RuntimeError("libpagedkv build failed\n" + msg)
    if force or procs or _stale(LIB, objs):
        tmp = LIB + ".tmp.%d" % os.getpid()
        subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
