"""Build the sm_103a attention library in-tree.

Compiles each CUDA translation unit in parallel with nvcc for
``arch=compute_103a,code=sm_103a`` and links them into
``attention_attn_fwd_gb300/_build/libattn_fwd_gb300.so``.
Usable as ``python -m attention_attn_fwd_gb300.build [--force] [-v]``.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libattn_fwd_gb300.so")
SOURCES = ["attn_api.cu", "attn_fwd_d64.cu", "attn_fwd_d128.cu",
           "attn_fwd_d64_packed.cu", "attn_fwd_d128_packed.cu",
           "attn_fwd_d128_fp8.cu", "attn_fwd_d128_fp8_packed.cu",
           "attn_noalloc.cu", "attn_bwd.cu", "attn_merge.cu"]
HEADERS = ["attn_fwd_kernel.cuh", "attn_fwd_launch.cuh", "attn_sync.cuh",
           "fast_div.h",
           "attn_bwd_kernel.cuh", "attn_merge_kernel.cuh",
           "sm103_ptx.cuh", "attn_launch.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required")
    return cand


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, h) for h in HEADERS]
    headers.append(os.path.join(ROOT, "include", "attn.h"))
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", CSRC, "-I", os.path.join(ROOT, "include")]
    if verbose:
        common += ["-Xptxas", "-v"]
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + headers):
            jobs.append([nvcc] + common + ["-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed: %s" % " ".join(cmd))
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + ".tmp%d" % os.getpid()
        subprocess.run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs,
                       check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
