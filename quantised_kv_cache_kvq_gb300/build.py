"""Build libkvq.so (the CUDA library behind include/kvq.h) in-tree for sm_103a.

Translation units compile in parallel with nvcc; the quantise-and-pack unit is built
with --fmad=false so its binary32 arithmetic is never contracted into fused
multiply-adds (its codes must match the documented arithmetic bit for bit).
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libkvq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
          "--expt-relaxed-constexpr"]
UNITS = {
    "kvq_api.cu": [],
    "kvq_append.cu": ["--fmad=false"],
    "kvq_decode_kivi2.cu": [],
    "kvq_decode_kivi4.cu": [],
    "kvq_decode_kivi8.cu": [],
    "kvq_decode_kivi2_steal.cu": [],
    "kvq_decode_kivi4_steal.cu": [],
    "kvq_decode_kivi8_steal.cu": [],
    "kvq_decode_kivi2_paged.cu": [],
    "kvq_decode_kivi4_paged.cu": [],
    "kvq_decode_kivi8_paged.cu": [],
    "kvq_decode_kivi2_paged_steal.cu": [],
    "kvq_decode_kivi4_paged_steal.cu": [],
    "kvq_decode_kivi8_paged_steal.cu": [],
    "kvq_decode_kivi2_sparse.cu": [],
    "kvq_decode_kivi4_sparse.cu": [],
    "kvq_decode_kivi8_sparse.cu": [],
    "kvq_decode_kivi2_sparse_paged.cu": [],
    "kvq_decode_kivi4_sparse_paged.cu": [],
    "kvq_decode_kivi8_sparse_paged.cu": [],
    "kvq_decode_kivi2_rope.cu": [],
    "kvq_decode_kivi4_rope.cu": [],
    "kvq_decode_kivi8_rope.cu": [],
    "kvq_decode_kivi2_rope_paged.cu": [],
    "kvq_decode_kivi4_rope_paged.cu": [],
    "kvq_decode_kivi8_rope_paged.cu": [],
    "kvq_decode_rows.cu": [],
    "kvq_decode_fp8.cu": [],
    "kvq_decode_rope.cu": [],
    "kvq_noalloc.cu": [],
}


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvq.so")
    return cand


def _sources():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "kvq.h")]


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in _sources())


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    for src, flags in UNITS.items():
        obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *COMMON, *flags, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        jobs.append((cmd, obj))
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        futs = [ex.submit(subprocess.run, cmd, capture_output=True, text=True) for cmd, _ in jobs]
        for (cmd, _), f in zip(jobs, futs):
            r = f.result()
            if verbose or r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed: " + " ".join(cmd))
    tmp = LIB + ".tmp%d" % os.getpid()
    link = [nvcc, *ARCH, "-shared", "-o", tmp] + [obj for _, obj in jobs]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("link failed: " + " ".join(link))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv,
                extra=("-Xptxas", "-v") if "--ptxas" in sys.argv else ()))
