"""Build libdeltalog.so in-tree for sm_103a (GB300).

Each translation unit is compiled by nvcc in parallel; the shared library is
linked against the shared CUDA runtime so that it shares the process's runtime
(and primary context) with PyTorch.  Rebuilds only when a source or header is
newer than the library.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libdeltalog.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CU_SOURCES = ["replay_prep.cu", "append_decode.cu", "append_fused_ne8.cu", "append_fused_ne16.cu",
              "append_fused_ne32.cu", "eager_step.cu", "slot_ops.cu", "prefill.cu", "prefill_tc.cu", "capi.cu",
              "noalloc.cu"]
CPP_SOURCES = ["slot_table.cpp"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdeltalog")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "deltalog.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force=False, verbose=False):
    """Compile and link; returns the library path."""
    if not force and not _stale():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    common = ["-std=c++17", "-O3", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]
    jobs = []
    for src in CU_SOURCES:
        obj = os.path.join(OUT_DIR, src + ".o")
        jobs.append([nvcc] + common + ARCH + ["-lineinfo", "-c", os.path.join(CSRC, src), "-o", obj]
                    + (["-Xptxas", "-v"] if verbose else []))
    for src in CPP_SOURCES:
        obj = os.path.join(OUT_DIR, src + ".o")
        jobs.append([nvcc] + common + ["-x", "c++", "-c", os.path.join(CSRC, src), "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        return cmd, r.returncode, r.stdout

    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(run, jobs))
    failed = [(c, out) for c, rc, out in results if rc != 0]
    if verbose:
        for c, rc, out in results:
            sys.stdout.write(out)
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + out for c, out in failed)
        raise RuntimeError("libdeltalog build failed:\n" + msg)
    objs = [os.path.join(OUT_DIR, s + ".o") for s in CU_SOURCES + CPP_SOURCES]
    tmp = LIB + ".%d.tmp" % os.getpid()
    link = [nvcc, "-shared", "-cudart", "shared"] + ARCH + objs + ["-o", tmp]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("libdeltalog link failed:\n" + " ".join(link) + "\n" + r.stdout)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
