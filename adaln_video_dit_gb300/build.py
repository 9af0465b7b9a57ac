"""Build libadaln.so in-tree (sm_103a) with nvcc.

Each translation unit is compiled in parallel, then linked into one shared
library beside this file.  No cmake, no torch extension machinery: the
library exports a plain C ABI (include/adaln.h).
"""
import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libadaln.so")
LIB_TUNING = os.path.join(HERE, "libadaln_tuning.so")
SOURCES = ["api.cu", "fwd.cu", "bwd.cu", "host.cu", "noalloc.cu", "selftest.cu"]
HEADERS = ["common.cuh", "ring.cuh", "internal.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
              "-I" + os.path.join(ROOT, "include")]


def nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _deps():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "adaln.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale(lib):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force=False, verbose=False, ptxas_info=False, tuning=False):
    """Compile libadaln.so if missing or stale; return its path.

    tuning=True builds libadaln_tuning.so instead, with -DADALN_TUNING: that
    copy reads the launch-shape sweep variables ADALN_RING_KB,
    ADALN_CTAS_PER_SM and ADALN_FWD_SCHED.  The release library (and the
    binding, which loads only libadaln.so) reads no environment variable."""
    lib = LIB_TUNING if tuning else LIB
    if not force and not _stale(lib):
        return lib
    out_dir = OUT_DIR + ("_tuning" if tuning else "")
    os.makedirs(out_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if tuning:
        extra.append("-DADALN_TUNING")

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib



def _strip_comments(text):
    """C/C++ source without comments and blank-space differences (string and
    character literals kept), so that edits to comments keep the hash."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_hash():
    """sha256 over the CUDA sources and headers with comments removed
    (identifies a kernel build's code)."""
    import hashlib
    h = hashlib.sha256()
    for f in sorted(_deps()):
        if f.endswith(".py"):
            continue
        with open(f, encoding="utf-8") as fh:
            h.update(os.path.basename(f).encode())
            h.update(_strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]
if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                ptxas_info="--ptxas" in sys.argv, tuning="--tuning" in sys.argv))
