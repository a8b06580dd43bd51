"""Build the ekv shared library (csrc/*.cu -> libekv.so) in tree with nvcc for sm_103a.

No CMake: each translation unit is compiled in parallel, then linked with the static
CUDA runtime. The result is written atomically next to this file.

A second library, libekv_waittest.so, is built beside it for the tests only: the
decode translation units compiled with EKV_TEST_WAIT_TIMEOUT (a 5 ms bound on the
pipeline waits and an entry point that makes one wait run out), linked with the other
objects of the production build. Nothing but the tests loads it.
"""

import concurrent.futures
import os
import shutil
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libekv.so")
TEST_LIB = os.path.join(HERE, "libekv_waittest.so")
SOURCES = ["ekv_api.cu", "decode_simt.cu", "decode_mma.cu", "gather_demote.cu", "noalloc.cu", "prefill_mma.cu", "prefill_tc05.cu"]
# translation units that see DecodeParams or the wait bound: rebuilt for the test library
TEST_SOURCES = ["ekv_api.cu", "decode_simt.cu", "decode_mma.cu", "noalloc.cu"]
TEST_DEFINE = "-DEKV_TEST_WAIT_TIMEOUT"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the ekv CUDA library cannot be built")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))]
    return files + [os.path.join(INCLUDE, "ekv.h"), os.path.abspath(__file__)]


def up_to_date():
    for lib in (LIB, TEST_LIB):
        if not os.path.exists(lib):
            return False
        t = os.path.getmtime(lib)
        if not all(os.path.getmtime(f) <= t for f in _inputs()):
            return False
    return True


def _link(cc, objs, lib):
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=HERE)
    os.close(fd)
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        os.unlink(tmp)
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)


def build(force=False, verbose=False, ptxas_info=False):
    """Compile and link libekv.so and the tests' libekv_waittest.so; returns libekv.so's path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(job):
        src, test = job
        obj = os.path.join(BUILD_DIR, src.replace(".cu", "_waittest.o" if test else ".o"))
        cmd = [cc] + FLAGS + extra + ([TEST_DEFINE] if test else []) + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}{' (test build)' if test else ''}:\n{r.stderr}")
        return obj, r.stderr

    jobs = [(s, False) for s in SOURCES] + [(s, True) for s in TEST_SOURCES]
    # the largest translation units first, so the pool is not left waiting on one of them
    jobs.sort(key=lambda j: -os.path.getsize(os.path.join(CSRC, j[0])))
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        results = dict(zip(jobs, ex.map(compile_one, jobs)))
    if verbose or ptxas_info:
        for (src, test), (_, log) in results.items():
            if log and not test:
                sys.stderr.write(log)
    _link(cc, [results[(s, False)][0] for s in SOURCES], LIB)
    _link(cc, [results[(s, s in TEST_SOURCES)][0] for s in SOURCES], TEST_LIB)
    return LIB


def ensure_built():
    return build(force=False)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
