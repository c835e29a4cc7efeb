"""Build libdsample.so in-tree for sm_103a with nvcc (no CMake, no torch extension).

The Gumbel bound table is generated first, then each translation unit is
compiled in parallel and linked into vocab_wide_logit_gb300/_build/libdsample.so.
"""
import concurrent.futures
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libdsample.so")
INCLUDE = os.path.join(ROOT, "include")
SOURCES = ["ds_api.cu", "k_greedy.cu", "k_sample_warp.cu", "k_sample_cluster.cu", "k_sample_stream.cu",
           "k_merge.cu", "k_reveal.cu", "k_log_softmax.cu"]
HEADERS = ["ds_device.cuh", "ds_sample_common.cuh", "ds_warp_common.cuh", "ds_launch.h", "gen_gumbel_bounds.py"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    table = os.path.join(OUT, "gumbel_bounds.inc")
    gen = os.path.join(CSRC, "gen_gumbel_bounds.py")
    if force or _stale(table, [gen]):
        subprocess.run([sys.executable, gen, table], check=True)
    common = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "dsample.h"), table,
                                                        os.path.abspath(__file__)]
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                    "-I", OUT, "--expt-relaxed-constexpr"]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OUT, src.replace(".cu", ".o"))
        if force or ptxas_verbose or _stale(o, [s] + common):
            jobs.append([nvcc()] + flags + ["-c", s, "-o", o])
    if jobs:
        with concurrent.futures.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
        for cmd, r in zip(jobs, results):
            if verbose or ptxas_verbose or r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed: " + " ".join(cmd))
    objs = [os.path.join(OUT, s.replace(".cu", ".o")) for s in SOURCES]
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + ".tmp%d" % os.getpid()
        subprocess.run([nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"], check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="--ptxas" in sys.argv))
