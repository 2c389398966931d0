"""Build libkvattn.so in-tree for sm_103a with nvcc (no cmake, no torch).

Every translation unit is compiled in parallel into ``_build/`` and linked
into ``continuous_batching_kv_gb300/libkvattn.so`` with the static CUDA
runtime, so the library loads on a machine without a GPU (its host-side
calls work there; device calls return an error).

    python continuous_batching_kv_gb300/build.py [--force] [--verbose]

(run as a script: importing the package first would look for the library).
"""

import argparse
import concurrent.futures as cf
import os
import re
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libkvattn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def nvcc():
    p = os.path.join(CUDA_HOME, "bin", "nvcc")
    return p if os.path.exists(p) else (shutil.which("nvcc") or "nvcc")


def sources():
    out = []
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cpp")):
            out.append(os.path.join(CSRC, f))
    return out


def headers():
    hs = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs


# Kernels that split their registers between warpgroups (setmaxnreg): the split
# in the source assumes this launch register count per thread, and an increase
# beyond what the launch holds would wait forever, so the build refuses any
# other count.
REG_SPLIT = {"k_prefill.cu": ("k_prefill", 168)}


def _check_regs(src, log):
    name, want = REG_SPLIT[os.path.basename(src)]
    lines = log.splitlines()
    for i, line in enumerate(lines):
        if "Compiling entry function" in line and name in line:
            for nxt in lines[i + 1:i + 6]:
                m = re.search(r"Used (\d+) registers", nxt)
                if m:
                    if int(m.group(1)) != want:
                        raise RuntimeError("%s: ptxas allocated %s registers per thread, the register split "
                                           "assumes %d" % (name, m.group(1), want))
                    return
    raise RuntimeError("%s: no ptxas register count found for %s" % (src, name))


def _compile(src, verbose):
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
    check = os.path.basename(src) in REG_SPLIT
    if src.endswith(".cu") and (verbose or check):
        cmd[1:1] = ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    if check:
        _check_regs(src, r.stderr)
    return obj, r.stderr


def build(force=False, verbose=False):
    """Compile and link libkvattn.so; skip when it is newer than every source."""
    srcs = sources()
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(p) for p in srcs + headers() + [__file__])
        if os.path.getmtime(LIB) >= newest:
            return LIB
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose), srcs))
    if verbose:
        for obj, log in results:
            if log.strip():
                sys.stderr.write(log)
    objs = [o for o, _ in results]
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose))
