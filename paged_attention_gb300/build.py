"""Build the C-ABI shared library for sm_103a (nvcc, in-tree).

Every ``csrc/*.cu`` file is compiled in parallel with
``-gencode arch=compute_103a,code=sm_103a -lineinfo`` and linked into
``paged_attention_gb300/_build/libpa_gb300.so`` (CUDA runtime linked
statically; the driver API is reached through cudaGetDriverEntryPoint).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import re
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libpa_gb300.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-I", INCLUDE, "-I", CSRC]


# Kernels that move registers between warpgroups with setmaxnreg: the block
# must be launched with exactly this many registers per thread, or the
# warpgroups' requests would not add up to what the block holds and
# setmaxnreg.inc could wait forever.  Checked on every build from ptxas -v.
REGISTER_BUDGETS = {"pa_prefill.cu": ("prefill_kernel", 168),
                    "pa_decode_fp8.cu": ("decode_fp8_kernel", 168)}


def check_register_budget(src: str, ptxas_log: str) -> None:
    kernel, want = REGISTER_BUDGETS[src]
    current = None
    seen = 0
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and current and kernel in current:
            seen += 1
            if int(m.group(1)) != want:
                raise RuntimeError(f"{current}: ptxas allocated {m.group(1)} registers, the "
                                   f"setmaxnreg split assumes {want}")
    if seen == 0:
        raise RuntimeError(f"{src}: no ptxas register report for {kernel}")


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path:
        return path
    for cand in ("/usr/local/cuda/bin/nvcc",):
        if os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _fingerprint() -> str:
    h = hashlib.sha256()
    files = _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [
        os.path.join(INCLUDE, "pa.h"), os.path.abspath(__file__)]
    for f in files:
        with open(f, "rb") as fh:
            h.update(f.encode() + fh.read())
    h.update(" ".join(ARCH + NVCC_FLAGS).encode())
    return h.hexdigest()


# Sources that decide what one kernel does on the device (its own file, the
# shared device helpers, the launcher / tensor-map code and the ABI header).
KERNEL_SOURCES = {
    "pa_decode_splitk": ("pa_decode.cu", "pa_decode_fp8.cu", "pa_decode_fp8_tc.cu",
                         "pa_decode_common.cuh"),
    # pa_prefill also runs the decode kernel on the decode part of a mixed batch
    "pa_prefill": ("pa_prefill.cu", "pa_decode.cu", "pa_decode_common.cuh"),
}


def _code_only(text: str) -> str:
    """C/C++ source without comments or blank-line and trailing-space noise."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif text[i] in "\"'":
            q, j = text[i], i + 1
            while j < n and text[j] != q:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    lines = [ln.rstrip() for ln in "".join(out).splitlines()]
    return "\n".join(ln for ln in lines if ln)


def kernel_fingerprint(kernel: str) -> str:
    """Short hash of the code (comments stripped) of one entry point's kernel
    sources; stored beside counters taken from that kernel so stale counters
    can be recognised, while a comment edit keeps them valid."""
    h = hashlib.sha256()
    files = [os.path.join(CSRC, f) for f in KERNEL_SOURCES[kernel]] + [
        os.path.join(CSRC, "pa_internal.cuh"), os.path.join(CSRC, "pa_api.cu"),
        os.path.join(INCLUDE, "pa.h")]
    for f in files:
        with open(f, encoding="utf-8") as fh:
            h.update(os.path.basename(f).encode() + _code_only(fh.read()).encode())
    h.update(" ".join(ARCH + NVCC_FLAGS[:4]).encode())
    return h.hexdigest()[:16]


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    """Compile and link the library; returns its path.  Skips work when the
    sources are unchanged since the last build."""
    os.makedirs(OUT_DIR, exist_ok=True)
    stamp = os.path.join(OUT_DIR, "stamp.txt")
    fp = _fingerprint() + " ".join(extra_flags or [])
    if not force and os.path.exists(LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read() == fp:
                return LIB_PATH
    cc = nvcc()
    flags = ARCH + NVCC_FLAGS + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(OUT_DIR, os.path.basename(src) + ".o")
        extra = ["-Xptxas", "-v"] if os.path.basename(src) in REGISTER_BUDGETS else []
        cmd = [cc, *flags, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if extra:
            check_register_budget(os.path.basename(src), r.stdout + r.stderr)
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(stamp, "w") as f:
        f.write(fp)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
