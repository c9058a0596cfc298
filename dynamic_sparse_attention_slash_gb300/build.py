"""Builds libmsa.so (the C-ABI library) in-tree with nvcc for sm_103a, and its
bounds-checking twin libmsa_checked.so (compiled with MSA_CHECKED: every index
the kernels read from index data is range-checked, and a bad one is reported
in the device status word instead of being used).

Translation units compile in parallel into ``_build/`` at the repository root;
the shared libraries are written next to this file.  A rebuild happens only
when a source or header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libmsa.so")
CHECKED_LIB_PATH = os.path.join(PKG_DIR, "libmsa_checked.so")

SOURCES = ["msa_api.cu", "estimate.cu", "topk.cu", "vs_index.cu", "bs_index.cu", "hip_index.cu",
           "prefill.cu", "prefill_tile.cu", "v_f16.cu", "static_scratch.cu", "kv_select.cu",
           "recall.cu", "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libmsa.so")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "msa.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib: str = None) -> bool:
    lib = lib or LIB_PATH
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _compile(job: tuple) -> tuple[str, str]:
    src, build_dir, extra = job
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _variants(checked: bool | None):
    """(library path, object folder, extra flags) of the builds asked for:
    checked None = both, False = the ordinary library, True = the checked one."""
    plain = (LIB_PATH, BUILD_DIR, [])
    chk = (CHECKED_LIB_PATH, os.path.join(BUILD_DIR, "checked"), ["-DMSA_CHECKED"])
    return {None: [plain, chk], False: [plain], True: [chk]}[checked]


def build(force: bool = False, verbose: bool = False, checked: bool | None = False) -> str:
    """Compiles every CUDA translation unit and links libmsa.so (checked=False),
    libmsa_checked.so (True) or both (None), all translation units of all
    variants in parallel; returns the path of the first library built."""
    todo = [v for v in _variants(checked) if force or not up_to_date(v[0])]
    if not todo:
        return _variants(checked)[0][0]
    jobs = []
    for lib, bdir, extra in todo:
        os.makedirs(bdir, exist_ok=True)
        jobs += [(src, bdir, extra) for src in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(_compile, jobs))
    if verbose:
        for _, log in results:
            print(log)
    for n, (lib, bdir, _) in enumerate(todo):
        part = results[n * len(SOURCES):(n + 1) * len(SOURCES)]
        with open(os.path.join(bdir, "ptxas.log"), "w") as f:
            for src, (_, log) in zip(SOURCES, part):
                f.write(f"==== {src}\n{log}\n")
        tmp = lib + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in part]]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return _variants(checked)[0][0]


if __name__ == "__main__":
    print(build(force=True, verbose=True, checked=None))
