"""Build libspecverify.so in place (nvcc, sm_103a only, one -gencode).

The four translation units compile in parallel into ``_build/`` beside the
package and link into ``libspecverify.so`` next to this file.  A rebuild
happens only when a source or header is newer than the library.
"""
from __future__ import annotations

import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(HERE, "libspecverify.so")

SOURCES = ["sv_api.cu", "sv_attention.cu", "sv_attention_tc.cu", "sv_vocab.cu", "sv_compact.cu",
           "sv_noalloc.cu", "sv_step.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", f"-I{INCLUDE}"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _inputs():
    return ([os.path.join(CSRC, s) for s in SOURCES] + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, defines=(), lib_path: str = LIB_PATH,
          build_dir: str = BUILD_DIR) -> str:
    """Compile the library; `defines` (e.g. SV_PHASE_STAMPS) go to every
    translation unit, for a diagnostic build at another `lib_path`."""
    if not force and up_to_date(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *[f"-D{d}" for d in defines], "-c",
               os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            print(out.decode(errors="replace"))
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = lib_path + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, "-shared", *ARCH, *objs, "-o", tmp])
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB_PATH)
