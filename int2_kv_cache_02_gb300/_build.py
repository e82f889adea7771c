"""In-tree build of liboscar.so and liboscar_synth.so for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into a
shared library next to this file (the CUDA runtime is linked statically).
A library is rebuilt only when a source or header is newer than it.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")

LIBS = {
    "liboscar.so": ["rotate.cu", "quantize.cu", "decode_int2.cu", "decode_int2_pad.cu", "decode_bf16.cu",
                    "combine.cu", "api.cu", "decode_static.cu"],
    "liboscar_synth.so": ["synth.cu"],
}
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: liboscar cannot be built")


def _deps() -> list[str]:
    out = []
    for d in (CSRC, INCLUDE):
        for f in os.listdir(d):
            if f.endswith((".h", ".cuh", ".cu")):
                out.append(os.path.join(d, f))
    return out


def lib_path(name: str = "liboscar.so") -> str:
    return os.path.join(PKG, name)


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False) -> dict[str, str]:
    """Builds both libraries if stale; returns {library: path}."""
    os.makedirs(BUILD, exist_ok=True)
    deps = _deps()
    paths = {}
    for lib, srcs in LIBS.items():
        target = lib_path(lib)
        paths[lib] = target
        if not force and not _stale(target, deps):
            continue
        with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
            results = list(ex.map(_compile, srcs))
        with open(os.path.join(BUILD, lib + ".ptxas.log"), "w") as f:
            for (obj, log), src in zip(results, srcs):
                f.write(f"== {src}\n{log}\n")
        tmp = target + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {lib} failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, target)
        if verbose:
            print(f"built {target}", file=sys.stderr)
    return paths


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
