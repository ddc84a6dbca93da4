"""Build the in-tree CUDA libraries with nvcc for sm_103a.

``libvpce.so``       the vocab-parallel cross-entropy C ABI (include/vpce.h)
``libvpce_synth.so`` the device twin of the seeded input generator

Each translation unit compiles in parallel; the results go to
``vocab_sharded_lm_gb300/_lib/`` (git-ignored).  Rebuilds only what changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "_lib")
OBJDIR = os.path.join(PKG, "_lib", "obj")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]

LIBS = {
    "libvpce.so": ["vpce_api.cu", "vpce_forward.cu", "vpce_backward.cu", "vpce_fused.cu", "vpce_static.cu",
                   "vpce_gemm.cu", "vpce_gemm_bwd.cu", "vpce_embed.cu", "vpce_lmhead_bwd.cu"],
    "libvpce_synth.so": ["synth_gen.cu"],
}
HEADERS = ["vpce_device.cuh", "vpce_kernels.cuh", "vpce_chunk.cuh", "vpce_tc.cuh"]
LINK: dict[str, list[str]] = {}


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _mtime(paths) -> float:
    return max(os.path.getmtime(p) for p in paths)


def _compile(nvcc: str, src: str, obj: str, deps) -> tuple[str, str]:
    if os.path.exists(obj) and os.path.getmtime(obj) >= _mtime([src] + deps):
        return obj, ""
    cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose: bool = False) -> dict:
    """Compile every library; returns {library name: path}."""
    nvcc = _nvcc()
    os.makedirs(OBJDIR, exist_ok=True)
    deps = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "vpce.h")]
    jobs = {}
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        for lib, srcs in LIBS.items():
            for s in srcs:
                src = os.path.join(CSRC, s)
                obj = os.path.join(OBJDIR, s.replace(".cu", ".o"))
                jobs[(lib, s)] = ex.submit(_compile, nvcc, src, obj, deps)
        logs = {k: f.result() for k, f in jobs.items()}
    if verbose:
        for (lib, s), (_, log) in logs.items():
            if log:
                sys.stderr.write(f"--- {s}\n{log}")
    out = {}
    cudalib = _cuda_lib_dir(nvcc)
    for lib, srcs in LIBS.items():
        objs = [logs[(lib, s)][0] for s in srcs]
        target = os.path.join(LIBDIR, lib)
        if not (os.path.exists(target) and os.path.getmtime(target) >= _mtime(objs)):
            tmp = target + ".tmp"
            cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
                   "-Xlinker", f"-rpath,{cudalib}"] + LINK.get(lib, [])
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed for {lib}:\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, target)
        out[lib] = target
    return out


if __name__ == "__main__":
    for k, v in build(verbose="-v" in sys.argv).items():
        print(k, v)
