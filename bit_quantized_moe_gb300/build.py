"""Build libqmv.so in-tree for sm_103a with nvcc.

    python bit_quantized_moe_gb300/build.py [--force] [--verbose-ptxas] [--phase-probe]

(run as a script or loaded by file path: importing the package itself needs
the built library).

Every translation unit under csrc/ is compiled in parallel to an object file
under _build/, then linked into _build/libqmv.so (CUDA runtime linked
as a shared library, so that it binds to the runtime PyTorch already loaded and
both agree on the current device). A unit is rebuilt
when it or any header in csrc/ or include/ is newer than its object.

--phase-probe builds the diagnostic variant (-DQMV_PHASE_PROBE: per-warp
%globaltimer stamps at the phases of each matvec launch) into
_build/probe/libqmv.so instead; the product library is never built with it.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libqmv.so")
PROBE_BUILD = os.path.join(BUILD, "probe")
PROBE_LIB = os.path.join(PROBE_BUILD, "libqmv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", CSRC, "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return found


def _sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _headers_mtime() -> float:
    m = 0.0
    for d in (CSRC, INCLUDE):
        for f in os.listdir(d):
            if f.endswith((".h", ".cuh")):
                m = max(m, os.path.getmtime(os.path.join(d, f)))
    return m


def _compile(src: str, force: bool, verbose_ptxas: bool, out_dir: str = BUILD,
             defines: tuple = ()) -> tuple[str, str]:
    path = os.path.join(CSRC, src)
    obj = os.path.join(out_dir, src + ".o")
    if (not force and os.path.exists(obj)
            and os.path.getmtime(obj) >= max(os.path.getmtime(path), _headers_mtime())):
        return obj, ""
    cmd = [nvcc(), *ARCH, *COMMON, *defines, "-c", path, "-o", obj]
    if verbose_ptxas and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None,
          phase_probe: bool = False) -> str:
    out_dir = PROBE_BUILD if phase_probe else BUILD
    lib = PROBE_LIB if phase_probe else LIB
    defines = ("-DQMV_PHASE_PROBE",) if phase_probe else ()
    os.makedirs(out_dir, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=jobs or min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, force, verbose_ptxas, out_dir, defines), srcs))
    objs = [o for o, _ in results]
    if verbose_ptxas:
        for (o, log), s in zip(results, srcs):
            if log:
                sys.stderr.write(f"--- {s}\n{log}")
    if (force or not os.path.exists(lib)
            or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs)):
        tmp = lib + ".tmp"
        libdir = os.path.join(os.path.dirname(os.path.dirname(nvcc())), "lib64")
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "shared",
               "-Xlinker", f"-rpath,{libdir}"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("--phase-probe", action="store_true")
    args = ap.parse_args(argv)
    print(build(force=args.force, verbose_ptxas=args.verbose_ptxas, phase_probe=args.phase_probe))
    return 0


if __name__ == "__main__":
    sys.exit(main())
