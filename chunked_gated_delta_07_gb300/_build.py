"""Builds libgdr.so in-tree from csrc/*.cu with nvcc for sm_103a only.

Each translation unit compiles in its own nvcc process (in parallel) into
``_build/``; the shared library is linked next to this file.  A unit is
recompiled only when it or a header is newer than its object.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build", "gdr")
LIB = os.path.join(HERE, "libgdr.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdr.so")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


# Checking builds, each into its own directory and library:
#   debug: device-side index checks (GDR_DEBUG); a failed one is reported by
#          gdr_get_status as GDR_ERR_BOUNDS instead of touching memory
#   asan:  the host code under AddressSanitizer and UndefinedBehaviorSanitizer (load
#          it in a process that preloads the sanitizer runtimes)
VARIANTS = {
    "debug": ["-DGDR_DEBUG"],
    "asan": ["-Xcompiler", "-fsanitize=address", "-Xcompiler", "-fsanitize=undefined",
             "-Xcompiler", "-fno-omit-frame-pointer", "-Xcompiler", "-fno-sanitize-recover=undefined", "-g"],
}


def variant_lib(variant: str) -> str:
    return os.path.join(HERE, f"libgdr_{variant}.so")


def build(verbose: bool = False, extra_flags: list[str] | None = None,
          variant: str | None = None) -> str:
    if variant is not None:
        return _build_into(os.path.join(ROOT, "_build", f"gdr_{variant}"), variant_lib(variant),
                           VARIANTS[variant], ["-Xcompiler", "-fsanitize=address", "-Xcompiler", "-fsanitize=undefined"]
                           if variant == "asan" else [], verbose)
    return _build_into(BUILD, LIB, list(extra_flags or []), [], verbose, force=bool(extra_flags))


def _build_into(build_dir, lib, extra, link_extra, verbose, force=False):
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr_mtime = max([os.path.getmtime(h) for h in _headers()] + [0.0])
    flags = NVCC_FLAGS + ARCH + extra
    procs, objs = [], []
    for src in srcs:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if (os.path.exists(obj) and os.path.getmtime(obj) >= os.path.getmtime(src)
                and os.path.getmtime(obj) >= hdr_mtime and not force):
            continue
        cmd = [nvcc(), "-c", src, "-o", obj] + flags
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"), flush=True)
    if failed:
        msg = "\n".join(f"--- {s}\n{o}" for s, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    if (procs or not os.path.exists(lib)
            or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs)):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"] + link_extra
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True))
