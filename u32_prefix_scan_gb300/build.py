"""Build libu32scan.so (the CUDA library) in-tree for sm_103a.

Each .cu under csrc/ is compiled to an object in parallel with nvcc, then
linked into u32_prefix_scan_gb300/libu32scan.so. The CUDA runtime is linked
statically, so the library needs only the driver at run time.
"""

from __future__ import annotations

import os
import pathlib
import shutil
import subprocess
import sys

PKG = pathlib.Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = ROOT / "_build"
SO = PKG / "libu32scan.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and pathlib.Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libu32scan.so")


def sources() -> list[pathlib.Path]:
    return sorted(CSRC.glob("*.cu"))


def _stale() -> bool:
    if not SO.exists():
        return True
    newest = max(p.stat().st_mtime for p in list(CSRC.iterdir()) + list(INCLUDE.glob("*.h")))
    return SO.stat().st_mtime < newest


def build(force: bool = False, verbose: bool = False) -> pathlib.Path:
    """Compile and link the library if any source is newer than it."""
    if not force and not _stale():
        return SO
    nvcc = _nvcc()
    BUILD.mkdir(exist_ok=True)
    procs = []
    for src in sources():
        obj = BUILD / (src.stem + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-c", str(src), "-o", str(obj)]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((src, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    objs, failed = [], []
    for src, obj, p in procs:
        out = p.communicate()[0].decode()
        if verbose or p.returncode:
            sys.stderr.write(out)
        (failed if p.returncode else objs).append(src if p.returncode else obj)
    if failed:
        raise RuntimeError(f"nvcc failed on {[f.name for f in failed]}")
    tmp = SO.with_name(f"{SO.name}.tmp{os.getpid()}")
    subprocess.check_call([nvcc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs)])
    os.replace(tmp, SO)
    return SO


def build_variant(tag: str, defines: list[str], verbose: bool = False) -> pathlib.Path:
    """Compile the library with extra preprocessor definitions (other launch
    shapes: the U32SCAN_* macros of the kernel files) into
    _build/variants/<tag>/libu32scan.so, if its sources or definitions
    changed since the last build. For tests that compare launch shapes; the
    package itself always loads the default library."""
    out = BUILD / "variants" / tag
    so = out / SO.name
    stamp = out / "defines.txt"
    want = " ".join(defines)
    if so.exists() and stamp.exists() and stamp.read_text() == want:
        newest = max(p.stat().st_mtime for p in list(CSRC.iterdir()) + list(INCLUDE.glob("*.h")))
        if so.stat().st_mtime >= newest:
            return so
    nvcc = _nvcc()
    out.mkdir(parents=True, exist_ok=True)
    procs = []
    for src in sources():
        obj = out / (src.stem + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *defines, "-c", str(src), "-o", str(obj)]
        procs.append((src, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    objs = []
    for src, obj, p in procs:
        text = p.communicate()[0].decode()
        if verbose or p.returncode:
            sys.stderr.write(text)
        if p.returncode:
            raise RuntimeError(f"nvcc failed on {src.name} with {defines}")
        objs.append(obj)
    tmp = so.with_name(f"{so.name}.tmp{os.getpid()}")
    subprocess.check_call([nvcc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs)])
    os.replace(tmp, so)
    stamp.write_text(want)
    return so


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(SO)
