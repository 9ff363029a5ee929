"""Builds libpsgd.so in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in its own nvcc process, in parallel, then
linked into one shared library.  Used by ``__graft_entry__.build()``.

Whether to rebuild is decided by content, not by file times: a SHA-256 over
every source file, the public header, this script, the compiler flags and
``nvcc --version`` is compiled into the library (``psgd_build_id()``), and an
existing ``libpsgd.so`` is reused only when it carries that exact hash and was
built for this machine's architecture.  ``-Xptxas -v`` register, spill and
shared-memory lines of every kernel are written to ``_build/ptxas.log``.
"""

from __future__ import annotations

import concurrent.futures
import hashlib
import os
import platform
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpsgd.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
PTXAS_LOG = os.path.join(BUILD, "ptxas.log")

SOURCES = ["psgd_api.cu", "psgd_misc.cu", "psgd_static.cu", "psgd_group.cu"] + \
          [f"kern_rp{r}.cu" for r in (1, 2, 4, 8, 16, 32)]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v", "-I", INCLUDE]
HASH_MARKER = b"psgd-source-hash:"

# ELF e_machine of the machines this builds on
_ELF_MACHINE = {"x86_64": 62, "aarch64": 183, "arm64": 183}


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libpsgd.so")
    return cand


def source_hash() -> str:
    """SHA-256 (hex, 32 chars) of everything the library is built from."""
    h = hashlib.sha256()
    for f in sorted(os.listdir(CSRC)):
        path = os.path.join(CSRC, f)
        if os.path.isfile(path):
            h.update(f.encode() + b"\0")
            with open(path, "rb") as fh:
                h.update(fh.read())
    for path in (os.path.join(INCLUDE, "psgd.h"), os.path.abspath(__file__)):
        with open(path, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(ARCH + FLAGS + SOURCES).encode())
    try:
        h.update(subprocess.run([_nvcc(), "--version"], capture_output=True, text=True).stdout.encode())
    except Exception:
        h.update(b"nvcc-unknown")
    return h.hexdigest()[:32]


def library_hash(path: str = LIB):
    """The source hash compiled into an existing library file, or None when it
    is missing, has none, or was built for another architecture."""
    try:
        with open(path, "rb") as fh:
            data = fh.read()
    except OSError:
        return None
    if len(data) < 20 or data[:4] != b"\x7fELF":
        return None
    want = _ELF_MACHINE.get(platform.machine())
    got = int.from_bytes(data[18:20], "little")
    if want is not None and got != want:
        return None
    i = data.find(HASH_MARKER)
    if i < 0:
        return None
    j = i + len(HASH_MARKER)
    return data[j:j + 32].decode("ascii", "replace")


def build(force: bool = False, verbose: bool = False) -> str:
    want = source_hash()
    if not force and library_hash() == want:
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        extra = [f'-DPSGD_SOURCE_HASH="{want}"'] if src == "psgd_api.cu" else []
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        return src, r.stderr

    workers = min(len(SOURCES), max(1, os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        results = list(ex.map(compile_one, SOURCES))
    with open(PTXAS_LOG, "w") as log:
        log.write(f"source hash {want}\n")
        for src, err in results:
            log.write(f"==== {src}\n{err}")
    if verbose:
        for src, err in results:
            spills = [ln for ln in err.splitlines() if "spill" in ln and not ln.strip().startswith("0 bytes")]
            bad = [ln for ln in spills if " 0 bytes spill stores, 0 bytes spill loads" not in ln]
            if bad:
                print(f"{src}: " + "\n".join(bad), file=sys.stderr)
    objs = [os.path.join(BUILD, s.replace(".cu", ".o")) for s in SOURCES]
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    if library_hash() != want:
        raise RuntimeError("the built library does not carry its source hash")
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
