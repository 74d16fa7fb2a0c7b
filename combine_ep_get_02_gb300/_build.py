"""Build the CUDA library ``_lib/libep_get.so`` in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel; the result links the CUDA runtime
statically, so the library needs nothing but the driver at run time.
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIB_DIR, "libep_get.so")
# the same library with every computed row index checked against its buffer
# (-DEP_CHECKED): for tests; an index outside latches EP_ERR_BOUNDS
LIB_CHECKED = os.path.join(LIB_DIR, "libep_get_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC,
         "--expt-relaxed-constexpr"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    hdr = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hdr += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return sources() + hdr + [os.path.abspath(__file__)]


# translation unit that holds each kernel (and its launcher)
KERNEL_UNITS = {"layout_kernel": "layout.cu", "layout_rows_kernel": "layout.cu", "dispatch_kernel": "dispatch.cu",
                "dispatch_bulk_kernel": "dispatch_bulk.cu", "combine_kernel": "combine.cu"}


def kernel_sources(kernel: str) -> list:
    """The kernel's translation unit and the library headers it includes, recursively."""
    import re
    seen, stack = [], [os.path.join(CSRC, KERNEL_UNITS[kernel])]
    while stack:
        p = stack.pop()
        if p in seen:
            continue
        seen.append(p)
        for name in re.findall(r'#include\s+"([^"]+)"', open(p).read()):
            q = os.path.join(CSRC, name)
            if os.path.exists(q):
                stack.append(q)
    return sorted(seen)


def _code_only(text: str) -> str:
    """C/C++ source without comments and blank lines (what the compiler sees)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())


def source_hash(kernel: str = None) -> str:
    """Short hash of one kernel's code (its unit and the csrc headers it
    includes, comments left out), or of every source and header when no kernel
    is named."""
    import hashlib
    files = kernel_sources(kernel) if kernel else [p for p in sorted(_deps()) if p.endswith((".cu", ".cuh", ".h"))]
    h = hashlib.sha256()
    for p in files:
        h.update(os.path.basename(p).encode())
        h.update(_code_only(open(p).read()).encode())
    return h.hexdigest()[:16]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = False) -> str:
    lib = LIB_CHECKED if checked else LIB
    if not force and up_to_date(lib):
        return lib
    nvcc = _nvcc()
    obj_dir = os.path.join(LIB_DIR, "obj_checked" if checked else "obj")
    os.makedirs(obj_dir, exist_ok=True)
    if checked:
        extra_flags = (*extra_flags, "-DEP_CHECKED")

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    flags = [a for a in sys.argv[1:] if a.startswith("-X") or a.startswith("--")]
    print(build(force=True, verbose=True, extra_flags=flags))
