"""Build the C-ABI library ``_lib/libea.so`` for sm_103a with nvcc.

Translation units are compiled in parallel, then linked into one shared library
(CUDA runtime linked statically; the driver's tensor-map encoder is looked up at
run time, so the library loads on a machine without a GPU driver).

``build(checked=True)`` builds the bounds-checked variant ``_lib/libea_checked.so``
(``-DEA_CHECKS``: every global access whose index depends on data or on the work
decomposition is tested first and reported in the workspace error word instead
of being made), which the tests run in place of a memory checker.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libea.so")
CHECKED_LIB = os.path.join(OUT_DIR, "libea_checked.so")
ROOT = os.path.dirname(HERE)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "nvcc")
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + os.path.join(ROOT, "include")]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _deps():
    inc = os.path.join(ROOT, "include")
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(inc, f) for f in os.listdir(inc)]


def _compile(src, extra, obj_dir=OUT_DIR):
    obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
    cmd = [NVCC] + ARCH + COMMON + extra + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False, extra=None, checked: bool = False) -> str:
    """Compile every source under csrc/ and link libea.so (libea_checked.so with
    checked=True); returns its path."""
    lib = CHECKED_LIB if checked else LIB
    obj_dir = os.path.join(OUT_DIR, "checked") if checked else OUT_DIR
    os.makedirs(obj_dir, exist_ok=True)
    newest = max(os.path.getmtime(p) for p in _deps())
    if not force and extra is None and os.path.exists(lib) and os.path.getmtime(lib) >= newest:
        return lib
    extra = list(extra or []) + (["-DEA_CHECKS"] if checked else [])
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(lambda s: _compile(s, extra, obj_dir), srcs))
    if verbose:
        for (obj, err) in results:
            if err.strip():
                print(err)
    objs = [o for o, _ in results]
    tmp = lib + ".tmp.%d" % os.getpid()
    cmd = [NVCC] + ARCH + ["-shared", "-Xcompiler", "-fPIC", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    extra = ["-Xptxas", "-v"] if "-v" in sys.argv else None
    print(build(force=True, verbose=True, extra=extra))
