"""Build libsparse_lookup.so from csrc/*.cu with nvcc for sm_103a.

Each translation unit is compiled to an object in parallel, then the objects
are linked into one shared library next to this file (git-ignored).  The CUDA
runtime is linked statically so the library only needs the driver.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsparse_lookup.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hs + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in sources() + headers() + [__file__])


def common_flags(extra=()):
    return ARCH + ["-O3", "-std=c++17", "-lineinfo", "-I", INCLUDE, "-I", CSRC,
                   "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr"] + list(extra)


def build(force: bool = False, verbose: bool = False, extra=(), out: str = None) -> str:
    """Compile and link; `extra` adds nvcc flags, `out` writes the library
    elsewhere (objects then go to a build folder of their own)."""
    lib_path = out or LIB
    build_dir = BUILD if out is None else lib_path + ".objs"
    if out is None and not force and not is_stale():
        return LIB
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        cmd = [cc] + common_flags(extra) + ["-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        for obj, log in ex.map(compile_one, sources()):
            objs.append(obj)
            if verbose and log:
                print(log)
    tmp = lib_path + ".tmp.%d" % os.getpid()
    cmd = [cc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
