"""Build libarnorm.so (the CUDA kernels and the C ABI) for sm_103a, in tree.

Each .cu file compiles to an object in parallel; the objects link into
``allreduce_sum_residual_gb300/libarnorm.so``.  Only nvcc is needed (no
cmake); the same command works on x86_64 and aarch64 hosts.
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libarnorm.so")
# The checking build: the same sources with device-side bounds checks
# compiled in (AR_CHECK=1); a failed check records AR_ERR_BOUNDS in the
# device status word and skips the access.  For tests, not for production.
CHECK_OBJ_DIR = os.path.join(PKG, "_build_check")
CHECK_LIB = os.path.join(PKG, "libarnorm_check.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "-Xptxas", "-warn-spills", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libarnorm.so")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), check: bool = False) -> str:
    """Compile and link libarnorm.so (with ``check``: libarnorm_check.so, the
    checking build) unless it is newer than every source."""
    lib_path, obj_dir = (CHECK_LIB, CHECK_OBJ_DIR) if check else (LIB, OBJ_DIR)
    extra_flags = tuple(extra_flags) + (("-DAR_CHECK=1",) if check else ())
    if not force and up_to_date(lib_path):
        return lib_path
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + f".tmp{os.getpid()}"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {os.path.basename(lib_path)} failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv, check="--check" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "-v" in sys.argv else []))
