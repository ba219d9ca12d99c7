"""Build libspecverify.so (the C-ABI CUDA library) in-tree for sm_103a.

Each translation unit under ``csrc/`` is compiled by nvcc in parallel, then
linked into ``draft_verify_acceptance_gb300/libspecverify.so``.  Register and
shared-memory usage reported by ptxas is written to ``_build/ptxas.log``.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libspecverify.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["spec_verify.cu", "verify_greedy.cu", "verify_sample.cu", "verify_sample_fused.cu", "verify_sample_seq.cu", "verify_sample_ee.cu", "verify_sample_2p.cu", "verify_draft_sample.cu", "verify_scd.cu", "rejection_cut.cu",
           "spec_verify_static.cu"]


def _nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecverify.so")
    return exe


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "spec_verify.h"))
    files.append(os.path.abspath(__file__))
    return files


LIB_DEBUG = os.path.join(HERE, "libspecverify_debug.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")


def _stale(lib):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile and link the library if any source is newer than it.

    debug=True builds the test variant libspecverify_debug.so with
    -DSPEC_DEBUG: the kernels' index checks skip an out-of-range global access
    and report SPEC_DEBUG_BOUNDS in the status word instead of faulting.  The
    same optional flag SPEC_NVTX (environment variable SPEC_NVTX=1 at build
    time) wraps every entry point in an NVTX range."""
    lib, bdir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    if not force and not _stale(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    wanted = {src.replace(".cu", ".o") for src in SOURCES}
    for f in os.listdir(bdir):  # objects of sources no longer in the library
        if f.endswith(".o") and f not in wanted:
            os.remove(os.path.join(bdir, f))
    nvcc = _nvcc()
    common = [nvcc, "-std=c++17", "-O3", *ARCH, "-lineinfo", "-Xptxas", "-v",
              "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", os.path.join(ROOT, "include")]
    if debug:
        common.append("-DSPEC_DEBUG")
    if os.environ.get("SPEC_NVTX") == "1":
        common.append("-DSPEC_NVTX")

    def compile_one(src):
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        r = subprocess.run(common + ["-c", os.path.join(CSRC, src), "-o", obj],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    with open(os.path.join(bdir, "ptxas.log"), "w") as f:
        for _, log in results:
            f.write(log)
    tmp = lib + ".tmp"
    r = subprocess.run([nvcc, "-shared", *ARCH, "-o", tmp] + [o for o, _ in results],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print(open(os.path.join(bdir, "ptxas.log")).read())
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
