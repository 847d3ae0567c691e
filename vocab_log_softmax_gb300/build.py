"""Builds libvls.so (the CUDA kernels and their C ABI) in-tree for sm_103a.

    python -m vocab_log_softmax_gb300.build [--force] [--jobs N]

Each ``csrc/*.cu`` translation unit is compiled by nvcc in parallel, then
linked into ``vocab_log_softmax_gb300/lib/libvls.so`` with the CUDA runtime
linked statically, so the library needs no ``libcudart`` at load time.

The same objects also make ``lib/libvls_test.so``, the test build: only the
C layer (``api.cu``) is compiled a second time, with ``VLS_TEST_HOOKS``, which
adds the hooks of ``include/vls_test.h`` (injected host-side failures, a
shorter wait limit for the tensor-core kernels, other launch geometries).
The kernels are the same objects in both libraries.
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
LIB_DIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIB_DIR, "libvls.so")
TEST_LIB = os.path.join(LIB_DIR, "libvls_test.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
    "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC,
]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libvls")
    return path


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def headers() -> list[str]:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]


def _newest(paths) -> float:
    return max(os.path.getmtime(p) for p in paths)


def _compile(src: str, extra: list[str], suffix: str = "") -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + suffix + ".o")
    cmd = [nvcc()] + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj


def _link(objs: list[str], out: str) -> None:
    tmp = out + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)


def build(force: bool = False, jobs: int | None = None, extra: list[str] | None = None,
          verbose: bool = False) -> str:
    """Compiles and links libvls.so and libvls_test.so if any source is newer
    than them; returns the path of libvls.so."""
    srcs = sources()
    newest = _newest(srcs + headers())
    if (not force and all(os.path.exists(p) and os.path.getmtime(p) >= newest for p in (LIB, TEST_LIB))):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    api = os.path.join(CSRC, "api.cu")
    jobs = jobs or min(len(srcs) + 1, os.cpu_count() or 4)
    extra = list(extra or [])
    units = [(s, extra, "") for s in srcs] + [(api, extra + ["-DVLS_TEST_HOOKS"], ".test")]
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda u: _compile(*u), units))
    product, test_api = objs[:-1], objs[-1]
    _link(product, LIB)
    _link([test_api if o.endswith("api.cu.o") else o for o in product], TEST_LIB)
    if verbose:
        print(f"built {LIB} and {TEST_LIB}", file=sys.stderr)
    return LIB


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--jobs", type=int, default=None)
    ap.add_argument("--ptxas-verbose", action="store_true", help="print registers / spills per kernel")
    args = ap.parse_args()
    extra = ["-Xptxas", "-v"] if args.ptxas_verbose else []
    if args.ptxas_verbose:
        # ptxas -v goes to stderr of each nvcc call; run serially to keep it readable
        os.makedirs(BUILD, exist_ok=True)
        for s in sources():
            cmd = [nvcc()] + NVCC_FLAGS + extra + ["-c", s, "-o", os.path.join(BUILD, os.path.basename(s) + ".o")]
            r = subprocess.run(cmd, capture_output=True, text=True)
            print(r.stderr)
            if r.returncode:
                sys.exit(r.returncode)
    print(build(force=args.force, jobs=args.jobs, verbose=True))


if __name__ == "__main__":
    main()
