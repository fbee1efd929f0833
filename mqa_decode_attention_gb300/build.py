"""Build libmqa_decode.so in-tree with nvcc for sm_103a.

Each .cu file is compiled in parallel to an object, then the objects are
linked into ``mqa_decode_attention_gb300/lib/libmqa_decode.so``. Extra nvcc
flags (for instance ``-DMQA_MMA_STAGES_D128=4``) can be passed in
``extra_flags``; ``out_dir`` lets a tuning build go elsewhere.
"""

from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG_DIR, "lib")
LIB_NAME = "libmqa_decode.so"
SOURCES = ["abi.cu", "append_rope.cu", "combine.cu", "decode_fma.cu", "decode_mma.cu", "decode_mma_paged.cu", "decode_mma_u8.cu",
           "noalloc.cu", "attn_tc05.cu", "attn_tc05_keys.cu", "attn_tc05_widen.cu",
           "attn_tc05_prefill.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-diag-suppress", "177"]


def nvcc() -> str:
    cand = [os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc"), shutil.which("nvcc")]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def lib_path(out_dir: str | None = None) -> str:
    return os.path.join(out_dir or LIB_DIR, LIB_NAME)


def build(verbose: bool = False, extra_flags: list[str] | None = None, out_dir: str | None = None,
          ptxas_verbose: bool = False) -> str:
    out_dir = out_dir or LIB_DIR
    obj_dir = os.path.join(out_dir, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    extra = list(extra_flags or [])
    if ptxas_verbose:
        extra += ["-Xptxas", "-v"]
    cc = nvcc()

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, *extra, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            if log.strip():
                print(log)
    out = lib_path(out_dir)
    tmp = out + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import sys

    print(build(verbose=True, ptxas_verbose="-v" in sys.argv))
