"""Builds libquestsparse.so in-tree with nvcc for sm_103a.

Each translation unit compiles in its own process (in parallel); the objects
link into one shared library with the CUDA runtime linked statically, so the
library needs nothing beyond the NVIDIA driver at run time.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libquestsparse.so")
OBJDIR = os.path.join(HERE, "_build")
# (source, object name, defines): qs_probe.cu compiles once for its host
# part and once per (KV dtype, head size) pair of kernel variants
PROBE_VARIANTS = [("F32", 128), ("F32", 64), ("BF16", 128), ("BF16", 64), ("F16", 128),
                  ("F16", 64), ("I8", 128)]
SOURCES = ([(f, os.path.splitext(f)[0], []) for f in
            ["qs_api.cu", "qs_metadata.cu", "qs_select.cu", "qs_probe.cu", "qs_attention.cu",
             "qs_importance.cu", "qs_importance_tc.cu", "qs_attention_noalloc.cu",
             "qs_step_fused.cu"]] +
           [("qs_probe.cu", "qs_probe_%s_%d" % (t, d), ["-DQS_PROBE_KT=%s" % t, "-DQS_PROBE_D=%d" % d])
            for t, d in PROBE_VARIANTS])
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills"]


def nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _inputs():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(ROOT, "include", "questsparse.h"))
    return deps


def _compile(job, verbose):
    src, name, defines = job
    obj = os.path.join(OBJDIR, name + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *defines, "-I", os.path.join(ROOT, "include"), "-c",
           os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    newest = max(os.path.getmtime(p) for p in _inputs())
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest:
        return LIB
    os.makedirs(OBJDIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), max(4, os.cpu_count() or 4))) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
