"""Builds libar.so, the engine's C-ABI shared library, in the package folder.

    python -m collective_reduction_gb300.build

Every translation unit is compiled by nvcc for sm_103a in parallel and linked
with the static CUDA runtime.  Float code is compiled without contraction
(-fmad=false) and without flushing subnormals, so the kernels perform exactly
the adds and multiplies the schedules name.
"""

import os
import shutil
import subprocess
import sys
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libar.so")
SOURCES = ["kernels.cu", "noalloc.cu", "schedule.cpp", "lower.cpp", "api.cpp", "bufcheck.cpp", "cost.cpp", "jit.cpp"]
# headers the run-time compiled DAG kernels include, embedded into jit.cpp
JIT_HEADERS = [os.path.join(INCLUDE, "ar.h")] + [os.path.join(CSRC, h) for h in ("devprog.hpp", "kargs.hpp",
                                                                                  "device.cuh")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found: the engine needs the CUDA toolkit to build")
    return p


def write_jit_headers(path, defines=()):
    """The JIT headers as C++ raw string literals, by include name; the
    build's -D macros lead the first one, so the run-time compiled kernels
    see the configuration the compiled ones do."""
    names, bodies = [], []
    prefix = "".join(f"#define {d.split('=', 1)[0]} {d.split('=', 1)[1] if '=' in d else 1}\n" for d in defines)
    for h in JIT_HEADERS:
        with open(h) as f:
            text = f.read()
        if h == JIT_HEADERS[0]:
            text = prefix + text
        if ")ARJIT\"" in text:
            raise RuntimeError(f"{h} contains the raw-string delimiter")
        names.append(os.path.basename(h))
        bodies.append(text)
    with open(path, "w") as f:
        f.write(f"constexpr int kJitHeaderCount = {len(names)};\n")
        f.write("const char* const kJitHeaderNames[] = {" + ", ".join(f'"{n}"' for n in names) + "};\n")
        f.write("const char* const kJitHeaders[] = {\n")
        for b in bodies:
            f.write('R"ARJIT(' + b + ')ARJIT",\n')
        f.write("};\n")


def build(verbose=False, defines=(), out=None):
    """Compile and link; `defines` are extra -D macros, `out` another path."""
    nv = nvcc()
    common = ["-std=c++17", "-O3", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    common += [f"-D{d}" for d in defines]
    with tempfile.TemporaryDirectory(prefix="ar_build_") as tmp:
        write_jit_headers(os.path.join(tmp, "jit_headers.inc"), defines)
        common += ["-I", tmp]
        procs, objs = [], []
        for src in SOURCES:
            obj = os.path.join(tmp, src + ".o")
            cmd = [nv, "-c", os.path.join(CSRC, src), "-o", obj] + common
            if src.endswith(".cu"):
                cmd += ARCH + ["-lineinfo", "-fmad=false", "-ftz=false", "-prec-div=true",
                               "-prec-sqrt=true", "-Xptxas", "-v" if verbose else "-O3"]
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
            objs.append(obj)
        failed = []
        for src, p in procs:
            log, _ = p.communicate()
            text = log.decode(errors="replace")
            if p.returncode != 0:
                failed.append(f"--- {src} ---\n{text}")
            elif verbose and text.strip():
                sys.stderr.write(text)
        if failed:
            raise RuntimeError("libar build failed:\n" + "\n".join(failed))
        tmp_lib = os.path.join(tmp, "libar.so")
        link = [nv, "-shared", "-o", tmp_lib] + objs + ARCH + ["-cudart", "static", "-ldl"]
        r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError("libar link failed:\n" + r.stdout.decode(errors="replace"))
        dest = out or LIB
        shutil.move(tmp_lib, dest)
    return dest


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
