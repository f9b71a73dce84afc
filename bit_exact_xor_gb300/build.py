"""Build libdcr.so in-tree: nvcc for sm_103a, one object per translation unit
compiled in parallel, then one shared-library link."""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libdcr.so")
SOURCES = ["plan.cpp", "pipeline.cpp", "encode.cu", "apply.cu", "dense.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", os.path.join(HERE, "..", "include")]


def build(verbose=False):
    bdir = os.path.join(HERE, "_build")
    os.makedirs(bdir, exist_ok=True)
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(bdir, src.rsplit(".", 1)[0] + ".o")
        cmd = ["nvcc"] + ARCH + FLAGS + (["-Xptxas", "-v"] if verbose and src.endswith(".cu") else []) + [
            "-x", "cu" if src.endswith(".cu") else "c++", "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    logs = []
    for cmd, p in procs:
        out, _ = p.communicate()
        logs.append(out.decode())
        if p.returncode != 0:
            raise RuntimeError("nvcc failed: %s\n%s" % (" ".join(cmd), out.decode()))
    link = ["nvcc"] + ARCH + ["-shared", "-o", OUT] + objs + ["-lcudart"]
    p = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if p.returncode != 0:
        raise RuntimeError("link failed:\n" + p.stdout.decode())
    return "".join(logs)


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
