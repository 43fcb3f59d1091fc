"""Builds libtri.so in-tree with nvcc for sm_103a."""
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "tri.cu")
OUT = os.path.join(PKG, "libtri.so")
CSRC = ("tri.cu", "tri_device.cuh", "tri_path.cuh", "tri_mma.cuh", "tri_calib.cuh", "tri_curve.cuh", "tri_decode.cuh")
DEPS = [os.path.join(PKG, "csrc", f) for f in CSRC] + [
    os.path.join(ROOT, "include", "tri.h")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def command(out=OUT, extra=()):
    return [nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
            "-shared", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
            "-I", os.path.join(ROOT, "include"), *extra, "-o", out, SRC, "-lcudart"]


def up_to_date() -> bool:
    if not os.path.exists(OUT):
        return False
    t = os.path.getmtime(OUT)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    if force or not up_to_date():
        cmd = command(extra=("-Xptxas", "-v") if verbose else ())
        tmp = OUT + ".tmp"
        cmd[cmd.index(OUT)] = tmp
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + r.stdout + r.stderr)
        if verbose:
            sys.stderr.write(r.stderr)
        os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(OUT)
