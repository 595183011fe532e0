"""Builds tests/c/forward_from_c.c, a plain C caller of the library, with gcc
(not a test module)."""
import glob
import os
import shutil
import subprocess

from mixture_experts_routed_gate_gb300 import _build

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "c", "forward_from_c.c")


def cuda_home() -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(_build.nvcc())))


def cudart_dir() -> str:
    home = cuda_home()
    for cand in [os.path.join(home, "lib64"), *glob.glob(os.path.join(home, "targets", "*", "lib"))]:
        if glob.glob(os.path.join(cand, "libcudart.so*")):
            return cand
    raise RuntimeError(f"libcudart.so not found under {home}")


def build(out_dir: str) -> str:
    """Compile and link the C caller against include/ and the built library."""
    gcc = shutil.which("gcc")
    if gcc is None:
        raise RuntimeError("gcc not found")
    lib = _build.build()
    lib_dir = os.path.dirname(lib)
    exe = os.path.join(out_dir, "forward_from_c")
    cmd = [gcc, "-std=c11", "-O2", "-Wall", "-Werror", SRC, "-I", _build.INCLUDE, "-I",
           os.path.join(cuda_home(), "include"), "-o", exe, "-L", lib_dir, "-lmoe_routed_gb300",
           "-L", cudart_dir(), "-lcudart", f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{cudart_dir()}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"gcc failed:\n{r.stdout}\n{r.stderr}")
    return exe
