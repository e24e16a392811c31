"""Build gen/libdlrm_gen.so (host generator loop + device fill kernel) for sm_103a."""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))


def build(verbose: bool = False) -> str:
    out = os.path.join(HERE, "libdlrm_gen.so")
    src = os.path.join(HERE, "gen.cu")
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cmd = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
           "-Xcompiler", "-fPIC,-fopenmp", "-shared", "-o", out, src, "-lgomp"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    return out


if __name__ == "__main__":
    build(verbose=True)
    sys.exit(0)
