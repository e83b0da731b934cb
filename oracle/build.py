"""Compile the plain-C oracle into two shared libraries (fp64 and fp32).

Test infrastructure: builds oracle/_build/libgpt2_oracle_f64.so and
libgpt2_oracle_f32.so from oracle/gpt2_oracle.c with gcc.  Rebuilds only
when the source is newer than the library.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gpt2_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")


def lib_path(real: str = "double") -> str:
    tag = "f64" if real == "double" else "f32"
    return os.path.join(OUT_DIR, f"libgpt2_oracle_{tag}.so")


def build(force: bool = False) -> None:
    os.makedirs(OUT_DIR, exist_ok=True)
    for real in ("double", "float"):
        out = lib_path(real)
        if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
            continue
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               f"-DREAL={real}", SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)


if __name__ == "__main__":
    build(force="--force" in sys.argv)
    print(lib_path("double"))
    print(lib_path("float"))
