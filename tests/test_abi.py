"""Host-side checks of the C-ABI library (no GPU): it builds for sm_103a, loads,
exports every function declared in include/*.h, the Python binding declares a
signature for each, and shape validation answers without touching a device."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


def _declared():
    names = set()
    for f in os.listdir(INCLUDE):
        if not f.endswith(".h"):
            continue
        src = open(os.path.join(INCLUDE, f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for m in re.finditer(r"\b(gpt2\w*)\s*\(", src):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    from scratch_gpt_step_train_b300 import build, gpt2
    build.build()
    return gpt2.lib()


def test_every_declared_symbol_is_exported(lib):
    from scratch_gpt_step_train_b300 import gpt2, kernels
    names = _declared()
    assert len(names) >= 20
    out = subprocess.run(["nm", "-D", "--defined-only", gpt2.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = sorted(n for n in names if n not in exported)
    assert not missing, missing
    bound = set(gpt2.SIGNATURES) | set(kernels.SIGNATURES)
    unbound = sorted(n for n in names if n not in bound)
    assert not unbound, unbound
    kernels.klib()
    for n in names:
        assert hasattr(lib, n)


def test_library_is_built_for_sm103a_only():
    """every object is compiled with exactly one target, sm_103a (the build
    passes no other -gencode / -arch flag)"""
    from scratch_gpt_step_train_b300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert not any(f.startswith(("-arch", "--gpu-architecture", "-gencode", "-code"))
                   for f in build.FLAGS)


@pytest.mark.gpu
def test_loaded_kernels_are_sm103(lib):
    """the runtime reports binary version 10.3 for the loaded GEMM kernel"""
    from scratch_gpt_step_train_b300 import kernels
    import torch
    torch.cuda.init()
    assert kernels.klib().gpt2k_binary_arch() == 103


def test_no_oracle_dependency_in_product():
    """the product package never imports or links the oracle"""
    pkg = os.path.join(ROOT, "scratch_gpt_step_train_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in txt.lower(), f


def test_workspace_shape_validation(lib):
    ws = lib.gpt2_workspace_bytes
    assert ws(12, 12, 768, 50257, 1024, 16, 1) > 0
    assert ws(2, 2, 16, 2, 3, 12, 0) > 0
    assert ws(2, 3, 16, 2, 3, 12, 0) == 0          # C % H
    assert ws(2, 2, 12, 64, 8, 2, 1) == 0          # bf16 needs C % 8 == 0
    assert ws(2, 2, 96, 64, 8, 2, 0) == 0          # head size 48 not supported
    assert ws(0, 2, 16, 2, 3, 12, 0) == 0
    assert ws(2, 2, 16, 2, 3, 0, 0) == 0
    # grows with the micro-batch, bf16 smaller than fp32 at the same shape
    assert ws(2, 2, 64, 100, 16, 4, 0) > ws(2, 2, 64, 100, 16, 2, 0)
    assert ws(2, 2, 64, 100, 16, 4, 1) < ws(2, 2, 64, 100, 16, 4, 0)


def test_workspace_fits_1558M_on_one_gpu(lib):
    """the 1558M micro-batch B=16, T=1024 workspace fits in 270 GB of HBM"""
    b = lib.gpt2_workspace_bytes(48, 25, 1600, 50257, 1024, 16, 1)
    assert 40e9 < b < 150e9, b
