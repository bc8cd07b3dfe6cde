"""The C ABI from a plain C program: tests/c/abi_smoke.c is compiled with gcc
against include/spec_verify.h, linked with libspec_verify.so and the CUDA
runtime, and run on the GPU (a greedy batch whose answer is fixed by
construction, the sampler, and a rejected argument)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
gpu = pytest.mark.gpu


@gpu
def test_plain_c_caller(tmp_path):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_45_gb300 import _native

    lib = _native.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.path.dirname(os.path.dirname(_native.nvcc_path()))
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "abi_smoke")
    cudalib = next((d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"),
                                os.path.join(cuda, "targets", "sbsa-linux", "lib"))
                    if os.path.exists(os.path.join(d, "libcudart.so"))), os.path.join(cuda, "lib64"))
    cmd = [cc, "-O2", "-std=c11", "-o", exe, os.path.join(ROOT, "tests", "c", "abi_smoke.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           "-L", libdir, "-l:" + os.path.basename(lib), "-L", cudalib, "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudalib}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip().endswith("OK"), run.stdout + run.stderr
