"""The C ABI used from a plain C program (tests/c/abi_smoke.c), compiled with
gcc against include/zero_gb300.h and linked with libzero_gb300.so (and the
oracle, for its reference values)."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def smoke_exe(zlib, tmp_path_factory):
    import oracle
    oracle.build()
    out = str(tmp_path_factory.mktemp("c") / "abi_smoke")
    lib_dir = os.path.dirname(zlib.lib_path)
    cuda_lib = "/usr/local/cuda/lib64"
    subprocess.check_call([
        "gcc", "-std=c11", "-O2", "-ffp-contract=off", "-I", os.path.join(ROOT, "include"),
        os.path.join(ROOT, "tests", "c", "abi_smoke.c"), os.path.join(ROOT, "oracle", "zero_oracle.c"),
        "-L", lib_dir, "-lzero_gb300", f"-Wl,-rpath,{lib_dir}",
        "-L", cuda_lib, "-lcudart", f"-Wl,-rpath,{cuda_lib}", "-lm", "-o", out])
    return out


def test_host_calls_from_c(smoke_exe):
    r = subprocess.run([smoke_exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


@pytest.mark.gpu
def test_fused_step_from_c(smoke_exe):
    r = subprocess.run([smoke_exe, "--gpu"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
