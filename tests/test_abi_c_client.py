"""The C ABI from plain C: tests/abi_c/nrc_client.c is compiled as C11
(-Wall -Wextra -Werror -pedantic) against include/nrc.h alone and linked
against libnrc.so.  Without a GPU it runs the host-only calls; on a GPU it runs
the pre-norm block on device buffers and its output is compared with the
oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "abi_c", "nrc_client.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")

pytestmark = pytest.mark.skipif(shutil.which("gcc") is None or
                                not os.path.exists(os.path.join(CUDA, "include",
                                                                "cuda_runtime_api.h")),
                                reason="needs gcc and the CUDA headers")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    from normalization_convolution_blocks_gb300 import build
    lib = build.build()
    out = str(tmp_path_factory.mktemp("abi_c") / "nrc_client")
    libdir = os.path.dirname(lib)
    cudalib = next((p for p in (os.path.join(CUDA, "lib64"), os.path.join(CUDA, "lib"))
                    if os.path.isdir(p)), os.path.join(CUDA, "lib64"))
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           SRC, "-o", out, "-L", libdir, "-lnrc", "-L", cudalib, "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudalib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return out


def test_c_client_host_only_calls(client):
    r = subprocess.run([client, "queries"], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert "queries ok" in r.stdout


@pytest.mark.gpu
def test_c_client_runs_the_block_on_the_gpu(client, tmp_path):
    from gpu_util import assert_f32, need_gpu
    need_gpu()
    import oracle
    from normalization_convolution_blocks_gb300 import synthetic as syn
    inp = syn.prenorm_block_inputs(2, 64, 700, 16, seed=31)
    (tmp_path / "dims.txt").write_text(f"2 64 700 16 {inp.eps!r}\n")
    for name, t in (("x", inp.x), ("rm", inp.running_mean), ("rv", inp.running_var),
                    ("gamma", inp.gamma), ("beta", inp.beta), ("w", inp.weight),
                    ("bias", inp.bias)):
        t.contiguous().numpy().astype(np.float32).tofile(tmp_path / f"{name}.bin")
    r = subprocess.run([client, "block", str(tmp_path)], capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    got = np.fromfile(tmp_path / "out.bin", dtype=np.float32).reshape(inp.x.shape)
    ref = oracle.prenorm_block(inp.x, inp.running_mean, inp.running_var, inp.gamma, inp.beta,
                               inp.eps, inp.weight, inp.bias, inp.dilation)
    assert_f32(got.astype(np.float64), ref, "C client block")
