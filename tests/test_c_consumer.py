"""The C ABI from a plain C99 program (tests/c_consumer.c), no Python in
between: host-side checks on the CPU, and on a GPU a real call compared with
the C oracle."""
import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _compile(tmp_path, gpu: bool) -> str:
    from residual_rmsnorm_gb300 import build
    lib = build.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / ("c_consumer_gpu" if gpu else "c_consumer"))
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Werror", os.path.join(HERE, "c_consumer.c"),
           "-I", os.path.join(ROOT, "include"), "-o", exe, "-L", libdir, "-ltpar", f"-Wl,-rpath,{libdir}", "-lm"]
    if gpu:
        import oracle
        olib = oracle.build()
        odir = os.path.dirname(olib)
        cuda_lib = build.cuda_lib_dir()
        cuda_inc = os.path.join(os.path.dirname(cuda_lib), "include")
        cmd[2:2] = ["-DTPAR_C_CONSUMER_GPU"]
        cmd += ["-I", cuda_inc, "-L", odir, "-loracle", f"-Wl,-rpath,{odir}", "-L", cuda_lib, "-lcudart",
                f"-Wl,-rpath,{cuda_lib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_host_checks(tmp_path):
    exe = _compile(tmp_path, gpu=False)
    r = subprocess.run([exe, "host"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "c_consumer host: ok" in r.stdout


@pytest.mark.gpu
def test_c_program_gpu_call_matches_oracle(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = _compile(tmp_path, gpu=True)
    r = subprocess.run([exe, "gpu"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert "c_consumer gpu: ok" in r.stdout
