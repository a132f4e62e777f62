"""The C ABI used from plain C: compile tests/c_client/kvevict_client.c with
gcc against include/kvevict.h, link libkvevict.so and the CUDA runtime, run it.
The client drives the device-buffer and host-buffer paths and checks the
state's invariants and that both paths agree bit for bit."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_client_runs(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kv_cache_attention_02_gb300 as kvx
    lib = kvx.lib()   # builds the library if needed
    libdir = os.path.dirname(lib._name)
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = tmp_path / "kvevict_client"
    cmd = [gcc, "-std=c11", "-O2", "-Wall", "-o", str(exe),
           os.path.join(ROOT, "tests", "c_client", "kvevict_client.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           "-L", libdir, "-L", os.path.join(cuda, "lib64"),
           "-Wl,-rpath," + libdir, "-Wl,-rpath," + os.path.join(cuda, "lib64"),
           "-l:" + os.path.basename(lib._name), "-lcudart", "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr + r.stdout
    assert "ok" in r.stdout
