"""The C ABI from plain C: tests/c/c_abi_layer.c is compiled with gcc against include/moe.h,
linked against libmoe.so and the CUDA runtime, and run; its checksums must equal those of the
same forward and backward made through the Python binding on the inputs the program wrote
out (same library, same inputs: the results are bit-identical, the checksums agree to the
rounding of their own summation order)."""
import os
import shutil
import subprocess

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_mixture_experts_56_b300 as m
    m._native.lib()
    return m


def test_c_program_matches_python_binding(moe, tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    cuda = "/usr/local/cuda"
    libdir = os.path.dirname(moe.library_path())
    exe = str(tmp_path / "c_abi_layer")
    cmd = [gcc, "-O2", "-std=c11", "-o", exe, os.path.join(ROOT, "tests", "c", "c_abi_layer.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           "-L", libdir, "-lmoe", "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    p = subprocess.run([exe, str(tmp_path)], capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr
    fields = p.stdout.split()
    c_vals = {fields[i]: float(fields[i + 1]) for i in range(2, len(fields), 2)}

    T, d, f, n, k = 200, 256, 384, 8, 2
    dev = "cuda"

    def bf(name, shape):
        raw = np.fromfile(str(tmp_path / f"{name}.bin"), dtype=np.int16).reshape(shape)
        return torch.from_numpy(raw).view(torch.bfloat16).to(dev)

    x, dy, wg = bf("x", (T, d)), bf("dy", (T, d)), bf("wg", (d, n))
    w1, w3, w2 = bf("w1", (n, f, d)), bf("w3", (n, f, d)), bf("w2", (n, d, f))
    ws = moe.workspace(T, d, f, n, k, torch.bfloat16, dev)
    y = moe.moe_layer_forward(x, wg, w1, w3, w2, k, ws)
    g = moe.moe_layer_backward(x, wg, w1, w3, w2, k, dy,
                               moe.backward_workspace(T, d, f, n, k, torch.bfloat16, dev))
    torch.cuda.synchronize()
    py = {"sum_abs_y": y.double().abs().sum().item(),
          "sum_abs_dw2": g["dw2"].double().abs().sum().item(),
          "sum_abs_dwg": g["dw_gate"].double().abs().sum().item()}
    for key, v in py.items():
        assert abs(c_vals[key] - v) <= 1e-9 * max(1.0, abs(v)), (key, c_vals[key], v)
