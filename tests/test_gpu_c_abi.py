"""The C ABI from plain C: tests/c_abi/layer_step.c allocates its own device
buffers with cudaMalloc and runs a whole routed-layer step (repack, route +
permute, moe_mlp_fwd, combine, combine backward, moe_mlp_bwd, permute and
router backward, unpack) through include/moe.h; its results match the
oracle as the Python-driven layer's do: counts bit-exact, every float output
within the bf16 bound."""
import os
import subprocess

import numpy as np
import pytest
import torch

from tests import harness as H
from workloads import WORKLOADS, bf16_bits_to_f64, make_inputs, scaled

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def build_layer_step(out_dir):
    """gcc, C99, against include/moe.h, libmoe.so and the CUDA runtime."""
    from moe_expert_mlp_gb300.build import build_library
    lib = build_library()
    cuda = "/usr/local/cuda"
    exe = os.path.join(out_dir, "layer_step")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-O2",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c_abi", "layer_step.c"), "-o", exe,
           "-L", os.path.dirname(lib), "-lmoe", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           "-Wl,-rpath," + os.path.dirname(lib), "-Wl,-rpath," + os.path.join(cuda, "lib64")]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_layer_step_from_c_matches_oracle(tmp_path):
    wl = scaled(WORKLOADS["bf16_t4096_e64"], T=384, E=8, k=2, d=192, F=160, router_bias=False)
    inp = make_inputs(wl)
    exe = build_layer_step(str(tmp_path))
    fin, fout = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(fin, "wb") as f:
        f.write(np.array([wl.T, wl.E, wl.k, wl.d, wl.F], dtype=np.int32).tobytes())
        f.write(np.ascontiguousarray(inp["logits"], dtype=np.float32).tobytes())
        for key in ("x", "w1", "w2", "dout"):
            f.write(np.ascontiguousarray(inp[key]).view(np.uint16).tobytes())
    r = subprocess.run([exe, str(fin), str(fout)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    T, E, d, F = wl.T, wl.E, wl.d, wl.F
    raw = np.fromfile(fout, dtype=np.uint8)
    sizes = [("out", T * d * 2), ("dx", T * d * 2), ("dlogits", T * E * 4),
             ("dw1", E * 2 * F * d * 2), ("dw2", E * d * F * 2), ("counts", E * 4)]
    assert raw.size == sum(n for _, n in sizes)
    got, o = {}, 0
    for name, n in sizes:
        got[name] = raw[o:o + n]
        o += n
    fwd, bwd = H.run_oracle_routed(wl, inp)
    assert np.array_equal(got["counts"].view(np.int32), fwd["counts"])
    bf = lambda b, shape: bf16_bits_to_f64(b.view(np.uint16).reshape(shape))
    H.assert_close("out", bf(got["out"], (T, d)), fwd["out"])
    H.assert_close("dx", bf(got["dx"], (T, d)), bwd["dx"])
    H.assert_close("dlogits", got["dlogits"].view(np.float32).reshape(T, E), bwd["dlogits"])
    H.assert_close("dW1", bf(got["dw1"], (E, 2 * F, d)), bwd["dW1"])
    H.assert_close("dW2", bf(got["dw2"], (E, d, F)), bwd["dW2"])
