"""The C-ABI library builds, loads without a GPU, and exports every entry
point that include/moe.h declares; the binding refuses to run without it."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(moe_[a-z0-9_]+)\s*\(",
                            src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def libmoe():
    from moe_expert_mlp_gb300.build import build_library
    build_library()
    import moe_expert_mlp_gb300 as m
    return m.lib()


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for required in ("moe_repack_fc1", "moe_route_permute", "moe_mlp_fwd", "moe_mlp_bwd",
                     "moe_unpermute_combine", "moe_unpermute_combine_bwd", "moe_permute_bwd",
                     "moe_route_bwd", "moe_workspace_size", "moe_read_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(libmoe):
    for name in declared_entry_points():
        assert hasattr(libmoe, name), name
    import moe_expert_mlp_gb300 as m
    assert sorted(m.EXPORTS) == declared_entry_points()


def test_host_side_errors_without_gpu(libmoe):
    import ctypes
    import moe_expert_mlp_gb300 as m
    desc = m.make_desc(T=64, E=4, k=2, d=128, F=64)
    n = ctypes.c_size_t(0)
    assert libmoe.moe_workspace_size(ctypes.byref(desc), ctypes.byref(n)) == 0
    assert n.value >= 256
    assert libmoe.moe_workspace_size(None, ctypes.byref(n)) == 1            # MOE_ERR_NULL
    bad = m.make_desc(T=64, E=4, k=2, d=100, F=64)
    assert libmoe.moe_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == 2  # MOE_ERR_SHAPE
    bad = m.make_desc(T=64, E=4, k=2, d=128, F=64)
    bad.align = 32
    assert libmoe.moe_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == 3  # unsupported
    assert m.moe_fc1_padded_width(2880) == 2944 and m.moe_fc1_padded_width(1408) == 1408
    assert libmoe.moe_status_string(2) == b"sizes out of the supported range"


def test_block_scaled_calls_reject_bad_arguments_without_gpu(libmoe):
    """The MXFP8 / NVFP4 calls validate the descriptor and pointers on the
    host and enqueue nothing: wrong operand type, shapes the block-scaled
    MMA cannot take, missing buffers."""
    import ctypes
    import moe_expert_mlp_gb300 as m
    from moe_expert_mlp_gb300 import _lib as L
    ok_nv = m.make_desc(T=0, E=4, k=1, d=128, F=64, dtype="nvfp4")
    bf16 = m.make_desc(T=0, E=4, k=1, d=128, F=64)
    bad_f = m.make_desc(T=0, E=4, k=1, d=128, F=96, dtype="nvfp4")     # F % 64 != 0
    null = ctypes.c_void_p(None)
    # operand type must match the call
    assert libmoe.moe_fc1_glu_fwd_nv(ctypes.byref(bf16), *([null] * 9)) == 3
    assert libmoe.moe_fc2_wgrad_mx(ctypes.byref(ok_nv), *([null] * 6)) == 3
    # NVFP4 needs F % 64 == 0
    assert libmoe.moe_fc2_fwd_nv(ctypes.byref(bad_f), *([null] * 7)) == 2
    # valid descriptor, missing buffers
    assert libmoe.moe_fc2_fwd_nv(ctypes.byref(ok_nv), *([null] * 7)) == 1
    assert libmoe.moe_mlp_bwd_nv(ctypes.byref(ok_nv), *([null] * 16)) == 1
    assert libmoe.moe_quantize_nvfp4_bf16(null, 1, 32, 32, null, 0, null) == 1
    assert L.moe_nvfp4_scale_bytes(256, 256) == 4 * 2 * 512
    assert L.moe_nvfp4_scale_bytes(0, 64) == 0
    assert L.moe_mx_scale_bytes(256, 256) == 2 * 2 * 512


def test_noalloc_size_limit_boundary(libmoe):
    """moe_route_permute_noalloc accepts a histogram of exactly 256 KiB
    (ceil(T/256) * E = 65536 entries: T = 65536, E = 256) and rejects one
    chunk more with MOE_ERR_WORKSPACE before anything else.  The accepted
    case is given NULL buffers, so it stops at the next check (MOE_ERR_NULL
    with a GPU, MOE_ERR_CUDA without one) and launches nothing."""
    import ctypes
    import moe_expert_mlp_gb300 as m
    null = ctypes.c_void_p(None)
    at = m.make_desc(T=65536, E=256, k=1, d=64, F=32)
    over = m.make_desc(T=65536 + 1, E=256, k=1, d=64, F=32)
    assert libmoe.moe_route_permute_noalloc(ctypes.byref(over), *([null] * 13)) == 4
    assert libmoe.moe_route_permute_noalloc(ctypes.byref(at), *([null] * 13)) in (1, 6)
    assert libmoe.moe_route_permute_noalloc(None, *([null] * 13)) == 1


def test_fp32_calls_reject_bad_arguments_without_gpu(libmoe):
    """The fp32 / TF32 calls check the descriptor and pointers on the host:
    the bf16 GEMM calls refuse an fp32 descriptor and the *_tf32 calls a
    bf16 one (MOE_ERR_UNSUPPORTED), recompute_h is refused with fp32,
    missing buffers give MOE_ERR_NULL and a misaligned output
    MOE_ERR_SHAPE.  The fp32 workspace adds the backward's transposed
    operands: W1p^T, W2^T, x_perm^T, dY^T, A^T and dH^T in fp32."""
    import ctypes
    import moe_expert_mlp_gb300 as m
    null = ctypes.c_void_p(None)
    E, d, F, cap = 4, 128, 96, 1024
    f32 = m.make_desc(T=0, E=E, k=1, d=d, F=F, dtype="fp32", capacity=cap)
    bf16 = m.make_desc(T=0, E=E, k=1, d=d, F=F, capacity=cap)
    assert libmoe.moe_fc1_glu_fwd(ctypes.byref(f32), *([null] * 9)) == 3
    assert libmoe.moe_fc2_wgrad(ctypes.byref(f32), *([null] * 6)) == 3
    assert libmoe.moe_quantize_act_mx(ctypes.byref(f32), null, 128, null, null, null) == 3
    assert libmoe.moe_fc1_glu_fwd_tf32(ctypes.byref(bf16), *([null] * 9)) == 3
    rc = m.make_desc(T=0, E=E, k=1, d=d, F=F, dtype="fp32", capacity=cap, recompute_h=True)
    assert libmoe.moe_fc2_fwd_tf32(ctypes.byref(rc), *([null] * 7)) == 3
    assert libmoe.moe_fc2_fwd_tf32(ctypes.byref(f32), *([null] * 7)) == 1
    assert libmoe.moe_fc1_wgrad_tf32(ctypes.byref(f32), *([null] * 6)) == 1
    assert libmoe.moe_transpose_weights_tf32(ctypes.byref(f32), *([null] * 5)) == 1
    assert libmoe.moe_transpose_rows_f32(ctypes.byref(f32), null, 128, null, null, null) == 1
    p = ctypes.c_void_p(4096)                      # never dereferenced on the host
    odd = ctypes.c_void_p(4100)                    # not 16-byte aligned
    assert libmoe.moe_fc2_fwd_tf32(ctypes.byref(f32), p, p, p, p, null, odd, null) == 2
    n_f32, n_bf16 = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert libmoe.moe_workspace_size(ctypes.byref(f32), ctypes.byref(n_f32)) == 0
    assert libmoe.moe_workspace_size(ctypes.byref(bf16), ctypes.byref(n_bf16)) == 0
    W1 = 2 * 128                                   # 2 * F_pad
    r = lambda b: (b + 255) // 256 * 256
    extra = (r(E * d * W1 * 4) + r(E * F * d * 4) + 2 * r(d * cap * 4) + r(F * cap * 4)
             + r(W1 * cap * 4))
    assert n_f32.value == r(n_bf16.value) + extra


def test_header_and_c_caller_compile_as_c(libmoe, tmp_path):
    """include/moe.h is plain C: the C caller of tests/c_abi (a whole layer
    step on caller-owned device buffers) compiles as C99 with every warning
    an error and links against libmoe.so and the CUDA runtime."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None or not os.path.isdir("/usr/local/cuda/include"):
        pytest.skip("needs gcc and the CUDA headers")
    from tests.test_gpu_c_abi import build_layer_step
    exe = build_layer_step(str(tmp_path))
    assert os.path.exists(exe)
    r = subprocess.run(["nm", "-D", "--undefined-only", exe], capture_output=True, text=True)
    for name in ("moe_route_permute", "moe_mlp_fwd", "moe_mlp_bwd", "moe_unpermute_combine"):
        assert name in r.stdout, name
