"""C-ABI library: loads, exports every declared entry point, validates arguments.

These run without a GPU: argument checks happen before any CUDA call, so an
invalid call returns its status code on any host, and a valid call on a host
with no device returns NO_DEVICE instead of touching CUDA memory.
"""
import ctypes
import os
import re

import pytest

import diffusion_transformer_joint_causal_b300 as dit
from diffusion_transformer_joint_causal_b300 import build as dit_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dit_attn.h")


@pytest.fixture(scope="module", autouse=True)
def _built():
    dit_build.build()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(dit_attn_\w+)\s*\(", text, re.M)))


def test_header_declares_the_binding_symbols():
    assert _declared() == sorted(dit.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(dit.library_path())
    for name in _declared():
        assert hasattr(lib, name), name


def test_version_and_status_strings():
    assert dit.version() >= 100
    for code in range(7):
        assert dit.status_string(code)
    assert dit.status_string(99) == "unknown status"


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


A = 0x7f0000000000   # fake, 16-byte aligned addresses: never dereferenced by a rejected call
MB = 1 << 20


@pytest.mark.parametrize("args,expect", [
    ((0, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 64, 0.125), 1),            # null q
    ((A, A + MB, A + 2 * MB, 0, 1, 1, 8, 8, 64, 0.125), 1),                     # null out
    ((A, A + MB, A + 2 * MB, A + 3 * MB, 0, 1, 8, 8, 64, 0.125), 1),            # B = 0
    ((A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 0, 8, 64, 0.125), 1),            # Lq = 0
    ((A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 0, 64, 0.125), 1),            # Lk = 0
    ((A, A + MB, A + 2 * MB, A + 3 * MB, 1, -2, 8, 8, 64, 0.125), 1),           # H < 0
    ((A + 8, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 64, 0.125), 1),        # misaligned q
    ((A, A + MB, A + 2 * MB, A + 3 * MB + 2, 1, 1, 8, 8, 64, 0.125), 1),        # misaligned out
    ((A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 64, float("nan")), 1),     # NaN scale
    ((A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 64, float("inf")), 1),     # inf scale
    ((A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 64, 2.4e38), 1),           # scale*log2(e) > FLT_MAX
    ((A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 64, -2.4e38), 1),
    ((A, A + MB, A + 2 * MB, A + 512, 1, 1, 8, 8, 64, 0.125), 1),               # out overlaps q
    ((A, A + MB, A + 2 * MB, A + MB + 512, 1, 1, 8, 8, 64, 0.125), 1),          # out overlaps k
    ((A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 96, 0.125), 2),            # d = 96
    ((A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 256, 0.125), 2),           # d = 256
    ((A, A + MB, A + 2 * MB, A + 3 * MB, 65536, 65536, 8, 8, 64, 0.125), 2),    # B*H too large
    ((A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 2**31 - 1, 8, 64, 0.125), 2),    # Lq too large
])
def test_forward_rejects_bad_arguments(args, expect):
    assert dit.forward_ptr(*args) == expect


@pytest.mark.skipif(_has_gpu(), reason="a valid call with fake pointers must not reach a GPU")
@pytest.mark.parametrize("scale", [-0.5, 0.0, -2.3e38, 2.3e38, -1e-30])
def test_forward_accepts_every_usable_scale(scale):
    # softmax(scale * q k^T) v is defined for any finite scale; every sign
    # passes the argument checks (the call then stops at the device check)
    assert dit.forward_ptr(A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 128, scale) == 4
    assert dit.forward_qk8_ptr(*_qk8(scale=scale, q_scale=1.0, k_scale=1.0)) == 4
    assert dit.forward_fp8_ptr(*_fp8(scale=scale, q_scale=1.0, k_scale=1.0)) == 4


@pytest.mark.skipif(_has_gpu(), reason="checks the no-device path")
def test_no_device_paths():
    assert dit.forward_ptr(A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 64, 0.125) == 4
    lib = ctypes.CDLL(dit.library_path())
    assert lib.dit_attn_create() == 4
    assert lib.dit_attn_destroy() == 4
    assert lib.dit_attn_get_device_error(None) == 4
    with pytest.raises(dit.DitAttnError):
        dit.create()


def test_python_forward_checks_tensors():
    import torch
    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        dit.forward(x, x, x)                               # CPU tensors
    with pytest.raises(TypeError):
        dit.forward(x.float(), x, x)


def test_wait_timeout_check_validates_before_cuda():
    lib = ctypes.CDLL(dit.library_path())
    assert lib.dit_attn_check_wait_timeout(0, None) == 1
    assert lib.dit_attn_check_wait_timeout(2000000, None) == 1


@pytest.mark.parametrize("args,expect", [
    ((0, A, 0, 8, 128, 1e-6), 1),                    # null x
    ((A, 0, 0, 8, 128, 1e-6), 1),                    # null y
    ((A, A + MB, 0, 0, 128, 1e-6), 1),               # rows = 0
    ((A, A + MB, 0, 8, 128, -1.0), 1),               # negative eps
    ((A, A + MB, 0, 8, 128, float("nan")), 1),       # NaN eps
    ((A + 4, A + MB, 0, 8, 128, 1e-6), 1),           # misaligned x
    ((A, A + MB, A + 2 * MB + 8, 8, 128, 1e-6), 1),  # misaligned weight
    ((A, A + 512, 0, 8, 128, 1e-6), 1),              # partial overlap of x and y
    ((A, A + MB, 0, 8, 96, 1e-6), 2),                # d = 96
])
def test_rmsnorm_rejects_bad_arguments(args, expect):
    assert dit.rmsnorm_ptr(*args) == expect


@pytest.mark.skipif(_has_gpu(), reason="checks the no-device path")
def test_rmsnorm_no_device():
    assert dit.rmsnorm_ptr(A, A, 0, 8, 128, 1e-6) == 4      # in place is allowed


QK8 = (A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 128, 0.125, 0.02, 0.03)


def _qk8(**change):
    names = ("q8", "k8", "v", "out", "B", "H", "Lq", "Lk", "d", "scale", "q_scale", "k_scale")
    args = dict(zip(names, QK8))
    args.update(change)
    return tuple(args[n] for n in names)


@pytest.mark.parametrize("args,expect", [
    (_qk8(q8=0), 1),                                  # null q8
    (_qk8(v=0), 1),                                   # null v
    (_qk8(Lk=0), 1),                                  # Lk = 0
    (_qk8(k8=A + MB + 8), 1),                         # misaligned k8
    (_qk8(q_scale=float("nan")), 1),                  # NaN q_scale
    (_qk8(k_scale=-1.0), 1),                          # negative k_scale
    (_qk8(k_scale=float("inf")), 1),                  # inf k_scale
    (_qk8(scale=1e20, q_scale=1e20, k_scale=1e20), 1),  # combined scale overflows fp32
    (_qk8(scale=-1e20, q_scale=1e20, k_scale=1e20), 1),
    (_qk8(scale=2.4e36, q_scale=10.0, k_scale=10.0), 1),  # combined scale * log2(e) > FLT_MAX
    (_qk8(out=A + 512), 1),                           # out overlaps the 1 KB of q8
    (_qk8(d=64), 2),                                  # e4m3 path is d = 128 only
    (_qk8(d=96), 2),
    (_qk8(B=65536, H=65536), 2),                      # B*H too large
])
def test_forward_qk8_rejects_bad_arguments(args, expect):
    assert dit.forward_qk8_ptr(*args) == expect


@pytest.mark.skipif(_has_gpu(), reason="a valid call with fake pointers must not reach a GPU")
def test_forward_qk8_overlap_counts_e4m3_bytes():
    # q8 is 8*128 = 1 KB of e4m3 codes: an out placed right after it does not
    # overlap (a bf16-sized count would say it does), so the call passes every
    # argument check and stops at the device check.
    assert dit.forward_qk8_ptr(*_qk8(out=A + 1024)) == 4


@pytest.mark.parametrize("args,expect", [
    ((0, A + MB, 0, 8, 128, 1e-6, 1.0), 1),           # null x
    ((A, A + MB, 0, 8, 128, 1e-6, 0.0), 1),           # zero out_scale
    ((A, A + MB, 0, 8, 128, 1e-6, float("inf")), 1),  # inf out_scale
    ((A, A + MB, 0, 8, 128, -1.0, 1.0), 1),           # negative eps
    ((A, A + 8, 0, 8, 128, 1e-6, 1.0), 1),            # misaligned y8
    ((A, A, 0, 8, 128, 1e-6, 1.0), 1),                # in place is not allowed for e4m3
    ((A, A + 1024, 0, 8, 128, 1e-6, 1.0), 1),         # y8 overlaps x (2 KB of bf16)
    ((A, A + MB, 0, 8, 96, 1e-6, 1.0), 2),            # d = 96
])
def test_rmsnorm_e4m3_rejects_bad_arguments(args, expect):
    assert dit.rmsnorm_e4m3_ptr(*args) == expect


@pytest.mark.skipif(_has_gpu(), reason="checks the no-device path")
def test_e4m3_entry_points_no_device():
    assert dit.forward_qk8_ptr(*QK8) == 4
    assert dit.rmsnorm_e4m3_ptr(A, A + 2048, 0, 8, 128, 1e-6, 1.0) == 4   # y8 right after x


def test_python_e4m3_wrappers_check_tensors():
    import torch
    x = torch.zeros(1, 1, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        dit.forward_qk8(x, x, x, 1.0, 1.0)                # bf16 q8 / CPU tensors
    with pytest.raises(TypeError):
        dit.rmsnorm_e4m3(x, 1.0)                          # CPU tensor


WS = A + 8 * MB   # a fake, aligned workspace address clear of the fake tensors


@pytest.mark.parametrize("ws,nbytes,expect", [
    (WS, -1, 1),                 # negative size
    (0, 4096, 1),                # size without a pointer
    (WS + 8, 4096, 1),           # misaligned
    (A + 2 * MB, 4096, 1),       # overlaps v
    (A + 3 * MB + 512, 64, 1),   # overlaps out (8*64*2 bytes from A + 3 MB)
])
def test_forward_ws_rejects_bad_workspace(ws, nbytes, expect):
    args = (A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 64, 0.125)
    assert dit.forward_ws_ptr(*args, ws, nbytes) == expect
    qk8 = (A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 128, 0.125, 0.02, 0.03)
    assert dit.forward_qk8_ws_ptr(*qk8, ws, nbytes) == expect


def test_forward_ws_still_checks_tensors():
    assert dit.forward_ws_ptr(0, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 64, 0.125, WS, 4096) == 1
    assert dit.forward_ws_ptr(A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 96, 0.125, WS, 4096) == 2


def test_workspace_size_validates_before_cuda():
    lib = ctypes.CDLL(dit.library_path())
    lib.dit_attn_workspace_size.argtypes = [ctypes.c_int] * 6 + [ctypes.c_void_p]
    nb = ctypes.c_longlong(7)
    assert lib.dit_attn_workspace_size(1, 1, 8, 8, 128, 0, None) == 1            # no output pointer
    assert lib.dit_attn_workspace_size(0, 1, 8, 8, 128, 0, ctypes.byref(nb)) == 1 and nb.value == 0
    assert lib.dit_attn_workspace_size(1, 1, 8, 8, 96, 0, ctypes.byref(nb)) == 2
    assert lib.dit_attn_workspace_size(1, 1, 8, 8, 64, 1, ctypes.byref(nb)) == 2  # e4m3 is d=128 only


@pytest.mark.skipif(_has_gpu(), reason="checks the no-device path")
def test_workspace_entry_points_no_device():
    assert dit.forward_ws_ptr(A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 64, 0.125, WS, 4096) == 4
    assert dit.forward_ws_ptr(A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 64, 0.125, 0, 0) == 4
    with pytest.raises(dit.DitAttnError):
        dit.workspace_size(1, 24, 16896, 16896, 128)


# ----------------------------------------------------------------- e4m3 Q/K/V forward, quantise

FP8 = (A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 128, 0.125, 0.02, 0.03, 0.01)


def _fp8(**change):
    names = ("q8", "k8", "v8", "out", "B", "H", "Lq", "Lk", "d", "scale", "q_scale", "k_scale",
             "v_scale")
    args = dict(zip(names, FP8))
    args.update(change)
    return tuple(args[n] for n in names)


@pytest.mark.parametrize("args,expect", [
    (_fp8(v8=0), 1),                                  # null v8
    (_fp8(Lq=0), 1),                                  # Lq = 0
    (_fp8(v8=A + 2 * MB + 4), 1),                     # misaligned v8
    (_fp8(v_scale=0.0), 1),                           # v_scale must be > 0
    (_fp8(v_scale=-0.5), 1),
    (_fp8(v_scale=float("nan")), 1),
    (_fp8(v_scale=float("inf")), 1),
    (_fp8(v_scale=1e-45), 1),                         # 1 / v_scale overflows fp32
    (_fp8(q_scale=-1.0), 1),
    (_fp8(scale=1e20, q_scale=1e20, k_scale=1e20), 1),
    (_fp8(scale=-2.4e36, q_scale=10.0, k_scale=10.0), 1),
    (_fp8(out=A + 2 * MB + 512), 1),                  # out overlaps the 1 KB of v8
    (_fp8(d=64), 2),                                  # d = 128 only
    (_fp8(B=65536, H=65536), 2),
])
def test_forward_fp8_rejects_bad_arguments(args, expect):
    assert dit.forward_fp8_ptr(*args) == expect


@pytest.mark.parametrize("ws,nbytes,expect", [
    (WS, -1, 1), (0, 4096, 1), (WS + 8, 4096, 1),
    (A + 2 * MB, 4096, 1),       # overlaps v8
])
def test_forward_fp8_ws_rejects_bad_workspace(ws, nbytes, expect):
    assert dit.forward_fp8_ws_ptr(*FP8, ws, nbytes) == expect


@pytest.mark.skipif(_has_gpu(), reason="a valid call with fake pointers must not reach a GPU")
def test_fp8_entry_points_no_device():
    # v8 is 1 KB of e4m3 codes: an out right after it does not overlap
    assert dit.forward_fp8_ptr(*_fp8(out=A + 2 * MB + 1024)) == 4
    assert dit.forward_fp8_ws_ptr(*FP8, WS, 4096) == 4
    assert dit.quantize_e4m3_ptr(A, A + 2048, 1000, 2.0) == 4     # y8 right after x


@pytest.mark.parametrize("args,expect", [
    ((0, A + MB, 100, 1.0), 1),                       # null x
    ((A, 0, 100, 1.0), 1),                            # null y8
    ((A, A + MB, 0, 1.0), 1),                         # n = 0
    ((A, A + MB, -5, 1.0), 1),
    ((A, A + MB, 100, 0.0), 1),                       # out_scale must be > 0
    ((A, A + MB, 100, float("nan")), 1),
    ((A, A + MB, 100, float("inf")), 1),
    ((A + 2, A + MB, 100, 1.0), 1),                   # misaligned x
    ((A, A + MB + 8, 100, 1.0), 1),                   # misaligned y8
    ((A, A + 192, 100, 1.0), 1),                      # y8 overlaps x (200 bytes of bf16)
    ((A, A + MB, 1 << 50, 1.0), 2),                   # too large
])
def test_quantize_e4m3_rejects_bad_arguments(args, expect):
    assert dit.quantize_e4m3_ptr(*args) == expect


def test_workspace_size_variants_validate_before_cuda():
    lib = ctypes.CDLL(dit.library_path())
    lib.dit_attn_workspace_size.argtypes = [ctypes.c_int] * 6 + [ctypes.c_void_p]
    nb = ctypes.c_longlong(7)
    assert lib.dit_attn_workspace_size(1, 1, 8, 8, 128, 4, ctypes.byref(nb)) == 1 and nb.value == 0
    assert lib.dit_attn_workspace_size(1, 1, 8, 8, 128, -1, ctypes.byref(nb)) == 1
    assert lib.dit_attn_workspace_size(1, 1, 8, 8, 64, 2, ctypes.byref(nb)) == 2   # d = 128 only


def test_python_fp8_wrappers_check_tensors():
    import torch
    x = torch.zeros(1, 1, 8, 128, dtype=torch.bfloat16)
    x8 = torch.zeros(1, 1, 8, 128, dtype=torch.uint8)
    with pytest.raises(TypeError):
        dit.forward_fp8(x8, x8, x, 1.0, 1.0, 1.0)          # bf16 v / CPU tensors
    with pytest.raises(TypeError):
        dit.forward_fp8(x8, x8, x8, 1.0, 1.0, 1.0)         # CPU tensors
    with pytest.raises(TypeError):
        dit.quantize_e4m3(x, 1.0)                          # CPU tensor


def test_check_exp2_validates_before_cuda():
    lib = ctypes.CDLL(dit.library_path())
    lib.dit_attn_check_exp2.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_longlong, ctypes.c_int,
                                                                ctypes.c_void_p]
    assert lib.dit_attn_check_exp2(None, A + MB, A + 2 * MB, 8, 3, None) == 1      # null x
    assert lib.dit_attn_check_exp2(A, A + MB, A + 2 * MB, 0, 3, None) == 1         # n = 0
    assert lib.dit_attn_check_exp2(A, A + MB, A + 2 * MB, 8, 4, None) == 1         # degree 4
    assert lib.dit_attn_check_exp2(A + 2, A + MB, A + 2 * MB, 8, 3, None) == 1     # misaligned
    assert lib.dit_attn_check_exp2(A, A + 16, A + 2 * MB, 8, 3, None) == 1         # overlap
