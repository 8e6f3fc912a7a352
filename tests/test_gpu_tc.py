"""The tensor-core path: operand layouts of tcgen05.mma and path selection.

The layout self-test (a test-only library, tests/tc_selftest) multiplies two
bf16 tiles through the descriptor forms the chunked scan uses and compares with a plain fp32 matmul of the same
bf16 values (a hardware-layout check; the scan itself is checked against the
oracle in test_gpu_parity.py)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import selective_ssm_scan_gb300 as sss  # noqa: E402

DEV = torch.device("cuda:0")


def _selftest_lib():
    """The test-only library with the operand-layout kernels (built on demand
    from tests/tc_selftest/tc_selftest.cu; not part of libsss)."""
    import ctypes
    import importlib.util
    import os
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tc_selftest", "build.py")
    spec = importlib.util.spec_from_file_location("tc_selftest_build", here)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    lib = ctypes.CDLL(mod.build())
    lib.sss_test_tcgen05_layouts.restype = ctypes.c_int
    lib.sss_test_tcgen05_layouts.argtypes = [ctypes.c_void_p] * 5
    return lib


def test_tcgen05_operand_layouts():
    g = torch.Generator(device="cpu").manual_seed(5)
    A = torch.randn((128, 128), generator=g).to(torch.bfloat16).to(DEV)
    B = torch.randn((128, 128), generator=g).to(torch.bfloat16).to(DEV)
    out = torch.empty((9, 128, 128), dtype=torch.float32, device=DEV)
    status = torch.zeros((1,), dtype=torch.int32, device=DEV)
    lib = _selftest_lib()
    rc = lib.sss_test_tcgen05_layouts(A.data_ptr(), B.data_ptr(), out.data_ptr(),
                                      status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    assert int(status.item()) == 0
    ref = (A.double() @ B.double().T).float()
    names = ["K-major A and B", "MN-major A", "MN-major B", "A from tensor memory",
             "A from tensor memory, MN-major B", "MN-major A and B",
             "K-major A, N=128 MN-major B", "A from tensor memory, N=128 MN-major B",
             "MN-major A, N=128 MN-major B"]
    for i, name in enumerate(names):
        cols = 64 if 1 <= i <= 5 else 128
        err = (out[i, :, :cols] - ref[:, :cols]).abs().max().item()
        assert err <= 1e-3 * ref.abs().max().item(), f"{name}: max abs err {err}"


def test_scan_path_selection():
    bf, f32 = torch.bfloat16, torch.float32
    # head pairs share a B/C group: the two-head kernel
    assert sss.ssm_scan_path(8, 1024, 32, 64, 128, 1, f32, bf, bf) == 2
    assert sss.ssm_scan_path(8, 1024, 32, 64, 128, 1, bf, bf, bf) == 2
    assert sss.ssm_scan_path(2, 300, 8, 64, 128, 4, bf, bf, bf) == 2
    # an odd number of heads per group: one head per CTA
    assert sss.ssm_scan_path(2, 300, 3, 64, 128, 1, bf, bf, bf) == 1
    assert sss.ssm_scan_path(2, 300, 6, 64, 128, 2, bf, bf, bf) == 1
    assert sss.ssm_scan_path(1, 64, 2, 4, 8, 1, f32, f32, f32) == 0
    assert sss.ssm_scan_path(1, 64, 2, 64, 128, 1, f32, f32, f32) == 0
