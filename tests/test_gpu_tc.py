"""The tensor-core path: operand layouts of tcgen05.mma and path selection.

The layout self-test multiplies two bf16 tiles through the four descriptor
forms the chunked scan uses and compares with a plain fp32 matmul of the same
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


def test_tcgen05_operand_layouts():
    g = torch.Generator(device="cpu").manual_seed(5)
    A = torch.randn((128, 128), generator=g).to(torch.bfloat16).to(DEV)
    B = torch.randn((128, 128), generator=g).to(torch.bfloat16).to(DEV)
    sss.device_status(clear=True)
    out = sss.tcgen05_selftest(A, B)
    torch.cuda.synchronize()
    assert sss.device_status() == 0
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
