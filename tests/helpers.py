"""Shared test helpers: moving synth arrays to torch, tolerance checks.

Tolerances (the contract of the forward and the update):
  * fp32-input runs: max|gpu - ref| <= 1e-5 * max|ref| per tensor;
  * bf16-input runs: y elementwise |gpu - ref| <= 1e-2 + 2e-2 |ref|,
    final / pool SSM states max|gpu - ref| <= 1e-3 * max|ref|;
  * conv states, pool slots, indices and untouched bytes: bit-exact.
"""
import numpy as np

Y_ATOL, Y_RTOL = 1e-2, 2e-2
STATE_REL = 1e-3
F32_REL = 1e-5


def to_torch(arr, dev):
    import torch
    if arr.dtype == "bf16":
        return torch.from_numpy(arr.data.view(np.int16).copy()).view(torch.bfloat16).to(dev)
    return torch.from_numpy(arr.data.copy()).to(dev)


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_y_close(gpu, ref, what="y"):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    if gpu.size == 0:
        return
    excess = np.abs(gpu - ref) - (Y_ATOL + Y_RTOL * np.abs(ref))
    i = int(np.argmax(excess))
    assert excess.flat[i] <= 0, (f"{what}: {int((excess > 0).sum())} of {excess.size} outside "
                                 f"tolerance; worst at {np.unravel_index(i, ref.shape)} "
                                 f"gpu={gpu.flat[i]} ref={ref.flat[i]}")


def max_rel(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    if gpu.size == 0:
        return 0.0
    den = np.abs(ref).max()
    return float(np.abs(gpu - ref).max() / (den if den > 0 else 1.0))


def assert_rel(gpu, ref, tol, what):
    r = max_rel(gpu, ref)
    assert r <= tol, f"{what}: max rel error {r:.3e} > {tol:.1e}"
