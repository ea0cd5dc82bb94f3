"""Helpers shared by the GPU parity tests (device copies, tolerance checks)."""
import numpy as np

# bf16-output tolerance of the layer: max |err| <= 3e-2 RMS(oracle), mean |err| <= 5e-3 RMS(oracle)
MAX_REL = 3e-2
MEAN_REL = 5e-3


def dev(a):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).cuda()


def host(t, dtype=None):
    a = t.detach().cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


def bf16_dev_to_f32(t) -> np.ndarray:
    a = t.detach().cpu().numpy().view(np.uint16)
    return (a.astype(np.uint32) << np.uint32(16)).view(np.float32)


def rms(ref) -> float:
    return float(np.sqrt(np.mean(np.asarray(ref, dtype=np.float64) ** 2)))


def assert_close_rms(got, ref, max_rel=MAX_REL, mean_rel=MEAN_REL, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    r = rms(ref)
    err = np.abs(got - ref)
    if r == 0.0:
        assert err.max() == 0.0, f"{what}: expected exact zeros"
        return
    assert err.max() <= max_rel * r, f"{what}: max|err|/rms = {err.max() / r:.3e}"
    assert err.mean() <= mean_rel * r, f"{what}: mean|err|/rms = {err.mean() / r:.3e}"


# The gate/up intermediate h = SiLU(g) * u is a product of two near-Gaussian
# dot products (max |h| ~ 15-20 RMS). Its error is driven by the bf16(q * s)
# weight rounding of g and u (relative 2^-9 per weight, ~2^-9/sqrt(3) of a
# K-term dot product's size), multiplied by the other factor, so it scales with
# |g| and |u| rather than with |h|. Emulating exactly that arithmetic on the CPU
# (bf16 weights, exact accumulation, bf16 output) gives max |err| up to
# 0.053 RMS(h) on the test shapes, mean 0.0015 RMS; the bound for h is
# 8e-2 RMS max (1.5x that), 5e-3 RMS mean. The down rows y = W2 h are near
# Gaussian and keep the layer's own bound (emulated max 0.017 RMS).
H_MAX_REL = 8e-2


def assert_close_h(got, ref, what=""):
    assert_close_rms(got, ref, max_rel=H_MAX_REL, mean_rel=MEAN_REL, what=what)
