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


# Intermediate rows of the grouped GEMMs (h = SiLU(g) * u, y = W2 h) are stored
# in bf16 and are heavy-tailed (h is a product of two near-Gaussian values:
# max|h| is ~20 RMS), so their own storage rounding (half a bf16 ulp, 2^-9
# relative) can exceed a fixed fraction of the RMS. Their bound is per
# element: twice that rounding of the value itself, plus 1e-2 RMS for the
# bf16(q * s) weight rounding accumulated over K (~2^-9 / sqrt(3) RMS).
def assert_close_rows(got, ref, rel=2.0 ** -8, abs_rms=1e-2, mean_rel=MEAN_REL, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    r = rms(ref)
    err = np.abs(got - ref)
    bound = rel * np.abs(ref) + abs_rms * r
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"{what}: err {err[worst]:.3e} > bound {bound[worst]:.3e} at {worst}"
    assert err.mean() <= mean_rel * r, f"{what}: mean|err|/rms = {err.mean() / r:.3e}"
