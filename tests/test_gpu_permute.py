"""Step 2 on the GPU: expert-sorted permutation and gather, bit-exact vs the oracle."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import dev, host

pytestmark = pytest.mark.gpu


def run_permute(B, ids: np.ndarray, E: int, H: int = 64, gather: bool = True):
    import torch
    T, k = ids.shape
    idd = dev(ids.astype(np.int32))
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    srt = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    inv = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(256 + 4 * E * ((T * k + 4095) // 4096) + 256, dtype=torch.uint8, device="cuda")
    x = xp = None
    xh = None
    if gather:
        xh = np.random.default_rng(T).integers(0, 1 << 16, size=(T, H), dtype=np.uint16)
        x = dev(xh)
        xp = torch.zeros((T * k, H), dtype=torch.int16, device="cuda")
    B.moe_permute(idd, T, E, k, off, srt, inv, x, H, xp, ws)
    status = B.moe_check_status(ws)
    xp_nat = host(xp, np.uint16).copy() if gather else None
    if gather:
        # the same gather in the tensor-core K order: every block of 8 inputs as [0,4,1,5,2,6,3,7]
        B.moe_permute(idd, T, E, k, off, srt, inv, x, H, xp, ws, B.MOE_FLAG_ROWS_MMA_ORDER)
        got = host(xp, np.uint16)
        perm = np.array([0, 4, 1, 5, 2, 6, 3, 7])
        assert np.array_equal(got, xp_nat.reshape(T * k, H // 8, 8)[:, :, perm].reshape(T * k, H))
    return host(off), host(srt), host(inv), xp_nat, xh, status


@pytest.mark.parametrize("T,E,k,skew", [(16, 8, 2, None), (64, 384, 8, None), (4096, 384, 8, None),
                                        (1, 1, 1, None), (1000, 5, 3, None), (700, 64, 8, "one"),
                                        (5000, 1024, 2, None), (333, 33, 7, "half"),
                                        (512, 1024, 8, None),     # 4096 assignments: the one-block path's largest
                                        (513, 384, 8, "one")])    # 4104: two segments
def test_permute_bit_exact(cuda_lib, T, E, k, skew):
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    rng = np.random.default_rng(T * 7 + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    if skew == "one":
        logits[:, 3] += 50.0          # expert 3 in every token
    elif skew == "half":
        logits[:, : E // 2] -= 50.0   # half of the experts never chosen
    ids, _, _ = oracle.route(logits, k)
    off, srt, inv, xp, xh, status = run_permute(B, ids, E)
    r_off, r_srt, r_inv = oracle.permute(ids, E)
    assert status == B.MOE_OK
    assert np.array_equal(off, r_off)
    assert np.array_equal(srt, r_srt)
    assert np.array_equal(inv, r_inv)
    assert np.array_equal(xp, xh[r_srt])


def test_permute_out_of_range_ids_are_reported_not_written(cuda_lib):
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    E = 8
    ids = np.array([[0, 1], [9, 2], [-1, 3], [7, 7000]], dtype=np.int32)
    off, srt, inv, _, _, status = run_permute(B, ids, E, gather=False)
    assert status == B.MOE_ERR_DEVICE_BOUNDS
    valid = (ids >= 0) & (ids < E)
    assert np.all(inv.reshape(ids.shape)[~valid] == -1)
    assert off[-1] == valid.sum()
    counts = np.bincount(ids[valid], minlength=E)
    assert np.array_equal(np.diff(off), counts)
    kept = np.sort(inv.reshape(-1)[valid.reshape(-1)])
    assert np.array_equal(kept, np.arange(valid.sum()))
