"""moe_permute_static_scratch, the permutation entry point that allocates
nothing: it must give exactly what the oracle's permutation and moe_permute
give, call after call, with no device memory taken or freed by the call.

Collected last (file name) so that it also runs after every other GPU test in
the same process; it must pass alone as well."""
import gc

import numpy as np
import pytest

import oracle
from tests.gpu_util import dev, host

pytestmark = pytest.mark.gpu


def _ids(rng, T, E, k):
    # k distinct experts per token, as the router gives them
    return np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)


def _outputs(T, E, k, H):
    import torch
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    srt = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    inv = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    xp = torch.zeros((T * k, H), dtype=torch.int16, device="cuda")
    return off, srt, inv, xp


def _with_workspace(B, ids_d, x, T, E, k, H, flags):
    import torch
    off, srt, inv, xp = _outputs(T, E, k, H)
    ws = torch.zeros(256 + 4 * E * ((T * k + 4095) // 4096), dtype=torch.uint8, device="cuda")
    B.moe_permute(ids_d, T, E, k, off, srt, inv, x, H, xp, ws, flags)
    assert B.moe_check_status(ws) == B.MOE_OK
    return [host(t) for t in (off, srt, inv, xp)]


@pytest.mark.parametrize("T,E,k,H,flags", [(64, 384, 8, 7168, 0x4), (4096, 384, 8, 256, 0),
                                           (100_000, 384, 8, 64, 0x4), (333, 33, 7, 8, 0)])
def test_static_scratch_matches_moe_permute_twice_without_allocating(cuda_lib, T, E, k, H, flags):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    rng = np.random.default_rng(T + E)
    status = torch.zeros(64, dtype=torch.int32, device="cuda")   # must start at 0
    x = dev(rng.integers(0, 1 << 16, size=(T, H), dtype=np.uint16))
    xh = host(x, np.uint16)
    for call in range(2):
        # a different routing on each call: nothing may carry over through the shared scratch
        ids = _ids(rng, T, E, k)
        ids_d = dev(ids)
        want = _with_workspace(B, ids_d, x, T, E, k, H, flags)
        off, srt, inv, xp = _outputs(T, E, k, H)
        torch.cuda.synchronize()
        # garbage left by earlier tests is freed now, not by a collection inside the measured call
        gc.collect()
        gc.disable()
        try:
            used0 = torch.cuda.memory_allocated()
            free0 = torch.cuda.mem_get_info()[0]
            B.moe_permute_static_scratch(ids_d, T, E, k, off, srt, inv, x, H, xp, status, flags)
            torch.cuda.synchronize()
            used1 = torch.cuda.memory_allocated()
            free1 = torch.cuda.mem_get_info()[0]
        finally:
            gc.enable()
        # nothing of this process's memory came or went (the strict check) ...
        assert used1 == used0
        if call == 1:
            # ... and, after the first call's set-up, the device's free memory did not drop by an
            # allocation's worth; other processes may share this GPU, so this one is approximate
            assert free1 >= free0 - (2 << 20)
        assert B.moe_check_status(status) == B.MOE_OK
        got = [host(t) for t in (off, srt, inv, xp)]
        for name, g, w in zip(("expert_offsets", "sorted_token_ids", "inv_perm", "x_perm"), got, want):
            assert np.array_equal(g, w), f"call {call}: {name} differs from moe_permute"
        # and directly against the oracle's stable expert sort
        r_off, r_srt, r_inv = oracle.permute(ids, E)
        assert np.array_equal(got[0], r_off) and np.array_equal(got[1], r_srt) and np.array_equal(got[2], r_inv)
        rows = xh[r_srt]
        if flags & 0x4:      # x_perm rows in the tensor-core K order
            rows = rows.reshape(T * k, H // 8, 8)[:, :, [0, 4, 1, 5, 2, 6, 3, 7]].reshape(T * k, H)
        assert np.array_equal(got[3].view(np.uint16), rows)


def test_static_scratch_reports_out_of_range_ids(cuda_lib):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    T, E, k = 16, 8, 2
    ids = _ids(np.random.default_rng(1), T, E, k)
    ids[3, 1] = E          # outside [0, E)
    off, srt, inv, _ = _outputs(T, E, k, 8)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_permute_static_scratch(dev(ids), T, E, k, off, srt, inv, None, 0, None, status)
    assert B.moe_check_status(status) == B.MOE_ERR_DEVICE_BOUNDS
    assert host(inv)[3 * k + 1] == -1
    assert host(off)[E] == T * k - 1


def test_static_scratch_rejects_sizes_beyond_its_array(cuda_lib):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    E, k = 1024, 8
    # histograms of 4 * E * ceil(T*k / 4096) bytes: 1 MiB holds 256 segments of 1024 experts
    T_fit = 256 * 4096 // k
    T_over = T_fit + 1
    one = torch.zeros(8, dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoeError) as ex:
        B.moe_permute_static_scratch(one, T_over, E, k, one, one, one, None, 0, None, None)
    assert ex.value.code == B.MOE_ERR_WORKSPACE_TOO_SMALL
    assert 4 * E * ((T_fit * k + 4095) // 4096) == B.MOE_PERMUTE_STATIC_SCRATCH_BYTES
