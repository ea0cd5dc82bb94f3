"""The routed bank in host memory: moe_stage_experts copies exactly the experts
that received rows (the others' device places keep what they held), and
moe_forward_offload gives the bits of moe_forward on a resident bank."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import bf16_dev_to_f32, dev, host, assert_close_rms

pytestmark = pytest.mark.gpu


def pinned(a):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).pin_memory()


def banks(B, arrays, fill=True):
    """(host bank tensors, host moe_weights_t, device bank tensors filled with a pattern, device moe_weights_t)"""
    import torch
    ht = {k: pinned(arrays[k]) for k in ("w13", "s13", "w2", "s2")}
    dt = {k: torch.full_like(ht[k], 0x5A5A if ht[k].dtype == torch.int16 else 0x5A5A5A5A, device="cuda")
          for k in ht}
    return ht, B.host_weights(ht["w13"], ht["s13"], ht["w2"], ht["s2"]), dt, \
        B.weights(dt["w13"], dt["s13"], dt["w2"], dt["s2"])


def test_stage_copies_exactly_the_touched_experts(cuda_lib):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    shape = synth.LayerShape(E=33, top_k=5, H=288, I=96)
    arrays = synth.make_layer(shape, seed=21)
    ht, hw, dt, dw = banks(B, arrays)
    counts = np.zeros(33, dtype=np.int64)
    counts[[0, 5, 6, 31, 32]] = [3, 1, 7, 2, 9]              # first, middle pair, last two
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    B.moe_stage_experts(B.dims(33, 5, 288, 96), hw, dev(offsets), dw)
    torch.cuda.synchronize()
    for k in ("w13", "s13", "w2", "s2"):
        got = dt[k].cpu().numpy()
        want = ht[k].numpy()
        pattern = np.full_like(want[0], want.dtype.type(0x5A5A if want.dtype == np.int16 else 0x5A5A5A5A))
        for e in range(33):
            if counts[e] > 0:
                assert np.array_equal(got[e], want[e]), (k, e)
            else:
                assert np.array_equal(got[e], pattern), (k, e)


@pytest.mark.parametrize("E,k,H,I,T", [(33, 5, 288, 96, 37), (8, 2, 256, 128, 16), (64, 6, 512, 256, 3)])
def test_forward_offload_equals_resident_forward(cuda_lib, E, k, H, I, T):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    from w4a16_mixture_experts_sigmoid_gb300.layer import MoeW4A16Layer
    shape = synth.LayerShape(E=E, top_k=k, H=H, I=I)
    arrays = synth.make_layer(shape, seed=E + T)
    x, logits = synth.make_tokens(T, H, E, seed=E + T + 1)
    resident = MoeW4A16Layer.from_arrays(shape, arrays)
    want = resident.forward(dev(x), dev(logits))
    _, hw, _, dw = banks(B, arrays)
    ws = torch.zeros(B.moe_workspace_size(resident.dims, T), dtype=torch.uint8, device="cuda")
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    for _ in range(2):                      # a second call re-stages over the first one's copies
        B.moe_forward_offload(resident.dims, hw, dw, dev(x), dev(logits), T, out, ws)
        assert B.moe_check_status(ws) == B.MOE_OK
        assert torch.equal(out, want)
    assert_close_rms(bf16_dev_to_f32(out), oracle.moe_layer(x, logits, arrays, k)["out"], what="offload")


def test_any_device_accessible_bank_is_staged(cuda_lib):
    """The source bank only has to be readable by the GPU: a bank in device memory stages the same way
    (a device-to-device copy), so the call's contract is about addressability, not placement."""
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    shape = synth.LayerShape(E=8, top_k=2, H=256, I=128)
    arrays = synth.make_layer(shape, seed=2)
    src = {kk: dev(arrays[kk]) for kk in ("w13", "s13", "w2", "s2")}
    dst = {kk: torch.zeros_like(v) for kk, v in src.items()}
    counts = np.array([1, 0, 2, 0, 0, 0, 0, 3], dtype=np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    B.moe_stage_experts(B.dims(8, 2, 256, 128), B.weights(src["w13"], src["s13"], src["w2"], src["s2"]),
                        dev(offsets), B.weights(dst["w13"], dst["s13"], dst["w2"], dst["s2"]))
    torch.cuda.synchronize()
    for kk in src:
        for e in range(8):
            if counts[e]:
                assert torch.equal(dst[kk][e], src[kk][e])
            else:
                assert int(dst[kk][e].abs().sum()) == 0


@pytest.mark.slow
def test_full_size_decode_offload_bit_exact(cuda_lib):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    from w4a16_mixture_experts_sigmoid_gb300.layer import MoeW4A16Layer
    arrays = synth.make_layer(synth.FULL, seed=0)
    resident = MoeW4A16Layer.from_arrays(synth.FULL, arrays)
    x, logits = synth.make_tokens(64, 7168, 384, seed=0)
    want = resident.forward(dev(x), dev(logits))
    _, hw, _, dw = banks(B, arrays)
    ws = torch.zeros(B.moe_workspace_size(resident.dims, 64), dtype=torch.uint8, device="cuda")
    out = torch.empty((64, 7168), dtype=torch.int16, device="cuda")
    B.moe_forward_offload(resident.dims, hw, dw, dev(x), dev(logits), 64, out, ws)
    assert B.moe_check_status(ws) == B.MOE_OK
    assert torch.equal(out, want)
