"""The whole layer on the GPU (moe_forward and friends) vs the oracle on small
shapes: every token, every path, the edge cases, the shared expert, combine
alone, host-buffer entry, determinism and the bounded-wait status path."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close_layer, assert_close_rms, bf16_dev_to_f32, dev, host

pytestmark = pytest.mark.gpu


def make(E, k, H, I, T, seed=0, shared_I=0, skew=None):
    shape = synth.LayerShape(E=E, top_k=k, H=H, I=I, shared_I=shared_I)
    arrays = synth.make_layer(shape, seed=seed)
    x, logits = synth.make_tokens(T, H, E, seed=seed + 1)
    if skew == "one":
        logits[:, 0] += 40.0
    return shape, arrays, x, logits


def gpu_forward(shape, arrays, x, logits, flags=0):
    from w4a16_mixture_experts_sigmoid_gb300.layer import MoeW4A16Layer
    layer = MoeW4A16Layer.from_arrays(shape, arrays)
    out = layer.forward(dev(x), dev(logits), flags=flags)
    assert layer.check_status() == 0
    return bf16_dev_to_f32(out), layer


CASES = [
    (8, 2, 256, 128, 16, None),     # tiny layer
    (1, 1, 64, 32, 5, None),        # one expert
    (2, 2, 96, 64, 1, None),        # one token, k == E
    (33, 5, 288, 96, 37, None),     # ragged everything
    (8, 2, 256, 128, 300, "one"),   # expert 0 in every token: many token chunks
    (64, 6, 512, 256, 3, None),     # most experts empty
]


@pytest.mark.parametrize("case", CASES, ids=[f"E{c[0]}k{c[1]}H{c[2]}I{c[3]}T{c[4]}" for c in CASES])
@pytest.mark.parametrize("path", ["tmem", "smem", "simt"])
def test_forward_matches_oracle(cuda_lib, case, path):
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    E, k, H, I, T, skew = case
    flags = {"tmem": 0, "smem": B.MOE_FLAG_A_SMEM, "simt": B.MOE_FLAG_GEMM_SIMT}[path]
    shape, arrays, x, logits = make(E, k, H, I, T, seed=E + T, skew=skew)
    got, _ = gpu_forward(shape, arrays, x, logits, flags)
    ref = oracle.moe_layer(x, logits, arrays, k)["out"]
    if case[:5] == (8, 2, 256, 128, 16):
        assert_close_rms(got, ref, what=f"forward {path}")      # the tiny layer config: the stated bound
    else:
        assert_close_layer(got, ref, x, logits, arrays, k, what=f"forward {path}")


def test_forward_T0_is_a_noop(cuda_lib):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    shape, arrays, _, _ = make(8, 2, 256, 128, 1)
    from w4a16_mixture_experts_sigmoid_gb300.layer import MoeW4A16Layer
    layer = MoeW4A16Layer.from_arrays(shape, arrays)
    before = B.moe_launch_count()
    x = torch.empty((0, 256), dtype=torch.int16, device="cuda")
    lg = torch.empty((0, 8), dtype=torch.float32, device="cuda")
    out = torch.empty((0, 256), dtype=torch.int16, device="cuda")
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    B.moe_forward(layer.dims, layer.weights, x, lg, 0, out, ws)
    assert B.moe_launch_count() == before


def test_zero_weights_and_shared_only(cuda_lib):
    shape, arrays, x, logits = make(8, 2, 256, 128, 9, shared_I=64)
    arrays["w13"][:] = np.uint32(0x88888888).view(np.int32)
    arrays["w2"][:] = np.uint32(0x88888888).view(np.int32)
    got, _ = gpu_forward(shape, arrays, x, logits)
    ref = oracle.moe_layer(x, logits, arrays, 2, with_shared=True)["out"]
    assert_close_rms(got, ref, what="shared only")
    plain = dict(arrays)
    del plain["sh_gu"], plain["sh_d"]
    got0, _ = gpu_forward(synth.LayerShape(E=8, top_k=2, H=256, I=128), plain, x, logits)
    assert np.all(got0 == 0)


@pytest.mark.parametrize("Is,T", [(64, 5), (128, 40), (192, 70)])
@pytest.mark.parametrize("simt", [False, True])
def test_shared_expert_and_layer_with_shared(cuda_lib, Is, T, simt):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    shape, arrays, x, logits = make(8, 2, 256, 128, T, shared_I=Is)
    flags = B.MOE_FLAG_GEMM_SIMT if simt else 0
    got, layer = gpu_forward(shape, arrays, x, logits, flags)
    ref = oracle.moe_layer(x, logits, arrays, 2, with_shared=True)["out"]
    assert_close_rms(got, ref, what="layer + shared")
    out = torch.empty((T, 256), dtype=torch.int16, device="cuda")
    B.moe_shared_expert(layer.dims, layer.weights, dev(x), T, out, layer.workspace(T), flags)
    ref_s = np.stack([oracle.shared_expert(oracle.bf16_to_f32(x[t]), arrays["sh_gu"], arrays["sh_d"])
                      for t in range(T)])
    assert_close_rms(bf16_dev_to_f32(out), ref_s, what="shared expert")


def test_combine_alone_rounds_once(cuda_lib):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    rng = np.random.default_rng(3)
    T, k, E, H = 50, 4, 12, 264
    ids, w, _ = oracle.route(rng.standard_normal((T, E)).astype(np.float32), k)
    _, _, inv = oracle.permute(ids, E)
    y = synth.normal_bf16((T * k, H), 3.0, 1, 1)
    add = synth.normal_bf16((T, H), 1.0, 1, 2)
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    B.moe_combine(dev(y), dev(inv), dev(w), T, k, H, dev(add), out)
    ref = oracle.combine(oracle.bf16_to_f32(y), inv, w, oracle.bf16_to_f32(add))
    got = bf16_dev_to_f32(out)
    # one bf16 rounding of an fp32 sum: within half an ulp of bf16 (plus fp32 summation noise)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6 * np.abs(ref).max())


def test_combine_f32_rounds_once(cuda_lib):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    rng = np.random.default_rng(4)
    T, k, E, H = 61, 8, 40, 264
    ids, w, _ = oracle.route(rng.standard_normal((T, E)).astype(np.float32), k)
    _, _, inv = oracle.permute(ids, E)
    y = (rng.standard_normal((T * k, H)) * 30).astype(np.float32)
    add = rng.standard_normal((T, H)).astype(np.float32)
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    B.moe_combine_f32(dev(y), dev(inv), dev(w), T, k, H, dev(add), out)
    ref = oracle.combine(y, inv, w, add)
    got = bf16_dev_to_f32(out)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6 * np.abs(ref).max())
    out2 = torch.empty((T, H), dtype=torch.int16, device="cuda")
    B.moe_combine_f32(dev(y), dev(inv), dev(w), T, k, H, None, out2)
    ref2 = oracle.combine(y, inv, w)
    assert np.all(np.abs(bf16_dev_to_f32(out2) - ref2) <= 2.0 ** -8 * np.abs(ref2) + 1e-6 * np.abs(ref2).max())


def test_forward_host_equals_forward_and_is_deterministic(cuda_lib):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300.layer import MoeW4A16Layer
    shape, arrays, x, logits = make(33, 5, 288, 96, 37)
    layer = MoeW4A16Layer.from_arrays(shape, arrays)
    a = host(layer.forward(dev(x), dev(logits)), np.uint16).copy()
    b = host(layer.forward(dev(x), dev(logits)), np.uint16).copy()
    assert np.array_equal(a, b)
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    lh = torch.from_numpy(logits).pin_memory()
    oh = torch.empty((37, 288), dtype=torch.int16).pin_memory()
    layer.forward_host(xh, lh, oh)
    torch.cuda.synchronize()
    assert np.array_equal(oh.numpy().view(np.uint16), a)


def test_bounded_wait_expires_into_status_word(cuda_lib):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    B.moe_debug_expire_wait(ws, 5_000_000)              # 5 ms
    assert B.moe_check_status(ws) == B.MOE_ERR_DEVICE_TIMEOUT
    assert B.moe_check_status(ws) == B.MOE_OK          # reset after reading
    # the context is still usable
    shape, arrays, x, logits = make(8, 2, 256, 128, 16)
    got, _ = gpu_forward(shape, arrays, x, logits)
    assert_close_rms(got, oracle.moe_layer(x, logits, arrays, 2)["out"])
