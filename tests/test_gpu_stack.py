"""The layer stack on the GPU, x <- x + MoE_l(RMSNorm(x)), against the oracle.

Teacher-forced: each layer's GPU output is checked against the oracle's
stack_layer applied to that layer's GPU input, so errors do not compound
through the check; the whole stack in one call must equal the layer-by-layer
calls bit for bit."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close_rms, bf16_dev_to_f32, dev, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,H", [(37, 7168), (5, 256), (1, 8), (300, 512)])
def test_rmsnorm_within_one_bf16_step_of_the_oracle(cuda_lib, T, H):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    x = synth.normal_bf16((T, H), 3.0, T, 77)
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    B.moe_rmsnorm(dev(x), T, H, 1e-6, out)
    got = bf16_dev_to_f32(out).astype(np.float64)
    ref = oracle.rmsnorm(oracle.bf16_to_f32(x), 1e-6).astype(np.float64)
    # fp32 sums in another order may move the bf16 rounding by one step, never more
    step = np.abs(ref) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(got - ref) <= step)
    exact = oracle.bf16_to_f32(oracle.f32_to_bf16(ref.astype(np.float32)))
    assert np.mean(got == exact) > 0.99


def make_stack(shape, L, T, seed0=0):
    from w4a16_mixture_experts_sigmoid_gb300.layer import MoeW4A16Layer, MoeW4A16Stack
    arrays = [synth.make_layer(shape, seed=seed0 + l) for l in range(L)]
    layers = [MoeW4A16Layer.from_arrays(shape, a) for a in arrays]
    logits = [synth.make_tokens(T, shape.H, shape.E, seed=seed0 + l)[1] for l in range(L)]
    x, _ = synth.make_tokens(T, shape.H, shape.E, seed=seed0)
    return arrays, layers, MoeW4A16Stack(layers), x, logits


def teacher_forced(arrays, layers, stack_cls, x, logits, k, tokens=None):
    """Runs the layers one call each; checks every layer against the oracle. Returns the last output."""
    cur = dev(x)
    for l, (a, lay) in enumerate(zip(arrays, layers)):
        one = stack_cls([lay])
        nxt = one.forward(cur, [dev(logits[l])])
        assert one.check_status() == 0
        xin = host(cur, np.uint16)
        ref = oracle.stack_layer(xin, logits[l], a, k, tokens=tokens)
        got = bf16_dev_to_f32(nxt)[ref["tokens"]]
        assert_close_rms(got, ref["out"], what=f"layer {l}")
        cur = nxt
    return cur


def test_tiny_stack_teacher_forced_and_one_call_equals_chained(cuda_lib):
    from w4a16_mixture_experts_sigmoid_gb300.layer import MoeW4A16Stack
    arrays, layers, stack, x, logits = make_stack(synth.TINY, 3, 16)
    chained = teacher_forced(arrays, layers, MoeW4A16Stack, x, logits, synth.TINY.top_k)
    whole = stack.forward(dev(x), [dev(v) for v in logits])
    assert stack.check_status() == 0
    assert np.array_equal(host(whole), host(chained))
    # the layers add something of the residual's own size (the check is not on an identity)
    delta = bf16_dev_to_f32(whole).astype(np.float64) - oracle.bf16_to_f32(x)
    assert np.sqrt(np.mean(delta ** 2)) > 0.2 * np.sqrt(np.mean(oracle.bf16_to_f32(x).astype(np.float64) ** 2))


def test_stack_in_place(cuda_lib):
    arrays, layers, stack, x, logits = make_stack(synth.TINY, 2, 9, seed0=5)
    want = host(stack.forward(dev(x), [dev(v) for v in logits]))
    xd = dev(x)
    stack.forward(xd, [dev(v) for v in logits], out=xd)
    assert np.array_equal(host(xd), want)


@pytest.mark.slow
def test_full_size_twelve_layer_stack_teacher_forced(cuda_lib):
    """The benchmarked stack (12 full-size layers, T = 256; layer l's weights and logits seed l,
    x seed 0): every layer against the oracle on its own seeded 16-token sample, fed the GPU's
    input of that layer; then the whole stack in one call equals the chained calls bit for bit.
    One layer's host arrays exist at a time."""
    import os
    from w4a16_mixture_experts_sigmoid_gb300.layer import MoeW4A16Layer, MoeW4A16Stack
    shape, T, L = synth.FULL, 256, 12
    x, _ = synth.make_tokens(T, shape.H, shape.E, seed=0)
    layers, logits = [], []
    cur = dev(x)
    for l in range(L):
        arrays = synth.make_layer(shape, seed=l)
        lay = MoeW4A16Layer.from_arrays(shape, arrays)
        lg = synth.make_tokens(T, shape.H, shape.E, seed=l)[1]
        one = MoeW4A16Stack([lay])
        nxt = one.forward(cur, [dev(lg)])
        assert one.check_status() == 0
        tokens = np.sort(np.random.default_rng(l).choice(T, 16, replace=False))
        ref = oracle.stack_layer(host(cur, np.uint16), lg, arrays, shape.top_k, tokens=tokens,
                                 workers=os.cpu_count() or 1)
        assert_close_rms(bf16_dev_to_f32(nxt)[tokens], ref["out"], what=f"layer {l}")
        del arrays, ref
        layers.append(lay)
        logits.append(lg)
        cur = nxt
    stack = MoeW4A16Stack(layers)
    whole = stack.forward(dev(x), [dev(v) for v in logits])
    assert stack.check_status() == 0
    assert np.array_equal(host(whole), host(cur))


def test_tiny_stack_with_shared_experts_teacher_forced(cuda_lib):
    """Layers with a bf16 shared expert: x + (routed + shared)(RMSNorm(x)), every layer."""
    from w4a16_mixture_experts_sigmoid_gb300.layer import MoeW4A16Layer, MoeW4A16Stack
    shape = synth.LayerShape(E=8, top_k=2, H=256, I=128, shared_I=128)
    T, L = 12, 2
    arrays = [synth.make_layer(shape, seed=40 + l) for l in range(L)]
    layers = [MoeW4A16Layer.from_arrays(shape, a) for a in arrays]
    logits = [synth.make_tokens(T, shape.H, shape.E, seed=40 + l)[1] for l in range(L)]
    x, _ = synth.make_tokens(T, shape.H, shape.E, seed=40)
    cur = dev(x)
    for l in range(L):
        one = MoeW4A16Stack([layers[l]])
        nxt = one.forward(cur, [dev(logits[l])])
        assert one.check_status() == 0
        ref = oracle.stack_layer(host(cur, np.uint16), logits[l], arrays[l], shape.top_k, with_shared=True)
        assert_close_rms(bf16_dev_to_f32(nxt), ref["out"], what=f"layer {l}")
        cur = nxt
    whole = MoeW4A16Stack(layers).forward(dev(x), [dev(v) for v in logits])
    assert np.array_equal(host(whole), host(cur))
