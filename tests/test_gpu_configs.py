"""Full-size layers on the GPU (384 experts, top-8, hidden 7168, intermediate
2048, int4 group 32), in the launch configuration the benchmark times:
routing and permutation bit-exact on every token; layer outputs against the
oracle on every token of the decode batch, on a seeded 256-token sample of
the 4096-token prefill, on every token of the shared-expert sweep up to
T = 128 and a 128-token sample at T = 512."""
import os

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close_rms, bf16_dev_to_f32, dev, host

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def full_layer(cuda_lib):
    from w4a16_mixture_experts_sigmoid_gb300.layer import MoeW4A16Layer
    arrays = synth.make_layer(synth.FULL_WITH_SHARED, seed=0)
    routed = {k: arrays[k] for k in ("w13", "s13", "w2", "s2")}
    layer = MoeW4A16Layer.from_arrays(synth.FULL, routed)
    shared = MoeW4A16Layer(384, 8, 7168, 2048, layer.w13, layer.s13, layer.w2, layer.s2,
                           dev(arrays["sh_gu"]), dev(arrays["sh_d"]))
    return arrays, layer, shared


def routing_bit_exact(B, layer, x, logits):
    import torch
    T, E, k = logits.shape[0], 384, 8
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    B.moe_route(dev(logits), T, E, k, ids, w)
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    srt = torch.empty(T * k, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
    B.moe_permute(ids, T, E, k, off, srt, inv, None, 0, None, layer.workspace(T))
    r_ids, r_w, _ = oracle.route(logits, k)
    r_off, r_srt, r_inv = oracle.permute(r_ids, E)
    assert np.array_equal(host(ids), r_ids)
    assert np.array_equal(host(w).view(np.uint32), r_w.view(np.uint32))
    assert np.array_equal(host(off), r_off)
    assert np.array_equal(host(srt), r_srt)
    assert np.array_equal(host(inv), r_inv)
    return r_off


WORKERS = os.cpu_count() or 1


def sampled_parity(arrays, layer, x, logits, tokens, with_shared=False, flags=0):
    out = layer.forward(dev(x), dev(logits), flags=flags)
    assert layer.check_status() == 0
    got = bf16_dev_to_f32(out)[tokens]
    ref = oracle.moe_layer(x, logits, arrays, 8, tokens=tokens, with_shared=with_shared, workers=WORKERS)["out"]
    assert_close_rms(got, ref, what=f"{len(tokens)} tokens")
    return got


def test_decode_T64(full_layer):
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    arrays, layer, _ = full_layer
    x, logits = synth.make_tokens(64, 7168, 384, seed=0)
    off = routing_bit_exact(B, layer, x, logits)
    assert (np.diff(off) > 0).sum() > 250          # near-uniform load touches most experts
    sampled_parity(arrays, layer, x, logits, np.arange(64))


@pytest.mark.parametrize("variant", ["smem", "tokens32", "simt", "pair"])
def test_decode_T64_other_paths(full_layer, variant):
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    arrays, layer, _ = full_layer
    x, logits = synth.make_tokens(64, 7168, 384, seed=0)
    flags = {"smem": B.MOE_FLAG_A_SMEM, "tokens32": B.MOE_FLAG_TOKENS_PER_TILE(32),
             "simt": B.MOE_FLAG_GEMM_SIMT, "pair": B.MOE_FLAG_GEMM_PAIR}[variant]
    sampled_parity(arrays, layer, x, logits, np.arange(0, 64, 8), flags=flags)


def test_prefill_T4096_zipf(full_layer):
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    arrays, layer, _ = full_layer
    bias = synth.zipf_bias(384, 4096, 8, 1.1, 0)
    x, logits = synth.make_tokens(4096, 7168, 384, seed=0, bias=bias)
    off = routing_bit_exact(B, layer, x, logits)
    counts = np.sort(np.diff(off))[::-1]
    assert counts[0] > 2000 and counts[0] > 20 * np.median(counts)   # skewed load
    tokens = np.sort(np.random.default_rng(0).choice(4096, 256, replace=False))
    sampled_parity(arrays, layer, x, logits, tokens)


@pytest.mark.parametrize("T", [1, 8, 32, 128, 512])
def test_decode_sweep_with_shared_expert(full_layer, T):
    arrays, _, shared = full_layer
    x, logits = synth.make_tokens(T, 7168, 384, seed=T)
    tokens = np.arange(T) if T <= 128 else np.sort(np.random.default_rng(0).choice(T, 128, replace=False))
    sampled_parity(arrays, shared, x, logits, tokens, with_shared=True)
