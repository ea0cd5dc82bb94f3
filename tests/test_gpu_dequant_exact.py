"""The tensor-core kernels' int4 -> bf16 conversion, bit for bit.

A down GEMM over one-hot activation rows returns single dequantised weights: row j of expert e,
one-hot at input i, gives y[j, n] = W2_e[n, i] * 1 exactly in the fp32 output. Each must equal
bf16(q * s) of the oracle's exact product, rounded once to nearest even ("Kimi-K2.6" catalog
page, QUANT and PARAMS: symmetric int4, group size 32). The scales cover both forms of the
kernel's conversion: ordinary group scales, and larger, negative, subnormal, zero and boundary
scales that take the other form."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu

E, H, I = 2, 128, 512


def scale_bits(rng, special_share):
    """[E, H, I/32] bf16 scales: ordinary ones (the conversion's fma form), and with special_share
    > 0 a share of every class that needs its other form, placed at random."""
    n = E * H * (I // 32)
    s = synth.f32_to_bf16_bits(rng.uniform(0.005, 0.02, size=n).astype(np.float32))
    if special_share == 0:
        return s.reshape(E, H, I // 32)
    special = np.array([
        0x3C00, 0x3CFF,   # exponent field 120: 2^-7 .. below 2^-6 (ordinary form)
        0x3D00, 0x3D7F,   # exponent 122: 2^-5 and just below 2^-4 (other form)
        0x3CFF | 0x8000,  # negative, ordinary form
        0x0080, 0x0081,   # exponent 1: the smallest normal scales (ordinary form)
        0x0001, 0x007F, 0x8005,   # subnormal scales (other form)
        0x0000, 0x8000,   # zero scales
        0x3E80, 0x3F80, 0x40F0, 0xBF00, 0x4700,   # 0.25, 1, 7.5, -0.5, 32768
        0x3D4C, 0xBC23,   # 0.05, -0.00995
    ], dtype=np.uint16)
    idx = rng.choice(n, size=int(n * special_share), replace=False)
    s[idx] = special[rng.integers(0, len(special), size=idx.size)]
    return s.reshape(E, H, I // 32)


def problem(special_share, seed=0):
    rng = np.random.default_rng(seed)
    layer = {
        "w13": synth.random_words((E, 2 * I, H // 8), seed, 101),
        "s13": synth.uniform_bf16((E, 2 * I, H // 32), 0.005, 0.02, seed, 102),
        "w2": synth.random_words((E, H, I // 8), seed, 103),
        "s2": scale_bits(rng, special_share),
    }
    T = E * I                                   # one row per (expert, input): top_k = 1
    offsets = np.arange(E + 1, dtype=np.int32) * I
    rows = np.zeros((T, I), dtype=np.uint16)
    rows[np.arange(T), np.arange(T) % I] = 0x3F80   # bf16 1.0
    # the exact products q*s (exact in fp32: 4-bit by 8-bit significands), [E, H, I]
    exact = np.stack([oracle.dequant(layer["w2"][e], layer["s2"][e]) for e in range(E)])
    return layer, offsets, rows, exact


def impl_flags(B, impl):
    T = B.MOE_FLAG_TOKENS_PER_TILE
    return {"tmem-auto": 0, "tmem-16": T(16), "tmem-32": T(32), "tmem-128": T(128),
            "smem-32": B.MOE_FLAG_A_SMEM | T(32), "pair-16": B.MOE_FLAG_GEMM_PAIR | T(16),
            "pair-128": B.MOE_FLAG_GEMM_PAIR | T(128), "simt": B.MOE_FLAG_GEMM_SIMT}[impl]


@pytest.mark.parametrize("special_share", [0.0, 0.002, 0.33], ids=["ordinary", "few-special", "third-special"])
@pytest.mark.parametrize("impl", ["tmem-auto", "tmem-16", "tmem-32", "tmem-128", "smem-32", "pair-16",
                                  "pair-128", "simt"])
def test_dequantised_weights_are_bf16_of_q_times_s_bit_for_bit(cuda_lib, impl, special_share):
    """Tensor-core paths: bf16(q*s) rounded once. The CUDA-core baseline multiplies in fp32 and
    keeps the exact product q*s. Ordinary scales only, a few special ones (most warps' stages
    keep the fma form, some switch), and a third special (nearly every stage switches)."""
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    layer, offsets, rows, exact = problem(special_share)
    T = rows.shape[0]
    d = B.dims(E, 1, H, I)
    tens = {key: dev(v) for key, v in layer.items()}
    w = B.weights(tens["w13"], tens["s13"], tens["w2"], tens["s2"])
    ws = torch.zeros(B.moe_workspace_size(d, T), dtype=torch.uint8, device="cuda")
    y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    B.moe_w4a16_grouped_gemm(B.MOE_GEMM_DOWN, d, w, dev(rows), T, dev(offsets), y, ws,
                             impl_flags(B, impl) | B.MOE_FLAG_OUT_F32)
    assert B.moe_check_status(ws) == B.MOE_OK
    got = y.cpu().numpy().reshape(E, I, H).transpose(0, 2, 1)   # [E, H, I]
    want = exact if impl == "simt" else oracle.bf16_to_f32(oracle.f32_to_bf16(exact))
    gb, wb = got.view(np.uint32), want.view(np.uint32)
    zero = (wb & 0x7FFFFFFF) == 0
    assert np.array_equal(gb[~zero], wb[~zero]), f"{np.count_nonzero(gb[~zero] != wb[~zero])} weights differ"
    # a zero product's sign depends on the form (q*s against n*S + C); its value does not
    assert np.all((gb[zero] & 0x7FFFFFFF) == 0)
