"""Steps 3 and 4 on the GPU: the grouped W4A16 GEMMs vs the oracle, every row,
for the tensor-core kernel (A in tensor memory, A in shared memory, every
token-tile size) and the CUDA-core baseline, on shapes that span several
tiles and ragged tails."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close_rows, bf16_dev_to_f32, dev

pytestmark = pytest.mark.gpu

# (E, k, H, I, T, skew)
SHAPES = [
    (8, 2, 256, 128, 16, None),        # the tiny layer
    (5, 3, 288, 96, 37, None),         # K tails: H % 256 != 0, I % 64 != 0
    (3, 2, 512, 256, 200, None),       # several token chunks per expert
    (1, 1, 1024, 512, 300, None),      # one expert owns every row
    (16, 4, 2048, 1024, 64, "half"),   # deep K, empty experts
]


def impl_flags(B):
    T = B.MOE_FLAG_TOKENS_PER_TILE
    return {
        "tmem-auto": 0, "tmem-16": T(16), "tmem-32": T(32), "tmem-64": T(64), "tmem-128": T(128),
        "smem-16": B.MOE_FLAG_A_SMEM | T(16), "smem-32": B.MOE_FLAG_A_SMEM | T(32),
        "simt": B.MOE_FLAG_GEMM_SIMT,
    }


_cache = {}


def problem(E, k, H, I, T, skew):
    key = (E, k, H, I, T, skew)
    if key not in _cache:
        layer = synth.make_layer(synth.LayerShape(E=E, top_k=k, H=H, I=I), seed=E + H)
        logits = np.random.default_rng(T).standard_normal((T, E)).astype(np.float32)
        if skew == "half":
            logits[:, ::2] -= 60.0
        ids, _, _ = oracle.route(logits, k)
        offsets, _, _ = oracle.permute(ids, E)
        R = T * k
        a_gu = synth.normal_bf16((R, H), 1.0, 7, 100)
        a_dn = synth.normal_bf16((R, I), 4.0, 7, 101)
        ref_h = oracle.gateup_rows(a_gu, offsets, layer, range(R))
        ref_y = oracle.down_rows(a_dn, offsets, layer, range(R))
        _cache[key] = (layer, offsets, a_gu, a_dn, ref_h, ref_y)
    return _cache[key]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"E{s[0]}k{s[1]}H{s[2]}I{s[3]}T{s[4]}" for s in SHAPES])
@pytest.mark.parametrize("impl", ["tmem-auto", "tmem-16", "tmem-32", "tmem-64", "tmem-128", "smem-16", "smem-32",
                                  "simt"])
def test_grouped_gemms_match_oracle(cuda_lib, shape, impl):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    E, k, H, I, T, skew = shape
    layer, offsets, a_gu, a_dn, ref_h, ref_y = problem(*shape)
    flags = impl_flags(B)[impl]
    R = T * k
    d = B.dims(E, k, H, I)
    tens = {key: dev(v) for key, v in layer.items()}
    w = B.weights(tens["w13"], tens["s13"], tens["w2"], tens["s2"])
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    off = dev(offsets)
    h = torch.full((R, I), 0x7FC0, dtype=torch.int16, device="cuda")     # NaN fill: unwritten rows show up
    y = torch.full((R, H), 0x7FC0, dtype=torch.int16, device="cuda")
    B.moe_w4a16_grouped_gemm(B.MOE_GEMM_GATEUP_SILU, d, w, dev(a_gu), T, off, h, ws, flags)
    B.moe_w4a16_grouped_gemm(B.MOE_GEMM_DOWN, d, w, dev(a_dn), T, off, y, ws, flags)
    assert B.moe_check_status(ws) == B.MOE_OK
    assert_close_rows(bf16_dev_to_f32(h), ref_h, what=f"gate/up {impl}")
    assert_close_rows(bf16_dev_to_f32(y), ref_y, what=f"down {impl}")


def test_unsupported_tile_size_is_rejected(cuda_lib):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    layer, offsets, a_gu, _, _, _ = problem(*SHAPES[0])
    tens = {key: dev(v) for key, v in layer.items()}
    w = B.weights(tens["w13"], tens["s13"], tens["w2"], tens["s2"])
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    h = torch.empty((32, 128), dtype=torch.int16, device="cuda")
    for flags in (B.MOE_FLAG_TOKENS_PER_TILE(48), B.MOE_FLAG_A_SMEM | B.MOE_FLAG_TOKENS_PER_TILE(64)):
        with pytest.raises(B.MoeError) as e:
            B.moe_w4a16_grouped_gemm(0, B.dims(8, 2, 256, 128), w, dev(a_gu), 16, dev(offsets), h, ws, flags)
        assert e.value.code == B.MOE_ERR_UNSUPPORTED_SHAPE
