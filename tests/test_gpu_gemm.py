"""Steps 3 and 4 on the GPU: the grouped W4A16 GEMMs vs the oracle, every row,
for the tensor-core kernel (A in tensor memory, A in shared memory, every
token-tile size) and the CUDA-core baseline, on shapes that span several
tiles and ragged tails."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import GEMM_SHAPES, assert_close_h, assert_close_rms, bf16_dev_to_f32, dev, gemm_problem

pytestmark = pytest.mark.gpu

SHAPES = GEMM_SHAPES


def impl_flags(B):
    T = B.MOE_FLAG_TOKENS_PER_TILE
    return {
        "tmem-auto": 0, "tmem-16": T(16), "tmem-32": T(32), "tmem-64": T(64), "tmem-128": T(128),
        "smem-16": B.MOE_FLAG_A_SMEM | T(16), "smem-32": B.MOE_FLAG_A_SMEM | T(32),
        "simt": B.MOE_FLAG_GEMM_SIMT,
        "pair-auto": B.MOE_FLAG_GEMM_PAIR, "pair-16": B.MOE_FLAG_GEMM_PAIR | T(16),
        "pair-32": B.MOE_FLAG_GEMM_PAIR | T(32), "pair-64": B.MOE_FLAG_GEMM_PAIR | T(64),
        "pair-128": B.MOE_FLAG_GEMM_PAIR | T(128),
    }


problem = gemm_problem


@pytest.mark.parametrize("shape", SHAPES, ids=[f"E{s[0]}k{s[1]}H{s[2]}I{s[3]}T{s[4]}" for s in SHAPES])
@pytest.mark.parametrize("impl", ["tmem-auto", "tmem-16", "tmem-32", "tmem-64", "tmem-128", "smem-16", "smem-32",
                                  "simt", "pair-auto", "pair-16", "pair-32", "pair-64", "pair-128"])
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
    ws = torch.zeros(B.moe_workspace_size(d, T), dtype=torch.uint8, device="cuda")
    off = dev(offsets)
    h = torch.full((R, I), 0x7FC0, dtype=torch.int16, device="cuda")     # NaN fill: unwritten rows show up
    y = torch.full((R, H), 0x7FC0, dtype=torch.int16, device="cuda")
    B.moe_w4a16_grouped_gemm(B.MOE_GEMM_GATEUP_SILU, d, w, dev(a_gu), T, off, h, ws, flags)
    B.moe_w4a16_grouped_gemm(B.MOE_GEMM_DOWN, d, w, dev(a_dn), T, off, y, ws, flags)
    assert B.moe_check_status(ws) == B.MOE_OK
    assert_close_h(bf16_dev_to_f32(h), ref_h, what=f"gate/up {impl}")
    assert_close_rms(bf16_dev_to_f32(y), ref_y, what=f"down {impl}")


def test_unsupported_tile_size_is_rejected(cuda_lib):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    layer, offsets, a_gu, _, _, _ = problem(*SHAPES[0])
    tens = {key: dev(v) for key, v in layer.items()}
    w = B.weights(tens["w13"], tens["s13"], tens["w2"], tens["s2"])
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    h = torch.empty((32, 128), dtype=torch.int16, device="cuda")
    for flags in (B.MOE_FLAG_TOKENS_PER_TILE(48), B.MOE_FLAG_A_SMEM | B.MOE_FLAG_TOKENS_PER_TILE(64)):
        with pytest.raises(B.MoeError) as e:
            B.moe_w4a16_grouped_gemm(0, B.dims(8, 2, 256, 128), w, dev(a_gu), 16, dev(offsets), h, ws, flags)
        assert e.value.code == B.MOE_ERR_UNSUPPORTED_SHAPE


CHAIN_CASES = [(33, 5, 288, 96, 37),
               (33, 5, 288, 96, 1),      # one token
               (33, 5, 288, 96, 3),
               (384, 8, 256, 128, 2),    # the full expert count and top-k
               (384, 8, 256, 128, 8),
               (1024, 8, 256, 128, 3)]   # E = 1024: the widest routing registers


@pytest.mark.parametrize("case", CHAIN_CASES, ids=[f"E{c[0]}k{c[1]}T{c[4]}" for c in CHAIN_CASES])
@pytest.mark.parametrize("simt", [False, True])
def test_split_calls_in_mma_order_chain_like_forward(cuda_lib, simt, case):
    """route -> permute -> gate/up -> down (fp32 rows) -> combine with the tensor-core K order
    for the exchanged rows gives exactly the bits of moe_forward."""
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    from w4a16_mixture_experts_sigmoid_gb300.layer import MoeW4A16Layer
    E, k, H, I, T = case
    shape = synth.LayerShape(E=E, top_k=k, H=H, I=I)
    arrays = synth.make_layer(shape, seed=3)
    x, logits = synth.make_tokens(T, H, E, seed=4)
    layer = MoeW4A16Layer.from_arrays(shape, arrays)
    flags = B.MOE_FLAG_GEMM_SIMT if simt else 0
    ref = layer.forward(dev(x), dev(logits), flags=flags).clone()
    R = T * k
    ws = torch.zeros(B.moe_workspace_size(layer.dims, T), dtype=torch.uint8, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    srt = torch.empty(R, dtype=torch.int32, device="cuda")
    inv = torch.empty(R, dtype=torch.int32, device="cuda")
    xp = torch.empty((R, H), dtype=torch.int16, device="cuda")
    h = torch.empty((R, I), dtype=torch.int16, device="cuda")
    y = torch.empty((R, H), dtype=torch.float32, device="cuda")     # the layer keeps y in fp32
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    order = 0 if simt else B.MOE_FLAG_ROWS_MMA_ORDER
    B.moe_route(dev(logits), T, E, k, ids, w)
    B.moe_permute(ids, T, E, k, off, srt, inv, dev(x), H, xp, ws, order)
    B.moe_w4a16_grouped_gemm(0, layer.dims, layer.weights, xp, T, off, h, ws, flags | order)
    B.moe_w4a16_grouped_gemm(1, layer.dims, layer.weights, h, T, off, y, ws, flags | order | B.MOE_FLAG_OUT_F32)
    B.moe_combine_f32(y, inv, w, T, k, H, None, out)
    assert B.moe_check_status(ws) == B.MOE_OK
    assert torch.equal(out, ref)


def test_mma_order_rows_give_the_same_products(cuda_lib):
    """The same rows handed over in natural order (converted inside) and in the
    tensor-core K order give bit-identical GEMM outputs."""
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    E, k, H, I, T, skew = SHAPES[1]
    layer, offsets, a_gu, a_dn, _, _ = problem(*SHAPES[1])
    tens = {key: dev(v) for key, v in layer.items()}
    w = B.weights(tens["w13"], tens["s13"], tens["w2"], tens["s2"])
    d = B.dims(E, k, H, I)
    R = T * k
    ws = torch.zeros(B.moe_workspace_size(d, T), dtype=torch.uint8, device="cuda")
    perm = np.array([0, 4, 1, 5, 2, 6, 3, 7])
    def mma(a):
        K = a.shape[1]
        return a.reshape(R, K // 8, 8)[:, :, perm].reshape(R, K)
    y0 = torch.empty((R, H), dtype=torch.int16, device="cuda")
    y1 = torch.empty((R, H), dtype=torch.int16, device="cuda")
    B.moe_w4a16_grouped_gemm(1, d, w, dev(a_dn), T, dev(offsets), y0, ws, 0)
    B.moe_w4a16_grouped_gemm(1, d, w, dev(mma(a_dn)), T, dev(offsets), y1, ws, B.MOE_FLAG_ROWS_MMA_ORDER)
    assert torch.equal(y0, y1)
    h0 = torch.empty((R, I), dtype=torch.int16, device="cuda")
    h1 = torch.empty((R, I), dtype=torch.int16, device="cuda")
    B.moe_w4a16_grouped_gemm(0, d, w, dev(a_gu), T, dev(offsets), h0, ws, 0)
    B.moe_w4a16_grouped_gemm(0, d, w, dev(mma(a_gu)), T, dev(offsets), h1, ws, B.MOE_FLAG_ROWS_MMA_ORDER)
    assert torch.equal(dev(mma(h0.cpu().numpy())), h1)     # h comes back in the same K order


@pytest.mark.parametrize("pair", [False, True])
def test_small_and_large_experts_split_between_launches(cuda_lib, pair):
    """With many rows per expert on average the GEMMs run one launch with 32-token tiles for the
    experts with up to 32 rows and one with 128-token tiles for the rest: every row of both,
    including experts right at the boundary and an empty one, matches the oracle."""
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    counts = np.array([1, 31, 32, 33, 64, 0, 128, 200], dtype=np.int64)    # mean 61 rows: 128-token choice
    E, k, H, I = len(counts), 1, 256, 128
    R = int(counts.sum())
    T = R
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    layer = synth.make_layer(synth.LayerShape(E=E, top_k=k, H=H, I=I), seed=31)
    a_gu = synth.normal_bf16((R, H), 1.0, 7, 102)
    a_dn = synth.normal_bf16((R, I), 4.0, 7, 103)
    ref_h = oracle.gateup_rows(a_gu, offsets, layer, range(R))
    ref_y = oracle.down_rows(a_dn, offsets, layer, range(R))
    d = B.dims(E, k, H, I)
    tens = {key: dev(v) for key, v in layer.items()}
    w = B.weights(tens["w13"], tens["s13"], tens["w2"], tens["s2"])
    ws = torch.zeros(B.moe_workspace_size(d, T), dtype=torch.uint8, device="cuda")
    off = dev(offsets)
    h = torch.full((R, I), 0x7FC0, dtype=torch.int16, device="cuda")
    y = torch.full((R, H), 0x7FC0, dtype=torch.int16, device="cuda")
    fl = B.MOE_FLAG_GEMM_PAIR if pair else 0
    B.moe_w4a16_grouped_gemm(B.MOE_GEMM_GATEUP_SILU, d, w, dev(a_gu), T, off, h, ws, fl)
    B.moe_w4a16_grouped_gemm(B.MOE_GEMM_DOWN, d, w, dev(a_dn), T, off, y, ws, fl)
    assert B.moe_check_status(ws) == B.MOE_OK
    assert_close_h(bf16_dev_to_f32(h), ref_h, what="gate/up split")
    assert_close_rms(bf16_dev_to_f32(y), ref_y, what="down split")


@pytest.mark.parametrize("impl", ["tmem-auto", "simt"])
def test_down_rows_in_fp32_are_the_unrounded_bf16_rows(cuda_lib, impl):
    """MOE_FLAG_OUT_F32: the same down products, not rounded: rounding them to bf16 gives the
    bf16 output bit for bit, and they match the oracle more closely than y's own bound."""
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    E, k, H, I, T, skew = SHAPES[2]
    layer, offsets, a_gu, a_dn, ref_h, ref_y = problem(*SHAPES[2])
    flags = impl_flags(B)[impl]
    R = T * k
    d = B.dims(E, k, H, I)
    tens = {key: dev(v) for key, v in layer.items()}
    w = B.weights(tens["w13"], tens["s13"], tens["w2"], tens["s2"])
    ws = torch.zeros(B.moe_workspace_size(d, T), dtype=torch.uint8, device="cuda")
    y16 = torch.empty((R, H), dtype=torch.int16, device="cuda")
    y32 = torch.full((R, H), float("nan"), dtype=torch.float32, device="cuda")
    B.moe_w4a16_grouped_gemm(1, d, w, dev(a_dn), T, dev(offsets), y16, ws, flags)
    B.moe_w4a16_grouped_gemm(1, d, w, dev(a_dn), T, dev(offsets), y32, ws, flags | B.MOE_FLAG_OUT_F32)
    assert B.moe_check_status(ws) == B.MOE_OK
    y32h = y32.cpu().numpy()
    assert np.array_equal(oracle.f32_to_bf16(y32h), y16.cpu().numpy().view(np.uint16))
    assert_close_rms(y32h, ref_y, what="down fp32")
    with pytest.raises(B.MoeError):
        B.moe_w4a16_grouped_gemm(0, d, w, dev(a_gu), T, dev(offsets), y32, ws, flags | B.MOE_FLAG_OUT_F32)
