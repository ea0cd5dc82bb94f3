"""4-bit float weights on the GPU (E2M1 codes, E4M3 scale per 16 inputs, fp32
scale per matrix): the grouped GEMMs against the oracle's row views on every
row, for every tile size and the CTA-pair kernel; the whole layer against the
oracle; the split calls chaining to exactly the layer's bits."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close_h, assert_close_rms, bf16_dev_to_f32, dev, host

pytestmark = pytest.mark.gpu

SHAPES = [
    (8, 2, 256, 128, 16),        # the tiny layer's shape
    (5, 3, 288, 96, 37),         # K tails (scales through plain loads)
    (3, 2, 512, 256, 200),       # several token chunks per expert
    (16, 4, 2048, 1024, 64),     # deep K
]


def fp4_weights(B, layer):
    t = {k: dev(v) for k, v in layer.items() if k != "fmt"}
    return B.weights_fp4(t["w13"], t["s13"], t["g13"], t["w2"], t["s2"], t["g2"]), t


@pytest.mark.parametrize("shape", SHAPES, ids=[f"E{s[0]}k{s[1]}H{s[2]}I{s[3]}T{s[4]}" for s in SHAPES])
@pytest.mark.parametrize("impl", ["auto", "16", "32", "64", "128", "pair"])
def test_fp4_grouped_gemms_match_oracle(cuda_lib, shape, impl):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    E, k, H, I, T = shape
    layer = synth.make_layer_fp4(synth.LayerShape(E=E, top_k=k, H=H, I=I), seed=E + H)
    logits = np.random.default_rng(T).standard_normal((T, E)).astype(np.float32)
    ids, _, _ = oracle.route(logits, k)
    offsets, _, _ = oracle.permute(ids, E)
    R = T * k
    a_gu = synth.normal_bf16((R, H), 1.0, 7, 100)
    a_dn = synth.normal_bf16((R, I), 4.0, 7, 101)
    ref_h = oracle.gateup_rows(a_gu, offsets, layer, range(R))
    ref_y = oracle.down_rows(a_dn, offsets, layer, range(R))
    flags = {"auto": 0, "pair": B.MOE_FLAG_GEMM_PAIR}.get(impl, 0)
    if impl.isdigit():
        flags = B.MOE_FLAG_TOKENS_PER_TILE(int(impl))
    d = B.dims(E, k, H, I, group=16)
    w, _ = fp4_weights(B, layer)
    ws = torch.zeros(B.moe_workspace_size(d, T), dtype=torch.uint8, device="cuda")
    off = dev(offsets)
    h = torch.full((R, I), 0x7FC0, dtype=torch.int16, device="cuda")
    y = torch.full((R, H), float("nan"), dtype=torch.float32, device="cuda")
    B.moe_fp4_grouped_gemm(B.MOE_GEMM_GATEUP_SILU, d, w, dev(a_gu), T, off, h, ws, flags)
    B.moe_fp4_grouped_gemm(B.MOE_GEMM_DOWN, d, w, dev(a_dn), T, off, y, ws, flags | B.MOE_FLAG_OUT_F32)
    assert B.moe_check_status(ws) == B.MOE_OK
    assert_close_h(bf16_dev_to_f32(h), ref_h, what=f"fp4 gate/up {impl}")
    assert_close_rms(host(y), ref_y, what=f"fp4 down {impl}")


@pytest.mark.parametrize("E,k,H,I,T", [(8, 2, 256, 128, 16), (33, 5, 288, 96, 37), (64, 6, 512, 256, 300)])
def test_fp4_layer_matches_oracle_and_split_calls(cuda_lib, E, k, H, I, T):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    from w4a16_mixture_experts_sigmoid_gb300.layer import MoeFp4Layer
    shape = synth.LayerShape(E=E, top_k=k, H=H, I=I)
    layer_h = synth.make_layer_fp4(shape, seed=E + T)
    x, logits = synth.make_tokens(T, H, E, seed=E + T + 1)
    layer = MoeFp4Layer.from_arrays(shape, layer_h)
    out = layer.forward(dev(x), dev(logits))
    assert layer.check_status() == 0
    ref = oracle.moe_layer(x, logits, layer_h, k)["out"]
    assert_close_rms(bf16_dev_to_f32(out), ref, what="fp4 layer")
    # the same layer through the split calls, rows in the tensor-core K order, y in fp32
    R = T * k
    ws = layer.workspace(T)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    srt = torch.empty(R, dtype=torch.int32, device="cuda")
    inv = torch.empty(R, dtype=torch.int32, device="cuda")
    xp = torch.empty((R, H), dtype=torch.int16, device="cuda")
    h = torch.empty((R, I), dtype=torch.int16, device="cuda")
    y = torch.empty((R, H), dtype=torch.float32, device="cuda")
    o2 = torch.empty((T, H), dtype=torch.int16, device="cuda")
    order = B.MOE_FLAG_ROWS_MMA_ORDER
    B.moe_route(dev(logits), T, E, k, ids, w)
    B.moe_permute(ids, T, E, k, off, srt, inv, dev(x), H, xp, ws, order)
    B.moe_fp4_grouped_gemm(0, layer.dims, layer.weights, xp, T, off, h, ws, order)
    B.moe_fp4_grouped_gemm(1, layer.dims, layer.weights, h, T, off, y, ws, order | B.MOE_FLAG_OUT_F32)
    B.moe_combine_f32(y, inv, w, T, k, H, None, o2)
    assert B.moe_check_status(ws) == B.MOE_OK
    assert torch.equal(out, o2)


def test_fp4_rejects_what_it_does_not_run(cuda_lib):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    shape = synth.LayerShape(E=8, top_k=2, H=256, I=128)
    layer = synth.make_layer_fp4(shape, seed=1)
    w, _ = fp4_weights(B, layer)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    a = torch.zeros((32, 256), dtype=torch.int16, device="cuda")
    off = dev(np.array([0, 32] + [32] * 7, dtype=np.int32))
    h = torch.empty((32, 128), dtype=torch.int16, device="cuda")
    for flags, code in ((B.MOE_FLAG_GEMM_SIMT, B.MOE_ERR_UNSUPPORTED_SHAPE),
                        (B.MOE_FLAG_A_SMEM, B.MOE_ERR_UNSUPPORTED_SHAPE)):
        with pytest.raises(B.MoeError) as ex:
            B.moe_fp4_grouped_gemm(0, B.dims(8, 2, 256, 128, group=16), w, a, 16, off, h, ws, flags)
        assert ex.value.code == code
    with pytest.raises(B.MoeError) as ex:      # group 32 is the INT4 bank's
        B.moe_fp4_grouped_gemm(0, B.dims(8, 2, 256, 128), w, a, 16, off, h, ws, 0)
    assert ex.value.code == B.MOE_ERR_UNSUPPORTED_SHAPE


@pytest.mark.slow
def test_fp4_full_size_decode_T64(cuda_lib):
    import os
    from w4a16_mixture_experts_sigmoid_gb300.layer import MoeFp4Layer
    shape = synth.FULL
    arrays = synth.make_layer_fp4(shape, seed=0)
    layer = MoeFp4Layer.from_arrays(shape, arrays)
    x, logits = synth.make_tokens(64, shape.H, shape.E, seed=0)
    out = layer.forward(dev(x), dev(logits))
    assert layer.check_status() == 0
    ref = oracle.moe_layer(x, logits, arrays, 8, workers=os.cpu_count() or 1)["out"]
    assert_close_rms(bf16_dev_to_f32(out), ref, what="fp4 decode T=64, all tokens")


@pytest.mark.parametrize("impl", ["auto", "16", "128", "pair"])
def test_fp4_dequantised_weights_bit_for_bit(cuda_lib, impl):
    """One-hot down GEMMs (fp32 output) read single weights back: row j of expert e, one-hot at input
    i, gives e2m1 * e4m3 * g, the exact product of the code and the block scale times the matrix
    scale rounded once in fp32, as the oracle computes it. The scale bytes span every finite E4M3
    code, subnormal to 448."""
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    E, H, I = 2, 128, 512
    layer = synth.make_layer_fp4(synth.LayerShape(E=E, top_k=1, H=H, I=I), seed=5)
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)   # every finite code
    layer["s2"] = codes[np.random.default_rng(6).integers(0, codes.size, size=layer["s2"].shape)]
    T = E * I
    offsets = np.arange(E + 1, dtype=np.int32) * I
    rows = np.zeros((T, I), dtype=np.uint16)
    rows[np.arange(T), np.arange(T) % I] = 0x3F80   # bf16 1.0
    want = np.stack([oracle.dequant_fp4(layer["w2"][e], layer["s2"][e], layer["g2"][e]) for e in range(E)])
    flags = {"auto": 0, "pair": B.MOE_FLAG_GEMM_PAIR | B.MOE_FLAG_TOKENS_PER_TILE(128)}.get(impl, 0)
    if impl.isdigit():
        flags = B.MOE_FLAG_TOKENS_PER_TILE(int(impl))
    d = B.dims(E, 1, H, I, group=16)
    w, _ = fp4_weights(B, layer)
    ws = torch.zeros(B.moe_workspace_size(d, T), dtype=torch.uint8, device="cuda")
    y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    B.moe_fp4_grouped_gemm(B.MOE_GEMM_DOWN, d, w, dev(rows), T, dev(offsets), y, ws, flags | B.MOE_FLAG_OUT_F32)
    assert B.moe_check_status(ws) == B.MOE_OK
    got = host(y).reshape(E, I, H).transpose(0, 2, 1)
    gb, wb = got.view(np.uint32), np.ascontiguousarray(want).view(np.uint32)
    zero = (wb & 0x7FFFFFFF) == 0
    assert np.array_equal(gb[~zero], wb[~zero]), f"{np.count_nonzero(gb[~zero] != wb[~zero])} weights differ"
    assert np.all((gb[zero] & 0x7FFFFFFF) == 0)
