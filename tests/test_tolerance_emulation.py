"""Where the intermediate-h tolerance comes from (no GPU).

The grouped GEMMs feed the tensor cores bf16(q * s) weights, accumulate in
fp32 and round their outputs to bf16 once. This test emulates exactly that
arithmetic on the CPU (bf16-rounded weights, fp64 sums standing in for an
accumulation with no further rounding, one bf16 rounding of the output) on the
very inputs of the GPU GEMM tests, measures its error against the fp32 oracle,
and checks that the bounds the GPU tests use cover it: the h bound with the
stated margin, y within the layer's own bound.
"""
import numpy as np
import pytest

import oracle
from tests.gpu_util import GEMM_SHAPES, H_MARGIN, H_MAX_REL, MAX_REL, MEAN_REL, gemm_problem


def bf16_round(v):
    return oracle.bf16_to_f32(oracle.f32_to_bf16(np.asarray(v, dtype=np.float32))).astype(np.float64)


def emulate_rows(layer, offsets, a_gu, a_dn):
    """bf16 weights, exact sums, SiLU(g) * u in fp64, bf16 outputs: h and y of every row."""
    R = a_gu.shape[0]
    I = layer["w2"].shape[-1] * 8
    owner = np.searchsorted(offsets, np.arange(R), side="right") - 1
    h = np.zeros((R, I))
    y = np.zeros((R, layer["w2"].shape[1]))
    for e in np.unique(owner):
        rows = np.nonzero(owner == e)[0]
        W13 = bf16_round(oracle.dequant(layer["w13"][e], layer["s13"][e]))
        gu = oracle.bf16_to_f32(a_gu[rows]).astype(np.float64) @ W13.T
        g, u = gu[:, :I], gu[:, I:]
        h[rows] = bf16_round(g / (1.0 + np.exp(-g)) * u)
        W2 = bf16_round(oracle.dequant(layer["w2"][e], layer["s2"][e]))
        y[rows] = bf16_round(oracle.bf16_to_f32(a_dn[rows]).astype(np.float64) @ W2.T)
    return h, y


def rel_errors(got, ref):
    ref = np.asarray(ref, dtype=np.float64)
    r = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref)
    return err.max() / r, err.mean() / r


@pytest.fixture(scope="module")
def emulated():
    res = {}
    for shape in GEMM_SHAPES:
        layer, offsets, a_gu, a_dn, ref_h, ref_y = gemm_problem(*shape)
        h, y = emulate_rows(layer, offsets, a_gu, a_dn)
        res[shape] = (rel_errors(h, ref_h), rel_errors(y, ref_y))
    return res


def test_h_bound_covers_the_emulated_error_with_margin(emulated):
    worst_max = max(v[0][0] for v in emulated.values())
    worst_mean = max(v[0][1] for v in emulated.values())
    # the figure the bound rests on: h's emulated error is well above the layer's 3e-2 ...
    assert worst_max > MAX_REL
    # ... and the bound keeps the stated margin over it
    assert worst_max * H_MARGIN <= H_MAX_REL, worst_max
    assert worst_mean * H_MARGIN <= MEAN_REL, worst_mean


def test_y_keeps_the_layer_bound(emulated):
    worst_max = max(v[1][0] for v in emulated.values())
    worst_mean = max(v[1][1] for v in emulated.values())
    assert worst_max * H_MARGIN <= MAX_REL, worst_max
    assert worst_mean * H_MARGIN <= MEAN_REL, worst_mean


def test_emulation_reports(emulated, capsys):
    """The per-shape figures, printed for the record (-s shows them)."""
    with capsys.disabled():
        for shape, ((hm, ha), (ym, ya)) in emulated.items():
            print(f"\n{shape}: h max {hm:.4f} mean {ha:.5f} RMS; y max {ym:.4f} mean {ya:.5f} RMS")


def test_layer_emulation_tail_reaches_the_stated_bound():
    """On a small layer whose expert 0 takes every one of 300 tokens, the intended arithmetic itself
    lands at the stated 3e-2: the reason the extra test shapes compare against it."""
    import synth
    from tests.gpu_util import MAX_REL, emulated_layer, rms
    E, k, H, I, T = 8, 2, 256, 128, 300
    arrays = synth.make_layer(synth.LayerShape(E=E, top_k=k, H=H, I=I), seed=E + T)
    x, logits = synth.make_tokens(T, H, E, seed=E + T + 1)
    logits[:, 0] += 40.0
    ref = oracle.moe_layer(x, logits, arrays, k)["out"].astype(np.float64)
    emu = emulated_layer(x, logits, arrays, k)
    worst = np.abs(emu - ref).max() / rms(ref)
    assert 0.8 * MAX_REL < worst < 1.5 * MAX_REL, worst
