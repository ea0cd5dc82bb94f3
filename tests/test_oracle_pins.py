"""Pins of the CPU oracle to things other than itself (no GPU).

Each test checks the oracle against a closed form, a brute-force restatement
written independently here (pure Python, fp64 where it is arithmetic), an
invariant of the layer, or a value printed on the pages (tests/golden/).
"""
import math
import os
import struct

import numpy as np
import pytest

import oracle
from tests.conftest import GOLDEN

F32 = np.float32


# ---------------------------------------------------------------------------
# helpers written independently of the oracle
# ---------------------------------------------------------------------------

def bf16_bits_to_float(bits: int) -> float:
    return struct.unpack(">f", struct.pack(">I", (int(bits) & 0xFFFF) << 16))[0]


def brute_dequant_row(words_row, scales_row):
    """Pure-Python dequantisation of one row: list of floats."""
    out = []
    for c, w in enumerate(words_row):
        u = int(w) & 0xFFFFFFFF
        for j in range(8):
            q = ((u >> (4 * j)) & 0xF) - 8
            out.append(q * bf16_bits_to_float(scales_row[(8 * c + j) // 32]))
    return out


def brute_expert(x, w13, s13, w2, s2):
    """fp64 pure-Python gated-SiLU expert on one token."""
    I = len(w2[0]) * 8
    W13 = [brute_dequant_row(w13[n], s13[n]) for n in range(2 * I)]
    gu = [sum(a * b for a, b in zip(row, x)) for row in W13]
    h = [gu[i] / (1.0 + math.exp(-gu[i])) * gu[I + i] for i in range(I)]
    W2 = [brute_dequant_row(w2[n], s2[n]) for n in range(len(w2))]
    return [sum(a * b for a, b in zip(row, h)) for row in W2]


def rand_layer(E, H, I, seed, lo=0.005, hi=0.02):
    import synth
    return synth.make_layer(synth.LayerShape(E=E, top_k=1, H=H, I=I), seed=seed, scale_lo=lo, scale_hi=hi)


def ulp32(v):
    v = np.abs(np.asarray(v, dtype=np.float32))
    return (np.nextafter(v, F32(np.inf)) - v).astype(np.float64)


# ---------------------------------------------------------------------------
# weight format
# ---------------------------------------------------------------------------

def read_nibble_fixture():
    rows = []
    with open(os.path.join(GOLDEN, "nibble_layout.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            q = [int(v) for v in parts[:8]]
            word = np.array([int(parts[8], 16)], dtype=np.uint32).view(np.int32)[0]
            rows.append((q, word))
    return rows


def test_nibble_layout_worked_examples():
    for q, word in read_nibble_fixture():
        assert oracle.pack_int4(np.array([q]))[0, 0] == word
        assert list(oracle.unpack_int4(np.array([[word]], dtype=np.int32))[0]) == q


def test_pack_unpack_round_trip():
    rng = np.random.default_rng(3)
    q = rng.integers(-8, 8, size=(37, 96))
    assert np.array_equal(oracle.unpack_int4(oracle.pack_int4(q)), q)
    words = rng.integers(-2**31, 2**31, size=(5, 12), dtype=np.int64).astype(np.int32)
    assert np.array_equal(oracle.pack_int4(oracle.unpack_int4(words)), words)


def test_dequant_matches_brute_force():
    layer = rand_layer(1, 64, 32, seed=5)
    W = oracle.dequant(layer["w2"][0], layer["s2"][0])
    for n in (0, 7, 63):
        ref = brute_dequant_row(layer["w2"][0][n], layer["s2"][0][n])
        assert np.array_equal(W[n], np.array(ref, dtype=np.float32))   # exact products


def test_param_count_identity():
    """Three H x I int4 matrices per expert reproduce the page's int32-stored count."""
    vals = {}
    with open(os.path.join(GOLDEN, "kimi_k26_param_counts.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    per_expert = oracle.expert_int4_params(vals["hidden"], vals["moe_intermediate"])
    assert vals["moe_layers"] * vals["routed_experts"] * per_expert == vals["int32_stored_params"]
    # and the oracle's tensor shapes carry exactly that many int4 values
    layer = rand_layer(2, 64, 32, seed=1)
    n = layer["w13"][0].size * 8 + layer["w2"][0].size * 8
    assert n == oracle.expert_int4_params(64, 32)


# ---------------------------------------------------------------------------
# defined sigmoid
# ---------------------------------------------------------------------------

def test_sigmoid_special_values():
    s = oracle.sigmoid_def(np.array([0.0, -0.0, np.inf, -np.inf], dtype=np.float32))
    assert s[0] == F32(0.5) and s[1] == F32(0.5)
    assert s[2] == F32(1.0) and s[3] == F32(0.0)
    assert np.isnan(oracle.sigmoid_def(np.float32(np.nan)))
    assert oracle.exp_def(np.float32(0.0)) == F32(1.0)
    assert oracle.exp_def(np.float32(1.0)) == F32(math.e)      # within rounding: e rounds to the fp32 of e


def test_sigmoid_within_ulp_of_fp64():
    rng = np.random.default_rng(0)
    x = np.concatenate([np.linspace(-100, 100, 2_000_001, dtype=np.float32),
                        (rng.standard_normal(1_000_000) * 10).astype(np.float32),
                        (rng.standard_normal(200_000) * 1e-3).astype(np.float32)])
    s = oracle.sigmoid_def(x).astype(np.float64)
    ref = 1.0 / (1.0 + np.exp(-x.astype(np.float64)))
    keep = ref > 1e-37                               # fp32 normal range
    err = np.abs(s - ref)[keep] / ulp32(ref[keep])
    assert err.max() <= 3.0, err.max()
    t = np.linspace(-87, 88, 500_001, dtype=np.float32)
    e = oracle.exp_def(t).astype(np.float64)
    ref_e = np.exp(t.astype(np.float64))
    assert (np.abs(e - ref_e) / ulp32(ref_e)).max() <= 1.5


def test_sigmoid_monotone_and_symmetric():
    x = np.sort(np.random.default_rng(1).standard_normal(400_000).astype(np.float32) * 20)
    s = oracle.sigmoid_def(x)
    assert np.all(np.diff(s) >= 0)
    sym = s.astype(np.float64) + oracle.sigmoid_def(-x).astype(np.float64)
    assert np.abs(sym - 1.0).max() <= 4 * 2.0 ** -24


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------

def brute_topk(scores_row, k):
    """Rank by counting how many experts beat each one (O(E^2), pure Python)."""
    E = len(scores_row)
    key = [(-1.0 if math.isnan(v) else float(v)) for v in scores_row]
    rank = []
    for e in range(E):
        beaten_by = sum(1 for f in range(E) if key[f] > key[e] or (key[f] == key[e] and f < e))
        rank.append(beaten_by)
    ids = [None] * E
    for e, r in enumerate(rank):
        ids[r] = e
    return ids[:k]


@pytest.mark.parametrize("E,k", [(8, 2), (33, 5), (16, 16), (1, 1)])
def test_topk_matches_brute_force(E, k):
    rng = np.random.default_rng(E * 100 + k)
    logits = rng.standard_normal((40, E)).astype(np.float32)
    logits[0, :] = 0.0                                     # all tied
    if E >= 4:
        logits[1, :4] = [20.0, 25.0, 17.0, 30.0]           # distinct logits, equal fp32 scores
        logits[2, ::2] = np.inf
        logits[3, 1::2] = -np.inf
        logits[4, :] = np.float32(1.5)
    ids, w, s = oracle.route(logits, k)
    for t in range(logits.shape[0]):
        assert list(ids[t]) == brute_topk(s[t], k), t


def test_crafted_tie_goes_to_lowest_index():
    logits = np.full((1, 6), -3.0, dtype=np.float32)
    logits[0, [1, 2, 4]] = [20.0, 25.0, 30.0]             # sigmoid of each rounds to 1.0f
    ids, w, s = oracle.route(logits, 2)
    assert s[0, 1] == s[0, 2] == s[0, 4] == F32(1.0)
    assert list(ids[0]) == [1, 2]
    assert w[0, 0] == w[0, 1] == F32(0.5)


def test_weights_sum_to_one():
    rng = np.random.default_rng(7)
    for E, k in [(384, 8), (8, 2), (64, 6)]:
        logits = (rng.standard_normal((200, E)) * 4).astype(np.float32)
        _, w, _ = oracle.route(logits, k)
        assert np.abs(w.astype(np.float64).sum(1) - 1.0).max() <= k * 2.0 ** -24


def test_weights_when_every_score_underflows():
    logits = np.full((2, 5), -100.0, dtype=np.float32)
    ids, w, s = oracle.route(logits, 3)
    assert np.all(s == 0)
    assert list(ids[0]) == [0, 1, 2]
    assert np.all(w == F32(1.0) / F32(3))


def test_renormalisation_matches_fp64_within_rounding():
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((50, 32)).astype(np.float32)
    ids, w, s = oracle.route(logits, 4)
    for t in range(50):
        sel = [float(s[t, e]) for e in ids[t]]
        tot = sum(sel)
        for j in range(4):
            assert abs(float(w[t, j]) - sel[j] / tot) <= 3 * 2.0 ** -24


# ---------------------------------------------------------------------------
# permutation
# ---------------------------------------------------------------------------

def brute_permute(ids, E):
    T, k = ids.shape
    rows = []
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if ids[t, j] == e:
                    rows.append((t, j))
    counts = [sum(1 for (t, j) in rows if ids[t, j] == e) for e in range(E)]
    offsets = [0]
    for c in counts:
        offsets.append(offsets[-1] + c)
    inv = [0] * (T * k)
    for p, (t, j) in enumerate(rows):
        inv[t * k + j] = p
    return offsets, [t for (t, j) in rows], inv


@pytest.mark.parametrize("T,E,k", [(16, 8, 2), (37, 33, 5), (5, 1, 1), (64, 12, 12)])
def test_permute_matches_brute_force(T, E, k):
    rng = np.random.default_rng(T + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    ids, _, _ = oracle.route(logits, k)
    off, srt, inv = oracle.permute(ids, E)
    b_off, b_srt, b_inv = brute_permute(ids, E)
    assert list(off) == b_off and list(srt) == b_srt and list(inv) == b_inv


# ---------------------------------------------------------------------------
# expert MLP, combine, layer
# ---------------------------------------------------------------------------

def test_single_expert_top1_equals_dense_brute_force():
    import synth
    layer = rand_layer(1, 64, 32, seed=9)
    x_bits, logits = synth.make_tokens(3, 64, 1, seed=4)
    res = oracle.moe_layer(x_bits, logits, layer, k=1)
    assert np.all(res["weights"] == F32(1.0))
    for t in range(3):
        x = [bf16_bits_to_float(b) for b in x_bits[t]]
        ref = np.array(brute_expert(x, layer["w13"][0], layer["s13"][0], layer["w2"][0], layer["s2"][0]))
        got = res["out"][t].astype(np.float64)
        rms = np.sqrt(np.mean(ref ** 2))
        assert np.abs(got - ref).max() <= 1e-5 * rms + 1e-12


def brute_owner(offsets, r):
    """The expert owning expert-sorted row r, by a plain scan of the offsets."""
    owner = None
    for e in range(len(offsets) - 1):
        if offsets[e] <= r < offsets[e + 1]:
            assert owner is None
            owner = e
    assert owner is not None
    return owner


# Offsets with empty experts at the start, in the middle and at the end, and a
# second set whose last expert owns rows; every row sits next to a boundary.
ROW_OFFSETS = [[0, 0, 3, 3, 7, 8, 8], [0, 2, 2, 2, 5, 5, 6]]


@pytest.mark.parametrize("offsets", ROW_OFFSETS)
def test_gateup_rows_use_each_rows_own_expert(offsets):
    import synth
    E, H, I = len(offsets) - 1, 64, 32
    layer = rand_layer(E, H, I, seed=31)
    R = offsets[-1]
    a_bits = synth.normal_bf16((R, H), 1.0, 5, 0)
    rows = list(np.random.default_rng(1).permutation(R))          # any order of rows
    got = oracle.gateup_rows(a_bits, np.array(offsets, dtype=np.int32), layer, rows)
    for p, r in enumerate(rows):
        e = brute_owner(offsets, r)
        x = [bf16_bits_to_float(b) for b in a_bits[r]]
        W13 = [brute_dequant_row(layer["w13"][e][n], layer["s13"][e][n]) for n in range(2 * I)]
        gu = [sum(a * b for a, b in zip(row, x)) for row in W13]
        ref = np.array([gu[i] / (1.0 + math.exp(-gu[i])) * gu[I + i] for i in range(I)])
        assert np.abs(got[p] - ref).max() <= 1e-5 * np.sqrt(np.mean(ref ** 2)), (r, e)


@pytest.mark.parametrize("offsets", ROW_OFFSETS)
def test_down_rows_use_each_rows_own_expert(offsets):
    import synth
    E, H, I = len(offsets) - 1, 64, 32
    layer = rand_layer(E, H, I, seed=32)
    R = offsets[-1]
    h_bits = synth.normal_bf16((R, I), 4.0, 6, 0)
    rows = list(np.random.default_rng(2).permutation(R))
    got = oracle.down_rows(h_bits, np.array(offsets, dtype=np.int32), layer, rows)
    for p, r in enumerate(rows):
        e = brute_owner(offsets, r)
        h = [bf16_bits_to_float(b) for b in h_bits[r]]
        W2 = [brute_dequant_row(layer["w2"][e][n], layer["s2"][e][n]) for n in range(H)]
        ref = np.array([sum(a * b for a, b in zip(row, h)) for row in W2])
        assert np.abs(got[p] - ref).max() <= 1e-5 * np.sqrt(np.mean(ref ** 2)), (r, e)


def test_rows_of_neighbouring_experts_differ():
    """The experts of the row pins are distinct, so a row read with its neighbour's expert fails them."""
    E, H, I = 6, 64, 32
    layer = rand_layer(E, H, I, seed=31)
    import synth
    a = synth.normal_bf16((1, H), 1.0, 5, 0)
    outs = [oracle.gateup_rows(a, np.array([0] * e + [1] * (E + 1 - e), dtype=np.int32), layer, [0])[0]
            for e in range(1, E + 1)]
    for e in range(E - 1):
        assert np.abs(outs[e] - outs[e + 1]).max() > 0.1 * np.sqrt(np.mean(outs[e] ** 2))


def test_gate_and_up_are_not_interchangeable():
    """Swapping the gate and up halves changes the output (pins which half is the gate)."""
    layer = rand_layer(1, 64, 32, seed=2)
    x = oracle.bf16_to_f32(np.random.default_rng(0).integers(0x3000, 0x4000, 64).astype(np.uint16))
    y = oracle.expert_mlp(x, layer["w13"][0], layer["s13"][0], layer["w2"][0], layer["s2"][0])
    sw = np.concatenate([layer["w13"][0][32:], layer["w13"][0][:32]])
    ss = np.concatenate([layer["s13"][0][32:], layer["s13"][0][:32]])
    y2 = oracle.expert_mlp(x, sw, ss, layer["w2"][0], layer["s2"][0])
    assert not np.allclose(y, y2, rtol=1e-3)
    xs = [float(v) for v in x]
    ref = np.array(brute_expert(xs, layer["w13"][0], layer["s13"][0], layer["w2"][0], layer["s2"][0]))
    assert np.abs(y - ref).max() <= 1e-5 * np.sqrt(np.mean(ref ** 2))


def test_identical_experts_give_the_single_expert_output():
    import synth
    one = rand_layer(1, 64, 32, seed=12)
    layer = {key: np.repeat(v, 4, axis=0) for key, v in one.items()}
    x_bits, logits = synth.make_tokens(6, 64, 4, seed=8)
    res = oracle.moe_layer(x_bits, logits, layer, k=3)
    for t in range(6):
        y = oracle.expert_mlp(oracle.bf16_to_f32(x_bits[t]), one["w13"][0], one["s13"][0], one["w2"][0], one["s2"][0])
        assert np.abs(res["out"][t] - y).max() <= 4 * 2.0 ** -24 * np.abs(y).max()


def test_power_of_two_scale_doubles_exactly():
    layer = rand_layer(1, 64, 32, seed=13)
    x = oracle.bf16_to_f32(np.random.default_rng(1).integers(0x3000, 0x4000, 64).astype(np.uint16))
    y = oracle.expert_mlp(x, layer["w13"][0], layer["s13"][0], layer["w2"][0], layer["s2"][0])
    s2 = (oracle.bf16_to_f32(layer["s2"][0]) * 2).view(np.uint32) >> np.uint32(16)
    y2 = oracle.expert_mlp(x, layer["w13"][0], layer["s13"][0], layer["w2"][0], s2.astype(np.uint16))
    assert np.array_equal(y2, 2 * y)
    s13 = layer["s13"][0].copy()                      # double the up half only
    s13[32:] = ((oracle.bf16_to_f32(s13[32:]) * 2).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    y3 = oracle.expert_mlp(x, layer["w13"][0], s13, layer["w2"][0], layer["s2"][0])
    assert np.array_equal(y3, 2 * y)


def test_zero_weights_give_exact_zero_and_shared_only():
    import synth
    E, H, I = 3, 64, 32
    layer = rand_layer(E, H, I, seed=4)
    layer["w13"][:] = np.int32(np.uint32(0x88888888).view(np.int32))
    layer["w2"][:] = np.int32(np.uint32(0x88888888).view(np.int32))
    x_bits, logits = synth.make_tokens(4, H, E, seed=2)
    res = oracle.moe_layer(x_bits, logits, layer, k=2)
    assert np.all(res["out"] == 0)
    layer["sh_gu"] = synth.normal_bf16((2 * 32, H), 0.02, 0, 4)
    layer["sh_d"] = synth.normal_bf16((H, 32), 0.02, 0, 5)
    res = oracle.moe_layer(x_bits, logits, layer, k=2, with_shared=True)
    for t in range(4):
        x = [bf16_bits_to_float(b) for b in x_bits[t]]
        Wg = [[bf16_bits_to_float(b) for b in row] for row in layer["sh_gu"]]
        Wd = [[bf16_bits_to_float(b) for b in row] for row in layer["sh_d"]]
        gu = [sum(a * b for a, b in zip(r, x)) for r in Wg]
        h = [gu[i] / (1 + math.exp(-gu[i])) * gu[32 + i] for i in range(32)]
        ref = np.array([sum(a * b for a, b in zip(r, h)) for r in Wd])
        assert np.abs(res["out"][t] - ref).max() <= 1e-5 * np.abs(ref).max()


def test_combine_weighted_rank_order_sum():
    rng = np.random.default_rng(5)
    T, k, E, H = 7, 3, 5, 16
    ids, w, _ = oracle.route(rng.standard_normal((T, E)).astype(np.float32), k)
    off, srt, inv = oracle.permute(ids, E)
    y = rng.standard_normal((T * k, H)).astype(np.float32)
    out = oracle.combine(y, inv, w)
    for t in range(T):
        ref = [sum(float(w[t, j]) * float(y[inv[t * k + j], c]) for j in range(k)) for c in range(H)]
        assert np.abs(out[t] - np.array(ref)).max() <= 1e-6 * max(1.0, np.abs(ref).max())
    # the row of assignment (t, j) holds that token
    assert np.all(srt[inv] == np.repeat(np.arange(T), k))


def test_rmsnorm_unit_rms():
    x = np.random.default_rng(0).standard_normal((4, 256)).astype(np.float32) * 7
    n = oracle.rmsnorm(x)
    assert np.abs(np.sqrt(np.mean(n.astype(np.float64) ** 2, axis=1)) - 1).max() < 1e-5


# ---------------------------------------------------------------------------
# bf16 rounding and the layer stack
# ---------------------------------------------------------------------------

def nearest_bf16_bits(v: float) -> int:
    """Brute force: of the bf16 values bracketing v, the nearer; on a tie the one with an even pattern."""
    from fractions import Fraction
    u = struct.unpack(">I", struct.pack(">f", v))[0]
    lo = u >> 16
    cands = [lo, lo + 1]
    fv = Fraction(v)
    best = min(cands, key=lambda b: (abs(Fraction(bf16_bits_to_float(b)) - fv), b & 1))
    return best


def test_f32_to_bf16_rounds_to_nearest_even():
    one = 1.0
    cases = [one, one + 2.0 ** -8, one + 3 * 2.0 ** -8, one + 2.0 ** -8 + 2.0 ** -20, -(one + 2.0 ** -8),
             -(one + 3 * 2.0 ** -8), 3.0e38, 1e-40, 0.0, -0.0, 65504.0, 7.0]
    got = oracle.f32_to_bf16(np.array(cases, dtype=np.float32))
    assert got[0] == 0x3F80
    assert got[1] == 0x3F80            # tie -> even (down)
    assert got[2] == 0x3F82            # tie -> even (up)
    assert got[3] == 0x3F81            # just above the tie -> up
    assert got[4] == 0xBF80 and got[5] == 0xBF82
    assert got[8] == 0x0000 and got[9] == 0x8000
    vals = np.random.default_rng(3).standard_normal(2000).astype(np.float32) * np.float32(37.0)
    got = oracle.f32_to_bf16(vals)
    for v, g in zip(vals, got):
        assert int(g) == nearest_bf16_bits(float(v))
    assert oracle.f32_to_bf16(np.array([np.nan], dtype=np.float32))[0] & 0x7F80 == 0x7F80


def test_stack_layer_with_zero_weights_is_the_identity():
    import synth
    E, H, I = 3, 64, 32
    layer = rand_layer(E, H, I, seed=6)
    layer["w13"][:] = np.int32(np.uint32(0x88888888).view(np.int32))
    layer["w2"][:] = np.int32(np.uint32(0x88888888).view(np.int32))
    x_bits, logits = synth.make_tokens(5, H, E, seed=3)
    res = oracle.stack_layer(x_bits, logits, layer, k=2)
    assert np.array_equal(res["out"], oracle.bf16_to_f32(x_bits))


def test_stack_layer_single_expert_equals_brute_force():
    """E=1, top-1: x + MLP(bf16(x / sqrt(mean(x^2) + eps))), written out in fp64 loops."""
    import synth
    H, I, eps = 64, 32, 1e-6
    layer = rand_layer(1, H, I, seed=21)
    x_bits, logits = synth.make_tokens(3, H, 1, seed=5)
    res = oracle.stack_layer(x_bits, logits, layer, k=1, eps=eps)
    for t in range(3):
        x = [bf16_bits_to_float(b) for b in x_bits[t]]
        r = math.sqrt(sum(v * v for v in x) / H + eps)
        xn = [bf16_bits_to_float(nearest_bf16_bits(v / r)) for v in x]
        mlp = brute_expert(xn, layer["w13"][0], layer["s13"][0], layer["w2"][0], layer["s2"][0])
        ref = np.array([a + b for a, b in zip(x, mlp)])
        got = res["out"][t].astype(np.float64)
        # fp32 against fp64 normalisation may put a few inputs one bf16 step apart
        assert np.abs(got - ref).max() <= 1e-2 * np.sqrt(np.mean(np.array(mlp) ** 2)) + 1e-6
        assert np.abs(got - ref).mean() <= 1e-4 * np.sqrt(np.mean(np.array(mlp) ** 2)) + 1e-6


# ---------------------------------------------------------------------------
# the router's logit projection
# ---------------------------------------------------------------------------

def test_router_logits_match_fp64_dot_products():
    import synth
    T, E, H = 5, 7, 96
    x = synth.normal_bf16((T, H), 1.0, 3, 0)
    wg = synth.normal_bf16((E, H), 0.05, 3, 1)
    got = oracle.router_logits(x, wg)
    for t in range(T):
        xs = [bf16_bits_to_float(b) for b in x[t]]
        for e in range(E):
            ws = [bf16_bits_to_float(b) for b in wg[e]]
            exact = sum(a * b for a, b in zip(xs, ws))
            bound = H * 2.0 ** -24 * sum(abs(a * b) for a, b in zip(xs, ws))
            assert abs(float(got[t, e]) - exact) <= bound, (t, e)


def test_router_logits_scale_and_transpose():
    """Doubling the gate doubles every logit exactly; row e of the gate makes column e."""
    import synth
    x = synth.normal_bf16((4, 64), 1.0, 4, 0)
    wg = synth.normal_bf16((6, 64), 0.05, 4, 1)
    a = oracle.router_logits(x, wg)
    wg2 = oracle.f32_to_bf16(oracle.bf16_to_f32(wg) * 2)
    assert np.array_equal(oracle.router_logits(x, wg2), a * 2)
    one_hot = np.zeros((6, 64), dtype=np.uint16)
    one_hot[2, 5] = 0x3F80                         # bf16 1.0: column 2 is x[:, 5]
    b = oracle.router_logits(x, one_hot)
    assert np.array_equal(b[:, 2], oracle.bf16_to_f32(x[:, 5]))
    assert np.all(b[:, [0, 1, 3, 4, 5]] == 0)


def test_identical_gate_rows_tie_to_the_lowest_expert():
    import synth
    x = synth.normal_bf16((8, 64), 1.0, 5, 0)
    wg = synth.normal_bf16((10, 64), 0.05, 5, 1)
    wg[7] = wg[2]                                   # experts 2 and 7 score the same for every token
    ids, w, _, logits = oracle.route_projected(x, wg, 10)
    assert np.array_equal(logits[:, 2], logits[:, 7])
    for t in range(8):
        pos = list(ids[t])
        assert pos.index(2) < pos.index(7)
        assert w[t, pos.index(2)] == w[t, pos.index(7)]


# ---------------------------------------------------------------------------
# 4-bit float weights
# ---------------------------------------------------------------------------

def test_e2m1_codes():
    """The sixteen E2M1 codes, worked out by hand from sign / 2 exponent bits (bias 1) / 1 mantissa bit."""
    want = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    got = oracle.e2m1_to_f32(np.arange(16))
    assert list(got) == want
    assert np.signbit(got[8])


def test_e4m3_codes():
    """Hand-worked E4M3 values: 1.0, the largest finite 448, the smallest normal 2^-6, the smallest
    subnormal 2^-9, a subnormal with m = 6, a negative, and the NaN code."""
    cases = {0x38: 1.0, 0x7E: 448.0, 0x08: 2.0 ** -6, 0x01: 2.0 ** -9, 0x06: 6 * 2.0 ** -9, 0xC0: -2.0,
             0x3C: 1.5, 0x40: 2.0, 0x30: 0.5, 0x00: 0.0}
    for b, v in cases.items():
        assert float(oracle.e4m3_to_f32(np.array([b]))[0]) == v, hex(b)
    assert np.isnan(oracle.e4m3_to_f32(np.array([0x7F, 0xFF]))).all()
    # every finite code is exactly representable in bf16 (8 significant bits): the GPU's exact scale
    allv = oracle.e4m3_to_f32(np.arange(256))
    fin = allv[np.isfinite(allv)]
    assert np.array_equal(oracle.bf16_to_f32(oracle.f32_to_bf16(fin)), fin)


def test_fp4_dequant_matches_brute_force():
    rng = np.random.default_rng(5)
    words = rng.integers(0, 2 ** 32, size=(3, 8), dtype=np.uint64).astype(np.uint32).view(np.int32)
    scales = rng.integers(0x20, 0x48, size=(3, 4)).astype(np.uint8)
    g = np.float32(0.37)
    got = oracle.dequant_fp4(words, scales, g)
    e2m1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    for n in range(3):
        for c in range(8):
            u = int(words[n, c]) & 0xFFFFFFFF
            for j in range(8):
                i = 8 * c + j
                sb = int(scales[n, i // 16])
                e, m = (sb >> 3) & 15, sb & 7
                sv = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
                want = np.float32(e2m1[(u >> (4 * j)) & 15] * sv) * g     # exact product, one fp32 rounding by g
                assert got[n, i] == np.float32(want), (n, i)


def test_fp4_layer_single_expert_equals_dense_brute_force():
    import synth
    shape = synth.LayerShape(E=1, top_k=1, H=64, I=32)
    layer = synth.make_layer_fp4(shape, seed=3)
    x_bits, logits = synth.make_tokens(2, 64, 1, seed=4)
    res = oracle.moe_layer(x_bits, logits, layer, k=1)
    W13, W2 = oracle.expert_weights(layer, 0)
    for t in range(2):
        x = [bf16_bits_to_float(b) for b in x_bits[t]]
        gu = [sum(float(a) * b for a, b in zip(row, x)) for row in W13]
        h = [gu[i] / (1.0 + math.exp(-gu[i])) * gu[32 + i] for i in range(32)]
        ref = np.array([sum(float(a) * b for a, b in zip(row, h)) for row in W2])
        assert np.abs(res["out"][t] - ref).max() <= 1e-5 * np.sqrt(np.mean(ref ** 2))
