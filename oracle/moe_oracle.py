"""Plain, slow CPU oracle of the routed-expert W4A16 MoE layer.

TEST INFRASTRUCTURE ONLY (see the package docstring): only the tests,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may use it.

What the layer computes, and where it comes from:

* Shapes and weight format -- "Kimi-K2.6" (model-catalog page), GEOMETRY,
  QUANT and PARAMS paragraphs: hidden 7168, 384 routed experts, 8 per token,
  moe_intermediate_size 2048; routed experts are the INT4 bank, int4 weights
  held in int32 containers, compressed-tensors pack-quantized, symmetric,
  group size 32. The page's I32 parameter count equals
  60 layers x 384 experts x 3 x 7168 x 2048, i.e. three H x I matrices per
  expert: gate, up (together ``W13``, ``[2I, H]``) and down (``W2``, ``[H, I]``).
* MoE routing -- "feat(pytorch): support Kimi K2.6", Motivation/Changes
  (MoE routing, compressed-tensors W4A16 MoE). The pages do not spell the
  router out. Adopted reading: score = sigmoid of the fp32 logit; the k best
  scores win, the lowest expert index wins a tie; the k winning scores are
  renormalised to sum to one.
* Nibble format (pages silent; adopted reading): a weight q in [-8, 7] is
  stored as the nibble q + 8; word c of a row holds inputs 8c..8c+7, input
  8c + j in bits 4j..4j+3 (little nibble first). One bf16 scale per 32
  consecutive inputs of a row.
* Expert MLP (pages give three matrices, not the activation; adopted
  reading): y = W2 (SiLU(W_gate x) * (W_up x)).

Precision: routing is fp32 and every step is a separately rounded IEEE fp32
operation, so the result is bit-exact by definition. The expert MLPs are the
plain "dequantise to fp32, then matmul" per token per selected expert, with
numpy's fp32 BLAS as the matmul primitive; combine sums in fp32 in rank order.
"""
from __future__ import annotations

import math

import numpy as np

F32 = np.float32

__all__ = [
    "bf16_to_f32", "exp_def", "sigmoid_def", "route", "permute",
    "unpack_int4", "pack_int4", "dequant", "silu", "expert_mlp",
    "shared_expert", "combine", "moe_layer", "gateup_rows", "down_rows",
    "rmsnorm", "stack_layer", "f32_to_bf16", "expert_int4_params", "EXP_CONSTANTS",
    "router_logits", "route_projected", "mlp", "e2m1_to_f32", "e4m3_to_f32", "dequant_fp4", "expert_weights",
]


# ---------------------------------------------------------------------------
# bf16 storage
# ---------------------------------------------------------------------------

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 values (exact: bf16 is the top half of fp32)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16(v: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, rounded to nearest with ties to even (NaN stays NaN).

    Keep the top 16 bits after adding 0x7FFF plus the lowest kept bit: below
    half an ulp rounds down, above rounds up, an exact half rounds to the even
    neighbour.
    """
    u = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(np.asarray(v, dtype=np.float32))
    return np.where(nan, np.uint16(0x7FC0), r).astype(np.uint16)


# ---------------------------------------------------------------------------
# The defined fp32 sigmoid
#
# A bit-exact router needs a sigmoid whose every rounding is fixed, since two
# libraries' expf differ in the last bits. sigmoid_def(x) = 1 / (1 + e(-x)),
# e(t) computed from IEEE basic operations only:
#   * t > 88 -> +inf ; t < -87 -> 0 ; NaN -> NaN
#   * n = round-half-even(t * LOG2E)
#   * r = (t - n * LN2_HI) - n * LN2_LO     (Cody & Waite's split of ln 2:
#                                            LN2_HI has 14 significant bits, so
#                                            n * LN2_HI is exact for |n| < 2^10)
#   * p = Taylor polynomial of exp(r) of degree 7 in Horner form, coefficient
#         of r^m = fp32(1/m!)
#   * e = p * 2^n
# Each +, -, * and / is one fp32 operation rounded to nearest even; nothing is
# fused.
# ---------------------------------------------------------------------------

def _exp_constants():
    ln2 = math.log(2.0)
    ln2_hi = round(ln2 * 2.0 ** 14) / 2.0 ** 14        # exact in fp32 (14 bits)
    return {
        "LOG2E": F32(1.0 / ln2),
        "LN2_HI": F32(ln2_hi),
        "LN2_LO": F32(ln2 - ln2_hi),
        "C": [F32(1.0 / math.factorial(m)) for m in range(8)],   # C[m] = 1/m!
    }


EXP_CONSTANTS = _exp_constants()


def exp_def(t) -> np.ndarray:
    """The defined fp32 exponential e(t) (see the block comment above)."""
    t = np.asarray(t, dtype=np.float32)
    c = EXP_CONSTANTS
    with np.errstate(invalid="ignore", over="ignore"):
        finite = (t >= F32(-87.0)) & (t <= F32(88.0))
        tt = np.where(finite, t, F32(0.0)).astype(np.float32)
        n = np.rint(tt * c["LOG2E"]).astype(np.float32)          # round half to even
        r = (tt - n * c["LN2_HI"]) - n * c["LN2_LO"]
        p = c["C"][7]
        for m in range(6, -1, -1):
            p = p * r + c["C"][m]
        scale = np.ldexp(np.float32(1.0), n.astype(np.int32)).astype(np.float32)
        e = (p * scale).astype(np.float32)
        e = np.where(t > F32(88.0), F32(np.inf), e)
        e = np.where(t < F32(-87.0), F32(0.0), e)
        e = np.where(np.isnan(t), t, e)
    return e.astype(np.float32)


def sigmoid_def(x) -> np.ndarray:
    """Router score: fp32 1 / (1 + e(-x)), every operation rounded to nearest even."""
    x = np.asarray(x, dtype=np.float32)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        return (F32(1.0) / (F32(1.0) + exp_def(-x))).astype(np.float32)


# ---------------------------------------------------------------------------
# Routing and the expert-sorted permutation
# ---------------------------------------------------------------------------

def route(logits: np.ndarray, k: int):
    """Top-k sigmoid routing of every token.

    Returns (ids [T,k] int32, weights [T,k] fp32, scores [T,E] fp32).
    ids are in rank order: score descending, expert index ascending on ties.
    A NaN score ranks below every number. weights: S = s_0 + s_1 + ... summed
    in rank order in fp32; w_j = s_j / S; if S == 0 every weight is 1/k.
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    assert 1 <= k <= E
    s = sigmoid_def(logits)
    key = np.where(np.isnan(s), F32(-1.0), s).astype(np.float32)
    idx = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((idx, -key), axis=-1)           # primary: key desc; then index asc
    ids = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(s, ids.astype(np.int64), axis=1)
    S = sel[:, 0].copy()
    for j in range(1, k):
        S = (S + sel[:, j]).astype(np.float32)
    with np.errstate(invalid="ignore", divide="ignore"):
        w = (sel / S[:, None]).astype(np.float32)
    zero = S == F32(0.0)
    if zero.any():
        w[zero, :] = F32(1.0) / F32(k)
    return ids, w, s


def router_logits(x_bits: np.ndarray, wg_bits: np.ndarray) -> np.ndarray:
    """The router's logit projection: logits[t, e] = sum_i x[t, i] * Wg[e, i], fp32.

    The pages name MoE routing ("feat(pytorch): support Kimi K2.6", Motivation
    and Changes) over 384 experts of hidden 7168 ("Kimi-K2.6" catalog page,
    GEOMETRY) but print no router; the reading taken is the plain linear gate of
    a routed MoE: bf16 token activations x [T, H] and a bf16 gate matrix
    Wg [E, H], products summed in fp32 (numpy's fp32 BLAS as the matmul).
    """
    x = bf16_to_f32(x_bits)
    wg = bf16_to_f32(wg_bits)
    return (x @ wg.T).astype(np.float32)


def route_projected(x_bits: np.ndarray, wg_bits: np.ndarray, k: int):
    """route() of the projected logits: (ids, weights, scores, logits)."""
    logits = router_logits(x_bits, wg_bits)
    ids, w, s = route(logits, k)
    return ids, w, s, logits


def permute(ids: np.ndarray, E: int):
    """Stable expert-sorted order of the T*k assignments.

    Assignment i = t*k + j. Returns (offsets [E+1], sorted_token_ids [T*k],
    inv_perm [T*k]) with offsets the exclusive prefix sum of per-expert
    counts, rows of one expert in increasing i, sorted_token_ids[p] the token
    of row p and inv_perm[i] the row of assignment i.
    """
    ids = np.asarray(ids)
    T, k = ids.shape
    flat = ids.reshape(-1).astype(np.int64)
    order = np.argsort(flat, kind="stable")
    sorted_token_ids = (order // k).astype(np.int32)
    inv = np.empty(T * k, dtype=np.int32)
    inv[order] = np.arange(T * k, dtype=np.int32)
    counts = np.bincount(flat, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return offsets, sorted_token_ids, inv


# ---------------------------------------------------------------------------
# Weight format
# ---------------------------------------------------------------------------

# Byte b of a little-endian word holds two inputs: bits 0..3 the earlier one,
# bits 4..7 the next. This table lists (q_low, q_high) = (nibble - 8) for all
# 256 byte values, so unpacking is one table lookup per byte.
_BYTE_TO_Q = np.array([[(b & 15) - 8, (b >> 4) - 8] for b in range(256)], dtype=np.int8)
_BYTE_TO_QF = _BYTE_TO_Q.astype(np.float32)


def _word_bytes(words: np.ndarray) -> np.ndarray:
    """int32 words [..., W] -> their bytes [..., 4W], least significant byte of each word first."""
    return np.ascontiguousarray(np.asarray(words).astype("<u4", copy=False)).view(np.uint8)


def unpack_int4(words: np.ndarray) -> np.ndarray:
    """int32 words [..., W] -> signed int4 values [..., 8W] (input 8c+j from bits 4j..4j+3)."""
    b = _word_bytes(words)
    return _BYTE_TO_Q[b].reshape(*b.shape[:-1], b.shape[-1] * 2)


def pack_int4(q: np.ndarray) -> np.ndarray:
    """Signed int4 values [..., 8W] in [-8, 7] -> int32 words [..., W]."""
    q = np.asarray(q)
    assert q.shape[-1] % 8 == 0 and q.min() >= -8 and q.max() <= 7
    nib = (q.astype(np.int64) + 8).reshape(*q.shape[:-1], q.shape[-1] // 8, 8).astype(np.uint32)
    word = np.zeros(nib.shape[:-1], dtype=np.uint32)
    for j in range(8):
        word |= nib[..., j] << np.uint32(4 * j)
    return word.view(np.int32)


def dequant(words: np.ndarray, scale_bits: np.ndarray, group: int = 32) -> np.ndarray:
    """W[n, i] = q[n, i] * scale[n, i // group], in fp32 (exact: 4-bit x 8-bit significands)."""
    b = _word_bytes(words)
    q = _BYTE_TO_QF[b].reshape(*b.shape[:-1], -1, group)       # [..., groups, group]
    s = bf16_to_f32(scale_bits)[..., None]                     # [..., groups, 1]
    q *= s
    return q.reshape(*b.shape[:-1], b.shape[-1] * 2)


# ---------------------------------------------------------------------------
# 4-bit float weights (NVFP4-style checkpoints)
#
# The pages name an NVFP4 checkpoint of the previous model and an
# nvfp4-pack-quantized format ("Kimi k2.5 MLA based eagle3", its test command;
# "Probing the Depths...", Assumption 2) without spelling it out. The reading
# taken is the published NVFP4 layout: each weight an E2M1 float (sign, two
# exponent bits with bias 1, one mantissa bit) in the same nibble positions as
# the INT4 bank (input 8c + j in bits 4j..4j+3 of word c), one FP8 E4M3 scale
# per 16 consecutive inputs of a row, and one fp32 scale per matrix and expert:
#     W[n, i] = e2m1(nibble) * e4m3(scale[n, i // 16]) * g
# ---------------------------------------------------------------------------

def e2m1_to_f32(nibbles) -> np.ndarray:
    """E2M1 codes (0..15) -> fp32: (-1)^s * 2^(e-1) * (1 + m/2) for e > 0, (-1)^s * m/2 for e = 0."""
    n = np.asarray(nibbles).astype(np.int64)
    s = (n >> 3) & 1
    e = (n >> 1) & 3
    m = n & 1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, e - 1))
    return np.where(s == 1, -mag, mag).astype(np.float32)


def e4m3_to_f32(bits) -> np.ndarray:
    """FP8 E4M3 bytes -> fp32: (-1)^s * 2^(e-7) * (1 + m/8) for e > 0, (-1)^s * 2^-6 * m/8 for e = 0;
    the code with e = 15 and m = 7 is NaN (the format has no infinities)."""
    b = np.asarray(bits).astype(np.int64)
    s = (b >> 7) & 1
    e = (b >> 3) & 15
    m = b & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag).astype(np.float32)


_BYTE_TO_FP4 = np.array([[e2m1_to_f32(b & 15), e2m1_to_f32(b >> 4)] for b in range(256)], dtype=np.float32)


def dequant_fp4(words: np.ndarray, scale_bytes: np.ndarray, gscale, group: int = 16) -> np.ndarray:
    """W[n, i] = e2m1(nibble) * e4m3(scale[n, i // group]) * g, in fp32 (the first product is exact)."""
    b = _word_bytes(words)
    v = _BYTE_TO_FP4[b].reshape(*b.shape[:-1], -1, group)      # [..., groups, group]
    v *= e4m3_to_f32(scale_bytes)[..., None]
    v *= np.float32(gscale)
    return v.reshape(*b.shape[:-1], b.shape[-1] * 2)


def expert_weights(layer: dict, e: int):
    """The fp32 W13 [2I, H] and W2 [H, I] of expert e, dequantised from the layer's format
    (layer["fmt"] == "nvfp4" for 4-bit floats; INT4 group-32 otherwise)."""
    if layer.get("fmt") == "nvfp4":
        return (dequant_fp4(layer["w13"][e], layer["s13"][e], layer["g13"][e]),
                dequant_fp4(layer["w2"][e], layer["s2"][e], layer["g2"][e]))
    return dequant(layer["w13"][e], layer["s13"][e]), dequant(layer["w2"][e], layer["s2"][e])


def expert_int4_params(H: int, I: int) -> int:
    """Logical int4 weights of one routed expert: W13 [2I, H] plus W2 [H, I]."""
    return 2 * I * H + H * I


# ---------------------------------------------------------------------------
# Expert MLPs
# ---------------------------------------------------------------------------

def silu(v: np.ndarray) -> np.ndarray:
    v = np.asarray(v, dtype=np.float32)
    with np.errstate(over="ignore"):
        return (v * (F32(1.0) / (F32(1.0) + np.exp(-v)))).astype(np.float32)


def expert_mlp(x: np.ndarray, w13: np.ndarray, s13: np.ndarray, w2: np.ndarray, s2: np.ndarray) -> np.ndarray:
    """One routed expert: fp32 x [H] (one token) -> fp32 y [H], or x [n, H] -> y [n, H] (each row on its own).

    Dequantise W13 and W2 to fp32, then per token g, u = W13 x (gate rows
    first), h = SiLU(g) * u, y = W2 h. Several tokens only put several
    columns into the same matrix products.
    """
    I = w2.shape[-1] * 8
    X = np.asarray(x, dtype=np.float32)
    single = X.ndim == 1
    X = X.reshape(-1, X.shape[-1])
    W13 = dequant(w13, s13)                  # [2I, H]
    gu = (X @ W13.T).astype(np.float32)      # row t: W13 x_t
    h = (silu(gu[:, :I]) * gu[:, I:]).astype(np.float32)
    W2 = dequant(w2, s2)                     # [H, I]
    y = (h @ W2.T).astype(np.float32)
    return y[0] if single else y


def mlp(X: np.ndarray, W13: np.ndarray, W2: np.ndarray) -> np.ndarray:
    """Gated-SiLU MLP of fp32 rows X [n, H] with dequantised fp32 W13 [2I, H], W2 [H, I]."""
    I = W2.shape[1]
    gu = (X @ W13.T).astype(np.float32)
    h = (silu(gu[:, :I]) * gu[:, I:]).astype(np.float32)
    return (h @ W2.T).astype(np.float32)


def shared_expert(x: np.ndarray, wgu_bits: np.ndarray, wd_bits: np.ndarray) -> np.ndarray:
    """The bf16 shared expert (gate rows first in wgu): fp32 x [H] -> fp32 [H], or [n, H] -> [n, H]."""
    Is = wd_bits.shape[1]
    X = np.asarray(x, dtype=np.float32)
    single = X.ndim == 1
    X = X.reshape(-1, X.shape[-1])
    gu = (X @ bf16_to_f32(wgu_bits).T).astype(np.float32)
    h = (silu(gu[:, :Is]) * gu[:, Is:]).astype(np.float32)
    y = (h @ bf16_to_f32(wd_bits).T).astype(np.float32)
    return y[0] if single else y


def _map(fn, items, workers: int):
    """fn over items, on a thread pool when workers > 1 (numpy and BLAS release the GIL)."""
    items = list(items)
    if workers <= 1 or len(items) <= 1:
        return [fn(i) for i in items]
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(min(workers, len(items))) as ex:
        return list(ex.map(fn, items))


def combine(y_rows: np.ndarray, inv: np.ndarray, w: np.ndarray, addend: np.ndarray | None = None) -> np.ndarray:
    """out[t] = sum_j w[t,j] * y[inv[t*k+j]] (+ addend[t]), fp32 sums in rank order j."""
    T, k = w.shape
    y = np.asarray(y_rows, dtype=np.float32)
    out = np.zeros((T, y.shape[1]), dtype=np.float32)
    for j in range(k):
        out = (out + w[:, j:j + 1] * y[inv.reshape(T, k)[:, j]]).astype(np.float32)
    if addend is not None:
        out = (out + np.asarray(addend, dtype=np.float32)).astype(np.float32)
    return out


def moe_layer(x_bits: np.ndarray, logits: np.ndarray, layer: dict, k: int, tokens=None,
              with_shared: bool = False, workers: int = 1) -> dict:
    """The routed MoE layer: routing for every token, outputs for ``tokens``.

    Returns ids, weights, offsets, sorted_token_ids, inv_perm (all tokens) and
    ``out`` fp32 [len(tokens), H] for the requested tokens (all by default):
    out[t] = sum over rank j of w[t, j] * expert_{ids[t, j]}(x[t]), summed in
    rank order, plus the shared expert when asked. Each expert is dequantised
    once and applied to every requested token that selected it; ``workers``
    threads run different experts at the same time.
    """
    T = x_bits.shape[0]
    E = layer["w13"].shape[0]
    ids, w, _ = route(logits, k)
    offsets, sorted_ids, inv = permute(ids, E)
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    H = x_bits.shape[1]
    X = bf16_to_f32(x_bits[tokens])                  # [n, H]
    sel = ids[tokens]                                # [n, k]
    y = np.zeros((len(tokens), k, H), dtype=np.float32)

    def one_expert(e):
        r, j = np.nonzero(sel == e)
        W13, W2 = expert_weights(layer, e)
        y[r, j] = mlp(X[r], W13, W2)

    _map(one_expert, np.unique(sel), workers)
    out = np.zeros((len(tokens), H), dtype=np.float32)
    for j in range(k):
        out = (out + w[tokens, j:j + 1] * y[:, j]).astype(np.float32)
    if with_shared:
        out = (out + shared_expert(X, layer["sh_gu"], layer["sh_d"])).astype(np.float32)
    return {"ids": ids, "weights": w, "offsets": offsets, "sorted_token_ids": sorted_ids,
            "inv_perm": inv, "out": out, "tokens": tokens}


# ---------------------------------------------------------------------------
# Row-level views used to check the two grouped GEMMs on their own
# ---------------------------------------------------------------------------

def _expert_of_rows(offsets: np.ndarray, rows) -> np.ndarray:
    """Expert e of each row r: offsets[e] <= r < offsets[e + 1] (empty experts own no row)."""
    return np.searchsorted(np.asarray(offsets), np.asarray(rows), side="right") - 1


def gateup_rows(a_bits: np.ndarray, offsets: np.ndarray, layer: dict, rows, workers: int = 1) -> np.ndarray:
    """h = SiLU(W_gate x) * (W_up x) for expert-sorted activation rows ``rows`` -> fp32 [len(rows), I]."""
    I = layer["w2"].shape[-1] * 8
    rows = np.asarray(list(rows), dtype=np.int64)
    owner = _expert_of_rows(offsets, rows)
    out = np.zeros((len(rows), I), dtype=np.float32)

    def one_expert(e):
        sel = np.nonzero(owner == e)[0]
        W13 = expert_weights(layer, e)[0]
        gu = (bf16_to_f32(a_bits[rows[sel]]) @ W13.T).astype(np.float32)
        out[sel] = silu(gu[:, :I]) * gu[:, I:]

    _map(one_expert, np.unique(owner), workers)
    return out


def down_rows(h_bits: np.ndarray, offsets: np.ndarray, layer: dict, rows, workers: int = 1) -> np.ndarray:
    """y = W2 h for expert-sorted rows ``rows`` -> fp32 [len(rows), H]."""
    H = layer["w2"].shape[1]
    rows = np.asarray(list(rows), dtype=np.int64)
    owner = _expert_of_rows(offsets, rows)
    out = np.zeros((len(rows), H), dtype=np.float32)

    def one_expert(e):
        sel = np.nonzero(owner == e)[0]
        out[sel] = bf16_to_f32(h_bits[rows[sel]]) @ expert_weights(layer, e)[1].T

    _map(one_expert, np.unique(owner), workers)
    return out


# ---------------------------------------------------------------------------
# Layer stack (pre-norm residual chain)
# ---------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """Parameter-free RMSNorm of each row, fp32."""
    x = np.asarray(x, dtype=np.float32)
    ms = np.mean(x.astype(np.float32) * x, axis=-1, keepdims=True, dtype=np.float32)
    return (x / np.sqrt(ms + F32(eps))).astype(np.float32)


def stack_layer(x_bits: np.ndarray, logits: np.ndarray, layer: dict, k: int, eps: float = 1e-6, tokens=None,
                with_shared: bool = False, workers: int = 1) -> dict:
    """One block of the layer stack, x + MoE(RMSNorm(x)), for ``tokens`` (all by default).

    The pages give 60 MoE layers ("Kimi-K2.6", GEOMETRY) but not how they are
    joined; the reading used is the pre-norm residual with a parameter-free
    RMSNorm. The normalised activations enter the layer as bf16 (the layer's
    input type), the residual add is fp32. Returns moe_layer's dict with
    ``out`` = x + MoE(...) in fp32.
    """
    xn_bits = f32_to_bf16(rmsnorm(bf16_to_f32(x_bits), eps))
    res = moe_layer(xn_bits, logits, layer, k, tokens=tokens, with_shared=with_shared, workers=workers)
    res["out"] = (bf16_to_f32(x_bits[res["tokens"]]) + res["out"]).astype(np.float32)
    res["xn_bits"] = xn_bits
    return res
