"""Seeded synthetic inputs for the routed-expert W4A16 MoE layer.

This module only draws random numbers and lays them out in the storage
formats of the layer's inputs. It holds none of the layer's arithmetic (no
routing, no unpacking, no dequantisation, no matmul): the CUDA library and the
CPU oracle both consume exactly the arrays produced here, and each interprets
them on its own.

Storage formats (the layer's inputs, as the Kimi-K2.6 catalog page describes
them in its QUANT and PARAMS paragraphs: int4 weights held in int32
containers, pack-quantized, symmetric, group size 32; activations bf16):

* packed weights: int32 words, ``[E, rows, K/8]``. A nibble that is uniform
  over 0..15 makes the whole 32-bit word uniform, so a packed tensor is drawn
  directly as uniform random 32-bit words.
* scales: bf16 bit patterns (``uint16``), ``[E, rows, K/32]``, drawn
  U[0.005, 0.02] in fp32 and rounded to the nearest bf16 (ties to even).
* activations: bf16 bit patterns ``[T, H]`` drawn N(0, 1).
* router logits: fp32 ``[T, E]`` drawn N(0, 1), optionally plus a per-expert
  bias that skews expert popularity towards a Zipf law.

Large tensors are drawn in fixed-size chunks, each from its own
``SeedSequence([seed, tensor_id, chunk])`` stream, on a thread pool; the
result does not depend on the number of threads.
"""
from __future__ import annotations

import functools
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_CHUNK = 1 << 22  # elements per independently seeded chunk

# tensor ids: keep every tensor of a layer on its own stream
TID_W13, TID_S13, TID_W2, TID_S2, TID_SH_GU, TID_SH_D, TID_X, TID_LOGITS, TID_GATE, TID_G13, TID_G2 = range(11)


@dataclass(frozen=True)
class LayerShape:
    E: int        # routed experts
    top_k: int    # experts per token
    H: int        # hidden size (input of gate/up, output of down)
    I: int        # expert intermediate size
    group: int = 32
    shared_I: int = 0   # 0: no shared expert


TINY = LayerShape(E=8, top_k=2, H=256, I=128)
FULL = LayerShape(E=384, top_k=8, H=7168, I=2048)
FULL_WITH_SHARED = LayerShape(E=384, top_k=8, H=7168, I=2048, shared_I=2048)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _fill_chunks(out: np.ndarray, seed: int, tensor_id: int, draw) -> np.ndarray:
    """Fill ``out`` (flat, contiguous) chunk by chunk; ``draw(gen, n)`` makes n values."""
    flat = out.reshape(-1)
    n = flat.size
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def work(c: int) -> None:
        lo = c * _CHUNK
        hi = min(n, lo + _CHUNK)
        gen = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor_id, c])))
        flat[lo:hi] = draw(gen, hi - lo)

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returns uint16 bit patterns.

    NaN inputs are not expected here (the generators never produce them).
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def random_words(shape, seed: int, tensor_id: int) -> np.ndarray:
    """Uniform 32-bit words (every nibble uniform over 0..15), as int32."""
    out = np.empty(shape, dtype=np.uint32)
    _fill_chunks(out, seed, tensor_id,
                 lambda g, n: g.integers(0, 0xFFFFFFFF, size=n, dtype=np.uint32, endpoint=True))
    return out.view(np.int32)


def uniform_bf16(shape, lo: float, hi: float, seed: int, tensor_id: int) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)

    def draw(g, n):
        u = g.random(n, dtype=np.float32)
        return f32_to_bf16_bits(np.float32(lo) + np.float32(hi - lo) * u)

    return _fill_chunks(out, seed, tensor_id, draw)


def normal_bf16(shape, std: float, seed: int, tensor_id: int) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    return _fill_chunks(out, seed, tensor_id,
                        lambda g, n: f32_to_bf16_bits(np.float32(std) * g.standard_normal(n, dtype=np.float32)))


def normal_f32(shape, seed: int, tensor_id: int) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    return _fill_chunks(out, seed, tensor_id, lambda g, n: g.standard_normal(n, dtype=np.float32))


def make_layer(shape: LayerShape, seed: int = 0, scale_lo: float = 0.005, scale_hi: float = 0.02,
               shared_std: float = 0.02) -> dict:
    """Weights of one routed-expert layer (plus the bf16 shared expert if ``shared_I``)."""
    E, H, I, G = shape.E, shape.H, shape.I, shape.group
    assert H % G == 0 and I % G == 0 and G == 32
    w = {
        "w13": random_words((E, 2 * I, H // 8), seed, TID_W13),
        "s13": uniform_bf16((E, 2 * I, H // G), scale_lo, scale_hi, seed, TID_S13),
        "w2": random_words((E, H, I // 8), seed, TID_W2),
        "s2": uniform_bf16((E, H, I // G), scale_lo, scale_hi, seed, TID_S2),
    }
    if shape.shared_I:
        Is = shape.shared_I
        w["sh_gu"] = normal_bf16((2 * Is, H), shared_std, seed, TID_SH_GU)
        w["sh_d"] = normal_bf16((H, Is), shared_std, seed, TID_SH_D)
    return w


def uniform_u8(shape, lo: int, hi: int, seed: int, tensor_id: int) -> np.ndarray:
    """Bytes uniform over the codes lo..hi (inclusive)."""
    out = np.empty(shape, dtype=np.uint8)
    return _fill_chunks(out, seed, tensor_id,
                        lambda g, n: g.integers(lo, hi, size=n, dtype=np.uint8, endpoint=True))


def make_layer_fp4(shape: LayerShape, seed: int = 0) -> dict:
    """Weights of one routed-expert layer in the 4-bit float layout: E2M1 codes packed eight to an
    int32 word (every code uniform over the sixteen), one FP8 E4M3 scale byte per 16 inputs drawn
    uniform over the codes 0x30..0x47 (0.5 to 3.75), one fp32 scale per matrix and expert drawn
    U[0.004, 0.008]: weights of about the INT4 bank's magnitude."""
    E, H, I = shape.E, shape.H, shape.I
    assert H % 32 == 0 and I % 32 == 0
    g13 = np.empty(E, dtype=np.float32)
    g2 = np.empty(E, dtype=np.float32)
    _fill_chunks(g13, seed, TID_G13, lambda g, n: np.float32(0.004) + np.float32(0.004) * g.random(n, np.float32))
    _fill_chunks(g2, seed, TID_G2, lambda g, n: np.float32(0.004) + np.float32(0.004) * g.random(n, np.float32))
    return {
        "fmt": "nvfp4",
        "w13": random_words((E, 2 * I, H // 8), seed, TID_W13),
        "s13": uniform_u8((E, 2 * I, H // 16), 0x30, 0x47, seed, TID_S13),
        "g13": g13,
        "w2": random_words((E, H, I // 8), seed, TID_W2),
        "s2": uniform_u8((E, H, I // 16), 0x30, 0x47, seed, TID_S2),
        "g2": g2,
    }


def make_gate(E: int, H: int, seed: int = 0) -> np.ndarray:
    """Router gate matrix, bf16 bits [E, H], N(0, 1/H): with N(0, 1) activations the projected
    logits are about N(0, 1), the router logits of the decode workloads."""
    return normal_bf16((E, H), float(1.0 / np.sqrt(H)), seed, TID_GATE)


def make_tokens(T: int, H: int, E: int, seed: int = 0, bias: np.ndarray | None = None):
    """Activations x (bf16 bits [T, H]) and router logits (fp32 [T, E])."""
    x = normal_bf16((T, H), 1.0, seed, TID_X)
    logits = normal_f32((T, E), seed, TID_LOGITS)
    if bias is not None:
        logits = (logits + bias.astype(np.float32)[None, :]).astype(np.float32)
    return x, logits


# ---------------------------------------------------------------------------
# Zipf-skewed expert popularity (prefill workload)
# ---------------------------------------------------------------------------

def zipf_targets(E: int, T: int, k: int, s: float) -> np.ndarray:
    """Per-rank assignment counts proportional to rank^-s, capped at T per expert.

    A token picks an expert at most once, so no expert can hold more than T of
    the T*k assignments; the excess of capped ranks is water-filled onto the rest.
    """
    share = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    total = float(T * k)
    tgt = np.zeros(E)
    free = np.ones(E, dtype=bool)
    remaining = total
    for _ in range(E):
        t = remaining * share * free / share[free].sum()
        over = free & (t > T)
        if not over.any():
            tgt[free] = t[free]
            break
        tgt[over] = T
        free &= ~over
        remaining = total - tgt[~free].sum()
    return tgt


@functools.lru_cache(maxsize=8)
def zipf_bias(E: int, T: int, k: int, s: float = 1.1, seed: int = 0, steps: int = 200) -> np.ndarray:
    """Per-expert logit bias making expert popularity follow Zipf(s).

    The expert -> popularity-rank map is a seeded permutation. The bias is
    fitted by damped log-ratio steps on an independent calibration draw
    (seed + 1), selecting each token's k largest biased logits. The result is
    deterministic for its arguments.
    """
    rank_of = np.random.default_rng(seed).permutation(E)
    target = zipf_targets(E, T, k, s)[rank_of]
    cal = np.random.default_rng(seed + 1).standard_normal((T, E), dtype=np.float32)
    b = np.zeros(E, dtype=np.float64)
    for _ in range(steps):
        z = cal + b.astype(np.float32)[None, :]
        top = np.argpartition(-z, k - 1, axis=1)[:, :k]
        cnt = np.bincount(top.ravel(), minlength=E).astype(np.float64)
        b += 0.3 * (np.log(target + 0.5) - np.log(cnt + 0.5))
    return b.astype(np.float32)


# ---------------------------------------------------------------------------
# the workloads (names describe the workload; sizes are the layer's)
# ---------------------------------------------------------------------------

WORKLOADS = {
    "tiny": dict(shape=TINY, T=16, seed=0, skew=None),
    "decode_t64": dict(shape=FULL, T=64, seed=0, skew=None),
    "prefill_t4096_zipf": dict(shape=FULL, T=4096, seed=0, skew=1.1),
    "decode_sweep_shared": dict(shape=FULL_WITH_SHARED, T=(1, 8, 32, 128, 512), seed=0, skew=None),
    "stack12_t256": dict(shape=FULL, T=256, seed=0, skew=None, layers=12),
}
