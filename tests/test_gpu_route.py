"""Step 1 on the GPU: the defined sigmoid and top-k routing, bit-exact vs the oracle."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import dev, host

pytestmark = pytest.mark.gpu


def gpu_scores(B, x: np.ndarray) -> np.ndarray:
    import torch
    xd = dev(x.astype(np.float32))
    out = torch.empty_like(xd)
    B.moe_sigmoid_scores(xd, xd.numel(), out)
    return host(out)


def test_sigmoid_bit_identical_on_a_strided_sweep_of_all_fp32(cuda_lib):
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    # every 251st bit pattern (all exponents, both signs) plus a dense window around 0
    bits = np.arange(0, 1 << 32, 251, dtype=np.uint64).astype(np.uint32)
    dense = np.linspace(-100, 100, 2_000_001, dtype=np.float32).view(np.uint32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 87.0, -87.0, 88.0, -88.0, 20.0, 1e-45],
                       dtype=np.float32).view(np.uint32)
    for chunk in (bits[: len(bits) // 2], bits[len(bits) // 2:], dense, special):
        x = chunk.view(np.float32)
        g = gpu_scores(B, x)
        r = oracle.sigmoid_def(x)
        both_nan = np.isnan(g) & np.isnan(r)
        same = (g.view(np.uint32) == r.view(np.uint32)) | both_nan
        bad = np.flatnonzero(~same)
        assert bad.size == 0, f"{bad.size} mismatches, first x={x[bad[:5]]} gpu={g[bad[:5]]} cpu={r[bad[:5]]}"


@pytest.mark.slow
def test_sigmoid_bit_identical_on_every_fp32(cuda_lib):
    """All 2^32 bit patterns, in 128 chunks of 2^25: the GPU's score of each equals the oracle's,
    bit for bit (NaN inputs give NaN on both sides). The oracle's chunks run on a few host threads."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    n = 1 << 25

    def cpu(c):
        x = (np.arange(n, dtype=np.uint64) + np.uint64(c * n)).astype(np.uint32).view(np.float32)
        return oracle.sigmoid_def(x)

    with ThreadPoolExecutor(max(1, min(4, os.cpu_count() or 1))) as ex:
        refs = ex.map(cpu, range(128))
        for c, r in enumerate(refs):
            x = (np.arange(n, dtype=np.uint64) + np.uint64(c * n)).astype(np.uint32).view(np.float32)
            g = gpu_scores(B, x)
            same = (g.view(np.uint32) == r.view(np.uint32)) | (np.isnan(g) & np.isnan(r))
            bad = np.flatnonzero(~same)
            assert bad.size == 0, f"chunk {c}: {bad.size} mismatches, first x={x[bad[:5]]} gpu={g[bad[:5]]}"


def check_route(B, logits: np.ndarray, k: int):
    import torch
    T, E = logits.shape
    ld = dev(logits)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    B.moe_route(ld, T, E, k, ids, w)
    r_ids, r_w, _ = oracle.route(logits, k)
    g_ids, g_w = host(ids), host(w)
    assert np.array_equal(g_ids, r_ids), np.argwhere(g_ids != r_ids)[:5]
    same = (g_w.view(np.uint32) == r_w.view(np.uint32)) | (np.isnan(g_w) & np.isnan(r_w))
    assert same.all(), np.argwhere(~same)[:5]


@pytest.mark.parametrize("T,E,k", [(16, 8, 2), (64, 384, 8), (1, 1, 1), (37, 33, 5), (5, 1024, 8),
                                   (3, 64, 64), (300, 256, 8)])
def test_route_bit_exact(cuda_lib, T, E, k):
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    _, logits = synth.make_tokens(T, 32, E, seed=T + E)
    check_route(B, logits, k)


def test_route_zipf_prefill_bit_exact(cuda_lib):
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    bias = synth.zipf_bias(384, 4096, 8, 1.1, 0)
    _, logits = synth.make_tokens(4096, 32, 384, seed=0, bias=bias)
    check_route(B, logits, 8)


def test_route_crafted_ties_and_specials(cuda_lib):
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    E = 40
    logits = np.random.default_rng(0).standard_normal((8, E)).astype(np.float32)
    logits[0, :] = 0.0                                   # every score 0.5
    logits[1, [3, 7, 11]] = [20.0, 25.0, 30.0]           # scores round to 1.0f: index order wins
    logits[2, ::3] = np.inf
    logits[3, :] = -np.inf                               # every score 0 -> weights 1/k
    logits[4, :] = -100.0
    logits[5, 5] = np.nan                                # NaN ranks last
    logits[6, :] = np.float32(1.5)
    logits[7, ::2] = 88.5
    check_route(B, logits, 6)
    check_route(B, logits, E)
