"""The router's logit projection on the GPU: logits = x . Wg^T on the tensor cores
(and the CUDA-core path), against the oracle's fp32 projection within the
rounding bound of a sum of bf16 products in any order; the top-k selection
bit-exact against the oracle's routing of the same logits; and the layer from
x alone equal, bit for bit, to the layer fed those logits."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import dev, host

pytestmark = pytest.mark.gpu


def project(B, x, wg, T, E, H, k, flags=0):
    import torch
    ws = torch.zeros(B.moe_router_workspace_size(T, E, H), dtype=torch.uint8, device="cuda")
    logits = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    B.moe_route_project(dev(x), dev(wg), T, E, H, k, logits, ids, w, ws, flags)
    assert B.moe_check_status(ws) == B.MOE_OK
    return host(logits), host(ids), host(w)


def check_logits(got, x, wg):
    ref = oracle.router_logits(x, wg).astype(np.float64)
    X = np.abs(oracle.bf16_to_f32(x).astype(np.float64))
    W = np.abs(oracle.bf16_to_f32(wg).astype(np.float64))
    H = X.shape[1]
    bound = 2 * H * 2.0 ** -24 * (X @ W.T)          # two fp32 sums of the same products, any order
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= bound + 1e-30)


@pytest.mark.parametrize("T", [1, 8, 64, 300, 4096])
@pytest.mark.parametrize("simt", [False, True])
def test_projection_and_selection_full_size(cuda_lib, T, simt):
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    if simt and T == 4096:
        pytest.skip("the CUDA-core kernel is a baseline for small batches")
    E, H, k = 384, 7168, 8
    x, _ = synth.make_tokens(T, H, E, seed=T)
    wg = synth.make_gate(E, H, seed=1)
    logits, ids, w = project(B, x, wg, T, E, H, k, B.MOE_FLAG_GEMM_SIMT if simt else 0)
    check_logits(logits, x, wg)
    r_ids, r_w, _ = oracle.route(logits, k)         # the selection of these very logits: bit-exact
    assert np.array_equal(ids, r_ids)
    assert np.array_equal(w.view(np.uint32), r_w.view(np.uint32))
    assert 0.5 < np.std(logits) < 2.0                # the gate's scale gives ~N(0, 1) logits


@pytest.mark.parametrize("E,H,T,k", [(33, 96, 37, 5), (8, 256, 16, 2), (1024, 64, 9, 8), (5, 4096, 130, 5)])
def test_projection_odd_shapes(cuda_lib, E, H, T, k):
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    x, _ = synth.make_tokens(T, H, E, seed=E + H)
    wg = synth.make_gate(E, H, seed=E)
    logits, ids, w = project(B, x, wg, T, E, H, k)
    check_logits(logits, x, wg)
    r_ids, r_w, _ = oracle.route(logits, k)
    assert np.array_equal(ids, r_ids)
    assert np.array_equal(w.view(np.uint32), r_w.view(np.uint32))


def test_forward_project_equals_forward_on_the_same_logits(cuda_lib):
    import torch
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    from w4a16_mixture_experts_sigmoid_gb300.layer import MoeW4A16Layer
    shape = synth.LayerShape(E=33, top_k=5, H=288, I=96, shared_I=64)
    arrays = synth.make_layer(shape, seed=9)
    layer = MoeW4A16Layer.from_arrays(shape, arrays)
    T = 41
    x, _ = synth.make_tokens(T, shape.H, shape.E, seed=10)
    wg = synth.make_gate(shape.E, shape.H, seed=11)
    ws = torch.zeros(B.moe_workspace_size(layer.dims, T, shape.shared_I, B.MOE_FLAG_ROUTER_PROJECT),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((T, shape.H), dtype=torch.int16, device="cuda")
    B.moe_forward_project(layer.dims, layer.weights, dev(wg), dev(x), T, out, ws)
    assert B.moe_check_status(ws) == B.MOE_OK
    logits, _, _ = project(B, x, wg, T, shape.E, shape.H, shape.top_k)
    ref = layer.forward(dev(x), dev(logits))
    assert torch.equal(out, ref)
    # and too small a workspace (the layer's without the router's share) is refused
    small = torch.zeros(B.moe_workspace_size(layer.dims, T, shape.shared_I), dtype=torch.uint8, device="cuda")
    with pytest.raises(B.MoeError) as ex:
        B.moe_forward_project(layer.dims, layer.weights, dev(wg), dev(x), T, out, small)
    assert ex.value.code == B.MOE_ERR_WORKSPACE_TOO_SMALL
