"""Routed-expert W4A16 MoE layer (sigmoid top-k router) for GB300, sm_103a.

The compute lives in libmoe_w4a16.so (hand-written CUDA behind the C ABI of
include/moe_w4a16.h). ``binding`` exposes that ABI under the same names;
``layer.MoeW4A16Layer`` keeps one layer's device weights and workspace.
"""
from . import binding  # noqa: F401

__all__ = ["binding"]
