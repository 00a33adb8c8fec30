"""Helpers for the GPU parity tests: pools from workload specs, host->device inputs, errors.

The CUDA path is reached only through the C ABI (kvb.Pool); expected values
come only from the fp64 oracle.
"""
from __future__ import annotations

import math

import numpy as np

from kv_buffered_decoding_gb300 import inputs as I

TOL_F32 = 1e-5   # max normwise relative error, fp32 inputs
TOL_BF16 = 2e-3  # max normwise relative error, bf16 inputs with fp32 accumulation


def tol_for(layer):
    return TOL_F32 if layer.kv_dtype == "f32" else TOL_BF16


def rel_err(x, ref, tail: int = 2) -> float:
    """Worst per-tensor error: max_i |x_i - r_i| / max_i |r_i| (normwise, well defined
    near zeros) over every tensor made of the trailing ``tail`` axes, the worst over
    the leading axes (steps, requests, drafts).

    With tail = 2 a tensor is one output o_t of one request ([Hv, d_v]) or one value
    head's state ([d_k, d_v]), so stacked runs are never pooled into one error."""
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert x.shape == r.shape, (x.shape, r.shape)
    if r.ndim <= tail:
        return float(np.abs(x - r).max() / max(np.abs(r).max(), 1e-30))
    axes = tuple(range(r.ndim - tail, r.ndim))
    num = np.abs(x - r).max(axis=axes)
    den = np.maximum(np.abs(r).max(axis=axes), 1e-30)
    return float((num / den).max())


def kvb_mod():
    from kv_buffered_decoding_gb300 import kvb
    return kvb


def make_pool(layer, m, n_req, blocks_per_req, block_size=8, num_blocks=None, num_slots=None,
              max_blocks=None, scale=1.0):
    kvb = kvb_mod()
    variant = layer.variant
    dtype = kvb.KVB_BF16 if layer.kv_dtype == "bf16" else kvb.KVB_F32
    num_blocks = n_req * blocks_per_req if num_blocks is None else num_blocks
    num_slots = n_req if num_slots is None else num_slots
    max_blocks = blocks_per_req if max_blocks is None else max_blocks
    cfg = kvb.make_config(variant, dtype, layer.n_qk_heads, layer.n_v_heads, layer.d_k, layer.d_v,
                          m, block_size, num_blocks, num_slots, n_req, max(max_blocks, 1), scale)
    return kvb.Pool(cfg)


def dev(x, layer=None, f32=False):
    """numpy float32 -> CUDA tensor in the storage dtype (exact: values are already rounded)."""
    import torch
    if x is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if not f32 and layer is not None and layer.kv_dtype == "bf16":
        t = t.to(torch.bfloat16)
    return t.cuda()


def token_tensors(tok, layer, idx):
    """Device tensors of one step's tokens (tok fields indexed by idx)."""
    return (dev(tok["q"][idx], layer), dev(tok["k"][idx], layer), dev(tok["v"][idx], layer),
            dev(None if tok["log_g"] is None else tok["log_g"][idx], f32=True),
            dev(None if tok["beta"] is None else tok["beta"][idx], f32=True))


def blocks_needed(cap, bs):
    return max(1, math.ceil(cap / bs))
