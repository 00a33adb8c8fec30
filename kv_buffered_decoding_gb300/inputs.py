"""Seeded synthetic inputs for the KV-buffered decoding workloads.

This module is shared by the CUDA path's tests and benchmark and by the fp64
oracle's tests.  It holds no arithmetic of the method itself: only random
draws, rounding to the storage dtype, and the shapes and value distributions of
the workloads.  Everything is drawn with numpy's PCG64 generator from an
explicit seed, in float32, then rounded to the storage dtype; both sides
consume the rounded values (the oracle upcasts them to float64).

The workloads mirror the layer shapes named for KVBuffer ("KVBuffer:
IO-aware Serving for Linear Attention", abstract: Qwen3-Next-style
linear-attention layers served in SGLang).  The pages publish no dataset;
these draws stand in for real activations.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

PLAIN, GATED, GATED_DELTA = 0, 1, 2
VARIANT_NAMES = {PLAIN: "plain", GATED: "gated", GATED_DELTA: "gated_delta"}


# --------------------------------------------------------------------------
# dtype rounding (storage format only)
# --------------------------------------------------------------------------
def bf16_bits(x) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the raw 16-bit patterns."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    nan = np.isnan(a)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    r = np.where(nan, np.uint16(0x7FC0), r)
    return r.reshape(a.shape)


def bf16_to_f32(bits) -> np.ndarray:
    """Widen raw bfloat16 patterns to float32 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def bf16_round(x) -> np.ndarray:
    """Values of ``x`` rounded to bfloat16, returned as float32."""
    return bf16_to_f32(bf16_bits(x))


def round_to(x, kv_dtype: str) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    if kv_dtype == "bf16":
        return bf16_round(x)
    if kv_dtype == "f32":
        return x.copy()
    raise ValueError(f"unknown kv dtype {kv_dtype!r}")


# --------------------------------------------------------------------------
# layers and token draws
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class Layer:
    """Shape of one linear-attention layer."""
    variant: int
    n_qk_heads: int
    n_v_heads: int
    d_k: int
    d_v: int
    kv_dtype: str  # "f32" or "bf16"
    qk_dist: str = "normal"  # "normal": N(0,1)/sqrt(d_k); "l2norm": unit rows

    @property
    def group(self) -> int:
        return self.n_v_heads // self.n_qk_heads


def _softplus(x):
    return np.log1p(np.exp(-np.abs(x))) + np.maximum(x, 0.0)


def draw_tokens(rng: np.random.Generator, layer: Layer, prefix: tuple) -> dict:
    """Draw q, k, v, log_g, beta for tokens laid out as ``prefix + (heads, dim)``.

    q, k: prefix + (Hk, d_k); v: prefix + (Hv, d_v); log_g, beta: prefix + (Hv,)
    (None where the variant has no gate / no beta).  q, k, v are rounded to the
    layer's storage dtype; log_g and beta are float32.
    """
    prefix = tuple(prefix)
    hk, hv, dk, dv = layer.n_qk_heads, layer.n_v_heads, layer.d_k, layer.d_v
    q = rng.standard_normal(prefix + (hk, dk), dtype=np.float32)
    k = rng.standard_normal(prefix + (hk, dk), dtype=np.float32)
    v = rng.standard_normal(prefix + (hv, dv), dtype=np.float32) / np.float32(np.sqrt(dv))
    if layer.qk_dist == "l2norm":
        q = q / np.linalg.norm(q, axis=-1, keepdims=True)
        k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    else:
        q = q / np.float32(np.sqrt(dk))
        k = k / np.float32(np.sqrt(dk))
    out = {
        "q": round_to(q, layer.kv_dtype),
        "k": round_to(k, layer.kv_dtype),
        "v": round_to(v, layer.kv_dtype),
        "log_g": None,
        "beta": None,
    }
    if layer.variant == GATED:
        out["log_g"] = rng.uniform(-0.1, 0.0, size=prefix + (hv,)).astype(np.float32)
    elif layer.variant == GATED_DELTA:
        z = rng.standard_normal(prefix + (hv,)).astype(np.float64)
        out["log_g"] = (-_softplus(z) * 0.1).astype(np.float32)
        b = rng.standard_normal(prefix + (hv,)).astype(np.float64)
        out["beta"] = (1.0 / (1.0 + np.exp(-b))).astype(np.float32)
    return out


def draw_state(rng: np.random.Generator, layer: Layer, n: int, scale: float | None = None) -> np.ndarray:
    """An iid N(0, scale^2) float32 state for ``n`` requests: [n, Hv, d_k, d_v]."""
    if scale is None:
        scale = 1.0 / np.sqrt(layer.d_k)
    s = rng.standard_normal((n, layer.n_v_heads, layer.d_k, layer.d_v), dtype=np.float32)
    return (s * np.float32(scale)).astype(np.float32)


def slice_tokens(tok: dict, idx) -> dict:
    """Index every present field of a token dict with the same index."""
    return {key: (None if val is None else val[idx]) for key, val in tok.items()}


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------
@dataclass
class Workload:
    name: str
    layer: Layer
    batch: int
    m: int
    steps: int
    seed: int
    prefill: int = 0
    block_size: int = 8
    extra: dict = field(default_factory=dict)


GATED_LAYER = Layer(GATED, 16, 16, 128, 128, "bf16")
GDN_LAYER = Layer(GATED_DELTA, 16, 32, 128, 128, "bf16", qk_dist="l2norm")

WORKLOADS = {
    # 1 request, 1 head, d=64, fp32, ungated: 16-token prefill then 64 decode steps, flush every 4
    "ungated_d64_f32": Workload("ungated_d64_f32", Layer(PLAIN, 1, 1, 64, 64, "f32"),
                                batch=1, m=4, steps=64, seed=0, prefill=16),
    # scalar-gated, B=32, H=16, d=128, bf16; 1024-token prefill state; m swept
    "gated_B32_H16_d128": Workload("gated_B32_H16_d128", GATED_LAYER, batch=32, m=8, steps=256,
                                   seed=1, prefill=1024, extra={"m_sweep": (0, 2, 4, 8, 16)}),
    # gated delta rule, 16 q/k heads shared by 32 v heads, B=256, m=8, 512 steps
    "gdn_B256_Hk16_Hv32_d128": Workload("gdn_B256_Hk16_Hv32_d128", GDN_LAYER, batch=256, m=8,
                                        steps=512, seed=2),
    # speculative verify on the gated layer: B=64, T drafts per round, 200 rounds
    "verify_B64_gated": Workload("verify_B64_gated", GATED_LAYER, batch=64, m=8, steps=200, seed=3,
                                 prefill=1024, extra={"T_list": (4, 2, 6, 8)}),
    # mixed ragged batch on the gated layer: 256 short (buffer-only) + 256 long requests
    "mixed_B512_gated": Workload("mixed_B512_gated", GATED_LAYER, batch=512, m=8, steps=256, seed=4,
                                 extra={"n_short": 256, "short_cap": 64, "num_blocks": 4096}),
}
