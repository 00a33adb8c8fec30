"""GPU parity with an output scale: cfg.scale = 1/sqrt(d_k) on every kernel family.

The recurrence's output is o_t = scale * S_t^T q_t (the scale touches only the
output, never the state).  Every other parity test runs with scale = 1, so this
file repeats the main paths with scale = 1/sqrt(d_k) and q drawn without the
usual 1/sqrt(d_k) pre-scaling, and compares outputs and states with the fp64
oracle at the same scale:

* decode: the per-head kernel (small batch) and the persistent kernel (a batch
  large enough for it), gated delta rule, with folds; recurrent decoding (m = 0);
* verify + accept: tensor-core path (bf16, d = 128) and the FFMA path (fp32, d = 64);
* short context: tensor-core score path (bf16, d = 128) and fp32 / d = 64;
* chunked prefill: tcgen05 (bf16, d = 128) and mma.sync (fp32, d = 64);
* the temporary-state baseline.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
from kv_buffered_decoding_gb300 import inputs as I
from tests import oracle_pool
from tests.gpu_harness import blocks_needed, dev, make_pool, rel_err, token_tensors, tol_for

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _unscaled_q(rng, layer, tok):
    """Replace q by N(0, 1) draws rounded to the storage dtype (the kernel scales)."""
    q = rng.standard_normal(tok["q"].shape, dtype=np.float32)
    tok["q"] = I.round_to(q, layer.kv_dtype)
    return tok


def _scale(layer):
    return 1.0 / math.sqrt(layer.d_k)


GDN128 = I.Layer(I.GATED_DELTA, 2, 4, 128, 128, "bf16", qk_dist="l2norm")
GATED128 = I.Layer(I.GATED, 2, 2, 128, 128, "bf16")
GDN64_F32 = I.Layer(I.GATED_DELTA, 1, 2, 64, 64, "f32", qk_dist="l2norm")
GATED64_F32 = I.Layer(I.GATED, 1, 1, 64, 64, "f32")


@pytest.mark.parametrize("B,layer", [(4, GDN128), (160, I.WORKLOADS["gdn_B256_Hk16_Hv32_d128"].layer)],
                         ids=["per_head_kernel", "persistent_kernel"])
def test_decode_scale(B, layer):
    """Decode with folds (m = 8, 12 steps); the B=160 x 32-head batch takes the
    persistent kernel (at least 8 units per resident CTA)."""
    s = _scale(layer)
    m, steps = 8, 12
    rng = np.random.default_rng(900 + B)
    S0 = I.draw_state(rng, layer, B)
    tok = _unscaled_q(rng, layer, I.draw_tokens(rng, layer, (steps, B)))
    pool = make_pool(layer, m, B, 1, 8, scale=s)
    pool.state.copy_(torch.from_numpy(S0))
    for r in range(B):
        pool.set_request(r, r, [r])
    outs = np.stack([pool.decode(np.arange(B), *token_tensors(tok, layer, t)).cpu().numpy()
                     for t in range(steps)])
    torch.cuda.synchronize()
    st = pool.state.cpu().numpy()
    assert pool.get_error() is None
    tasks = [dict(S0=S0[p], hist={k_: (None if v_ is None else v_[:, p]) for k_, v_ in tok.items()},
                  out=outs[:, p], state=st[p], fold_at=np.full(len(p), m - 1),
                  variant=layer.variant, scale=s)
             for p in oracle_pool.chunks(B, 16)]
    res = oracle_pool.run(oracle_pool.decode_errors, tasks)
    tol = tol_for(layer)
    assert max(r_[0].max() for r_ in res) <= tol
    assert max(r_[1].max() for r_ in res) <= tol


def test_recurrent_scale():
    layer, B, steps = GDN128, 3, 5
    s = _scale(layer)
    rng = np.random.default_rng(910)
    S0 = I.draw_state(rng, layer, B)
    tok = _unscaled_q(rng, layer, I.draw_tokens(rng, layer, (steps, B)))
    pool = make_pool(layer, 0, B, 1, 8, scale=s)
    pool.state.copy_(torch.from_numpy(S0))
    for r in range(B):
        pool.set_request(r, r, [])
    outs = np.stack([pool.decode(np.arange(B), *token_tensors(tok, layer, t)).cpu().numpy()
                     for t in range(steps)])
    o_ref, S_ref, _ = oracle.decode_sequence(S0, tok, layer.variant, s)
    tol = tol_for(layer)
    assert rel_err(outs, o_ref) <= tol
    assert rel_err(pool.state.cpu().numpy(), S_ref) <= tol


@pytest.mark.parametrize("layer", [GDN128, GATED128, GDN64_F32], ids=["gdn_bf16_d128", "gated_bf16_d128",
                                                                       "gdn_f32_d64"])
def test_verify_scale(layer):
    """Three rounds of verify (T = 4) + accept; outputs every round, states at the end."""
    s = _scale(layer)
    B, m, T = 6, 8, 4
    nb = blocks_needed(m - 1 + T, 8)
    rng = np.random.default_rng(920 + layer.d_k + layer.variant)
    S0 = I.draw_state(rng, layer, B)
    pool = make_pool(layer, m, B, nb, 8, scale=s)
    pool.state.copy_(torch.from_numpy(S0))
    for r in range(B):
        pool.set_request(r, r, list(range(r * nb, (r + 1) * nb)))
    S_hist = S0.astype(np.float64)
    tol = tol_for(layer)
    req = np.arange(B)
    for rnd in range(3):
        tok = _unscaled_q(rng, layer, I.draw_tokens(rng, layer, (B, T)))
        o = pool.verify(req, dev(tok["q"], layer), dev(tok["k"], layer), dev(tok["v"], layer),
                        dev(tok["log_g"], f32=True), dev(tok["beta"], f32=True))
        j = rng.integers(0, T + 1, size=B)
        pool.accept(req, j)
        drafts = {key: (None if val is None else np.swapaxes(val, 0, 1)) for key, val in tok.items()}
        o_ref = oracle.verify(S_hist, drafts, layer.variant, s)
        assert rel_err(np.swapaxes(o.cpu().numpy(), 0, 1), o_ref) <= tol, rnd
        S_hist = oracle.accept(S_hist, drafts, j, layer.variant, s)
    pool.flush(req)
    torch.cuda.synchronize()
    assert rel_err(pool.state.cpu().numpy(), S_hist) <= tol
    assert pool.get_error() is None


@pytest.mark.parametrize("layer", [GATED128, GDN128, GATED64_F32], ids=["gated_bf16_d128", "gdn_bf16_d128",
                                                                         "gated_f32_d64"])
def test_short_context_scale(layer):
    """Short-context requests decoding 20 tokens from their buffers alone."""
    s = _scale(layer)
    B, steps = 4, 20
    rng = np.random.default_rng(930 + layer.d_k + layer.variant)
    pool = make_pool(layer, 8, B, 3, 8, num_slots=0, scale=s)
    for r in range(B):
        pool.set_request(r, -1, [3 * r, 3 * r + 1, 3 * r + 2])
    tok = _unscaled_q(rng, layer, I.draw_tokens(rng, layer, (steps, B)))
    outs = np.stack([pool.short_ctx(np.arange(B), *token_tensors(tok, layer, t)).cpu().numpy()
                     for t in range(steps)])
    tol = tol_for(layer)
    for r in range(B):
        hist = {k_: (None if v_ is None else v_[:, r]) for k_, v_ in tok.items()}
        o_ref = oracle.short_context(hist, layer.variant, layer.d_k, layer.d_v, s)
        assert rel_err(outs[:, r], o_ref) <= tol, r
    assert pool.get_error() is None


@pytest.mark.parametrize("layer", [GDN128, GATED128, GDN64_F32], ids=["tcgen05_gdn", "tcgen05_gated",
                                                                       "mma_sync_gdn_f32"])
def test_prefill_scale(layer):
    """Prompts of 130 and 64 tokens from S = 0: every prompt output and the state."""
    s = _scale(layer)
    lengths = np.array([130, 64])
    B, L = 2, 130
    rng = np.random.default_rng(940 + layer.d_k + layer.variant)
    pool = make_pool(layer, 8, B, 1, 8, scale=s)
    for r in range(B):
        pool.set_request(r, r, [r])
    tok = _unscaled_q(rng, layer, I.draw_tokens(rng, layer, (B, L)))
    o = pool.prefill(np.arange(B), *token_tensors(tok, layer, slice(None)), lengths=lengths,
                     from_zero=True).cpu().numpy()
    torch.cuda.synchronize()
    st = pool.state.cpu().numpy()
    tol = tol_for(layer)
    zero = np.zeros((layer.n_v_heads, layer.d_k, layer.d_v))
    for r in range(B):
        n = int(lengths[r])
        prompt = {k_: (None if v_ is None else v_[r, :n]) for k_, v_ in tok.items()}
        o_ref, S_r, _ = oracle.decode_sequence(zero, prompt, layer.variant, s)
        assert rel_err(o[r, :n], o_ref) <= tol, r
        assert rel_err(st[r], S_r) <= tol, r
    assert pool.get_error() is None


def test_tempstate_scale():
    layer, B, T = GDN128, 3, 4
    s = _scale(layer)
    rng = np.random.default_rng(950)
    S0 = I.draw_state(rng, layer, B)
    pool = make_pool(layer, 0, B, 1, 8, scale=s)
    pool.state.copy_(torch.from_numpy(S0))
    for r in range(B):
        pool.set_request(r, r, [])
    tok = _unscaled_q(rng, layer, I.draw_tokens(rng, layer, (B, T)))
    o, temp = pool.verify_tempstate(np.arange(B), dev(tok["q"], layer), dev(tok["k"], layer),
                                    dev(tok["v"], layer), dev(tok["log_g"], f32=True),
                                    dev(tok["beta"], f32=True))
    drafts = {key: np.swapaxes(val, 0, 1) for key, val in tok.items()}
    o_ref, _, states = oracle.decode_sequence(S0, drafts, layer.variant, s, keep_states=range(T))
    tol = tol_for(layer)
    assert rel_err(np.swapaxes(o.cpu().numpy(), 0, 1), o_ref) <= tol
    tp = temp.cpu().numpy()
    for j in range(T):
        assert rel_err(tp[:, j], states[j]) <= tol, j
