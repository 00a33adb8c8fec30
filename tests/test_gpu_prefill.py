"""GPU parity: chunked prefill (kvb_prefill) against the fp64 recurrence.

Ragged prompts (one token, exactly one chunk, several chunks with a ragged
tail, empty) run through fresh states (from S = 0) and through existing
states; every prompt token's output and the final state are compared with the
oracle's per-token recurrence, rows past a prompt stay untouched, and the
request then decodes on from the prefilled state.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from kv_buffered_decoding_gb300 import inputs as I
from tests.gpu_harness import dev, kvb_mod, make_pool, rel_err, token_tensors, tol_for

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

LAYERS = [
    I.Layer(I.GATED_DELTA, 2, 4, 128, 128, "bf16", qk_dist="l2norm"),
    I.Layer(I.GATED, 2, 2, 128, 128, "bf16"),
    I.Layer(I.PLAIN, 1, 2, 64, 64, "bf16"),
    I.Layer(I.GATED_DELTA, 1, 2, 64, 64, "f32", qk_dist="l2norm"),
    I.Layer(I.GATED, 1, 1, 128, 128, "f32"),
]
IDS = ["gated_delta_d128_bf16", "gated_d128_bf16", "plain_d64_bf16", "gated_delta_d64_f32",
       "gated_d128_f32"]


def _prompt(tok, b, n):
    return {key: (None if val is None else val[b, :n]) for key, val in tok.items()}


@pytest.mark.parametrize("layer", LAYERS, ids=IDS)
@pytest.mark.parametrize("from_zero", [True, False], ids=["fresh", "continued"])
def test_prefill_matches_recurrence(layer, from_zero):
    rng = np.random.default_rng(300 + layer.variant * 10 + layer.d_k + int(from_zero))
    lengths = np.array([150, 1, 64, 0, 129])
    B, L = len(lengths), int(lengths.max())
    pool = make_pool(layer, 4, B, 1, 8)
    S0 = I.draw_state(rng, layer, B)
    pool.state.copy_(torch.from_numpy(S0))
    for r in range(B):
        pool.set_request(r, B - 1 - r, [r])
    tok = I.draw_tokens(rng, layer, (B, L))
    o = torch.full((B, L, layer.n_v_heads, layer.d_v), float("nan"), device="cuda")
    pool.prefill(np.arange(B), *token_tensors(tok, layer, slice(None)), o=o, lengths=lengths,
                 from_zero=from_zero)
    torch.cuda.synchronize()
    o = o.cpu().numpy()
    st = pool.state.cpu().numpy()
    tol = tol_for(layer)
    zero = np.zeros((layer.n_v_heads, layer.d_k, layer.d_v))
    S_ref = []
    for r in range(B):
        start = zero if from_zero else S0[B - 1 - r].astype(np.float64)
        n = int(lengths[r])
        if n:
            o_ref, S_r, _ = oracle.decode_sequence(start, _prompt(tok, r, n), layer.variant)
            assert rel_err(o[r, :n], o_ref) <= tol, r
        else:
            S_r = start
        assert np.all(np.isnan(o[r, n:])), r
        assert rel_err(st[B - 1 - r], S_r) <= tol if np.abs(S_r).max() > 0 else \
            np.all(st[B - 1 - r] == 0.0), r
        S_ref.append(S_r)
    assert np.array_equal(pool.get_lengths(), np.zeros(B))

    # decode on from the prefilled states (buffered, fold at m = 4)
    for t in range(5):
        dt = I.draw_tokens(rng, layer, (B,))
        od = pool.decode(np.arange(B), *token_tensors(dt, layer, slice(None))).cpu().numpy()
        for r in range(B):
            one = {key: (None if val is None else val[r:r + 1]) for key, val in dt.items()}
            o_ref, S_ref[r], _ = oracle.decode_sequence(S_ref[r], one, layer.variant)
            assert rel_err(od[r], o_ref[0]) <= tol, (t, r)
    assert pool.get_error() is None


def test_prefill_unaligned_buffers_rejected():
    """Token buffers must start on a 16-byte boundary (the prefill kernels stage
    tiles with 16-byte copies and TMA): an output or key buffer 4 bytes off it is
    refused with KVB_E_ARG before any launch, the output and the state stay as
    they were, and an aligned call then runs normally."""
    kvb = kvb_mod()
    layer = I.Layer(I.GATED_DELTA, 2, 4, 128, 128, "bf16", qk_dist="l2norm")
    rng = np.random.default_rng(305)
    B, L = 2, 70
    pool = make_pool(layer, 4, B, 1, 8)
    for r in range(B):
        pool.set_request(r, r, [r])
    S0 = I.draw_state(rng, layer, B)
    pool.state.copy_(torch.from_numpy(S0))
    tok = I.draw_tokens(rng, layer, (B, L))
    q, k, v, log_g, beta = token_tensors(tok, layer, slice(None))
    n_o = B * L * layer.n_v_heads * layer.d_v
    big = torch.full((n_o + 1,), float("nan"), device="cuda")
    o_bad = big[1:].view(B, L, layer.n_v_heads, layer.d_v)
    assert o_bad.data_ptr() % 16 == 4
    kbig = torch.empty(k.numel() + 2, dtype=k.dtype, device="cuda")
    k_bad = kbig[2:].view(k.shape)
    k_bad.copy_(k)
    assert k_bad.data_ptr() % 16 == 4
    for args in ((q, k, v, log_g, beta, o_bad), (q, k_bad, v, log_g, beta, None)):
        with pytest.raises(kvb.KvbError) as ex:
            pool.prefill(np.arange(B), *args[:5], o=args[5], from_zero=True)
        assert ex.value.status == kvb.KVB_E_ARG
    torch.cuda.synchronize()
    assert torch.isnan(big).all()
    assert np.array_equal(pool.state.cpu().numpy(), S0)
    o = pool.prefill(np.arange(B), q, k, v, log_g, beta, from_zero=True).cpu().numpy()
    zero = np.zeros((layer.n_v_heads, layer.d_k, layer.d_v))
    for r in range(B):
        o_ref, _, _ = oracle.decode_sequence(zero, _prompt(tok, r, L), layer.variant)
        assert rel_err(o[r], o_ref) <= tol_for(layer), r
    assert pool.get_error() is None


def test_prefill_long_prompt_gated_delta():
    """Sixteen chunks (1024 tokens): rounding does not build up across chunks."""
    layer = I.Layer(I.GATED_DELTA, 1, 2, 128, 128, "bf16", qk_dist="l2norm")
    rng = np.random.default_rng(301)
    B, L = 2, 1024
    pool = make_pool(layer, 8, B, 1, 8)
    for r in range(B):
        pool.set_request(r, r, [r])
    tok = I.draw_tokens(rng, layer, (B, L))
    o = pool.prefill(np.arange(B), *token_tensors(tok, layer, slice(None))).cpu().numpy()
    st = pool.state.cpu().numpy()
    tol = tol_for(layer)
    zero = np.zeros((layer.n_v_heads, layer.d_k, layer.d_v))
    for r in range(B):
        o_ref, S_r, _ = oracle.decode_sequence(zero, _prompt(tok, r, L), layer.variant)
        assert rel_err(o[r], o_ref) <= tol, r
        assert rel_err(st[r], S_r) <= tol, r


def test_prefill_errors():
    kvb = kvb_mod()
    layer = I.Layer(I.GATED, 1, 1, 64, 64, "bf16")
    rng = np.random.default_rng(302)
    pool = make_pool(layer, 4, 3, 1, 8, num_slots=2)
    pool.set_request(0, 0, [0])
    pool.set_request(1, -1, [1])
    pool.set_request(2, 1, [2])
    tok = I.draw_tokens(rng, layer, (1, 8))
    args = token_tensors(tok, layer, slice(None))
    dtok = I.draw_tokens(rng, layer, (1,))
    pool.decode([2], *token_tensors(dtok, layer, slice(None)))
    for req, lengths, code in (([1], None, kvb.KVB_E_STATE),      # no state slot
                               ([2], None, kvb.KVB_E_STATE),      # buffer not empty
                               ([0], [9], kvb.KVB_E_ARG)):        # longer than L
        with pytest.raises(kvb.KvbError) as ex:
            pool.prefill(req, *args, lengths=lengths)
        assert ex.value.status == code
    pool.flush([2])
    pool.prefill([2], *args)
    assert pool.get_error() is None


def test_prefill_wait_timeout_reports_and_recovers():
    """The tensor-core prefill waits for its tensor-core products with bounded polls.
    A test hook caps every wait on the products of a CTA's first chunk at one
    non-blocking poll, so one of them runs out while its products are still in
    flight (the delta rule's block products are issued only after the first
    block's solve, right before the next warpgroup looks): each CTA records a
    timeout (kind 2) in the error word, waits with the full bound for the products
    and copies in flight, releases its tensor memory and returns; nothing faults.
    The same context then runs a normal prefill that matches the recurrence."""
    kvb = kvb_mod()
    layer = I.Layer(I.GATED_DELTA, 2, 4, 128, 128, "bf16", qk_dist="l2norm")
    B, L = 2, 50
    rng = np.random.default_rng(333)
    pool = make_pool(layer, 8, B, 1, 8)
    for r in range(B):
        pool.set_request(r, r, [r])
    tok = I.draw_tokens(rng, layer, (B, L))
    kvb.set_prefill_wait_limit(1)
    try:
        pool.prefill(np.arange(B), *token_tensors(tok, layer, slice(None)), from_zero=True)
        err = pool.get_error()
    finally:
        kvb.set_prefill_wait_limit(0)
    assert err is not None and err[0] == 2, err
    assert 0 <= err[1] < B and 0 <= err[2] < layer.n_v_heads
    o = pool.prefill(np.arange(B), *token_tensors(tok, layer, slice(None)), from_zero=True)
    torch.cuda.synchronize()
    o = o.cpu().numpy()
    st = pool.state.cpu().numpy()
    zero = np.zeros((layer.n_v_heads, layer.d_k, layer.d_v))
    for r in range(B):
        o_ref, S_r, _ = oracle.decode_sequence(zero, _prompt(tok, r, L), layer.variant)
        assert rel_err(o[r], o_ref) <= tol_for(layer), r
        assert rel_err(st[r], S_r) <= tol_for(layer), r
    assert pool.get_error() is None
