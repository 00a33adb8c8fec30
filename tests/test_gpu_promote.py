"""GPU parity: short-to-long promotion (kvb_promote).

Short-context requests of ragged lengths (0 up to their whole 32-slot buffer)
decode from the buffer alone, are promoted to a state slot, and continue with
kvb_decode (auto-fold at m) and a verify/accept round.  The promoted state must
equal the fp64 recurrence from S = 0 over the request's history (all zeros for
an empty history, exactly), and every later output the recurrence over the
whole history.  Lengths are compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from kv_buffered_decoding_gb300 import inputs as I
from tests.gpu_harness import kvb_mod, make_pool, rel_err, token_tensors, tol_for

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _append(hist, tok, idx):
    for key, val in tok.items():
        if val is not None:
            hist.setdefault(key, []).append(val[idx])


def _stack(hist):
    return {key: np.stack(val) for key, val in hist.items()}


@pytest.mark.parametrize("layer,m", [
    (I.Layer(I.GATED_DELTA, 2, 4, 64, 64, "bf16", qk_dist="l2norm"), 4),
    (I.Layer(I.GATED, 2, 2, 128, 128, "bf16"), 8),
    (I.Layer(I.PLAIN, 1, 1, 64, 64, "f32"), 3),
], ids=["gated_delta_d64", "gated_d128", "plain_d64_f32"])
def test_promote_then_decode(layer, m):
    kvb = kvb_mod()
    rng = np.random.default_rng(40 + m)
    R, nb, bs = 6, 4, 8
    cap = nb * bs
    pool = make_pool(layer, m, R, nb, bs, num_blocks=R * nb + 4, num_slots=R + 1)
    blocks = rng.permutation(R * nb + 4)
    for r in range(R):
        pool.set_request(r, -1, [int(b) for b in blocks[r * nb:(r + 1) * nb]])
    lengths = np.array([0, 1, 5, 17, cap, 9])
    hist = [dict() for _ in range(R)]
    tol = tol_for(layer)
    for t in range(cap):
        rows = np.nonzero(lengths > t)[0]
        tok = I.draw_tokens(rng, layer, (len(rows),))
        o = pool.short_ctx(rows, *token_tensors(tok, layer, slice(None))).cpu().numpy()
        for i, r in enumerate(rows):
            _append(hist[r], tok, i)
        if t in (0, 16, cap - 1):
            for i, r in enumerate(rows):
                o_ref = oracle.short_context(_stack(hist[r]), layer.variant, layer.d_k,
                                             layer.d_v)
                assert rel_err(o[i], o_ref[-1]) <= tol, (t, r)
    assert np.array_equal(pool.get_lengths(), lengths)

    # promote every request into slots in a shuffled order (slot R stays free)
    slots = rng.permutation(R)
    req = np.arange(R)
    pool.state.fill_(float("nan"))  # whatever the slots held before must not matter
    pool.promote(req, slots)
    torch.cuda.synchronize()
    assert np.array_equal(pool.get_lengths(), np.zeros(R))
    assert np.array_equal(pool.get_device_lengths(), np.zeros(R))
    st = pool.state.cpu().numpy()
    S = []
    for r in range(R):
        if lengths[r] == 0:
            assert np.all(st[slots[r]] == 0.0)
            S.append(np.zeros((layer.n_v_heads, layer.d_k, layer.d_v)))
        else:
            _, S_r, _ = oracle.decode_sequence(
                np.zeros((layer.n_v_heads, layer.d_k, layer.d_v)), _stack(hist[r]), layer.variant)
            assert rel_err(st[slots[r]], S_r) <= tol, r
            S.append(S_r)
    assert np.all(np.isnan(st[R]))  # the unused slot is untouched

    # the promoted requests continue as state-backed requests
    n = np.zeros(R, dtype=np.int64)
    for t in range(2 * m + 1):
        tok = I.draw_tokens(rng, layer, (R,))
        o = pool.decode(req, *token_tensors(tok, layer, slice(None))).cpu().numpy()
        for r in range(R):
            one = {key: (None if val is None else val[r:r + 1]) for key, val in tok.items()}
            o_ref, S[r], _ = oracle.decode_sequence(S[r], one, layer.variant)
            assert rel_err(o[r], o_ref[0]) <= tol, (t, r)
        n = (n + 1) % m
        assert np.array_equal(pool.get_lengths(), n)
    T = 3
    tok = I.draw_tokens(rng, layer, (R, T))
    o = pool.verify(req, *token_tensors(tok, layer, slice(None))).cpu().numpy()
    acc = rng.integers(0, T + 1, size=R)
    pool.accept(req, acc)
    for r in range(R):
        dr = {key: (None if val is None else val[r]) for key, val in tok.items()}
        assert rel_err(o[r], oracle.verify(S[r], dr, layer.variant)) <= tol, r
    pool.flush(req)
    torch.cuda.synchronize()
    st = pool.state.cpu().numpy()
    for r in range(R):
        acc_tok = {key: (None if val is None else val[r, :acc[r]]) for key, val in tok.items()}
        _, S_r, _ = oracle.decode_sequence(S[r], acc_tok, layer.variant)
        assert rel_err(st[slots[r]], S_r) <= tol, r
    assert pool.get_error() is None

    # errors: already state-backed; slot owned or listed twice; out of range
    with pytest.raises(kvb.KvbError) as ex:
        pool.promote([0], [R])
    assert ex.value.status == kvb.KVB_E_STATE
    pool.release_request(1)
    pool.set_request(1, -1, [int(b) for b in blocks[nb:2 * nb]])
    for sl, code in (([slots[2]], kvb.KVB_E_RANGE), ([R + 1], kvb.KVB_E_RANGE),
                     ([-1], kvb.KVB_E_RANGE)):
        with pytest.raises(kvb.KvbError) as ex:
            pool.promote([1], sl)
        assert ex.value.status == code
    pool.promote([1], [R])
    torch.cuda.synchronize()
    assert np.all(pool.state[R].cpu().numpy() == 0.0)
