"""GPU parity: the persistent buffered decode and fold (launches large enough for them).

Batches of 200 requests x 32 value heads (6400 units, at least 8 per resident
CTA on a 152-SM part) take the persistent kernel; the staggered warm-up
launches of random subsets take the per-head kernel, so both run on the same
pool.  Every variant and both input dtypes; m = 9 reaches the largest staged
buffer (8 tokens).  Sampled requests are compared with the fp64 oracle (every
output, the state after the last fold), and all lengths bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from kv_buffered_decoding_gb300 import inputs as I
from tests.gpu_harness import make_pool, rel_err, token_tensors, tol_for

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


@pytest.mark.parametrize("layer,m", [
    (I.Layer(I.GATED_DELTA, 8, 32, 128, 128, "bf16", qk_dist="l2norm"), 9),
    (I.Layer(I.GATED, 16, 32, 128, 128, "f32"), 8),
    (I.Layer(I.PLAIN, 32, 32, 128, 128, "bf16"), 4),
    (I.Layer(I.GATED_DELTA, 16, 32, 128, 128, "f32", qk_dist="l2norm"), 8),
], ids=["gated_delta_bf16_m9", "gated_f32_m8", "plain_bf16_m4", "gated_delta_f32_m8"])
def test_persistent_decode(layer, m):
    B, bs = 200, 8
    nb = -(-m // bs)
    rng = np.random.default_rng(700 + m + layer.variant)
    pool = make_pool(layer, m, B, nb, bs, num_blocks=B * nb + 16)
    S0 = I.draw_state(rng, layer, B)
    pool.state.copy_(torch.from_numpy(S0))
    perm = rng.permutation(B * nb + 16)
    for r in range(B):
        pool.set_request(r, r, [int(x) for x in perm[r * nb:(r + 1) * nb]])
    sample = np.array([0, 1, 57, 99, 150, 199])
    hist = {r: [] for r in sample}  # per-step token dicts of the sampled rows

    def one(tok, i):
        return {key: (None if val is None else val[i:i + 1]) for key, val in tok.items()}

    # staggered start: request r first decodes r % m tokens in ragged subset launches
    occ = np.arange(B) % m
    for s in range(m - 1):
        rows = np.nonzero(occ > s)[0]
        tok = I.draw_tokens(rng, layer, (len(rows),))
        pool.decode(rows, *token_tensors(tok, layer, slice(None)))
        for i, r in enumerate(rows):
            if r in hist:
                hist[r].append(one(tok, i))
    n = occ.copy()
    assert np.array_equal(pool.get_lengths(), n)
    tol = tol_for(layer)
    req = np.arange(B)
    outs = {r: [] for r in sample}
    steps = 2 * m + 3
    for t in range(steps):
        tok = I.draw_tokens(rng, layer, (B,))
        o = pool.decode(req, *token_tensors(tok, layer, slice(None))).cpu().numpy()
        for r in sample:
            hist[r].append(one(tok, r))
            outs[r].append(o[r])
        n = (n + 1) % m
        assert np.array_equal(pool.get_lengths(), n), t
    torch.cuda.synchronize()
    st = pool.state.cpu().numpy()
    for r in sample:
        seq = {key: (None if hist[r][0][key] is None
                     else np.concatenate([h[key] for h in hist[r]])) for key in hist[r][0]}
        total = seq["v"].shape[0]
        o_ref, _, states = oracle.decode_sequence(S0[r], seq, layer.variant,
                                                  keep_states=range(total))
        assert rel_err(np.stack(outs[r]), o_ref[total - steps:]) <= tol, r
        last_fold = total - int(n[r]) - 1
        assert rel_err(st[r], states[last_fold]) <= tol, r
    assert np.array_equal(pool.get_device_lengths(), n)
    assert pool.get_error() is None


@pytest.mark.parametrize("layer,promote", [
    (I.Layer(I.GATED_DELTA, 8, 32, 128, 128, "bf16", qk_dist="l2norm"), False),
    (I.Layer(I.GATED, 16, 32, 128, 128, "f32"), False),
    (I.Layer(I.PLAIN, 32, 32, 128, 128, "bf16"), False),
    (I.Layer(I.GATED_DELTA, 8, 32, 128, 128, "bf16", qk_dist="l2norm"), True),
    (I.Layer(I.GATED, 16, 32, 128, 128, "bf16"), True),
], ids=["flush_gated_delta_bf16", "flush_gated_f32", "flush_plain_bf16",
        "promote_gated_delta_bf16", "promote_gated_bf16"])
def test_persistent_fold(layer, promote):
    """Flush (or promote) of 200 requests x 32 heads holding 0..8 buffered tokens.

    With every row at most 8 tokens long and at least 8 units per resident CTA
    the fold takes the streaming kernel.  Promotion starts from S = 0 whatever
    the slot held (the slots are filled with NaN first)."""
    B, bs, m = 200, 8, 9
    rng = np.random.default_rng(720 + layer.variant + 10 * promote)
    pool = make_pool(layer, m, B, 2, bs, num_blocks=2 * B + 8, num_slots=B + 1)
    perm = rng.permutation(2 * B + 8)
    S0 = np.zeros((B, layer.n_v_heads, layer.d_k, layer.d_v), dtype=np.float32)
    if not promote:
        S0 = I.draw_state(rng, layer, B)
        pool.state[:B].copy_(torch.from_numpy(S0))
    for r in range(B):
        pool.set_request(r, -1 if promote else r, [int(x) for x in perm[2 * r:2 * r + 2]])
    lengths = rng.integers(0, 9, size=B)
    lengths[:3] = [0, 8, 1]
    hist = [[] for _ in range(B)]
    for t in range(8):
        rows = np.nonzero(lengths > t)[0]
        tok = I.draw_tokens(rng, layer, (len(rows),))
        args = token_tensors(tok, layer, slice(None))
        if promote:
            pool.short_ctx(rows, *args)
        else:
            pool.decode(rows, *args)
        for i, r in enumerate(rows):
            hist[r].append({key: (None if val is None else val[i:i + 1])
                            for key, val in tok.items()})
    assert np.array_equal(pool.get_lengths(), lengths)
    req = np.arange(B)
    slots = rng.permutation(B) if promote else req
    if promote:
        pool.state.fill_(float("nan"))
        pool.promote(req, slots)
    else:
        pool.flush(req)
    torch.cuda.synchronize()
    st = pool.state.cpu().numpy()
    tol = tol_for(layer)
    for r in list(range(0, B, 7)) + [1, 2, B - 1]:
        if lengths[r] == 0:
            if promote:
                assert np.all(st[slots[r]] == 0.0), r
            else:
                assert np.array_equal(st[r], S0[r]), r
            continue
        seq = {key: (None if hist[r][0][key] is None
                     else np.concatenate([h[key] for h in hist[r]])) for key in hist[r][0]}
        _, S_ref, _ = oracle.decode_sequence(S0[r], seq, layer.variant)
        assert rel_err(st[slots[r]], S_ref) <= tol, r
    if promote:
        assert np.all(np.isnan(st[B]))
    assert np.array_equal(pool.get_lengths(), np.zeros(B))
    assert np.array_equal(pool.get_device_lengths(), np.zeros(B))
    assert pool.get_error() is None


def _stack(hist):
    return {key: np.stack(val) for key, val in hist.items()}


@pytest.mark.parametrize("layer,B,bs", [
    (I.Layer(I.GATED_DELTA, 8, 32, 128, 128, "bf16", qk_dist="l2norm"), 160, 4),
    (I.Layer(I.GATED, 16, 16, 128, 128, "f32"), 200, 4),
    (I.Layer(I.PLAIN, 16, 16, 128, 128, "bf16"), 200, 4),
    (I.Layer(I.GATED_DELTA, 16, 16, 128, 128, "f32", qk_dist="l2norm"), 120, 4),
    (I.Layer(I.GATED, 16, 16, 128, 128, "bf16"), 200, 8),
    (I.Layer(I.PLAIN, 8, 16, 128, 128, "bf16"), 160, 16),
], ids=["gated_delta_bf16", "gated_f32", "plain_bf16", "gated_delta_f32", "gated_bf16_bs8",
        "plain_bf16_grouped_bs16"])
def test_short_ctx_large_batch(layer, B, bs):
    """Short-context decode of B requests (no state) growing to ragged lengths
    1..64 in 64-slot buffers, launches from B rows down to a handful.  With 4-token
    blocks the ids beyond the row descriptor's come from the block table; 8- and
    16-token blocks (the bench's size, and a grouped layer) cover whole blocks per
    id.  Sampled outputs against the oracle's buffer-only decode, all lengths bit
    for bit."""
    nb = 64 // bs
    cap = nb * bs
    rng = np.random.default_rng(740 + layer.variant + B)
    pool = make_pool(layer, 8, B, nb, bs, num_blocks=B * nb + 8, num_slots=1)
    blocks = rng.permutation(B * nb + 8)
    for r in range(B):
        pool.set_request(r, -1, [int(x) for x in blocks[r * nb:(r + 1) * nb]])
    lengths = rng.integers(1, cap + 1, size=B)
    lengths[:2] = [cap, 1]
    sample = [0, 1, 5, 77, B - 1]
    hist = {r: {} for r in sample}
    tol = tol_for(layer)
    for t in range(cap):
        rows = np.nonzero(lengths > t)[0]
        tok = I.draw_tokens(rng, layer, (len(rows),))
        o = pool.short_ctx(rows, *token_tensors(tok, layer, slice(None))).cpu().numpy()
        for i, r in enumerate(rows):
            if r in hist:
                for key, val in tok.items():
                    if val is not None:
                        hist[r].setdefault(key, []).append(val[i])
                if t in (0, 9, 31, 47, cap - 1) or t == lengths[r] - 1:
                    o_ref = oracle.short_context(_stack(hist[r]), layer.variant, layer.d_k,
                                                 layer.d_v)
                    assert rel_err(o[i], o_ref[-1]) <= tol, (t, r)
        assert np.array_equal(pool.get_lengths(), np.minimum(lengths, t + 1)), t
    assert np.array_equal(pool.get_device_lengths(), lengths)
    assert pool.get_error() is None
