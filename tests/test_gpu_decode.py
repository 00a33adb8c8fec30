"""GPU parity: buffered decode, fold, recurrent baseline, against the fp64 oracle.

Workloads (seeded, synthetic):
* ungated, 1 request, 1 head, d=64, fp32: 16-token prefill (verify + accept,
  which folds all 16), then 64 decode steps with m = 4; every output, the
  state after the prefill, after every fold and at the end.
* scalar-gated, B=32, H=16, d=128, bf16, 1024-token prefill state, 256 steps,
  m in {0, 2, 4, 8, 16} (m = 0 is the recurrent baseline).
* gated delta rule, 16 q/k heads shared by 32 value heads, d=128, bf16: a
  small batch compared in full, and the full B=256, m=8 launch with outputs
  and states of sampled requests compared (requests are independent).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from kv_buffered_decoding_gb300 import inputs as I
from tests.gpu_harness import (blocks_needed, dev, make_pool, rel_err, token_tensors, tol_for)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _buffered_keys_at(pool, block_ids, n, bs):
    """Keys stored for token slots 0..n-1 of a request owning `block_ids`."""
    kb = pool.kbuf.float().cpu().numpy()
    return np.stack([kb[block_ids[p // bs], :, p % bs] for p in range(n)]) if n else None


def test_ungated_fp32_prefill_and_decode():
    w = I.WORKLOADS["ungated_d64_f32"]
    layer = w.layer
    rng = np.random.default_rng(w.seed)
    n_tok = w.prefill + w.steps
    tok = I.draw_tokens(rng, layer, (n_tok, 1))
    S_zero = np.zeros((1, 1, layer.d_k, layer.d_v))
    o_ref, S_end, states = oracle.decode_sequence(S_zero, tok, layer.variant,
                                                  keep_states=range(n_tok))
    cap = 16
    pool = make_pool(layer, w.m, 1, blocks_needed(cap, w.block_size), w.block_size)
    pool.state.zero_()
    pool.set_request(0, 0, [1, 0])  # blocks in reverse order: the table must be honoured
    tol = tol_for(layer)

    # prefill: 16 drafts verified together, all accepted -> one fold of 16 tokens
    P = w.prefill
    pre = {k_: (None if v_ is None else v_[:P].transpose(1, 0, *range(2, v_.ndim)))
           for k_, v_ in tok.items()}
    q, k, v, g, b = (dev(pre["q"], layer), dev(pre["k"], layer), dev(pre["v"], layer), None, None)
    o = pool.verify([0], q, k, v, g, b)
    assert rel_err(o.cpu().numpy()[0], o_ref[:P, 0]) <= tol
    pool.accept([0], [P])
    assert pool.get_lengths()[0] == 0
    torch.cuda.synchronize()
    assert rel_err(pool.state[0].cpu().numpy(), states[P - 1][0]) <= tol

    n = 0
    for t in range(P, n_tok):
        q, k, v, g, b = token_tensors(tok, layer, t)
        o = pool.decode([0], q, k, v, g, b)
        assert rel_err(o.cpu().numpy(), o_ref[t]) <= tol, t
        n = (n + 1) % w.m
        assert pool.get_lengths()[0] == n
        if n == 0:
            assert rel_err(pool.state[0].cpu().numpy(), states[t][0]) <= tol, t
    assert np.array_equal(pool.get_device_lengths(), pool.get_lengths())
    assert pool.get_error() is None
    # 64 decode steps = 16 full cycles: the stored state is the oracle's final state
    assert rel_err(pool.state[0].cpu().numpy(), S_end[0]) <= tol
    # two more tokens stay buffered, in block 1 (the first block of the table)
    for t in range(2):
        q, k, v, g, b = token_tensors(tok, layer, n_tok - 2 + t)
        pool.decode([0], q, k, v, g, b)
    got = _buffered_keys_at(pool, [1, 0], 2, w.block_size)
    assert np.array_equal(got, tok["k"][n_tok - 2:, 0])
    assert pool.get_lengths()[0] == 2


@pytest.fixture(scope="module")
def gated_case():
    w = I.WORKLOADS["gated_B32_H16_d128"]
    layer = w.layer
    rng = np.random.default_rng(w.seed)
    B = w.batch
    pre = I.draw_tokens(rng, layer, (w.prefill, B))
    S0 = oracle.gated_prefill_closed_form(pre, layer.variant).astype(np.float32)
    tok = I.draw_tokens(rng, layer, (w.steps, B))
    o_ref, S_end, states = oracle.decode_sequence(S0, tok, layer.variant,
                                                  keep_states=range(w.steps))
    return w, S0, tok, o_ref, states


@pytest.mark.parametrize("m", [0, 2, 4, 8, 16])
def test_gated_sweep_m(gated_case, m):
    w, S0, tok, o_ref, states = gated_case
    layer = w.layer
    B, bs = w.batch, w.block_size
    nbpr = blocks_needed(max(m, 1), bs) if m > 0 else 0
    pool = make_pool(layer, m, B, max(nbpr, 1), bs)
    pool.state.copy_(torch.from_numpy(S0))
    perm = np.random.default_rng(99).permutation(B * max(nbpr, 1))
    for r in range(B):
        pool.set_request(r, r, perm[r * nbpr:(r + 1) * nbpr] if nbpr else [])
    req = np.arange(B)
    tol = tol_for(layer)
    worst = 0.0
    last_fold = -1
    for t in range(w.steps):
        q, k, v, g, b = token_tensors(tok, layer, t)
        o = pool.decode(req, q, k, v, g, b)
        worst = max(worst, rel_err(o.cpu().numpy(), o_ref[t]))
        if m == 0 or (t + 1) % m == 0:
            last_fold = t
            if t % 64 == 63 or m == 0 and t % 64 == 0:
                torch.cuda.synchronize()
                assert rel_err(pool.state.cpu().numpy(), states[t]) <= tol, t
    assert worst <= tol, worst
    torch.cuda.synchronize()
    assert rel_err(pool.state.cpu().numpy(), states[last_fold]) <= tol
    expect_len = 0 if m == 0 else w.steps % m
    assert (pool.get_lengths() == expect_len).all()
    assert np.array_equal(pool.get_device_lengths(), pool.get_lengths())
    # fold what is left: the state becomes the oracle's final state
    if m > 0:
        pool.flush(req)
        torch.cuda.synchronize()
        assert rel_err(pool.state.cpu().numpy(), states[w.steps - 1]) <= tol
        assert (pool.get_lengths() == 0).all()
    assert pool.get_error() is None


def _gdn_run(B, steps, sample, seed, stagger=False):
    w = I.WORKLOADS["gdn_B256_Hk16_Hv32_d128"]
    layer = w.layer
    rng = np.random.default_rng(seed)
    S0 = I.draw_state(rng, layer, B)
    tok = I.draw_tokens(rng, layer, (steps, B))
    bs, m = w.block_size, w.m
    pool = make_pool(layer, m, B, blocks_needed(m, bs), bs)
    pool.state.copy_(torch.from_numpy(S0))
    perm = np.random.default_rng(seed + 1).permutation(B)
    for r in range(B):
        pool.set_request(r, r, [int(perm[r])])
    # staggered start: request r first decodes (r % m) tokens alone (ragged launches)
    warm = {}
    if stagger:
        occ = np.arange(B) % m
        wtok = I.draw_tokens(rng, layer, (m - 1, B))
        for s in range(m - 1):
            rows = np.nonzero(occ > s)[0]
            q, k, v, g, b = token_tensors(wtok, layer, (s, rows))
            pool.decode(rows, q, k, v, g, b)
        warm = {"tok": wtok, "occ": occ}
        assert np.array_equal(pool.get_lengths(), occ)
    outs = []
    req = np.arange(B)
    for t in range(steps):
        q, k, v, g, b = token_tensors(tok, layer, t)
        outs.append(pool.decode(req, q, k, v, g, b).cpu().numpy()[sample])
    torch.cuda.synchronize()
    return w, layer, S0, tok, np.stack(outs), pool, warm, perm


def _gdn_oracle(layer, S0, tok, sample, warm, steps, m):
    """Oracle outputs for the sampled requests (history = warm-up tokens, then the steps)."""
    o_all, states_all = [], []
    for r in sample:
        hist = {}
        if warm:
            nw = int(warm["occ"][r])
            for key, val in tok.items():
                wv = warm["tok"][key]
                hist[key] = None if val is None else np.concatenate([wv[:nw, r], val[:steps, r]])
        else:
            hist = {key: (None if val is None else val[:steps, r]) for key, val in tok.items()}
        n_hist = hist["v"].shape[0]
        o, _, st = oracle.decode_sequence(S0[r], hist, layer.variant, keep_states=range(n_hist))
        offset = n_hist - steps
        o_all.append(o[offset:])
        states_all.append((st, offset))
    return np.stack(o_all, axis=1), states_all


def test_gdn_small_batch_full_compare():
    B, steps = 4, 40
    sample = np.arange(B)
    w, layer, S0, tok, outs, pool, warm, perm = _gdn_run(B, steps, sample, seed=20)
    o_ref, st = _gdn_oracle(layer, S0, tok, sample, warm, steps, w.m)
    assert rel_err(outs, o_ref) <= tol_for(layer)
    last_fold = (steps // w.m) * w.m - 1
    for i, r in enumerate(sample):
        states, off = st[i]
        assert rel_err(pool.state[r].cpu().numpy(), states[off + last_fold]) <= tol_for(layer)
    assert pool.get_error() is None


@pytest.mark.parametrize("stagger", [False, True])
def test_gdn_full_size_sampled(stagger):
    """B=256, m=8: the launch configuration the benchmark times; 3 full cycles."""
    B, steps = 256, 24
    sample = np.array([0, 1, 37, 100, 127, 128, 200, 255])
    w, layer, S0, tok, outs, pool, warm, perm = _gdn_run(B, steps, sample, seed=21,
                                                          stagger=stagger)
    o_ref, st = _gdn_oracle(layer, S0, tok, sample, warm, steps, w.m)
    assert rel_err(outs, o_ref) <= tol_for(layer)
    lengths = pool.get_lengths()
    for i, r in enumerate(sample):
        states, off = st[i]
        n_tot = off + steps
        n_buf = n_tot % w.m
        assert lengths[r] == n_buf
        last_fold = n_tot - n_buf - 1
        assert rel_err(pool.state[r].cpu().numpy(), states[last_fold]) <= tol_for(layer)
        # bit-exact placement: buffered slot p holds the key of token (last_fold + 1 + p)
        if n_buf:
            got = _buffered_keys_at(pool, [int(perm[r])], n_buf, w.block_size)
            if warm:
                nw = int(warm["occ"][r])
                hist_k = np.concatenate([warm["tok"]["k"][:nw, r], tok["k"][:steps, r]])
            else:
                hist_k = tok["k"][:steps, r]
            assert np.array_equal(got, hist_k[last_fold + 1:last_fold + 1 + n_buf])
    assert np.array_equal(pool.get_device_lengths(), lengths)
    assert pool.get_error() is None
