"""GPU parity: buffered decode, fold, recurrent baseline, against the fp64 oracle.

Workloads (seeded, synthetic):
* ungated, 1 request, 1 head, d=64, fp32: 16-token prefill (verify + accept,
  which folds all 16), then 64 decode steps with m = 4; every output, the
  state after the prefill, after every fold and at the end.
* scalar-gated, B=32, H=16, d=128, bf16, 1024-token prefill state, 256 steps,
  m in {0, 2, 4, 8, 16} (m = 0 is the recurrent baseline).
* gated delta rule, 16 q/k heads shared by 32 value heads, d=128, bf16, the
  full B=256, m=8 launch for 64 steps (8 buffer cycles), from a cycle-aligned
  and from a staggered start: every request's output at every step and every
  request's state after its last fold.

Errors are taken per tensor (one request's output o_t, one request's state)
and the worst over the run is compared with the tolerance.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from kv_buffered_decoding_gb300 import inputs as I
from tests import oracle_pool
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
        worst = max(worst, oracle_pool.rel_err_rows(o.cpu().numpy(), o_ref[t], 1).max())
        if m == 0 or (t + 1) % m == 0:
            last_fold = t
            if t % 64 == 63 or m == 0 and t % 64 == 0:
                torch.cuda.synchronize()
                assert oracle_pool.rel_err_rows(pool.state.cpu().numpy(), states[t], 1).max() <= tol, t
    assert worst <= tol, worst
    torch.cuda.synchronize()
    assert oracle_pool.rel_err_rows(pool.state.cpu().numpy(), states[last_fold], 1).max() <= tol
    expect_len = 0 if m == 0 else w.steps % m
    assert (pool.get_lengths() == expect_len).all()
    assert np.array_equal(pool.get_device_lengths(), pool.get_lengths())
    # fold what is left: the state becomes the oracle's final state
    if m > 0:
        pool.flush(req)
        torch.cuda.synchronize()
        assert oracle_pool.rel_err_rows(pool.state.cpu().numpy(), states[w.steps - 1], 1).max() <= tol
        assert (pool.get_lengths() == 0).all()
    assert pool.get_error() is None


def _gdn_full(B, steps, seed, stagger, scale=1.0):
    """Run B requests of the gated-delta layer for ``steps`` decode steps on the GPU
    (after ``r % m`` warm-up tokens for request r when staggered) and compare every
    output and every final state with the oracle, per tensor."""
    w = I.WORKLOADS["gdn_B256_Hk16_Hv32_d128"]
    layer = w.layer
    rng = np.random.default_rng(seed)
    S0 = I.draw_state(rng, layer, B)
    tok = I.draw_tokens(rng, layer, (steps, B))
    bs, m = w.block_size, w.m
    pool = make_pool(layer, m, B, blocks_needed(m, bs), bs, scale=scale)
    pool.state.copy_(torch.from_numpy(S0))
    perm = np.random.default_rng(seed + 1).permutation(B)
    for r in range(B):
        pool.set_request(r, r, [int(perm[r])])
    occ = np.arange(B) % m if stagger else np.zeros(B, dtype=np.int64)
    wtok = I.draw_tokens(rng, layer, (m - 1, B))
    for s in range(m - 1):  # warm-up tokens on subsets of the rows: ragged launches
        rows = np.nonzero(occ > s)[0]
        if len(rows):
            pool.decode(rows, *token_tensors(wtok, layer, (s, rows)))
    assert np.array_equal(pool.get_lengths(), occ.astype(np.int32))
    req = np.arange(B)
    outs = np.empty((steps, B, layer.n_v_heads, layer.d_v), dtype=np.float32)
    for t in range(steps):
        outs[t] = pool.decode(req, *token_tensors(tok, layer, t)).cpu().numpy()
    torch.cuda.synchronize()
    states = pool.state.cpu().numpy()
    lengths = pool.get_lengths()
    n_tot = occ + steps
    assert np.array_equal(lengths, (n_tot % m).astype(np.int32))
    assert np.array_equal(pool.get_device_lengths(), lengths)
    assert pool.get_error() is None

    # one oracle task per chunk of requests with the same warm-up length
    tasks = []
    for o in np.unique(occ):
        same = np.nonzero(occ == o)[0]
        for part in np.array_split(same, max(1, len(same) // 16)):
            hist = {}
            for key, val in tok.items():
                hist[key] = None if val is None else np.concatenate([wtok[key][:o, part], val[:, part]])
            nt = int(o) + steps
            last_fold = nt - nt % m - 1
            tasks.append(dict(S0=S0[part], hist=hist, out=outs[:, part], state=states[part],
                              fold_at=np.full(len(part), last_fold), variant=layer.variant,
                              scale=scale, rows=part))
    results = oracle_pool.run(oracle_pool.decode_errors, tasks)
    err_o = np.zeros(B)
    err_s = np.zeros(B)
    for task, (eo, es) in zip(tasks, results):
        err_o[task["rows"]] = eo
        err_s[task["rows"]] = es
    tol = tol_for(layer)
    assert err_o.max() <= tol, (err_o.max(), int(err_o.argmax()))
    assert err_s.max() <= tol, (err_s.max(), int(err_s.argmax()))

    # bit-exact placement: buffered slot p of a request holds the key of its
    # (last fold + 1 + p)-th history token, for every request
    kb = pool.kbuf.float().cpu().numpy()
    for r in range(B):
        nb = int(lengths[r])
        if nb == 0:
            continue
        o = int(occ[r])
        hist_k = np.concatenate([wtok["k"][:o, r], tok["k"][:, r]])
        got = np.stack([kb[perm[r], :, p] for p in range(nb)])
        assert np.array_equal(got, hist_k[len(hist_k) - nb:]), r
    pool.close()
    return err_o.max(), err_s.max()


@pytest.mark.parametrize("layer", [
    I.Layer(I.GATED, 2, 4, 128, 128, "f32"),
    I.Layer(I.GATED_DELTA, 2, 4, 128, 128, "f32", qk_dist="l2norm"),
], ids=["gated_f32", "gated_delta_f32"])
@pytest.mark.parametrize("m", [5, 8, 12])
def test_fold_ranks_f32_d128(layer, m):
    """Folds of rank 5 to 12 on an fp32 pool at d = 128, in the per-head decode and flush
    kernels. Above rank 4 the rank update runs as tf32 tensor-core products with the fp32
    keys split into two parts (three products per tile); ranks above 8 take two k-steps.
    Every output and the state after every fold match the recurrence, and so does the state
    after a final flush of m - 1 tokens."""
    rng = np.random.default_rng(800 + m + 10 * layer.variant)
    B, bs = 3, 4
    steps = 3 * m - 1  # two folds, then m - 1 tokens left for the flush
    nb = blocks_needed(m, bs)
    pool = make_pool(layer, m, B, nb, bs)
    S0 = I.draw_state(rng, layer, B)
    pool.state.copy_(torch.from_numpy(S0))
    for r in range(B):
        pool.set_request(r, r, list(range(r * nb, (r + 1) * nb)))
    tok = I.draw_tokens(rng, layer, (steps, B))
    o_ref, _, states = oracle.decode_sequence(S0.astype(np.float64), tok, layer.variant,
                                              keep_states=range(steps))
    tol = tol_for(layer)
    req = np.arange(B)
    for t in range(steps):
        o = pool.decode(req, *token_tensors(tok, layer, t)).cpu().numpy()
        assert rel_err(o, o_ref[t]) <= tol, t
        if (t + 1) % m == 0:
            assert rel_err(pool.state.cpu().numpy(), states[t]) <= tol, t
    assert (pool.get_lengths() == m - 1).all()
    pool.flush(req)
    assert rel_err(pool.state.cpu().numpy(), states[steps - 1]) <= tol
    assert pool.get_error() is None


def test_gdn_small_batch_full_compare():
    _gdn_full(4, 40, seed=20, stagger=True)


@pytest.mark.parametrize("stagger", [False, True])
def test_gdn_full_size(stagger):
    """B=256, m=8: the launch configuration the benchmark times; 64 steps = 8
    buffer cycles; every request's output every step, every state."""
    _gdn_full(256, 64, seed=21, stagger=stagger)
