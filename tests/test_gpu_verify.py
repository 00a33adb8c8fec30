"""GPU parity: speculative verify of T drafts and accept of a prefix (no temporary states).

Workload: the scalar-gated layer (16 heads, d=128, bf16) with a 1024-token
prefill state, B=64 requests, m=8, T in {4, 2, 6, 8} drafts per round and an
accepted prefix length drawn uniformly from [0, T] per request and round,
200 rounds for every T.  Every round compares every request's draft outputs
with the oracle (recurrent output after the accepted history plus drafts
0..j) and the buffer lengths bit for bit with an independent host model
(n += j; fold all when n >= m); every request's state (the one of its last
fold) at checkpoints and, after a closing flush, the recurrent replay of
accepted tokens only.  Errors are per tensor (one request's draft output,
one request's state), the worst over the run.
"""
from __future__ import annotations

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

@pytest.fixture(scope="module")
def prefill_state():
    w = I.WORKLOADS["verify_B64_gated"]
    rng = np.random.default_rng(w.seed)
    pre = I.draw_tokens(rng, w.layer, (w.prefill, w.batch))
    return oracle.gated_prefill_closed_form(pre, w.layer.variant).astype(np.float32)


def _bt(x):
    """[B, T, ...] -> [T, B, ...] for the oracle."""
    return None if x is None else np.swapaxes(x, 0, 1)


@pytest.mark.parametrize("T", [4, 2, 6, 8])
def test_verify_accept_rounds(prefill_state, T):
    """Config: B=64, m=8, 200 rounds of verify + accept of a random prefix.  Every
    request's draft outputs every round; every request's state at checkpoints and
    after a closing flush; lengths bit for bit every round."""
    w = I.WORKLOADS["verify_B64_gated"]
    layer, B, m, bs, rounds = w.layer, w.batch, w.m, w.block_size, w.steps
    cap = m - 1 + T
    nb = blocks_needed(cap, bs)
    pool = make_pool(layer, m, B, nb, bs)
    pool.state.copy_(torch.from_numpy(prefill_state))
    perm = np.random.default_rng(w.seed + 100 + T).permutation(B * nb)
    for r in range(B):
        pool.set_request(r, r, perm[r * nb:(r + 1) * nb])
    rng = np.random.default_rng(w.seed * 1000 + T)
    req = np.arange(B)
    tok = I.draw_tokens(rng, layer, (rounds, B, T))
    acc = rng.integers(0, T + 1, size=(rounds, B))
    n_model = np.zeros(B, dtype=np.int64)
    outs = np.empty((rounds, B, T, layer.n_v_heads, layer.d_v), dtype=np.float32)
    fold_rounds = np.zeros((rounds, B), dtype=bool)
    checkpoints = {}
    for rnd in range(rounds):
        o = pool.verify(req, dev(tok["q"][rnd], layer), dev(tok["k"][rnd], layer),
                        dev(tok["v"][rnd], layer), dev(tok["log_g"][rnd], f32=True), None)
        pool.accept(req, acc[rnd])
        outs[rnd] = o.cpu().numpy()
        n_model = n_model + acc[rnd]
        folded = n_model >= m
        n_model[folded] = 0
        fold_rounds[rnd] = folded
        assert np.array_equal(pool.get_lengths(), n_model.astype(np.int32)), rnd
        if rnd % 25 == 24:
            torch.cuda.synchronize()
            checkpoints[rnd] = pool.state.cpu().numpy()
    assert np.array_equal(pool.get_device_lengths(), pool.get_lengths())
    pool.flush(req)  # fold whatever is buffered: states = replay of accepted tokens only
    torch.cuda.synchronize()
    final = pool.state.cpu().numpy()
    assert pool.get_error() is None
    pool.close()

    tasks = []
    for part in oracle_pool.chunks(B, 4):
        drafts = {key: (None if val is None else np.moveaxis(val[:, part], 1, 2))
                  for key, val in tok.items()}  # [rounds, T, r, ...]
        tasks.append(dict(S0=prefill_state[part], drafts=drafts, acc=acc[:, part],
                          out=outs[:, part], fold_rounds=fold_rounds[:, part],
                          checkpoints={k_: v_[part] for k_, v_ in checkpoints.items()},
                          final=final[part], variant=layer.variant))
    res = oracle_pool.run(oracle_pool.verify_errors, tasks)
    err_o = np.concatenate([r_[0] for r_ in res])
    err_ck = np.concatenate([r_[1] for r_ in res])
    err_f = np.concatenate([r_[2] for r_ in res])
    tol = tol_for(layer)
    assert err_o.max() <= tol, (err_o.max(), int(err_o.argmax()))
    assert err_ck.max() <= tol, (err_ck.max(), int(err_ck.argmax()))
    assert err_f.max() <= tol, (err_f.max(), int(err_f.argmax()))
    assert fold_rounds.sum() > B  # folds happened throughout


def test_accept_zero_and_full():
    """j = 0 leaves length and state untouched; j = T equals T decode steps."""
    w = I.WORKLOADS["verify_B64_gated"]
    layer, m, bs, T = w.layer, 8, 8, 4
    B = 3
    rng = np.random.default_rng(7)
    S0 = I.draw_state(rng, layer, B, scale=0.05)
    pool = make_pool(layer, m, B, 2, bs)
    pool.state.copy_(torch.from_numpy(S0))
    for r in range(B):
        pool.set_request(r, r, [2 * r + 1, 2 * r])
    tok = I.draw_tokens(rng, layer, (B, T))
    args = (dev(tok["q"], layer), dev(tok["k"], layer), dev(tok["v"], layer),
            dev(tok["log_g"], f32=True), None)
    pool.verify(np.arange(B), *args)
    pool.accept(np.arange(B), [0, T, 2])
    torch.cuda.synchronize()
    assert list(pool.get_lengths()) == [0, T, 2]
    assert torch.equal(pool.state[0].cpu(), torch.from_numpy(S0[0]))  # untouched, bit for bit
    # request 1 then decodes: its history is exactly the 4 accepted drafts
    nxt = I.draw_tokens(rng, layer, (1, B))
    o = pool.decode([1], dev(nxt["q"][0, 1:2], layer), dev(nxt["k"][0, 1:2], layer),
                    dev(nxt["v"][0, 1:2], layer), dev(nxt["log_g"][0, 1:2], f32=True), None)
    hist = {key: np.concatenate([np.swapaxes(tok[key], 0, 1)[:, 1], nxt[key][:, 1]])
            for key in ("q", "k", "v", "log_g")}
    hist["beta"] = None
    o_ref, _, _ = oracle.decode_sequence(S0[1], hist, layer.variant)
    assert rel_err(o.cpu().numpy()[0], o_ref[-1]) <= tol_for(layer)
    assert pool.get_error() is None


@pytest.mark.parametrize("T", [4, 6])
def test_verify_gated_delta_d128(T):
    """Gated delta rule at d=128 with grouped heads (the tensor-core verify path for
    bf16): 30 rounds of verify + random prefix accept; outputs every round, state at
    every fold and after a final flush."""
    layer = I.Layer(I.GATED_DELTA, 2, 4, 128, 128, "bf16", qk_dist="l2norm")
    B, m, bs = 8, 8, 8
    nb = blocks_needed(m - 1 + T, bs)
    rng = np.random.default_rng(40 + T)
    S0 = I.draw_state(rng, layer, B)
    pool = make_pool(layer, m, B, nb, bs)
    pool.state.copy_(torch.from_numpy(S0))
    perm = rng.permutation(B * nb)
    for r in range(B):
        pool.set_request(r, r, perm[r * nb:(r + 1) * nb])
    req = np.arange(B)
    S_hist = S0.astype(np.float64)
    n_model = np.zeros(B, dtype=np.int64)
    tol = tol_for(layer)
    for rnd in range(30):
        tok = I.draw_tokens(rng, layer, (B, T))
        o = pool.verify(req, dev(tok["q"], layer), dev(tok["k"], layer), dev(tok["v"], layer),
                        dev(tok["log_g"], f32=True), dev(tok["beta"], f32=True))
        j = rng.integers(0, T + 1, size=B)
        pool.accept(req, j)
        drafts = {key: _bt(val) for key, val in tok.items()}
        o_ref = oracle.verify(S_hist, drafts, layer.variant)
        assert oracle_pool.rel_err_rows(np.swapaxes(o.cpu().numpy(), 0, 1), o_ref, 2).max() <= tol, rnd
        S_hist = oracle.accept(S_hist, drafts, j, layer.variant)
        n_model = n_model + j
        folded = n_model >= m
        n_model[folded] = 0
        assert np.array_equal(pool.get_lengths(), n_model.astype(np.int32)), rnd
        if folded.any():
            torch.cuda.synchronize()
            st = pool.state.cpu().numpy()
            assert oracle_pool.rel_err_rows(st[folded], S_hist[folded], 1).max() <= tol, rnd
    pool.flush(req)
    torch.cuda.synchronize()
    assert oracle_pool.rel_err_rows(pool.state.cpu().numpy(), S_hist, 1).max() <= tol
    assert pool.get_error() is None


GDN_SMALL = I.Layer(I.GATED_DELTA, 2, 4, 128, 128, "bf16", qk_dist="l2norm")


GATED_SMALL = I.Layer(I.GATED, 2, 4, 128, 128, "bf16")


@pytest.mark.parametrize("name,T,m", [("gdn", 1, 8), ("gdn", 4, 8), ("gdn", 8, 8), ("gdn", 12, 8),
                                      ("gated", 9, 8), ("gated", 16, 1)])
def test_verify_tc_shapes(name, T, m):
    """The tensor-core verify (the state tile by TMA, the mat-vecs as one tcgen05
    product; chunks of at most 16 tokens and at most 16 vectors: 2T for the delta rule,
    T without it) and, past those limits (T = 12 with the delta rule), the mma.sync
    kernel: ragged buffers of 0..m-1 tokens (empty at m = 1, so that 16 drafts make a
    16-token chunk, the launch shape with one pipeline per CTA), stateless
    (short-context) requests verifying against S = 0, and more (row, head) units than
    the persistent grid holds, so every CTA walks several.  Every draft output and,
    after accept and a closing flush, every state."""
    layer = GDN_SMALL if name == "gdn" else GATED_SMALL
    B, n_short, bs = 100, 10, 8
    n_long = B - n_short
    nb = blocks_needed(m - 1 + T, bs)
    rng = np.random.default_rng(60 + T + 100 * layer.variant)
    pool = make_pool(layer, m, B, nb, bs, num_slots=n_long)
    S0 = I.draw_state(rng, layer, n_long)
    pool.state.copy_(torch.from_numpy(S0))
    perm = rng.permutation(B * nb)
    for r in range(B):
        pool.set_request(r, r if r < n_long else -1, perm[r * nb:(r + 1) * nb])
    occ = np.arange(B) % m
    wtok = I.draw_tokens(rng, layer, (m - 1, B))
    for s in range(m - 1):
        rows = np.nonzero(occ > s)[0]
        lrows, srows = rows[rows < n_long], rows[rows >= n_long]
        if len(lrows):
            pool.decode(lrows, *token_tensors(wtok, layer, (s, lrows)))
        if len(srows):
            pool.short_ctx(srows, *token_tensors(wtok, layer, (s, srows)))
    assert np.array_equal(pool.get_lengths(), occ.astype(np.int32))
    req = np.arange(B)
    tok = I.draw_tokens(rng, layer, (B, T))
    o = pool.verify(req, *token_tensors(tok, layer, slice(None))).cpu().numpy()
    j = rng.integers(0, T + 1, size=B)
    pool.accept(req, j)
    tol = tol_for(layer)
    zero = np.zeros((layer.n_v_heads, layer.d_k, layer.d_v))
    S_acc = []
    for r in range(B):
        hist = {key: (None if tok[key] is None else
                      np.concatenate([wtok[key][:occ[r], r], tok[key][r]]))
                for key in tok}
        start = S0[r].astype(np.float64) if r < n_long else zero
        o_ref, _, states = oracle.decode_sequence(start, hist, layer.variant,
                                                  keep_states=range(occ[r] + T))
        assert rel_err(o[r], o_ref[occ[r]:]) <= tol, r
        S_acc.append(states[occ[r] + j[r] - 1] if occ[r] + j[r] > 0 else start)
    expect = occ + j
    expect[(expect >= m) & (req < n_long)] = 0
    assert np.array_equal(pool.get_lengths(), expect.astype(np.int32))
    pool.flush(req[:n_long])
    torch.cuda.synchronize()
    st = pool.state.cpu().numpy()
    for r in range(n_long):
        assert rel_err(st[r], S_acc[r]) <= tol, r
    assert pool.get_error() is None


def test_verify_tc_corrupt_table():
    """One-slot blocks put the drafts' slots past the row descriptor's first eight
    blocks, so the tensor-core verify reads them from the device block table.  A
    corrupted entry there is caught by the kernel's own check: the unit records
    (kind 1, request, value) and writes nothing, and the other request verifies
    normally."""
    layer = GDN_SMALL
    rng = np.random.default_rng(71)
    pool = make_pool(layer, 16, 2, 16, 1)
    S0 = I.draw_state(rng, layer, 2)
    pool.state.copy_(torch.from_numpy(S0))
    pool.set_request(0, 0, list(range(16)))
    pool.set_request(1, 1, list(range(16, 32)))
    pre = I.draw_tokens(rng, layer, (10, 2))
    for t in range(10):
        pool.decode([0, 1], *token_tensors(pre, layer, t))
    torch.cuda.synchronize()
    # the block table is the first region of the metadata: request 0, block 10 (slot 10)
    bad = torch.tensor([12345], dtype=torch.int32).view(torch.uint8).cuda()
    pool._meta_mem[40:44].copy_(bad)
    tok = I.draw_tokens(rng, layer, (2, 4))
    o = torch.full((2, 4, layer.n_v_heads, layer.d_v), float("nan"), device="cuda")
    pool.verify([0, 1], *token_tensors(tok, layer, slice(None)), o=o)
    o = o.cpu().numpy()
    assert pool.get_error() == (1, 0, 12345)
    assert np.all(np.isnan(o[0]))
    hist = {key: (None if tok[key] is None else np.concatenate([pre[key][:, 1], tok[key][1]]))
            for key in tok}
    o_ref, _, _ = oracle.decode_sequence(S0[1], hist, layer.variant)
    assert rel_err(o[1], o_ref[10:]) <= tol_for(layer)
