"""GPU parity under random interleavings of every call (seeded).

A small pool with long requests (state + buffer) and short requests (buffer only)
runs a random sequence of decode, short-context decode, verify + accept, flush and
retire/admit operations on random subsets of requests (ragged lengths and folds in
the middle of a launch).  An independent host model keeps each request's full
history: outputs are checked against the fp64 oracle run on that history, buffer
lengths bit for bit after every operation, and the stored state of a long request
whenever its buffer is empty.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from kv_buffered_decoding_gb300 import inputs as I
from tests.gpu_harness import dev, make_pool, rel_err, tol_for

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


class Req:
    def __init__(self, kind, slot, blocks, S0, cap):
        self.kind, self.slot, self.blocks, self.cap = kind, slot, blocks, cap
        self.S = S0.astype(np.float64)  # state after every accepted token
        self.n = 0


@pytest.mark.parametrize("layer,m,seed", [
    (I.Layer(I.GATED_DELTA, 2, 4, 64, 64, "bf16", qk_dist="l2norm"), 5, 1),
    (I.Layer(I.GATED, 2, 2, 128, 128, "bf16"), 4, 2),
], ids=["gated_delta_d64", "gated_d128"])
def test_random_interleavings(layer, m, seed):
    rng = np.random.default_rng(seed)
    n_long, n_short, bs, nb_req = 6, 4, 4, 4
    R = n_long + n_short
    cap = nb_req * bs
    pool = make_pool(layer, m, R, nb_req, bs, num_blocks=R * nb_req + 8, num_slots=n_long)
    S0 = I.draw_state(rng, layer, n_long)
    pool.state.copy_(torch.from_numpy(S0))
    free = list(rng.permutation(R * nb_req + 8))
    reqs = {}

    def admit(r):
        blocks = [int(free.pop()) for _ in range(nb_req)]
        if r < n_long:
            st = pool.state[r].cpu().numpy()
            reqs[r] = Req("long", r, blocks, st, cap)
            pool.set_request(r, r, blocks)
        else:
            reqs[r] = Req("short", -1, blocks, np.zeros((layer.n_v_heads, layer.d_k, layer.d_v)), cap)
            pool.set_request(r, -1, blocks)

    for r in range(R):
        admit(r)
    tol = tol_for(layer)

    def tok_dict(t):
        return {key: (None if val is None else val) for key, val in t.items()}

    def check_lengths():
        lens = pool.get_lengths()
        for r, q in reqs.items():
            assert lens[r] == q.n, (r, lens[r], q.n)

    for step in range(60):
        op = rng.choice(["decode", "short", "verify", "flush", "recycle"], p=[0.35, 0.2, 0.3, 0.1, 0.05])
        if op in ("decode", "short"):
            kind = "long" if op == "decode" else "short"
            cand = [r for r, q in reqs.items() if q.kind == kind and q.n + 1 <= q.cap]
            if not cand:
                continue
            rows = np.array(sorted(rng.choice(cand, size=rng.integers(1, len(cand) + 1), replace=False)))
            tok = I.draw_tokens(rng, layer, (len(rows),))
            args = (dev(tok["q"], layer), dev(tok["k"], layer), dev(tok["v"], layer),
                    dev(tok["log_g"], f32=True), dev(tok["beta"], f32=True))
            o = (pool.decode(rows, *args) if op == "decode" else pool.short_ctx(rows, *args)).cpu().numpy()
            for i, r in enumerate(rows):
                q = reqs[r]
                one = {key: (None if val is None else val[i:i + 1]) for key, val in tok.items()}
                o_ref, S_new, _ = oracle.decode_sequence(q.S, one, layer.variant)
                assert rel_err(o[i], o_ref[0]) <= tol, (step, op, r)
                q.S = S_new
                q.n += 1
                if q.kind == "long" and q.n >= m:
                    q.n = 0
        elif op == "verify":
            T = int(rng.integers(1, 5))
            cand = [r for r, q in reqs.items() if q.n + T <= q.cap]
            if not cand:
                continue
            rows = np.array(sorted(rng.choice(cand, size=rng.integers(1, len(cand) + 1), replace=False)))
            tok = I.draw_tokens(rng, layer, (len(rows), T))
            o = pool.verify(rows, dev(tok["q"], layer), dev(tok["k"], layer), dev(tok["v"], layer),
                            dev(tok["log_g"], f32=True), dev(tok["beta"], f32=True)).cpu().numpy()
            j = rng.integers(0, T + 1, size=len(rows))
            pool.accept(rows, j)
            for i, r in enumerate(rows):
                q = reqs[r]
                dr = {key: (None if val is None else val[i]) for key, val in tok.items()}
                o_ref = oracle.verify(q.S, dr, layer.variant)
                assert rel_err(o[i], o_ref) <= tol, (step, op, r)
                if j[i]:
                    acc = {key: (None if val is None else val[:j[i]]) for key, val in dr.items()}
                    _, q.S, _ = oracle.decode_sequence(q.S, acc, layer.variant)
                q.n += int(j[i])
                if q.kind == "long" and q.n >= m:
                    q.n = 0
        elif op == "flush":
            rows = [r for r, q in reqs.items() if q.kind == "long"]
            rows = np.array(sorted(rng.choice(rows, size=rng.integers(1, len(rows) + 1), replace=False)))
            pool.flush(rows)
            for r in rows:
                reqs[r].n = 0
        else:  # retire a short request, admit a fresh one in its place
            shorts = [r for r, q in reqs.items() if q.kind == "short"]
            r = int(rng.choice(shorts))
            pool.release_request(r)
            free[:0] = reqs[r].blocks
            admit(r)
        check_lengths()
        torch.cuda.synchronize()
        st = pool.state.cpu().numpy()
        for r, q in reqs.items():
            if q.kind == "long" and q.n == 0:
                assert rel_err(st[q.slot], q.S) <= tol, (step, op, r)
    assert np.array_equal(pool.get_device_lengths(), pool.get_lengths())
    assert pool.get_error() is None
