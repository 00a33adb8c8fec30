"""Property test (CPU): random operation sequences on the brute-force buffered model
equal the recurrent oracle.

For any variant, flush threshold m, sequence of decode / verify(T) + accept(j) /
flush operations and token values, the buffered algorithm's outputs and its
state after every fold equal the per-token recurrence on the accepted history.
This extends the oracle pin for the buffered form to arbitrary interleavings.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from tests.buffered_model import BufferedHead

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")


@hyp.settings(max_examples=60, deadline=None)
@hyp.given(variant=st.sampled_from([0, 1, 2]), m=st.integers(1, 6),
           ops=st.lists(st.tuples(st.sampled_from(["decode", "verify", "flush"]),
                                  st.integers(1, 4), st.integers(0, 4)), min_size=1, max_size=12),
           seed=st.integers(0, 2 ** 31 - 1))
def test_buffered_model_equals_recurrence(variant, m, ops, seed):
    rng = np.random.default_rng(seed)
    dk, dv = 4, 3
    S0 = rng.standard_normal((dk, dv))
    head = BufferedHead(S0, variant, m)
    S_hist = S0[None, None].copy()

    def draw(T):
        k = rng.standard_normal((T, 1, 1, dk))
        k = k / np.linalg.norm(k, axis=-1, keepdims=True)
        return {"q": rng.standard_normal((T, 1, 1, dk)), "k": k,
                "v": rng.standard_normal((T, 1, 1, dv)),
                "log_g": None if variant == 0 else rng.uniform(-0.4, 0.0, (T, 1, 1)),
                "beta": rng.uniform(0.1, 0.9, (T, 1, 1)) if variant == 2 else None}

    def scal(x, t):
        return None if x is None else x[t, 0, 0]

    for op, T, j in ops:
        if op == "decode":
            tok = draw(1)
            o = head.decode(tok["q"][0, 0, 0], tok["k"][0, 0, 0], tok["v"][0, 0, 0],
                            scal(tok["log_g"], 0), scal(tok["beta"], 0))
            o_ref, S_hist, _ = oracle.decode_sequence(S_hist, tok, variant)
            assert np.abs(o - o_ref[0, 0, 0]).max() <= 1e-10
        elif op == "verify":
            tok = draw(T)
            drafts = [(tok["q"][t, 0, 0], tok["k"][t, 0, 0], tok["v"][t, 0, 0],
                       scal(tok["log_g"], t), scal(tok["beta"], t)) for t in range(T)]
            o = head.verify(drafts)
            assert np.abs(o - oracle.verify(S_hist, tok, variant)[:, 0, 0]).max() <= 1e-10
            jj = min(j, T)
            head.accept(jj)
            S_hist = oracle.accept(S_hist, tok, np.array([jj]), variant)
        else:
            head.flush()
        assert np.abs(head.current_state() - S_hist[0, 0]).max() <= 1e-10
        if not head.buf:
            assert np.abs(head.S - S_hist[0, 0]).max() <= 1e-10
